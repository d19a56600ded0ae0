"""The C-ABI library builds, loads without a GPU, and exports every entry point
that include/biv.h declares (no compute call is made here)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "biv.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(biv_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib_path():
    from invariant_forward_bitwise_gb300 import build
    return build.build()


def test_header_declares_entry_points():
    names = _declared()
    assert "biv_gemm" in names and "biv_attention" in names and "biv_logprob" in names
    assert len(names) >= 20


def test_library_exports_every_declared_symbol(lib_path):
    import ctypes
    lib = ctypes.CDLL(lib_path)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_header(lib_path):
    from invariant_forward_bitwise_gb300 import biv
    assert sorted(biv.EXPORTS) == _declared()
    lib = biv.load(lib_path)
    assert lib.biv_version() >= 100
    assert isinstance(lib.biv_last_error(), bytes)


def test_host_validation_without_gpu(lib_path):
    """Argument checks run on the host and launch nothing."""
    import ctypes as C
    from invariant_forward_bitwise_gb300 import biv
    lib = biv.load(lib_path)
    d = biv.GemmDesc()
    d.M, d.N, d.K = 4, 8, 12          # K*2 not a multiple of 16 -> rejected
    d.a_dtype = d.b_dtype = d.c_dtype = biv.BF16
    st = lib.biv_gemm(C.byref(d), None, 0, None)
    assert st == biv.BIV_ERR_INVALID and b"K" in lib.biv_last_error()
    st = lib.biv_add_rmsnorm(None, 0, None, 0, None, None, 0, 3, 12, 1e-6, None)
    assert st == biv.BIV_ERR_INVALID
    st = lib.biv_topk(None, 0, None, 1, 10, 11, None, None)
    assert st == biv.BIV_ERR_INVALID
    # zero-sized work is a no-op
    assert lib.biv_silu_mul(None, 0, None, 0, 0, 8, None) == biv.BIV_OK
