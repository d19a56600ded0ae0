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


def _gemm_plan(lib, biv, M, N, K):
    """Workspace bytes and partials layout the planner picks (host only)."""
    import ctypes as C
    d = biv.GemmDesc()
    d.M, d.N, d.K = M, N, K
    d.a_dtype = d.b_dtype = d.c_dtype = biv.BF16
    d.lda, d.ldb, d.ldc = K, K, N
    d.A, d.B, d.C = 0x100000, 0x200000, 0x300000   # never dereferenced: no launch here
    n = C.c_size_t(0)
    assert lib.biv_gemm_workspace(C.byref(d), C.byref(n)) == biv.BIV_OK, lib.biv_last_error()
    p = biv.Partials()
    ws = C.c_void_p(0x1000) if n.value else None
    assert lib.biv_gemm_partials(C.byref(d), ws, C.byref(p)) == biv.BIV_OK, lib.biv_last_error()
    return n.value, p


def test_gemm_plan_on_host(lib_path):
    """The K-chunk schedule depends on K alone (max(8, ceil(KB/8)) blocks of
    64 per chunk); few-row calls leave their chunks to a fold across CTAs,
    and the workspace holds exactly chunks x M x ldp FP32 partials."""
    from invariant_forward_bitwise_gb300 import biv
    lib = biv.load(lib_path)
    for M in (1, 16, 64):
        for N, K, chunks in ((12288, 2048, 4), (2048, 6144, 8), (4096, 2048, 4), (2048, 2048, 4)):
            n, p = _gemm_plan(lib, biv, M, N, K)
            ldp = (N + 127) // 128 * 128
            assert (p.chunks, p.ld, p.chunk_stride) == (chunks, ldp, M * ldp), (M, N, K)
            assert n == chunks * M * ldp * 4
    # one chunk (K <= 512): nothing to fold across CTAs
    assert _gemm_plan(lib, biv, 1, 4096, 512)[0] == 0
    # prefill-sized calls fold inside the CTA: no workspace
    for N, K in ((12288, 2048), (2048, 6144), (151936, 2048)):
        n, p = _gemm_plan(lib, biv, 16384, N, K)
        assert n == 0 and p.chunks == 0


def test_partials_consumers_reject_bad_layouts(lib_path):
    """The ops that fold GEMM partials check the layout on the host."""
    import ctypes as C
    from invariant_forward_bitwise_gb300 import biv
    lib = biv.load(lib_path)
    bad = [biv.Partials(0x1000, 9, 2048, 64 * 2048),      # more than 8 chunks
           biv.Partials(0x1004, 4, 2048, 64 * 2048),      # base not 16-byte aligned
           biv.Partials(0x1000, 4, 2047, 64 * 2047)]      # row pitch not a multiple of 4
    for p in bad:
        st = lib.biv_add_rmsnorm_partials(C.byref(p), None, 0, C.c_void_p(0x2000), C.c_void_p(0x3000),
                                          2048, 4, 2048, C.c_float(1e-6), None)
        assert st == biv.BIV_ERR_INVALID
        st = lib.biv_silu_mul_partials(C.byref(p), C.c_void_p(0x3000), 1024, 4, 1024, None)
        assert st == biv.BIV_ERR_INVALID
