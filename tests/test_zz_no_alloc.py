"""biv_attention_noalloc: attention for callers that cannot allocate device
memory themselves (for example code living inside another runtime's memory
budget, or a hook that must not call cudaMalloc while its caller holds a
lock).  It must give exactly what biv_attention gives with a caller-provided
workspace, call after call, although every call reuses the library's one
fixed scratch array.  This file is collected last on purpose."""
import ctypes as C
import math

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from invariant_forward_bitwise_gb300 import biv, build
    build.build()
    biv.load()
    return biv


def _case(B, seed, lens, Hq=16, Hkv=8, D=128, kv_split=128, fp8=False, mode=0):
    """A paged cache (bf16, or e4m3 codes with per-(token, head) scales) with
    several splits per row, so that scratch is used."""
    g = synth.rng(seed)
    npages = [(L + 63) // 64 for L in lens]
    total = sum(npages)
    perm = g.permutation(total)
    bt = np.zeros((len(lens), max(npages)), np.int32)
    at = 0
    for i, n in enumerate(npages):
        bt[i, :n] = perm[at:at + n]
        at += n
    kc = torch.zeros(total, 64, Hkv, D, dtype=torch.uint8 if fp8 else torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.zeros(total, 64, Hkv, dtype=torch.float32, device="cuda") if fp8 else None
    vs = torch.zeros_like(ks) if fp8 else None
    for i, L in enumerate(lens):
        pos = np.arange(L)
        slot = torch.from_numpy(bt[i][pos // 64].astype(np.int64) * 64 + pos % 64).cuda()
        k = synth.normal_bf16(g, (L, Hkv * D)).cuda()
        v = synth.normal_bf16(g, (L, Hkv * D)).cuda()
        if fp8:
            B.biv_kv_fp8_quant(k, v, Hkv * D, slot, L, Hkv, D, kc, vc, ks, vs)
        else:
            B.biv_kv_store_bf16(k, v, Hkv * D, slot, L, Hkv, D, kc, vc)
    rows = [(i, p) for i, L in enumerate(lens) for p in (L - 1, L // 2)]
    T = len(rows)
    q = synth.normal_bf16(g, (T, Hq * D)).cuda()
    keep = dict(kc=kc, vc=vc, ks=ks, vs=vs, q=q, bt=torch.from_numpy(bt).cuda(),
                seq=torch.tensor([r[0] for r in rows], dtype=torch.int32, device="cuda"),
                pos=torch.tensor([r[1] for r in rows], dtype=torch.int32, device="cuda"),
                qb=torch.tensor(np.stack([np.arange(T), np.ones(T)], 1).astype(np.int32).ravel(),
                                device="cuda"))
    d = B.AttnDesc()
    d.q, d.q_stride = q.data_ptr(), q.stride(0)
    d.T, d.Hq, d.Hkv, d.D = T, Hq, Hkv, D
    d.row_seq, d.row_pos = keep["seq"].data_ptr(), keep["pos"].data_ptr()
    d.qblocks, d.nqblocks, d.max_rows_per_block = keep["qb"].data_ptr(), T, 1
    d.kv_dtype = B.E4M3 if fp8 else B.BF16
    d.k_cache, d.v_cache = kc.data_ptr(), vc.data_ptr()
    if fp8:
        d.k_scale, d.v_scale = ks.data_ptr(), vs.data_ptr()
    d.mode = mode
    d.block_table, d.max_pages = keep["bt"].data_ptr(), bt.shape[1]
    d.page, d.kv_split, d.max_ctx = 64, kv_split, max(lens)
    d.scale = 1.0 / math.sqrt(D)
    d.num_pages = total
    return d, keep


def _run(B, d, out, noalloc):
    d.out, d.out_stride = out.data_ptr(), out.stride(0)
    lib = B.load()
    if noalloc:
        st = lib.biv_attention_noalloc(C.byref(d), None)
    else:
        n = B.biv_attention_workspace(d)
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
        st = lib.biv_attention(C.byref(d), C.c_void_p(ws.data_ptr()), ws.numel(), None)
        torch.cuda.synchronize()
    assert st == B.BIV_OK, lib.biv_last_error()
    torch.cuda.synchronize()


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16kv", "fp8kv"])
@pytest.mark.parametrize("mode", [0, 1], ids=["invariant", "fast"])
def test_noalloc_matches_workspace_attention_twice(B, fp8, mode):
    """Bitwise equal to biv_attention with a caller workspace in the same mode
    (FAST sizes its split, and so its scratch, from the GPU's SM count)."""
    for seed, lens in [(1, [700, 300, 1000]), (2, [129, 900])]:
        d, keep = _case(B, seed, lens, fp8=fp8, mode=mode)
        assert B.biv_attention_workspace(d) > 0          # the split partials need scratch
        T, width = d.T, d.Hq * d.D
        ref = torch.full((T, width), float("nan"), dtype=torch.bfloat16, device="cuda")
        _run(B, d, ref, noalloc=False)
        for _ in range(2):                                # two calls in a row share the array
            got = torch.full((T, width), float("nan"), dtype=torch.bfloat16, device="cuda")
            _run(B, d, got, noalloc=True)
            assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("mode", [0, 1], ids=["invariant", "fast"])
def test_noalloc_rejects_requests_beyond_the_fixed_array(B, mode):
    d, keep = _case(B, 3, [200], mode=mode)
    # descriptor only: rejected before any launch.  One query block keeps the
    # FAST split small too (it splits finer when few CTAs would run).
    d.T, d.nqblocks = 4096, 1
    d.max_ctx, d.kv_split = 65536, 64
    assert B.biv_attention_workspace(d) > 64 << 20   # guard: never launch this descriptor
    lib = B.load()
    st = lib.biv_attention_noalloc(C.byref(d), None)
    assert st == B.BIV_ERR_WORKSPACE
    assert b"scratch" in lib.biv_last_error()
