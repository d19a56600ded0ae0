"""Paged attention: parity with the oracle's plain softmax, and bitwise
invariance of a row across prefill blocks, decode, block partitions and batch
mix (one attention operator for every path)."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import ops
from oracle.codecs import bf16_to_f32

pytestmark = pytest.mark.gpu
REL = 1e-2


@pytest.fixture(scope="module")
def B():
    from invariant_forward_bitwise_gb300 import biv, build
    build.build()
    biv.load()
    return biv


def host_f32(t):
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return bf16_to_f32(t.view(torch.int16).numpy().view(np.uint16))
    return t.float().numpy()


def bits(t):
    return t.detach().contiguous().view(torch.uint8).cpu().numpy()


def rel_err(got, ref):
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(np.asarray(got, np.float64) - ref)) / max(np.max(np.abs(ref)), 1e-30))


class Paged:
    """Sequences' K/V in a shuffled paged cache (64-token pages)."""

    def __init__(self, B, g, lens, Hkv, D, fp8=False):
        self.B, self.lens, self.Hkv, self.D, self.fp8 = B, lens, Hkv, D, fp8
        npages = [(L + 63) // 64 for L in lens]
        total = sum(npages) + 3
        perm = g.permutation(total)
        self.bt = np.zeros((len(lens), max(npages)), np.int32)
        at = 0
        for i, n in enumerate(npages):
            self.bt[i, :n] = perm[at:at + n]
            at += n
        self.k = [synth.normal_bf16(g, (L, Hkv, D)) for L in lens]
        self.v = [synth.normal_bf16(g, (L, Hkv, D)) for L in lens]
        shape = (total, 64, Hkv, D)
        if fp8:
            self.kc = torch.zeros(shape, dtype=torch.uint8, device="cuda")
            self.vc = torch.zeros(shape, dtype=torch.uint8, device="cuda")
            self.ks = torch.zeros(shape[:3], dtype=torch.float32, device="cuda")
            self.vs = torch.zeros(shape[:3], dtype=torch.float32, device="cuda")
        else:
            # stale NaN everywhere that no token wrote: masked slots must not leak
            self.kc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
            self.vc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
            self.ks = self.vs = None
        for i, L in enumerate(lens):
            pos = np.arange(L)
            slot = (self.bt[i][pos // 64].astype(np.int64) * 64 + pos % 64)
            kd, vd = self.k[i].cuda().reshape(L, -1), self.v[i].cuda().reshape(L, -1)
            if fp8:
                B.biv_kv_fp8_quant(kd, vd, Hkv * D, torch.from_numpy(slot).cuda(), L, Hkv, D,
                                   self.kc, self.vc, self.ks, self.vs)
            else:
                B.biv_kv_store_bf16(kd, vd, Hkv * D, torch.from_numpy(slot).cuda(), L, Hkv, D,
                                    self.kc, self.vc)
        self.bt_d = torch.from_numpy(self.bt).cuda()

    def oracle_kv(self, i):
        k = self.k[i].float().numpy()
        v = self.v[i].float().numpy()
        if self.fp8:
            k, v = ops.kv_roundtrip(k), ops.kv_roundtrip(v)
        return k, v


def run_attn(B, pc, q, rows, blocks, Hq, kv_split=1024, mode=0, topk_idx=None, topk=0, tma=True,
             max_ctx=None):
    """rows: list of (seq, pos); blocks: list of (first row, count)."""
    T = len(rows)
    D = pc.D
    out = torch.full((T, Hq * D), float("nan"), dtype=torch.bfloat16, device="cuda")
    row_seq = torch.tensor([r[0] for r in rows], dtype=torch.int32, device="cuda")
    row_pos = torch.tensor([r[1] for r in rows], dtype=torch.int32, device="cuda")
    qb = torch.tensor(np.array(blocks, np.int32).ravel(), dtype=torch.int32, device="cuda")
    d = B.AttnDesc()
    d.q, d.q_stride = q.data_ptr(), q.stride(0)
    d.out, d.out_stride = out.data_ptr(), out.stride(0)
    d.T, d.Hq, d.Hkv, d.D = T, Hq, pc.Hkv, D
    d.row_seq, d.row_pos = row_seq.data_ptr(), row_pos.data_ptr()
    d.qblocks, d.nqblocks = qb.data_ptr(), len(blocks)
    d.max_rows_per_block = max(b[1] for b in blocks)
    d.kv_dtype = B.E4M3 if pc.fp8 else B.BF16
    d.k_cache, d.v_cache = pc.kc.data_ptr(), pc.vc.data_ptr()
    d.k_scale = pc.ks.data_ptr() if pc.fp8 else None
    d.v_scale = pc.vs.data_ptr() if pc.fp8 else None
    d.block_table, d.max_pages = pc.bt_d.data_ptr(), pc.bt.shape[1]
    d.page, d.kv_split = 64, kv_split
    d.max_ctx = max(r[1] for r in rows) + 1 if max_ctx is None else max_ctx
    if topk_idx is not None:
        d.topk_idx, d.topk_stride, d.topk = topk_idx.data_ptr(), topk_idx.stride(0), topk
    d.scale = 1.0 / math.sqrt(D)
    d.mode = mode
    d.num_pages = pc.kc.shape[0] if tma else 0
    n = B.biv_attention_workspace(d)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda") if n else None
    B.biv_attention(d, ws)
    torch.cuda.synchronize()
    return out


def blocks_of(rows, per):
    out, i = [], 0
    while i < len(rows):
        j = i
        while j < len(rows) and j - i < per and rows[j][0] == rows[i][0]:
            j += 1
        out.append((i, j - i))
        i = j
    return out


@pytest.mark.parametrize("D,Hq,Hkv,fp8,split", [(128, 16, 8, False, 1024), (128, 16, 8, True, 128),
                                                 (64, 4, 2, False, 64), (80, 32, 4, False, 192),
                                                 (128, 32, 1, True, 256)])
def test_prefill_parity_and_decode_invariance(B, D, Hq, Hkv, fp8, split):
    g = synth.rng(D + Hq + split)
    lens = [37, 300, 64, 129]
    pc = Paged(B, g, lens, Hkv, D, fp8)
    G = Hq // Hkv
    rows = [(i, p) for i, L in enumerate(lens) for p in range(L)]
    q = synth.normal_bf16(g, (len(rows), Hq * D)).cuda()
    per = max(1, 64 // G)
    out = run_attn(B, pc, q, rows, blocks_of(rows, per), Hq, kv_split=split)
    got = host_f32(out).reshape(len(rows), Hq, D)
    qh = host_f32(q).reshape(len(rows), Hq, D)
    at = 0
    for i, L in enumerate(lens):
        k, v = pc.oracle_kv(i)
        ref = ops.attention(qh[at:at + L], k, v, np.arange(L), np.arange(L), 1.0 / math.sqrt(D))
        assert rel_err(got[at:at + L], ref) < REL, i
        at += L
    # decode: one row per sequence at its last position, one row per block
    last = [sum(lens[:i + 1]) - 1 for i in range(len(lens))]
    drows = [rows[j] for j in last]
    qd = q[torch.tensor(last, device="cuda")]
    dout = run_attn(B, pc, qd, drows, [(j, 1) for j in range(len(drows))], Hq, kv_split=split)
    assert np.array_equal(bits(dout), bits(out[torch.tensor(last, device="cuda")]))
    # another block partition of the same prefill rows
    out2 = run_attn(B, pc, q, rows, blocks_of(rows, max(1, per // 3)), Hq, kv_split=split)
    assert np.array_equal(bits(out2), bits(out))


@pytest.mark.parametrize("D,Hq,Hkv,split", [(128, 16, 8, 1024), (128, 16, 8, 128), (64, 4, 2, 64),
                                           (128, 8, 8, 256), (64, 32, 4, 192)])
def test_tcgen05_prefill_equals_mma_sync_kernel(B, monkeypatch, D, Hq, Hkv, split):
    """Prefill blocks of up to 128 query vectors on tcgen05 give the bits of
    the mma.sync kernel on blocks of up to 64 (ragged lengths, stale NaN in
    unwritten page slots, one to twelve KV splits merged), and stay within the
    oracle's tolerance."""
    g = synth.rng(D * 3 + Hq + split)
    lens = [37, 300, 64, 129, 700]
    pc = Paged(B, g, lens, Hkv, D)
    G = Hq // Hkv
    rows = [(i, p) for i, L in enumerate(lens) for p in range(L)]
    q = synth.normal_bf16(g, (len(rows), Hq * D)).cuda()
    out_tc = run_attn(B, pc, q, rows, blocks_of(rows, 128 // G), Hq, kv_split=split)
    monkeypatch.setenv("BIV_ATTN_PREFILL_TC", "0")
    out_ms = run_attn(B, pc, q, rows, blocks_of(rows, max(1, 64 // G)), Hq, kv_split=split)
    assert np.array_equal(bits(out_tc), bits(out_ms))
    at = sum(lens[:4])
    k, v = pc.oracle_kv(4)
    ref = ops.attention(host_f32(q).reshape(len(rows), Hq, D)[at:], k, v, np.arange(700),
                        np.arange(700), 1.0 / math.sqrt(D))
    assert rel_err(host_f32(out_tc).reshape(len(rows), Hq, D)[at:], ref) < REL


def test_prefill_cta_shape_changes_no_bit(B, monkeypatch):
    """The two-stage prefill CTA gives the bits of the default one-stage CTA."""
    g = synth.rng(77)
    lens = [300, 129]
    Hq, Hkv, D = 16, 8, 128
    pc = Paged(B, g, lens, Hkv, D, False)
    rows = [(i, p) for i, L in enumerate(lens) for p in range(L)]
    q = synth.normal_bf16(g, (len(rows), Hq * D)).cuda()
    blocks = blocks_of(rows, 64 // (Hq // Hkv))
    out1 = run_attn(B, pc, q, rows, blocks, Hq)
    monkeypatch.setenv("BIV_ATTN_PREFILL_STAGES", "2")
    out2 = run_attn(B, pc, q, rows, blocks, Hq)
    assert np.array_equal(bits(out1), bits(out2))


def test_fast_mode_close_not_required_equal(B):
    g = synth.rng(3)
    lens = [2000, 900]
    pc = Paged(B, g, lens, 8, 128)
    rows = [(0, 1999), (1, 899)]
    q = synth.normal_bf16(g, (2, 16 * 128)).cuda()
    inv = run_attn(B, pc, q, rows, [(0, 1), (1, 1)], 16)
    fast = run_attn(B, pc, q, rows, [(0, 1), (1, 1)], 16, mode=B.MODE_FAST)
    assert rel_err(host_f32(fast), host_f32(inv)) < 1e-2


def test_sparse_topk_attention(B):
    g = synth.rng(4)
    L, D, Hq = 700, 128, 32
    pc = Paged(B, g, [L], 1, D)
    qpos = [699, 650, 100]
    topk = 256
    idx = np.full((3, topk), -1, np.int32)
    for r, p in enumerate(qpos):
        cand = g.permutation(p + 1)[:min(topk, p + 1) - (r == 0) * 10]
        idx[r, :cand.size] = np.sort(cand)
    rows = [(0, p) for p in qpos]
    q = synth.normal_bf16(g, (3, Hq * D)).cuda()
    out = run_attn(B, pc, q, rows, [(0, 1), (1, 1), (2, 1)], Hq, kv_split=128,
                   topk_idx=torch.from_numpy(idx).cuda(), topk=topk)
    k, v = pc.oracle_kv(0)
    ref = ops.sparse_attention(host_f32(q).reshape(3, Hq, D), k, v, idx, np.array(qpos), 1 / math.sqrt(D))
    assert rel_err(host_f32(out).reshape(3, Hq, D), ref) < REL
    # the same row alone
    one = run_attn(B, pc, q[1:2], rows[1:2], [(0, 1)], Hq, kv_split=128,
                   topk_idx=torch.from_numpy(idx[1:2]).cuda(), topk=topk)
    assert np.array_equal(bits(one), bits(out[1:2]))
    # dense top-k that lists every position equals causal attention
    full = np.tile(np.arange(topk, dtype=np.int32), (1, 1))
    rows2 = [(0, 200)]
    o_sparse = run_attn(B, pc, q[:1], rows2, [(0, 1)], Hq, kv_split=128,
                        topk_idx=torch.from_numpy(np.where(full <= 200, full, -1)).cuda(), topk=topk)
    o_dense = run_attn(B, pc, q[:1], rows2, [(0, 1)], Hq, kv_split=128)
    assert rel_err(host_f32(o_sparse), host_f32(o_dense)) < 1e-2


@pytest.mark.parametrize("D", [64, 128])
def test_tma_loader_equals_thread_loader(B, D):
    """Whole-page TMA loads and thread-issued loads feed the same arithmetic."""
    g = synth.rng(50 + D)
    lens = [200, 77]
    pc = Paged(B, g, lens, 2, D)
    rows = [(i, p) for i, L in enumerate(lens) for p in range(L)]
    q = synth.normal_bf16(g, (len(rows), 4 * D)).cuda()
    blocks = blocks_of(rows, 32)
    a = run_attn(B, pc, q, rows, blocks, 4, kv_split=128, tma=True)
    b = run_attn(B, pc, q, rows, blocks, 4, kv_split=128, tma=False)
    assert np.array_equal(bits(a), bits(b))
    last = [sum(lens[:i + 1]) - 1 for i in range(len(lens))]
    dec = run_attn(B, pc, q[torch.tensor(last, device="cuda")], [rows[j] for j in last],
                   [(j, 1) for j in range(len(last))], 4, kv_split=128, tma=True)
    assert np.array_equal(bits(dec), bits(a[torch.tensor(last, device="cuda")]))


@pytest.mark.parametrize("D", [64, 128])
def test_grouped_dsplit_cta_changes_no_bit(B, monkeypatch, D):
    """Blocks of 17-32 query vectors on the thread loader run two vector
    groups of two warps (split keys in S, split head dimension in P.V); they
    give the bits of the four-warp CTA: sparse MQA rows (32 heads on one KV
    head, several 64-key tiles and splits, a short list) and dense blocks of
    12 rows at G = 2 with ragged tails."""
    g = synth.rng(91 + D)
    L, Hq = 700, 32
    pc = Paged(B, g, [L], 1, D)
    qpos = [699, 650, 100, 5]
    topk = 320
    idx = np.full((len(qpos), topk), -1, np.int32)
    for r, p in enumerate(qpos):
        cand = g.permutation(p + 1)[:min(topk, p + 1)]
        idx[r, :cand.size] = np.sort(cand)
    rows = [(0, p) for p in qpos]
    q = synth.normal_bf16(g, (len(qpos), Hq * D)).cuda()
    blocks = [(i, 1) for i in range(len(qpos))]
    kw = dict(kv_split=128, topk_idx=torch.from_numpy(idx).cuda(), topk=topk)
    got = run_attn(B, pc, q, rows, blocks, Hq, **kw)
    monkeypatch.setenv("BIV_ATTN_GROUP_DSPLIT", "0")
    ref = run_attn(B, pc, q, rows, blocks, Hq, **kw)
    assert np.array_equal(bits(got), bits(ref))
    monkeypatch.delenv("BIV_ATTN_GROUP_DSPLIT")
    # dense, thread loader: 12-row blocks of 16 q / 8 kv heads (24 vectors)
    lens = [300, 129, 70]
    pc2 = Paged(B, g, lens, 8, D)
    rows2 = [(i, p) for i, n in enumerate(lens) for p in range(n)]
    q2 = synth.normal_bf16(g, (len(rows2), 16 * D)).cuda()
    blocks2 = blocks_of(rows2, 12)
    got2 = run_attn(B, pc2, q2, rows2, blocks2, 16, kv_split=256, tma=False)
    monkeypatch.setenv("BIV_ATTN_GROUP_DSPLIT", "0")
    ref2 = run_attn(B, pc2, q2, rows2, blocks2, 16, kv_split=256, tma=False)
    assert np.array_equal(bits(got2), bits(ref2))
    # and both equal the one-row blocks of the same rows
    one = run_attn(B, pc2, q2, rows2, [(i, 1) for i in range(len(rows2))], 16, kv_split=256, tma=False)
    assert np.array_equal(bits(got2), bits(one))


@pytest.mark.parametrize("stages,dsplit", [("1", "1"), ("2", "2"), ("3", "4"), ("1", "4")])
@pytest.mark.parametrize("D", [64, 128])
def test_decode_cta_shape_changes_no_bit(B, monkeypatch, stages, dsplit, D):
    """The decode CTAs' TMA pipeline depth and the number of warps that split
    the head dimension are speed choices: every one gives the bits of one
    warp with a two-stage pipeline, over several 64-key tiles and splits."""
    g = synth.rng(77 + D)
    lens = [700, 130, 1500]
    pc = Paged(B, g, lens, 8, D)
    last = [(i, L - 1) for i, L in enumerate(lens)]
    q = synth.normal_bf16(g, (len(last), 16 * D)).cuda()
    blocks = [(j, 1) for j in range(len(last))]
    monkeypatch.setenv("BIV_ATTN_DECODE_STAGES", "2")
    monkeypatch.setenv("BIV_ATTN_DECODE_DSPLIT", "1")
    ref = run_attn(B, pc, q, last, blocks, 16, kv_split=1024, tma=True)
    monkeypatch.setenv("BIV_ATTN_DECODE_STAGES", stages)
    monkeypatch.setenv("BIV_ATTN_DECODE_DSPLIT", dsplit)
    got = run_attn(B, pc, q, last, blocks, 16, kv_split=1024, tma=True)
    assert np.array_equal(bits(got), bits(ref))
    # and the prefill CTA shape gives the same row bits (one operator for both)
    rows = [(i, p) for i, L in enumerate(lens) for p in range(L)]
    qp = synth.normal_bf16(g, (len(rows), 16 * D)).cuda()
    full = run_attn(B, pc, qp, rows, blocks_of(rows, 32), 16, kv_split=1024, tma=True)
    idx = [sum(lens[:i + 1]) - 1 for i in range(len(lens))]
    dec = run_attn(B, pc, qp[torch.tensor(idx, device="cuda")], last, blocks, 16, kv_split=1024, tma=True)
    assert np.array_equal(bits(dec), bits(full[torch.tensor(idx, device="cuda")]))


@pytest.mark.parametrize("tma", [True, False], ids=["tma", "threads"])
def test_row_beyond_max_ctx_is_reported_and_isolated(B, tma):
    """A row whose position lies past the splits that max_ctx provides for
    (the caller broke the bound) is reported on the device error word and
    gets NaN output; it touches no workspace slot, and the other rows of the
    call keep the bits they have when the bound holds."""
    g = synth.rng(41)
    Hq, Hkv, D = 16, 8, 128
    pc = Paged(B, g, [700], Hkv, D)
    q = synth.normal_bf16(g, (3, Hq * D)).cuda()
    rows = [(0, 699), (0, 100), (0, 200)]
    blocks = [(0, 1), (1, 1), (2, 1)]
    assert B.biv_poll_error() == 0
    good = run_attn(B, pc, q, rows, blocks, Hq, kv_split=128, tma=tma)
    assert B.biv_poll_error() == 0
    for max_ctx in (201, 100):           # 2 splits; 1 split (no workspace at all)
        bad = run_attn(B, pc, q, rows, blocks, Hq, kv_split=128, tma=tma, max_ctx=max_ctx)
        assert B.biv_poll_error() == 2
        assert B.biv_poll_error() == 0
        assert torch.isnan(bad[0].float()).all()
        ok = [1, 2] if max_ctx == 201 else [1]
        assert np.array_equal(bits(bad[ok]), bits(good[ok]))


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16kv", "fp8kv"])
def test_decode_row_at_16k_context_parity(B, fp8):
    """One decode row of a 16384-token sequence: 16 splits of 1024 keys merged
    in ascending order, against the oracle's plain softmax over every key."""
    g = synth.rng(16384 + fp8)
    Hq, Hkv, D, L = 16, 8, 128, 16384
    pc = Paged(B, g, [L], Hkv, D, fp8=fp8)
    q = synth.normal_bf16(g, (1, Hq * D)).cuda()
    out = run_attn(B, pc, q, [(0, L - 1)], [(0, 1)], Hq, kv_split=1024)
    k, v = pc.oracle_kv(0)
    ref = ops.attention(host_f32(q).reshape(1, Hq, D), k, v, np.array([L - 1]), np.arange(L),
                        1 / math.sqrt(D))
    assert rel_err(host_f32(out).reshape(1, Hq, D), ref) < REL
