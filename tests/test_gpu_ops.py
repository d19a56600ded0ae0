"""Per-op parity of the CUDA path against the CPU oracle, plus bitwise row
invariance (a row computed alone equals the same row inside any batch).

Tolerances: integer/byte outputs bit-exact; floating-point outputs within the
relative error 1e-2 of the oracle (max |gpu - oracle| / max |oracle| per
output tensor), the per-op bar of the method's statement.
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import ops
from oracle.codecs import bf16_to_f32, e4m3_to_f32

pytestmark = pytest.mark.gpu

REL = 1e-2


@pytest.fixture(scope="module")
def B():
    from invariant_forward_bitwise_gb300 import biv, build
    build.build()
    biv.load()
    return biv


def dev(x, dtype=None):
    t = torch.as_tensor(x)
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host_f32(t):
    """bf16/float CUDA tensor -> float32 numpy (bf16 decoded by the oracle codec)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return bf16_to_f32(t.view(torch.int16).numpy().view(np.uint16))
    return t.float().numpy()


def rel_err(got, ref):
    ref = np.asarray(ref, np.float64)
    den = max(np.max(np.abs(ref)), 1e-30)
    return float(np.max(np.abs(np.asarray(got, np.float64) - ref)) / den)


def bits(t):
    return t.detach().contiguous().view(torch.uint8).cpu().numpy()


def rnd_bf16(g, *shape, std=1.0):
    return synth.normal_bf16(g, shape, std)


# ------------------------------------------------------------------ RMSNorm --
@pytest.mark.parametrize("d", [256, 2048, 2560, 4096, 128, 8192])
def test_add_rmsnorm_parity_and_row_invariance(B, d):
    g = synth.rng(d)
    rows = 37
    x, r, w = rnd_bf16(g, rows, d), rnd_bf16(g, rows, d), rnd_bf16(g, d)
    xd, rd, wd = dev(x), dev(r), dev(w)
    y = torch.empty_like(xd)
    B.biv_add_rmsnorm(xd, rd, wd, y, 1e-6)
    r_ref, y_ref = ops.add_rmsnorm(x.float().numpy(), r.float().numpy(), w.float().numpy(), 1e-6)
    assert np.array_equal(host_f32(rd), r_ref)          # bf16(x + r) is exact
    assert rel_err(host_f32(y), y_ref) < REL
    # no-residual form
    y2 = torch.empty_like(xd)
    B.biv_add_rmsnorm(xd, None, wd, y2, 1e-6)
    assert rel_err(host_f32(y2), ops.rmsnorm(x.float().numpy(), w.float().numpy(), 1e-6)) < REL
    # row 11 alone == row 11 in the batch, bit for bit
    r1 = dev(r[11:12])
    y1 = torch.empty_like(xd[11:12])
    B.biv_add_rmsnorm(xd[11:12], r1, wd, y1, 1e-6)
    assert np.array_equal(bits(y1), bits(y[11:12])) and np.array_equal(bits(r1), bits(rd[11:12]))


def test_silu_mul_parity(B):
    g = synth.rng(5)
    gu = rnd_bf16(g, 19, 2 * 688, std=2.0)
    y = torch.empty(19, 688, dtype=torch.bfloat16, device="cuda")
    B.biv_silu_mul(dev(gu), y)
    assert rel_err(host_f32(y), ops.silu_mul(gu.float().numpy())) < REL


def test_embed_and_bad_id(B):
    g = synth.rng(6)
    table = rnd_bf16(g, 100, 64)
    ids = np.array([3, 0, 99, 42], np.int32)
    h = torch.empty(4, 64, dtype=torch.bfloat16, device="cuda")
    B.biv_embed(dev(ids), dev(table), h)
    assert np.array_equal(bits(h), bits(table[ids]))
    assert B.biv_poll_error() == 0
    B.biv_embed(dev(np.array([1, 100], np.int32)), dev(table), h[:2])
    assert B.biv_poll_error() == 2                      # bad index reported, then cleared
    assert B.biv_poll_error() == 0


# --------------------------------------------------------------------- RoPE --
@pytest.mark.parametrize("D,qk", [(128, True), (64, False), (80, False)])
def test_qk_norm_rope_parity(B, D, qk):
    g = synth.rng(7)
    T, Hq, Hkv, max_pos = 9, 4, 2, 5000
    qkv = rnd_bf16(g, T, (Hq + 2 * Hkv) * D)
    pos = np.array([0, 1, 5, 77, 128, 1000, 4095, 4999, 3], np.int32)
    qw = rnd_bf16(g, D) if qk else None
    kw = rnd_bf16(g, D) if qk else None
    tab = torch.empty(2 * max_pos * (D // 2), dtype=torch.float32, device="cuda")
    B.biv_rope_table(1e6, D, max_pos, tab)
    cos, sin = ops.rope_table(1e6, D, max_pos)
    got_tab = tab.cpu().numpy().reshape(2, max_pos, D // 2)
    assert np.max(np.abs(got_tab[0] - cos)) < 1e-6 and np.max(np.abs(got_tab[1] - sin)) < 1e-6
    qd = dev(qkv)
    B.biv_qk_norm_rope(qd, T, Hq, Hkv, D, dev(qw) if qk else None, dev(kw) if qk else None, tab,
                       max_pos, dev(pos), 1e-6)
    x = qkv.float().numpy()
    q = x[:, :Hq * D].reshape(T, Hq, D)
    k = x[:, Hq * D:(Hq + Hkv) * D].reshape(T, Hkv, D)
    qr = ops.qk_norm_rope(q, pos, qw.float().numpy() if qk else None, 1e-6, cos, sin)
    kr = ops.qk_norm_rope(k, pos, kw.float().numpy() if qk else None, 1e-6, cos, sin)
    got = host_f32(qd)
    assert rel_err(got[:, :Hq * D].reshape(T, Hq, D), qr) < REL
    assert rel_err(got[:, Hq * D:(Hq + Hkv) * D].reshape(T, Hkv, D), kr) < REL
    assert np.array_equal(got[:, (Hq + Hkv) * D:], x[:, (Hq + Hkv) * D:])   # v untouched


# ------------------------------------------------------------------- FP8 KV --
@pytest.mark.parametrize("D", [128, 64, 80])
def test_kv_fp8_quant_codes_bit_exact_and_gather(B, D):
    g = synth.rng(8)
    T, Hkv, page = 70, 2, 64
    k, v = rnd_bf16(g, T, Hkv * D, std=3.0), rnd_bf16(g, T, Hkv * D)
    k[5] = 0   # amax = 0 row -> scale 1, codes 0
    pages = 4
    slot = np.arange(T, dtype=np.int64) + 64 * 1      # start on page 1
    kc = torch.zeros(pages, page, Hkv, D, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.zeros(pages, page, Hkv, dtype=torch.float32, device="cuda")
    vs = torch.zeros_like(ks)
    kd, vd = dev(k), dev(v)
    B.biv_kv_fp8_quant(kd, vd, Hkv * D, dev(slot), T, Hkv, D, kc, vc, ks, vs)
    c_ref, s_ref = ops.fp8_quant_rows(k.float().numpy().reshape(T, Hkv, D))
    got_c = kc.view(-1, Hkv, D)[64:64 + T].cpu().numpy()
    got_s = ks.view(-1, Hkv)[64:64 + T].cpu().numpy()
    assert np.array_equal(got_c, c_ref) and np.array_equal(got_s, s_ref)
    # gather + dequant of 2 sequences sharing the pages
    bt = dev(np.array([[1, 2, 0, 0], [1, 0, 0, 0]], np.int32))
    ctx = dev(np.array([T, 10], np.int32))
    row0 = dev(np.array([0, T], np.int64))
    out = torch.empty(T + 10, Hkv, D, dtype=torch.bfloat16, device="cuda")
    B.biv_kv_fp8_gather(kc, ks, bt, ctx, row0, Hkv, D, page, out)
    ref = ops.fp8_dequant_rows(c_ref, s_ref)
    assert np.array_equal(host_f32(out[:T]), ref) and np.array_equal(host_f32(out[T:]), ref[:10])


def test_kv_store_bf16(B):
    g = synth.rng(9)
    T, Hkv, D = 5, 2, 64
    qkv = rnd_bf16(g, T, 4 * Hkv * D)
    kd = dev(qkv)
    kc = torch.zeros(2, 64, Hkv, D, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    slot = dev(np.array([0, 1, -1, 70, 127], np.int64))
    B.biv_kv_store_bf16(kd[:, :Hkv * D], kd[:, Hkv * D:], 4 * Hkv * D, slot, T, Hkv, D, kc, vc)
    kcf = kc.view(-1, Hkv * D)
    assert torch.equal(kcf[70], kd[3, :Hkv * D]) and torch.equal(kcf[2], torch.zeros_like(kcf[2]))
    assert torch.equal(vc.view(-1, Hkv * D)[127], kd[4, Hkv * D:2 * Hkv * D])


# ------------------------------------------------------------------ logprob --
@pytest.mark.parametrize("V", [4096, 151936])
def test_logprob_parity_and_invariance(B, V):
    g = synth.rng(10)
    T = 13
    z = (synth.normal_f32(g, (T, V)) * 3).astype(np.float32)
    tgt = g.integers(0, V, size=T).astype(np.int32)
    lp = torch.empty(T, dtype=torch.float32, device="cuda")
    zd = dev(z)
    B.biv_logprob(zd, dev(tgt), lp)
    ref = ops.logprob(z, tgt)
    assert np.max(np.abs(lp.cpu().numpy() - ref)) < 1e-4
    lp1 = torch.empty(1, dtype=torch.float32, device="cuda")
    B.biv_logprob(zd[7:8], dev(tgt[7:8]), lp1)
    assert np.array_equal(bits(lp1), bits(lp[7:8]))
    # uniform logits: exactly -log V up to float rounding
    B.biv_logprob(torch.zeros(2, V, device="cuda"), dev(np.array([0, 1], np.int32)), lp[:2])
    assert np.allclose(lp[:2].cpu().numpy(), -math.log(V), atol=1e-5)


@pytest.mark.parametrize("M,V,K", [(13, 4096, 256), (5, 4100, 96), (1, 151936, 2048),
                                   (300, 151936, 2048)])
def test_lm_head_logprob_parity_and_invariance(B, M, V, K):
    """The fused LM head + log-softmax gather: within 1e-4 of the oracle's
    logprob of the oracle's FP32 logits (peaked head, logit std about 3), a row
    alone or inside another batch keeps its bits, and a bad target is NaN and
    reported."""
    g = synth.rng(M + V + K)
    h, W = rnd_bf16(g, M, K), rnd_bf16(g, V, K, std=3.0 / math.sqrt(K))
    tgt = g.integers(0, V, size=M).astype(np.int32)
    hd, Wd, td = dev(h), dev(W), dev(tgt)
    ws = torch.empty(B.biv_lm_head_logprob_workspace(M, V), dtype=torch.uint8, device="cuda")
    lp = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda")
    B.biv_lm_head_logprob(hd, Wd, td, lp, ws)
    assert B.biv_poll_error() == 0
    got = lp.cpu().numpy()
    rows = np.arange(M) if M * V <= 1 << 22 else np.unique(np.r_[0, 7, M // 2, M - 1] % M)
    z = ops.gemm(h[rows].float().numpy(), W.float().numpy(), out="f32")
    ref = ops.logprob(z, tgt[rows])
    assert np.std(z) > 1.0
    assert np.max(np.abs(got[rows] - ref)) < 1e-4
    # a row alone, and a slice in the middle of the batch: the same bits
    r = min(7, M - 1)
    one = torch.empty(1, dtype=torch.float32, device="cuda")
    B.biv_lm_head_logprob(hd[r:r + 1], Wd, td[r:r + 1], one, ws)
    assert np.array_equal(bits(one), bits(lp[r:r + 1]))
    if M > 4:
        mid = torch.empty(M - 3, dtype=torch.float32, device="cuda")
        B.biv_lm_head_logprob(hd[2:M - 1], Wd, td[2:M - 1], mid, ws)
        assert np.array_equal(bits(mid), bits(lp[2:M - 1]))
    # zero weights: every logit 0, lp = -log V up to rounding
    B.biv_lm_head_logprob(hd[:1], torch.zeros_like(Wd), td[:1], one, ws)
    assert abs(one.item() + math.log(V)) < 1e-5
    # a target outside [0, V): NaN and error code 2, then cleared
    B.biv_lm_head_logprob(hd[:1], Wd, dev(np.array([V], np.int32)), one, ws)
    assert math.isnan(one.item()) and B.biv_poll_error() == 2
    assert B.biv_poll_error() == 0


# --------------------------------------------------------------------- GEMM --
GEMM_SHAPES = [(1, 64, 64), (5, 96, 80), (130, 512, 256), (200, 688, 256), (77, 256, 688),
               (257, 1000, 320), (64, 4096, 2048), (300, 2048, 6144)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_gemm_bf16_parity(B, M, N, K, out):
    g = synth.rng(M * 7 + N + K)
    a, b = rnd_bf16(g, M, K), rnd_bf16(g, N, K, std=0.05)
    ad, bd = dev(a), dev(b)
    c = torch.full((M, N), float("nan"), dtype=torch.bfloat16 if out == "bf16" else torch.float32,
                   device="cuda")
    B.biv_gemm(B.gemm_desc(ad, bd, c))
    ref = ops.gemm(a.float().numpy(), b.float().numpy(), out=out)
    got = host_f32(c)
    assert np.isfinite(got).all()
    assert rel_err(got, ref) < REL


@pytest.mark.parametrize("N,K", [(512, 256), (4096, 2048), (151936 // 8, 2048)])
def test_gemm_row_invariance(B, N, K):
    """Any row's bits are the same alone, in a batch of 300, or at another
    position of the 128-row tile."""
    g = synth.rng(N + K)
    M = 300
    a, b = rnd_bf16(g, M, K), rnd_bf16(g, N, K, std=0.05)
    ad, bd = dev(a), dev(b)
    full = torch.empty(M, N, dtype=torch.float32, device="cuda")
    B.biv_gemm(B.gemm_desc(ad, bd, full))
    for r in [0, 1, 127, 128, 200, 299]:
        one = torch.empty(1, N, dtype=torch.float32, device="cuda")
        B.biv_gemm(B.gemm_desc(ad[r:r + 1], bd, one))
        assert np.array_equal(bits(one), bits(full[r:r + 1])), r
    # shifted batch: row r lands at another tile position
    sub = torch.empty(M - 45, N, dtype=torch.float32, device="cuda")
    B.biv_gemm(B.gemm_desc(ad[45:], bd, sub))
    assert np.array_equal(bits(sub), bits(full[45:]))


def test_gemm_fast_mode_is_close_but_batch_dependent(B):
    g = synth.rng(11)
    M, N, K = 3, 2048, 6144
    a, b = rnd_bf16(g, M, K), rnd_bf16(g, N, K, std=0.05)
    ad, bd = dev(a), dev(b)
    inv = torch.empty(M, N, dtype=torch.float32, device="cuda")
    B.biv_gemm(B.gemm_desc(ad, bd, inv))
    d = B.gemm_desc(ad, bd, torch.empty(M, N, dtype=torch.float32, device="cuda"), mode=B.MODE_FAST)
    fast = torch.empty(M, N, dtype=torch.float32, device="cuda")
    d = B.gemm_desc(ad, bd, fast, mode=B.MODE_FAST)
    n = B.biv_gemm_workspace(d)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    B.biv_gemm(d, ws)
    assert n > 0                                     # FAST splits K at small M
    assert rel_err(fast.cpu().numpy(), inv.cpu().numpy()) < 1e-4


def test_gemm_fp8_block_scaled_parity(B):
    g = synth.rng(12)
    M, N, K = 200, 384, 512
    a = rnd_bf16(g, M, K)
    codes_b, sb = synth.fp8_block_weights(g, 1, N, K)
    ad = dev(a)
    ac = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    sa = torch.empty(M, K // 128, dtype=torch.float32, device="cuda")
    B.biv_act_quant_fp8(ad, ac, sa)
    ac_ref, sa_ref = ops.act_quant_fp8(a.float().numpy())
    assert np.array_equal(ac.cpu().numpy(), ac_ref) and np.array_equal(sa.cpu().numpy(), sa_ref)
    bc = dev(codes_b[0].view(torch.uint8))
    c = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    B.biv_gemm(B.gemm_desc(ac, bc, c, sa=sa, sb=dev(sb[0])))
    ref = ops.gemm_fp8_block(ac_ref, sa_ref, synth.fp8_bits(codes_b[0]), sb[0])
    assert rel_err(host_f32(c), ref) < REL
    one = torch.empty(1, N, dtype=torch.bfloat16, device="cuda")
    B.biv_gemm(B.gemm_desc(ac[150:151], bc, one, sa=sa[150:151], sb=dev(sb[0])))
    assert np.array_equal(bits(one), bits(c[150:151]))


@pytest.mark.parametrize("rows,I", [(1, 1408), (300, 1408), (7, 144)])
def test_silu_mul_quant_equals_two_calls(B, rows, I):
    """The fused SiLU-mul + FP8 activation quantisation writes the codes and
    scales of biv_silu_mul followed by biv_act_quant_fp8, bit for bit (a
    ragged last group included); they are the oracle's quantisation of that
    bf16 activation, which is within the SiLU-mul tolerance of the oracle's."""
    g = synth.rng(rows + I)
    gu = rnd_bf16(g, rows, 2 * I)
    gu[0, :I] = 0.0                                   # an all-zero first row: scale 1
    gud = dev(gu)
    act = torch.empty(rows, I, dtype=torch.bfloat16, device="cuda")
    q2 = torch.empty(rows, I, dtype=torch.uint8, device="cuda")
    s2 = torch.empty(rows, (I + 127) // 128, dtype=torch.float32, device="cuda")
    B.biv_silu_mul(gud, act)
    B.biv_act_quant_fp8(act, q2, s2)
    q1 = torch.full((rows, I), 0xAB, dtype=torch.uint8, device="cuda")
    s1 = torch.full((rows, (I + 127) // 128), float("nan"), dtype=torch.float32, device="cuda")
    B.biv_silu_mul_quant_fp8(gud, q1, s1)
    assert np.array_equal(bits(q1), bits(q2)) and np.array_equal(bits(s1), bits(s2))
    rq, rs = ops.act_quant_fp8(host_f32(act))
    assert np.array_equal(q1.cpu().numpy(), rq) and np.array_equal(s1.cpu().numpy(), rs)
    assert rel_err(host_f32(act), ops.silu_mul(gu.float().numpy())) < REL


def test_gemm_fp8_grouped(B):
    g = synth.rng(13)
    G, N, K = 4, 256, 384
    counts = [130, 0, 7, 257]
    M = sum(counts)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    a = rnd_bf16(g, M, K)
    codes_b, sb = synth.fp8_block_weights(g, G, N, K)
    ac = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    sa = torch.empty(M, K // 128, dtype=torch.float32, device="cuda")
    B.biv_act_quant_fp8(dev(a), ac, sa)
    c = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    bc = dev(codes_b.view(torch.uint8).reshape(G * N, K))
    B.biv_gemm(B.gemm_desc(ac, bc, c, sa=sa, sb=dev(sb), group_offsets=dev(offs), groups=G, M=M))
    ac_h, sa_h = ac.cpu().numpy(), sa.cpu().numpy()
    got = host_f32(c)
    for e in range(G):
        lo, hi = offs[e], offs[e + 1]
        if hi == lo:
            continue
        ref = ops.gemm_fp8_block(ac_h[lo:hi], sa_h[lo:hi], synth.fp8_bits(codes_b[e]), sb[e])
        assert rel_err(got[lo:hi], ref) < REL, e


@pytest.mark.parametrize("G,N,K", [(1, 640, 384), (5, 512, 1408), (3, 2816, 4096)])
def test_fp8_two_block_stages_change_no_bit(B, monkeypatch, G, N, K):
    """FP8 stages of two 128-wide K blocks (3-D TMA boxes; an odd block count
    leaves the last stage's second block as zero fill) and of one block feed
    the same MMAs and the same promotions: every output bit is the same; a
    group with no rows and N % 256 == 128 included."""
    g = synth.rng(G * 7 + N + K)
    counts = [0] if G == 1 else [150, 0, 300, 5, 129][:G]
    M = 333 if G == 1 else sum(counts)
    a = rnd_bf16(g, M, K)
    codes_b, sb = synth.fp8_block_weights(g, G, N, K)
    ac = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    sa = torch.empty(M, K // 128, dtype=torch.float32, device="cuda")
    B.biv_act_quant_fp8(dev(a), ac, sa)
    bc = dev(codes_b.view(torch.uint8).reshape(G * N, K))
    kw = {}
    if G > 1:
        offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        kw = dict(group_offsets=dev(offs), groups=G, M=M)
    outs = []
    for kpb in ["2", "1"]:
        monkeypatch.setenv("BIV_GEMM_KPB", kpb)
        c = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        B.biv_gemm(B.gemm_desc(ac, bc, c, sa=sa, sb=dev(sb if G > 1 else sb[0]), **kw))
        outs.append(bits(c))
    assert np.array_equal(outs[0], outs[1])
    lo = 0 if G == 1 else counts[0] + counts[1]
    hi = M if G == 1 else lo + counts[2]
    e = 0 if G == 1 else 2
    ref = ops.gemm_fp8_block(ac.cpu().numpy()[lo:hi], sa.cpu().numpy()[lo:hi],
                             synth.fp8_bits(codes_b[e]), sb[e])
    got = outs[0].view(np.uint16).reshape(M, N)[lo:hi]
    assert rel_err((got.astype(np.uint32) << 16).view(np.float32), ref) < REL


# -------------------------------------------------------------------- Top-K --
def test_topk_brute_force_ties(B):
    g = synth.rng(14)
    R, n, k = 40, 1000, 37
    s = g.integers(0, 4, size=(R, n)).astype(np.float32)
    s[3] = -np.inf
    s[4, :500] = -np.inf
    s[5, 7] = -0.0
    s[6] = 0.0
    nv = g.integers(0, n + 1, size=R).astype(np.int32)
    nv[:8] = n
    nv[8] = 10
    idx = torch.empty(R, k, dtype=torch.int32, device="cuda")
    B.biv_topk(dev(s), dev(nv), k, idx)
    assert np.array_equal(idx.cpu().numpy(), ops.topk_positions(s, nv, k))


def test_topk_indexer_shape(B):
    g = synth.rng(15)
    R, n, k = 64, 32768, 2048
    s = synth.normal_f32(g, (R, n))
    s[:, ::3] = np.round(s[:, ::3], 1)          # plenty of ties
    nv = (n - R + np.arange(R)).astype(np.int32)
    idx = torch.empty(R, k, dtype=torch.int32, device="cuda")
    sd = dev(s)
    B.biv_topk(sd, dev(nv), k, idx)
    got = idx.cpu().numpy()
    assert np.array_equal(got, ops.topk_positions(s, nv, k))           # all 64 rows
    # a row alone gives the same indices
    one = torch.empty(1, k, dtype=torch.int32, device="cuda")
    B.biv_topk(sd[40:41], dev(nv[40:41]), k, one)
    assert np.array_equal(one.cpu().numpy()[0], got[40])


def test_topk_range_refinement_distributions(B):
    """Rows whose keys sit in one bin, two values, the extremes of the float
    range (+inf, the largest and smallest normals, denormals), only negative
    scores, a ragged valid length: every row equals the oracle's selection."""
    g = synth.rng(16)
    R, n, k = 12, 5000, 300
    s = synth.normal_f32(g, (R, n))
    s[0] = 1.5                                            # one key value
    s[1] = np.where(g.random(n) < 0.5, 2.0, -2.0)         # two values
    s[2] = np.float32(3.4e38) * np.sign(s[2])             # +-max normal
    s[2, ::7] = np.inf
    s[3] = np.float32(1e-40) * g.integers(-3, 4, n)        # denormals and zeros
    s[4] = -np.abs(s[4]) - 1.0                            # all negative
    s[5] = np.ldexp(np.float32(1.0), g.integers(-120, 120, n)).astype(np.float32)  # exponents spread
    s[6] = np.float32(1.0) + np.float32(2.0 ** -23) * g.integers(0, 40, n)  # adjacent keys
    s[7, :] = -np.inf
    s[7, 10:20] = 0.5                                     # fewer valid than k
    s[8] = np.round(s[8] * 4) / 4                         # many ties at the threshold
    nv = np.full(R, n, np.int32)
    nv[9] = 1234
    nv[10] = k                                            # exactly k valid
    nv[11] = 0
    idx = torch.empty(R, k, dtype=torch.int32, device="cuda")
    B.biv_topk(dev(s), dev(nv), k, idx)
    assert np.array_equal(idx.cpu().numpy(), ops.topk_positions(s, nv, k))


def test_topk_many_rows_per_cta(B):
    """More rows than SMs, so each persistent CTA selects several rows in turn
    and its first round starts from the previous row's bin: rows whose scale
    jumps by 1e6 either way, rows with fewer than k valid scores, exactly k,
    and one key value follow one another; every row equals the oracle's."""
    g = synth.rng(18)
    R, n, k = 1400, 4096, 256
    s = synth.normal_f32(g, (R, n))
    scale = np.float32(10.0) ** g.choice([-6, -3, 0, 0, 0, 3, 6], size=R).astype(np.float32)
    s *= scale[:, None]
    s[::9] += np.float32(50.0)
    s[5::11] = np.round(s[5::11])                     # ties at the threshold
    s[7::13] = 2.5                                    # one key value
    nv = np.full(R, n, np.int32)
    nv[3::7] = g.integers(0, 2 * k, size=nv[3::7].size)   # some below k, some above
    nv[4::17] = k
    idx = torch.empty(R, k, dtype=torch.int32, device="cuda")
    B.biv_topk(dev(s), dev(nv), k, idx)
    got, ref = idx.cpu().numpy(), ops.topk_positions(s, nv, k)
    bad = np.nonzero((got != ref).any(axis=1))[0]
    assert bad.size == 0, f"rows differ: {bad[:20]} (of {bad.size})"


def test_topk_nan_never_chosen(B):
    """NaN scores of either sign and any payload are never chosen, as in the
    oracle (a NaN is not greater than -inf); the rest of the row is selected
    as if they were -inf."""
    g = synth.rng(17)
    R, n, k = 4, 3000, 200
    s = synth.normal_f32(g, (R, n))
    nan_bits = np.array([0x7FC00000, 0x7F800001, 0x7FFFFFFF, 0xFFC00000, 0xFF800001, 0xFFFFFFFF],
                        np.uint32)
    for r in range(R):
        pos = g.choice(n, size=300 + 100 * r, replace=False)
        s[r, pos] = nan_bits[g.integers(0, nan_bits.size, pos.size)].view(np.float32)
    s[3, 150:] = np.uint32(0x7FC00000).view(np.float32)   # fewer than k non-NaN scores
    nv = np.full(R, n, np.int32)
    idx = torch.empty(R, k, dtype=torch.int32, device="cuda")
    B.biv_topk(dev(s), dev(nv), k, idx)
    got = idx.cpu().numpy()
    assert np.array_equal(got, ops.topk_positions(s, nv, k))
    for r in range(R):
        chosen = got[r][got[r] >= 0]
        assert not np.isnan(s[r, chosen]).any()


def test_router_topk(B):
    g = synth.rng(16)
    R, E, k = 300, 64, 6
    z = (g.integers(-3, 4, size=(R, E)) * 0.5).astype(np.float32)
    idx = torch.empty(R, k, dtype=torch.int32, device="cuda")
    w = torch.empty(R, k, dtype=torch.float32, device="cuda")
    B.biv_router_topk(dev(z), k, idx, w)
    ri, rw = ops.router_topk(z, k)
    assert np.array_equal(idx.cpu().numpy(), ri)
    assert np.max(np.abs(w.cpu().numpy() - rw)) < 1e-6


def test_moe_dispatch_gather_combine(B):
    g = synth.rng(17)
    T, k, E, d = 50, 6, 8, 64
    idx = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    src = torch.empty(T * k, dtype=torch.int32, device="cuda")
    B.biv_moe_dispatch(dev(idx), E, offs, perm, src)
    flat = idx.ravel()
    ref_perm = np.concatenate([np.nonzero(flat == e)[0] for e in range(E)]).astype(np.int32)
    assert np.array_equal(perm.cpu().numpy(), ref_perm)
    assert np.array_equal(offs.cpu().numpy(), np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    inv = np.empty_like(ref_perm)
    inv[ref_perm] = np.arange(T * k)
    assert np.array_equal(src.cpu().numpy(), inv)
    # gather token rows into expert order, combine back in slot order
    h = rnd_bf16(g, T, d)
    hg = torch.empty(T * k, d, dtype=torch.bfloat16, device="cuda")
    B.biv_gather_rows(dev(h), perm, k, T * k, hg)
    assert np.array_equal(bits(hg), bits(h[torch.from_numpy(ref_perm // k).long()]))
    y = rnd_bf16(g, T * k, d)
    w = np.abs(synth.normal_f32(g, (T, k)))
    sh = rnd_bf16(g, T, d)
    out = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    B.biv_moe_combine(dev(y), src, dev(w), dev(sh), out)
    y_slots = y.float().numpy()[inv].reshape(T, k, d)
    assert rel_err(host_f32(out), ops.moe_combine(y_slots, w, sh.float().numpy())) < REL
    onehot = np.zeros((T, k), np.float32)
    onehot[:, 2] = 1
    B.biv_moe_combine(dev(y), src, dev(onehot), None, out)
    assert np.array_equal(host_f32(out), y_slots[:, 2])


def test_device_wait_timeout_reports_and_recovers(B):
    assert B.biv_poll_error() == 0
    B.biv_selftest_timeout(2_000_000)        # 2 ms bounded wait that nobody satisfies
    assert B.biv_poll_error() == 1           # timeout reported, word cleared
    assert B.biv_poll_error() == 0
    x = torch.ones(4, 64, dtype=torch.bfloat16, device="cuda")
    B.biv_add_rmsnorm(x, None, x[0], x.clone(), 1e-6)   # context still usable
    torch.cuda.synchronize()


@pytest.mark.parametrize("M,N,K,out", [(1, 2048, 2048, "bf16"), (77, 4096, 6144, "f32"),
                                       (300, 1000, 520, "bf16"), (4096, 2048, 2048, "bf16"),
                                       (1200, 151936 // 4, 256, "f32")])
def test_gemm_chunk_fold_in_cta_equals_fold_across_ctas(B, monkeypatch, M, N, K, out):
    """The fixed K-chunk schedule folded inside one CTA (registers) and across
    CTAs (per-chunk partials, folded in chunk order by a second kernel) must
    give the same bits, call after call on one workspace."""
    g = synth.rng(M + N + K)
    a, b = rnd_bf16(g, M, K), rnd_bf16(g, N, K, std=0.05)
    ad, bd = dev(a), dev(b)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    res = []
    for fold in ["cta", "partial", "partial"]:
        monkeypatch.setenv("BIV_GEMM_FOLD", fold)
        monkeypatch.setenv("BIV_GEMM_TILE_N", "128")
        c = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
        d = B.gemm_desc(ad, bd, c)
        n = B.biv_gemm_workspace(d)
        assert (n > 0) == (fold == "partial" and K > 512)
        ws = torch.full((max(n, 256),), 0xFF, dtype=torch.uint8, device="cuda")  # no initial value needed
        B.biv_gemm(d, ws)
        B.biv_gemm(d, ws)
        torch.cuda.synchronize()
        res.append(bits(c))
    monkeypatch.delenv("BIV_GEMM_FOLD")
    monkeypatch.delenv("BIV_GEMM_TILE_N")
    c = torch.empty(M, N, dtype=dt, device="cuda")
    B.biv_gemm(B.gemm_desc(ad, bd, c))                  # the planner's own choice
    res.append(bits(c))
    for r in res[1:]:
        assert np.array_equal(r, res[0])
    ref = ops.gemm(a.float().numpy(), b.float().numpy(), out=out)     # every row
    assert rel_err(host_f32(c), ref) < REL


def test_gemm_shared_workspace_across_shapes(B):
    """Calls of different shapes (different tile counts and chunk counts) on
    one workspace give what each gives on a fresh one."""
    g = synth.rng(5150)
    shapes = [(100, 512, 2048), (7, 8192, 688), (64, 2048, 6144), (3, 4096, 2048), (100, 512, 2048)]
    ws = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    for M, N, K in shapes:
        a, b = dev(rnd_bf16(g, M, K)), dev(rnd_bf16(g, N, K, std=0.05))
        c1 = torch.empty(M, N, dtype=torch.float32, device="cuda")
        c2 = torch.empty(M, N, dtype=torch.float32, device="cuda")
        d1, d2 = B.gemm_desc(a, b, c1), B.gemm_desc(a, b, c2)
        assert B.biv_gemm_workspace(d1) > 0
        B.biv_gemm(d1, ws)
        B.biv_gemm(d2, torch.zeros(B.biv_gemm_workspace(d2), dtype=torch.uint8, device="cuda"))
        torch.cuda.synchronize()
        assert np.array_equal(bits(c1), bits(c2)), (M, N, K)


@pytest.mark.parametrize("M,N,K", [(3, 512, 192), (100, 512, 2048), (7, 8192, 688), (300, 12288, 64),
                                   (4096, 1024, 256)])
def test_tcgen05_result_independent_of_tile_width(B, monkeypatch, M, N, K):
    """The hardware property the tile planner relies on: with the same K
    schedule an output element has the same bits whatever the MMA instruction
    width (tile N) of its CTA, whichever way the chunks are folded."""
    g = synth.rng(M * N + K)
    a, b = rnd_bf16(g, M, K), rnd_bf16(g, N, K, std=0.05)
    ad, bd = dev(a), dev(b)
    outs = []
    for bn in ["64", "128", "192", "256"]:
        monkeypatch.setenv("BIV_GEMM_TILE_N", bn)
        c = torch.empty(M, N, dtype=torch.float32, device="cuda")
        B.biv_gemm(B.gemm_desc(ad, bd, c))
        outs.append(bits(c))
    monkeypatch.delenv("BIV_GEMM_TILE_N")
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    ref = ops.gemm(a.float().numpy(), b.float().numpy(), out="f32")   # every row
    got = outs[0].view(np.float32).reshape(M, N)
    assert rel_err(got, ref) < REL


@pytest.mark.parametrize("M,N,K", [(1, 4096, 2048), (64, 2048, 6144), (256, 12288, 2048),
                                   (300, 1000, 576), (2048, 2048, 2048)])
@pytest.mark.parametrize("fold", ["cta", "partial"])
def test_two_block_stages_change_no_bit(B, monkeypatch, M, N, K, fold):
    """Pipeline stages of two K blocks (3-D TMA boxes) and of one K block feed
    the same MMAs in the same order: every output bit is the same, folded in
    the CTA or as partials (odd chunk tails included: K 576 is 9 blocks)."""
    g = synth.rng(M + N * 3 + K)
    a, b = rnd_bf16(g, M, K), rnd_bf16(g, N, K, std=0.05)
    ad, bd = dev(a), dev(b)
    monkeypatch.setenv("BIV_GEMM_FOLD", fold)
    outs = []
    for kpb in ["2", "1"]:
        monkeypatch.setenv("BIV_GEMM_KPB", kpb)
        d = B.gemm_desc(ad, bd, torch.empty(M, N, dtype=torch.float32, device="cuda"))
        ws = torch.empty(max(B.biv_gemm_workspace(d), 16), dtype=torch.uint8, device="cuda")
        c = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        B.biv_gemm(B.gemm_desc(ad, bd, c), ws)
        outs.append(bits(c))
    assert np.array_equal(outs[0], outs[1])
    rows = np.unique(np.r_[0, M // 2, M - 1])
    ref = ops.gemm(a[rows].float().numpy(), b.float().numpy(), out="f32")
    assert rel_err(outs[0].view(np.float32).reshape(M, N)[rows], ref) < REL


def test_partials_workspace_alignment_changes_no_bit(B, monkeypatch):
    """Partial mode stores its FP32 partials 32 bytes at a time when the
    workspace is 32-byte aligned and 16 bytes at a time otherwise: the
    outputs have the same bits either way."""
    g = synth.rng(77)
    M, N, K = 64, 4096, 2048
    a, b = rnd_bf16(g, M, K), rnd_bf16(g, N, K, std=0.05)
    ad, bd = dev(a), dev(b)
    monkeypatch.setenv("BIV_GEMM_FOLD", "partial")
    d = B.gemm_desc(ad, bd, torch.empty(M, N, dtype=torch.float32, device="cuda"))
    need = B.biv_gemm_workspace(d)
    assert need > 0
    big = torch.empty(need + 64, dtype=torch.uint8, device="cuda")
    assert big.data_ptr() % 32 == 0
    outs = []
    for off in (0, 16):
        c = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        B.biv_gemm(B.gemm_desc(ad, bd, c), big[off:off + need])
        outs.append(bits(c))
    assert np.array_equal(outs[0], outs[1])


# ------------------------------------------------- fused GEMM consumers --
def _deferred_gemm(B, ad, bd, M, N, ws):
    """GEMM whose fold is left to the consumer; returns the partials (chunks
    > 0) -- the shapes below are chosen so that the plan leaves partials."""
    c = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    d = B.gemm_desc(ad, bd, c)
    assert 0 < B.biv_gemm_workspace(d) <= ws.numel()
    d.defer_fold = 1
    B.biv_gemm(d, ws)
    P = B.biv_gemm_partials(d, ws)
    assert P.chunks > 1
    return P


@pytest.mark.parametrize("M,d_model,K", [(1, 2048, 2048), (37, 2048, 6144), (64, 1024, 3072)])
def test_add_rmsnorm_from_partials_equals_folded_gemm(B, M, d_model, K):
    """Residual add + RMSNorm reading the GEMM's chunk partials (the fold done
    in the consumer) gives the bits of the GEMM folding them itself followed
    by the plain op."""
    g = synth.rng(M * 7 + K)
    a, b = rnd_bf16(g, M, K), rnd_bf16(g, d_model, K, std=0.05)
    r, w = rnd_bf16(g, M, d_model), rnd_bf16(g, d_model)
    ad, bd, wd = dev(a), dev(b), dev(w)
    ws = torch.full((64 << 20,), 0xFF, dtype=torch.uint8, device="cuda")
    c = torch.empty(M, d_model, dtype=torch.bfloat16, device="cuda")
    B.biv_gemm(B.gemm_desc(ad, bd, c), ws)
    r1, y1 = dev(r), torch.empty(M, d_model, dtype=torch.bfloat16, device="cuda")
    B.biv_add_rmsnorm(c, r1, wd, y1, 1e-6)
    P = _deferred_gemm(B, ad, bd, M, d_model, ws)
    r2, y2 = dev(r), torch.empty_like(y1)
    B.biv_add_rmsnorm_partials(P, r2, wd, y2, M, 1e-6)
    torch.cuda.synchronize()
    assert np.array_equal(bits(r2), bits(r1)) and np.array_equal(bits(y2), bits(y1))


@pytest.mark.parametrize("kv_fp8", [False, True], ids=["bf16kv", "fp8kv"])
@pytest.mark.parametrize("D,qk,fold", [(128, True, False), (128, True, True), (64, False, True)])
def test_qkv_finalize_equals_separate_ops(B, kv_fp8, D, qk, fold):
    """QK-norm + RoPE + k/v cache store in one kernel (optionally folding the
    QKV GEMM's chunk partials first) gives the bits of the separate ops: the
    normed, rotated q and k rows, v untouched, the same cache codes/scales."""
    g = synth.rng(D + 3 * qk + 5 * fold + 11 * kv_fp8)
    T, Hq, Hkv, max_pos, K = 9, 4, 2, 5000, 2048
    W3 = (Hq + 2 * Hkv) * D
    pos = np.array([0, 1, 5, 77, 128, 1000, 4095, 4999, 3], np.int32)
    slot = np.array([64, 65, 3, 130, 200, 7, 66, 140, 0], np.int64)
    qw = dev(rnd_bf16(g, D)) if qk else None
    kw = dev(rnd_bf16(g, D)) if qk else None
    tab = torch.empty(2 * max_pos * (D // 2), dtype=torch.float32, device="cuda")
    B.biv_rope_table(1e6, D, max_pos, tab)
    pages, page = 4, 64
    cdt = torch.uint8 if kv_fp8 else torch.bfloat16

    def caches():
        kc = torch.zeros(pages, page, Hkv, D, dtype=cdt, device="cuda")
        ks = torch.zeros(pages, page, Hkv, dtype=torch.float32, device="cuda") if kv_fp8 else None
        return kc, torch.zeros_like(kc), ks, (torch.zeros_like(ks) if kv_fp8 else None)

    ws = torch.full((64 << 20,), 0xFF, dtype=torch.uint8, device="cuda")
    if fold:
        a, b = dev(rnd_bf16(g, T, K)), dev(rnd_bf16(g, W3, K, std=0.05))
        q1 = torch.empty(T, W3, dtype=torch.bfloat16, device="cuda")
        B.biv_gemm(B.gemm_desc(a, b, q1), ws)
    else:
        q1 = dev(rnd_bf16(g, T, W3))
    q2 = q1.clone()
    # separate ops
    kc1, vc1, ks1, vs1 = caches()
    B.biv_qk_norm_rope(q1, T, Hq, Hkv, D, qw, kw, tab, max_pos, dev(pos), 1e-6)
    kq, vq = q1[:, Hq * D:], q1[:, (Hq + Hkv) * D:]
    if kv_fp8:
        B.biv_kv_fp8_quant(kq, vq, q1.stride(0), dev(slot), T, Hkv, D, kc1, vc1, ks1, vs1)
    else:
        B.biv_kv_store_bf16(kq, vq, q1.stride(0), dev(slot), T, Hkv, D, kc1, vc1)
    # fused
    kc2, vc2, ks2, vs2 = caches()
    P = None
    if fold:
        q2.fill_(float("nan"))
        P = _deferred_gemm(B, a, b, T, W3, ws)
    B.biv_qkv_finalize(q2, T, Hq, Hkv, D, qw, kw, tab, max_pos, dev(pos), 1e-6, dev(slot),
                       B.E4M3 if kv_fp8 else B.BF16, kc2, vc2, ks2, vs2, partials=P)
    torch.cuda.synchronize()
    assert np.array_equal(bits(q2), bits(q1))
    for x, y in [(kc2, kc1), (vc2, vc1)] + ([(ks2, ks1), (vs2, vs1)] if kv_fp8 else []):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))


@pytest.mark.parametrize("M,I", [(1, 6144), (64, 6144), (5, 688)])
def test_silu_mul_from_partials_equals_folded_gemm(B, M, I):
    """SiLU-mul reading the gate/up GEMM's chunk partials gives the bits of
    the GEMM folding them itself followed by the plain op."""
    g = synth.rng(M + I)
    K = 2048
    a, b = dev(rnd_bf16(g, M, K)), dev(rnd_bf16(g, 2 * I, K, std=0.05))
    ws = torch.full((64 << 20,), 0xFF, dtype=torch.uint8, device="cuda")
    gu = torch.empty(M, 2 * I, dtype=torch.bfloat16, device="cuda")
    B.biv_gemm(B.gemm_desc(a, b, gu), ws)
    y1 = torch.empty(M, I, dtype=torch.bfloat16, device="cuda")
    B.biv_silu_mul(gu, y1)
    P = _deferred_gemm(B, a, b, M, 2 * I, ws)
    y2 = torch.full_like(y1, float("nan"))
    B.biv_silu_mul_partials(P, y2, M)
    torch.cuda.synchronize()
    assert np.array_equal(bits(y2), bits(y1))
