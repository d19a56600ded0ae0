"""Pins for the per-op oracle against closed forms, library routines and brute
force (CPU only).  Each check is chosen so that a plausible slip in the oracle
(a dropped term, a wrong sign or index, a transposed operand) fails."""
import math

import numpy as np
import pytest
import torch

from oracle import ops
from oracle.codecs import bf16_round, e4m3_to_f32, f32_to_e4m3
from oracle.ssd import ssd_chunked, ssd_sequential

F32 = np.float32


def bf(x):
    return bf16_round(np.asarray(x, F32))


def randn(g, *shape, std=1.0):
    return bf(g.standard_normal(shape).astype(F32) * std)


# ---------------------------------------------------------------- GEMM ----
def test_gemm_within_fp32_bound_of_fp64():
    g = np.random.default_rng(0)
    for M, N, K in [(1, 7, 5), (33, 65, 300), (130, 40, 688)]:
        a, b = randn(g, M, K), randn(g, N, K)
        ref = a.astype(np.float64) @ b.astype(np.float64).T
        bound = K * 2.0 ** -23 * (np.abs(a).astype(np.float64) @ np.abs(b).astype(np.float64).T)
        c = ops.gemm(a, b, out="f32")
        assert np.all(np.abs(c - ref) <= bound + 1e-30)
        cb = ops.gemm(a, b)
        assert np.all(np.abs(cb - ref) <= bound + np.abs(ref) * 2.0 ** -8 + 1e-30)


def test_gemm_accumulation_orders_within_fp32_bounds():
    """Every FP32 order the oracle offers stays within K * 2^-23 * sum|a||b|
    of the exact sum; round-toward-zero never rounds away from zero on
    same-sign terms; integer sums are exact in every order."""
    g = np.random.default_rng(30)
    a, b = randn(g, 4, 700), randn(g, 6, 700)
    ref = a.astype(np.float64) @ b.astype(np.float64).T
    bound = 700 * 2.0 ** -23 * (np.abs(a).astype(np.float64) @ np.abs(b).astype(np.float64).T)
    pos_a, pos_b = np.abs(a), np.abs(b)
    pos_ref = pos_a.astype(np.float64) @ pos_b.astype(np.float64).T
    ia = g.integers(-4, 5, size=(3, 50)).astype(F32)
    ib = g.integers(-4, 5, size=(2, 50)).astype(F32)
    for kind in ops.KINDS:
        with ops.accumulation(kind):
            assert np.all(np.abs(ops.gemm(a, b, out="f32") - ref) <= bound + 1e-30), kind
            if kind == "f32_rz":
                assert np.all(ops.gemm(pos_a, pos_b, out="f32") <= pos_ref)
            assert np.array_equal(ops.gemm(ia, ib, out="f32"), (ia @ ib.T).astype(F32))
    with pytest.raises(ValueError):
        with ops.accumulation("f16"):
            pass


def test_gemm_integer_exact_and_orientation():
    g = np.random.default_rng(1)
    a = g.integers(-4, 5, size=(9, 13)).astype(F32)
    b = g.integers(-4, 5, size=(6, 13)).astype(F32)
    c = ops.gemm(a, b, out="f32")
    assert np.array_equal(c, (a.astype(np.int64) @ b.astype(np.int64).T).astype(F32))
    # C[m, n] = sum_k A[m, k] B[n, k]: one-hot probes fix the orientation
    e = np.zeros((1, 13), F32); e[0, 4] = 1
    assert np.array_equal(ops.gemm(e, b, out="f32")[0], b[:, 4])


# ------------------------------------------------------------- RMSNorm ----
def test_rmsnorm_constant_vector_gives_sign_times_gain():
    g = np.random.default_rng(2)
    w = randn(g, 256) + 1
    for c in [3.0, -0.5, 1e-2]:
        y = ops.rmsnorm(np.full((1, 256), c, F32), w, 1e-6)
        assert np.allclose(y[0], bf(np.sign(c) * w / math.sqrt(1 + 1e-6 / c ** 2)), rtol=2 ** -7)


def test_rmsnorm_against_linalg_norm():
    g = np.random.default_rng(3)
    x, w = randn(g, 5, 2048), randn(g, 2048)
    rms = np.linalg.norm(x.astype(np.float64), axis=1, keepdims=True) / math.sqrt(2048)
    ref = x / np.sqrt(rms ** 2 + 1e-6) * w
    assert np.allclose(ops.rmsnorm(x, w, 1e-6), ref, rtol=2 ** -7, atol=1e-6)


def test_add_rmsnorm_residual_is_bf16_sum():
    g = np.random.default_rng(4)
    x, r, w = randn(g, 4, 256), randn(g, 4, 256), randn(g, 256)
    r2, y = ops.add_rmsnorm(x, r, w, 1e-6)
    tr = (torch.from_numpy(x).bfloat16() + torch.from_numpy(r).bfloat16()).float().numpy()
    assert np.array_equal(r2, tr)
    assert np.array_equal(y, ops.rmsnorm(tr, w, 1e-6))


# ------------------------------------------------------------- SiLU-mul ----
def test_silu_mul_against_torch_silu():
    g = np.random.default_rng(5)
    gu = randn(g, 3, 2 * 688, std=3)
    y = ops.silu_mul(gu)
    t = torch.from_numpy(gu).double()
    ref = (torch.nn.functional.silu(t[:, :688]) * t[:, 688:]).numpy()
    assert np.allclose(y, ref, rtol=2 ** -7, atol=1e-30)
    assert y.shape == (3, 688)


# ----------------------------------------------------------------- RoPE ----
def test_rope_table_is_complex_exponential():
    cos, sin = ops.rope_table(1e6, 128, 300)
    i = np.arange(64)
    z = np.exp(1j * np.outer(np.arange(300), np.power(1e6, -i / 64.0)))
    assert np.allclose(cos, z.real, atol=1e-6) and np.allclose(sin, z.imag, atol=1e-6)


def test_rope_rotation_properties():
    g = np.random.default_rng(6)
    cos, sin = ops.rope_table(1e4, 64, 600)
    q, k = randn(g, 1, 1, 64), randn(g, 1, 1, 64)
    # position 0 is the identity
    assert np.array_equal(ops.rope(q, np.array([0]), cos, sin), q)
    # pair (i, i+32) rotates as the complex number x_i + j x_{i+32}
    p = 37
    zq = (q[0, 0, :32] + 1j * q[0, 0, 32:]) * np.exp(1j * p * np.power(1e4, -np.arange(32) / 32.0))
    r = ops.rope(q, np.array([p]), cos, sin)[0, 0]
    assert np.allclose(r[:32], zq.real, atol=2e-2) and np.allclose(r[32:], zq.imag, atol=2e-2)
    # scores depend on the relative position only
    d1 = np.dot(ops.rope(q, np.array([500]), cos, sin).ravel(), ops.rope(k, np.array([490]), cos, sin).ravel())
    d2 = np.dot(ops.rope(q, np.array([12]), cos, sin).ravel(), ops.rope(k, np.array([2]), cos, sin).ravel())
    assert abs(d1 - d2) < 0.05 * (np.abs(q).sum() * np.abs(k).max())


def test_qk_norm_rope_is_head_norm_then_rotation():
    g = np.random.default_rng(12)
    T, H, D = 7, 3, 64
    x = randn(g, T, H, D, std=3.0)
    pos = g.integers(0, 500, size=T)
    cos, sin = ops.rope_table(1e4, D, 512)
    # no norm weight: RoPE alone
    assert np.array_equal(ops.qk_norm_rope(x, pos, None, 1e-6, cos, sin), ops.rope(x, pos, cos, sin))
    one = np.ones(D, F32)
    # at position 0 the rotation is the identity: each head normalised on its own
    y0 = ops.qk_norm_rope(x, np.zeros(T, np.int64), one, 1e-6, cos, sin).astype(np.float64)
    x64 = x.astype(np.float64)
    n = x64 / np.sqrt(np.mean(x64 * x64, axis=-1, keepdims=True) + 1e-6)
    assert np.all(np.abs(y0 - n) <= 2 ** -8 * np.abs(n) + 1e-30)
    # elsewhere the rotation keeps each head's RMS at 1 (a dropped sin or cos
    # term would not)
    y = ops.qk_norm_rope(x, pos, one, 1e-6, cos, sin).astype(np.float64)
    assert np.all(np.abs(np.sqrt(np.mean(y * y, axis=-1)) - 1.0) < 1e-2)


def test_kv_roundtrip_within_e4m3_half_spacing():
    """Per (token, head): s = amax / 448, x -> bf16(e4m3(x / s) * s).  e4m3
    keeps 3 mantissa bits, so the code is off by at most 2^-4 of the value
    (normal codes) or 2^-10 * s (subnormal codes), and the bf16 rounding adds
    at most 2^-8 of the result; more is a slip.  The amax element maps to code
    448 and comes back to the bf16 rounding, and an all-zero row stays zero."""
    g = np.random.default_rng(13)
    T, H, D = 40, 4, 128
    mag = np.power(10.0, g.uniform(-3, 3, size=(T, H, 1)))
    x = (g.standard_normal((T, H, D)) * mag).astype(F32)
    x[3, 2] = 0.0
    rt = ops.kv_roundtrip(x).astype(np.float64)
    x64 = x.astype(np.float64)
    s = np.max(np.abs(x64), axis=-1, keepdims=True) / 448.0
    e8 = np.maximum(np.abs(x64) * 2 ** -4, s * 2 ** -10)
    bound = (e8 + 2 ** -8 * (np.abs(x64) + e8)) * (1 + 1e-5)
    assert np.all(np.abs(rt - x64) <= bound)
    am = np.argmax(np.abs(x64), axis=-1)[..., None]
    ta, ra = np.take_along_axis(x64, am, -1), np.take_along_axis(rt, am, -1)
    nz = ta != 0
    assert np.all(np.abs(ra - ta)[nz] <= 2 ** -8 * (1 + 1e-5) * np.abs(ta)[nz])
    assert np.all(rt[3, 2] == 0.0)
    # finer than that: a random row is not returned unchanged
    assert not np.array_equal(rt, x64)


# ------------------------------------------------------------ attention ----
def test_attention_against_torch_sdpa_causal_gqa():
    g = np.random.default_rng(7)
    T, Hq, Hkv, D = 37, 4, 2, 64
    q, k, v = randn(g, T, Hq, D), randn(g, T, Hkv, D), randn(g, T, Hkv, D)
    pos = np.arange(T)
    scale = 1 / math.sqrt(D)
    o = ops.attention(q, k, v, pos, pos, scale)
    tq = torch.from_numpy(q).double().permute(1, 0, 2)
    tk = torch.from_numpy(k).double().permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
    tv = torch.from_numpy(v).double().permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=scale)
    assert np.allclose(o, ref.permute(1, 0, 2).numpy(), rtol=2 ** -7, atol=1e-3)


def test_attention_special_cases():
    g = np.random.default_rng(8)
    D = 64
    k, v = randn(g, 5, 1, D), randn(g, 5, 1, D)
    q = randn(g, 5, 2, D)
    # the first query sees only key 0: o = v0 exactly
    o = ops.attention(q, k, v, np.arange(5), np.arange(5), 0.125)
    assert np.array_equal(o[0, 0], v[0, 0]) and np.array_equal(o[0, 1], v[0, 0])
    # identical keys -> the mean of the visible values
    ke = np.repeat(k[:1], 5, axis=0)
    o = ops.attention(q, ke, v, np.arange(5), np.arange(5), 0.125)
    assert np.allclose(o[4, 0], bf(v[:, 0].mean(0)), rtol=2 ** -7, atol=1e-6)


def test_sparse_attention_with_all_positions_is_causal():
    g = np.random.default_rng(9)
    T, D = 20, 64
    q, k, v = randn(g, T, 4, D), randn(g, T, 1, D), randn(g, T, 1, D)
    idx = np.tile(np.arange(32, dtype=np.int32) - 0, (T, 1))
    idx[idx >= T] = -1
    ref = ops.attention(q, k, v, np.arange(T), np.arange(T), 0.125)
    assert np.array_equal(ops.sparse_attention(q, k, v, idx, np.arange(T), 0.125), ref)


# ---------------------------------------------------------------- Top-K ----
def _brute_topk(row, nv, k):
    items = [(-float(row[i]), i) for i in range(nv) if row[i] != -np.inf]
    items.sort()
    chosen = sorted(i for _, i in items[:k])
    return chosen + [-1] * (k - len(chosen))


def test_topk_positions_brute_force_with_ties():
    g = np.random.default_rng(10)
    for n, k in [(10, 3), (17, 17), (8, 12), (64, 5), (33, 32)]:
        s = g.integers(0, 3, size=(12, n)).astype(F32)
        s[3, :] = -np.inf
        s[4, ::2] = -np.inf
        s[5, 1] = -0.0
        nv = g.integers(0, n + 1, size=12)
        nv[0] = n
        got = ops.topk_positions(s, nv, k)
        for r in range(12):
            assert got[r].tolist() == _brute_topk(s[r], nv[r], k), (n, k, r)


def test_topk_positions_brute_force_extreme_values():
    """The oracle's selection on +inf, +-max normals, denormals, signed zeros
    and adjacent floats equals a plain sort by (score desc, position asc)."""
    g = np.random.default_rng(12)
    n, k = 200, 37
    rows = [np.float32(3.4e38) * np.sign(g.standard_normal(n)).astype(F32),
            (np.float32(1e-40) * g.integers(-3, 4, n)).astype(F32),
            (np.float32(1.0) + np.float32(2.0 ** -23) * g.integers(0, 9, n)).astype(F32),
            np.ldexp(np.float32(1.0), g.integers(-126, 127, n)).astype(F32),
            np.where(g.random(n) < 0.5, F32(0.0), F32(-0.0)).astype(F32)]
    rows[0][::7] = np.inf
    s = np.stack(rows)
    nv = np.array([n, n, 150, n, n])
    got = ops.topk_positions(s, nv, k)
    for r in range(s.shape[0]):
        assert got[r].tolist() == _brute_topk(s[r], nv[r], k), r


def test_router_brute_force_and_softmax_weights():
    g = np.random.default_rng(11)
    z = g.integers(-2, 3, size=(16, 64)).astype(F32) * F32(0.5)
    idx, w = ops.router_topk(z, 6)
    for r in range(16):
        order = sorted(range(64), key=lambda e: (-float(z[r, e]), e))[:6]
        assert idx[r].tolist() == order
    p = torch.softmax(torch.from_numpy(z).double(), dim=1).numpy()
    assert np.allclose(w, np.take_along_axis(p, idx.astype(np.int64), 1), rtol=1e-6)


# ------------------------------------------------------------------ FP8 ----
def test_fp8_block_gemm_exact_on_integers_with_pow2_scales():
    g = np.random.default_rng(12)
    M, N, K = 5, 200, 300
    a = g.integers(-8, 9, size=(M, K)).astype(F32)
    b = g.integers(-8, 9, size=(N, K)).astype(F32)
    ac, bc = f32_to_e4m3(a), f32_to_e4m3(b)
    assert np.array_equal(e4m3_to_f32(ac), a)
    kb, nb = 3, 2
    sa = np.exp2(g.integers(-3, 3, size=(M, kb))).astype(F32)
    sb = np.exp2(g.integers(-3, 3, size=(nb, kb))).astype(F32)
    ref = np.zeros((M, N))
    for j in range(kb):
        ks = slice(128 * j, min(K, 128 * j + 128))
        sbn = np.repeat(sb[:, j], 128)[:N]
        ref += sa[:, j:j + 1] * sbn[None, :] * (a[:, ks].astype(np.float64) @ b[:, ks].T)
    assert np.array_equal(ops.gemm_fp8_block(ac, sa, bc, sb, out="f32"), ref.astype(F32))


def test_act_quant_groups():
    g = np.random.default_rng(13)
    x = randn(g, 3, 300)
    x[1, 128:256] = 0
    c, s = ops.act_quant_fp8(x)
    assert c.shape == (3, 300) and s.shape == (3, 3)
    assert s[1, 1] == 1.0 and np.all(c[1, 128:256] == 0)
    for j in range(3):
        blk = x[:, 128 * j:128 * j + 128]
        assert np.array_equal(s[:, j], np.where(np.abs(blk).max(1) == 0, 1, np.abs(blk).max(1) / F32(448)).astype(F32))
    deq = e4m3_to_f32(c) * np.repeat(s, 128, axis=1)[:, :300]
    assert np.allclose(deq, x, rtol=2 ** -3, atol=1e-30)


def test_moe_combine_one_hot_and_order():
    g = np.random.default_rng(14)
    y = randn(g, 4, 6, 32)
    w = np.zeros((4, 6), F32)
    w[np.arange(4), [0, 5, 2, 3]] = 1
    assert np.array_equal(ops.moe_combine(y, w), y[np.arange(4), [0, 5, 2, 3]])
    sh = randn(g, 4, 32)
    w2 = np.full((4, 6), 0.25, F32)
    ref = bf(np.float64(0.25) * y.astype(np.float64).sum(1) + sh)
    assert np.allclose(ops.moe_combine(y, w2, sh), ref, rtol=2 ** -7, atol=1e-6)


def test_moe_combine_fixed_fp32_order():
    """The merge is one FP32 accumulator over slots 0..k-1 in order, the shared
    expert added last.  a = 1 + 2^-8 is the midpoint between two bf16 values
    and t = 3 * 2^-26 is three quarters of half an FP32 ulp of a: added to a
    one at a time, each t is lost and the sum stays on the midpoint (bf16
    rounds it to even, 1.0); two t added together first (1.5 half-ulps) push
    the sum past it (bf16 1.0078125).  So any other order shows in the bits."""
    a, t = F32(1 + 2 ** -8), F32(3 * 2 ** -26)
    one = np.ones((1, 3), F32)
    y = np.zeros((1, 3, 4), F32)
    y[0, :, 0] = [a, t, t]            # in slot order: a, then each t lost
    assert ops.moe_combine(y, one)[0, 0] == F32(1.0)
    assert ops.moe_combine(y[:, ::-1], one)[0, 0] == F32(1.0078125)   # the reverse order differs
    y2 = np.zeros((1, 2, 4), F32)
    y2[0, :, 0] = [t, a]              # slots t, a, then the shared expert t
    sh = np.zeros((1, 4), F32)
    sh[0, 0] = t
    assert ops.moe_combine(y2, one[:, :2], sh)[0, 0] == F32(1.0)


# ---------------------------------------------------------- log-softmax ----
def test_log_softmax_normalised_and_against_torch():
    g = np.random.default_rng(15)
    z = (g.standard_normal((6, 4096)) * 3).astype(F32)
    lp = ops.log_softmax(z)
    assert np.allclose(np.exp(lp.astype(np.float64)).sum(1), 1.0, atol=1e-5)
    ref = torch.log_softmax(torch.from_numpy(z).double(), dim=1).numpy()
    assert np.allclose(lp, ref, atol=1e-5)
    tgt = g.integers(0, 4096, size=6)
    assert np.allclose(ops.logprob(z, tgt), ref[np.arange(6), tgt], atol=1e-5)
    u = np.zeros((2, 151936), F32)
    assert np.allclose(ops.logprob(u, np.array([0, 5])), -math.log(151936), atol=1e-6)


def test_diff_stats_k3():
    a = np.array([-1.0, -2.0, -0.5], F32)
    assert ops.diff_stats(a, a) == {"max": 0.0, "mean": 0.0, "std": 0.0, "k3": 0.0}
    st = ops.diff_stats(a, a + F32(0.1))
    assert st["max"] > 0 and st["k3"] > 0


# ------------------------------------------------------------------ SSD ----
def _ssd_inputs(g, T, H=3, P=4, N=5):
    x = g.standard_normal((T, H, P))
    dt = np.log1p(np.exp(g.standard_normal((T, H)) - 1))
    A = -g.uniform(0.5, 4, size=H)
    B = g.standard_normal((T, N))
    C = g.standard_normal((T, N))
    D = g.standard_normal(H)
    return x, dt, A, B, C, D


def test_ssd_chunked_equals_sequential_fp64():
    g = np.random.default_rng(16)
    x, dt, A, B, C, D = _ssd_inputs(g, 75)
    y0, h0 = ssd_sequential(x, dt, A, B, C, D, dtype=np.float64, round_out=False)
    for Q, start in [(16, 0), (8, 5), (64, 0), (256, 200)]:
        y1, h1 = ssd_chunked(x, dt, A, B, C, D, Q, start_pos=start)
        assert np.allclose(y1, y0, rtol=1e-9, atol=1e-9) and np.allclose(h1, h0, rtol=1e-9, atol=1e-9)


def test_ssd_zero_decay_is_causal_linear_attention():
    g = np.random.default_rng(17)
    x, dt, A, B, C, D = _ssd_inputs(g, 30)
    A = np.zeros_like(A)
    dt = np.ones_like(dt)
    y, _ = ssd_sequential(x, dt, A, B, C, D, dtype=np.float64, round_out=False)
    CB = np.tril(C @ B.T)                                # [t, s], s <= t
    ref = np.einsum("ts,shp->thp", CB, x) + D[None, :, None] * x
    assert np.allclose(y, ref, rtol=1e-10, atol=1e-10)


def test_ssd_state_carry_and_fp32():
    g = np.random.default_rng(18)
    x, dt, A, B, C, D = _ssd_inputs(g, 40)
    y, h = ssd_sequential(x, dt, A, B, C, D, dtype=np.float64, round_out=False)
    ya, ha = ssd_sequential(x[:23], dt[:23], A, B[:23], C[:23], D, dtype=np.float64, round_out=False)
    yb, hb = ssd_sequential(x[23:], dt[23:], A, B[23:], C[23:], D, h0=ha, dtype=np.float64, round_out=False)
    assert np.allclose(np.concatenate([ya, yb]), y) and np.allclose(hb, h)
    y32, _ = ssd_sequential(x, dt, A, B, C, D, dtype=np.float32, round_out=False)
    assert np.allclose(y32, y, rtol=1e-4, atol=1e-4)
