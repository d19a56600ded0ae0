"""Pins for the Mamba-2 mixer, the hybrid stack and the NVFP4 codec of the
oracle (CPU only), against what the format definitions and the mathematics
fix: the e2m1 value table, softplus as log(1 + e^x), causal convolution
against numpy's full convolution, the gated norm's closed forms, and the
stack's decode equal to its prefill on the oracle's own recurrence ("Finish
RL Training Faster", section "一致性有多个层面": decode replays prefill)."""
import numpy as np
import pytest

import synth
from oracle import mamba, ops
from oracle.codecs import bf16_round, e2m1_to_f32, e4m3_to_f32, nvfp4_dequant

F32 = np.float32


def test_e2m1_table_is_the_ocp_fp4_grid():
    # sign bit 3, exponent bits 2-1 (bias 1), mantissa bit 0: the published
    # E2M1 values are +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    v = e2m1_to_f32(np.arange(16, dtype=np.uint8))
    assert v[:8].tolist() == grid
    assert v[8:].tolist() == [-x for x in grid]
    assert np.signbit(v[8])                       # code 8 is -0


def _pack(codes):
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def test_nvfp4_dequant_blocks_packing_and_bf16_exactness():
    g = np.random.default_rng(0)
    codes = g.integers(0, 16, size=(5, 48)).astype(np.uint8)
    sc = g.integers(0, 0x7F, size=(5, 3)).astype(np.uint8)
    w = nvfp4_dequant(_pack(codes), sc)
    assert np.array_equal(bf16_round(w), w)        # on the bf16 grid
    # element (n, k) uses its own code and the scale of its block of 16 along k
    for n in range(5):
        for k in range(48):
            assert w[n, k] == F32(e2m1_to_f32(codes[n, k]) * e4m3_to_f32(sc[n, k // 16]))
    # one-hot codes fix the block index and the nibble order: value 1.0
    # (code 2) at k = 17 (high nibble of byte 8) picks scale 1
    c1 = np.zeros((1, 48), np.uint8)
    c1[0, 17] = 2
    assert _pack(c1)[0, 8] == 0x20
    s1 = np.array([[0x38, 0x40, 0x48]], np.uint8)   # 1.0, 2.0, 4.0
    d1 = nvfp4_dequant(_pack(c1), s1)
    assert d1[0, 17] == 2.0 and np.count_nonzero(d1) == 1


def test_softplus_against_logaddexp():
    x = np.concatenate([np.linspace(-30, 30, 2001), [-88.0, 19.99, 20.0, 20.01, 50.0]]).astype(F32)
    ref = np.logaddexp(0.0, x.astype(np.float64))
    got = mamba.softplus(x)
    assert np.all(np.abs(got - ref) <= 4 * np.spacing(np.abs(ref).astype(F32)) + 1e-30)


def test_conv1d_causal_against_numpy_convolve():
    g = np.random.default_rng(1)
    T, Ch = 37, 9
    x = bf16_round(g.standard_normal((T, Ch)).astype(F32))
    w = bf16_round(g.standard_normal((Ch, 4)).astype(F32))
    b = bf16_round(g.standard_normal(Ch).astype(F32))
    got, st = mamba.conv1d_causal_silu(x, w, b)
    for c in range(Ch):
        # out[t] = b + sum_j w[j] x[t-3+j]: numpy's convolve flips its kernel
        lin = np.convolve(x[:, c].astype(np.float64), w[c, ::-1].astype(np.float64))[:T] + b[c]
        ref = lin / (1.0 + np.exp(-lin))
        assert np.allclose(got[:, c], ref, rtol=2 ** -7, atol=1e-6), c
    assert np.array_equal(st, x[-3:])


def test_conv1d_state_carries_across_calls_bitwise():
    g = np.random.default_rng(2)
    x = bf16_round(g.standard_normal((50, 6)).astype(F32))
    w = bf16_round(g.standard_normal((6, 4)).astype(F32))
    b = bf16_round(g.standard_normal(6).astype(F32))
    whole, _ = mamba.conv1d_causal_silu(x, w, b)
    parts, st = [], None
    for a, e in [(0, 1), (1, 2), (2, 20), (20, 21), (21, 50)]:
        o, st = mamba.conv1d_causal_silu(x[a:e], w, b, st)
        parts.append(o)
    assert np.array_equal(np.concatenate(parts), whole)


def test_conv1d_planted_kernel_flip_is_caught():
    g = np.random.default_rng(3)
    x = bf16_round(g.standard_normal((20, 4)).astype(F32))
    w = bf16_round(g.standard_normal((4, 4)).astype(F32))
    b = np.zeros(4, F32)
    good, _ = mamba.conv1d_causal_silu(x, w, b)
    bad, _ = mamba.conv1d_causal_silu(x, w[:, ::-1].copy(), b)
    lin = np.convolve(x[:, 0].astype(np.float64), w[0, ::-1].astype(np.float64))[:20]
    ref = lin / (1 + np.exp(-lin))
    assert np.allclose(good[:, 0], ref, rtol=2 ** -7, atol=1e-6)
    assert not np.allclose(bad[:, 0], ref, rtol=2 ** -7, atol=1e-6)


def test_gated_rmsnorm_closed_forms():
    g = np.random.default_rng(4)
    w = bf16_round((1 + 0.1 * g.standard_normal(64)).astype(F32))
    # silu(30) = 30 in FP32, so g = 30 c: a constant vector normalises to sign(c) w
    for c in (2.5, -0.75):
        y = mamba.gated_rmsnorm(np.full((1, 64), c, F32), np.full((1, 64), 30.0, F32), w, 1e-6)
        assert np.allclose(y[0], np.sign(c) * w, rtol=2 ** -7)
    # a zero gate gives exactly zero
    y0 = mamba.gated_rmsnorm(g.standard_normal((2, 64)).astype(F32), np.zeros((2, 64), F32), w, 1e-6)
    assert np.array_equal(y0, np.zeros_like(y0))
    # the gate multiplies before the norm: scaling y by 4 changes nothing
    y = bf16_round(g.standard_normal((3, 64)).astype(F32))
    z = bf16_round(g.standard_normal((3, 64)).astype(F32))
    assert np.allclose(mamba.gated_rmsnorm(4 * y, z, w, 1e-6), mamba.gated_rmsnorm(y, z, w, 1e-6),
                       rtol=2 ** -7, atol=1e-6)


def _tiny():
    cfg = synth.HYBRID_TINY
    W = synth.hybrid_weights(cfg, seed=0, random_gains=True, lm_scale=8.0)
    return cfg, mamba.HybridOracle(cfg, mamba.decode_hybrid_weights(synth.host_payload(W)), max_pos=512)


def test_hybrid_decode_and_chunked_prefill_equal_prefill():
    cfg, orc = _tiny()
    s = synth.hybrid_sequences(cfg, n=1, lo=40, hi=40, seed=3, prompt_frac=0.6)[0]
    full = orc.prefill_logprobs(s.tokens)
    assert np.array_equal(orc.decode_logprobs(s.tokens, s.prompt_len), full)
    assert np.array_equal(orc.decode_logprobs(s.tokens, s.prompt_len, chunk=7), full)
    z = orc.forward_rows(s.tokens[:-1], np.arange(s.length - 1), orc.new_state())
    lp = ops.log_softmax(z)
    assert np.allclose(np.exp(lp.astype(np.float64)).sum(1), 1.0, atol=1e-4)
    assert np.std(full) > 0.5                      # the x8 head is peaked


def test_hybrid_state_shapes_after_a_call():
    cfg, orc = _tiny()
    st = orc.new_state()
    toks = np.arange(10) % cfg.vocab
    orc.forward_rows(toks, np.arange(10), st)
    for kind, s_ in zip(cfg.pattern, st):
        if kind == "M":
            assert s_["conv"].shape == (3, cfg.conv_channels)
            assert s_["ssd"].shape == (cfg.ssd_heads, cfg.ssd_head_dim, cfg.state)
        else:
            assert s_["k"].shape == (10, cfg.kv_heads, cfg.head_dim)
