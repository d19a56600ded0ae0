"""Pins for the oracle's MoE block and its FP8 expert MLP (CPU only).

What the mathematics fixes, checked without retyping the oracle:

* a per-token restatement -- each token's selected experts recomputed one
  token at a time and merged in slot order by a plain loop -- equals the
  batched block bit for bit (catches a row/slot mix-up in the scatter);
* an FP8 expert lies within the RMS error that e4m3 activation rounding
  leaves of the same MLP in float64 on the dequantised weights with
  unquantised activations (catches gate/up swapped, a wrong SiLU, a
  transposed or misindexed block scale, a mis-weighted shared expert);
* the two activation quantisation points have closed-form consequences:
  an input whose 128-groups each hold one large element over a zero weight
  column and otherwise values below half the smallest e4m3 step gives an
  expert output of exactly 0, and so does the same construction one GEMM
  later, so skipping either quantisation (or moving it) is caught;
* mistakes planted in copies of the block on the CPU -- slots swapped, the
  shared expert weighted, gate and up exchanged -- fail these pins.

Sources: "Finish RL Training Faster: Bitwise-Consistent, High-Performance,
Agent-Driven", section "让训练前向使用推理的数值" (MoE with unified
quantisation rounding and per-row computation; expert outputs merged in FP32
in fixed slot order).
"""
import numpy as np
import pytest

import oracle.model as om
from oracle import ops
from oracle.codecs import bf16_round, e4m3_to_f32, f32_to_e4m3

F32 = np.float32


def _codes(g, shape):
    return f32_to_e4m3(np.clip(g.standard_normal(shape) * 64.0, -448, 448).astype(F32))


def _scales(g, n, k):
    nb, kb = (n + 127) // 128, (k + 127) // 128
    return (F32(0.02 / 64) * np.exp2(g.uniform(-1, 1, size=(nb, kb)))).astype(F32)


def _expert(g, d, I):
    return (_codes(g, (2 * I, d)), _scales(g, 2 * I, d), _codes(g, (d, I)), _scales(g, d, I))


def _block_inputs(seed, T=16, E=8, d=256, I=256):
    g = np.random.default_rng(seed)
    h = bf16_round(g.standard_normal((T, d)).astype(F32))
    wr = bf16_round((g.standard_normal((E, d)) * 0.05).astype(F32))
    experts = [_expert(g, d, I) for _ in range(E)]
    shared = _expert(g, d, I)
    return h, wr, experts, shared


def _deq(codes, scales):
    n, k = codes.shape
    s = np.repeat(np.repeat(np.asarray(scales, np.float64), 128, 0), 128, 1)[:n, :k]
    return e4m3_to_f32(codes).astype(np.float64) * s


def _dense_expert(x, wgu_c, sgu, wd_c, sd):
    """The expert MLP in float64 on dequantised weights and unquantised
    activations: silu(gate) * up, then the down projection."""
    x = np.asarray(x, np.float64)
    Wgu, Wd = _deq(wgu_c, sgu), _deq(wd_c, sd)
    I = Wgu.shape[0] // 2
    gu = x @ Wgu.T
    g, u = gu[:, :I], gu[:, I:]
    return (g / (1.0 + np.exp(-g)) * u) @ Wd.T


# e4m3 keeps 3 mantissa bits: rounding to nearest leaves a relative error
# uniform within +-2^-4 of a value placed uniformly in its binade, RMS about
# 2^-4 / sqrt(3) = 0.036.  Two activation quantisations in a row compound to
# about 0.05 (the bf16 roundings add 2^-9-sized terms).  A correct expert sits
# near that; the mistakes the pins guard against (gate and up exchanged, the
# SiLU replaced, a block scale misindexed, the shared expert mis-weighted)
# land at 0.3 and above.
REL_RMS = 0.12


def _rel_rms(got, ref):
    ref = np.asarray(ref, np.float64)
    return float(np.sqrt(np.mean((np.asarray(got, np.float64) - ref) ** 2) / np.mean(ref ** 2)))


def _per_token_moe(h, wr, experts, shared, k, idx, w):
    """Token by token: each selected expert recomputed on this row alone, then
    a plain FP32 loop over the slots in order, the shared expert last."""
    T, d = h.shape
    out = np.zeros((T, d), F32)
    for t in range(T):
        acc = np.zeros(d, F32)
        for s in range(k):
            ys = om.expert_mlp_fp8(h[t:t + 1], *experts[int(idx[t, s])])[0]
            acc = (acc + F32(w[t, s]) * ys).astype(F32)
        acc = (acc + om.expert_mlp_fp8(h[t:t + 1], *shared)[0]).astype(F32)
        out[t] = bf16_round(acc)
    return out


def _dense_moe(h, experts, shared, k, idx, w):
    T, d = h.shape
    ref = np.zeros((T, d))
    for t in range(T):
        for s in range(k):
            ref[t] += float(w[t, s]) * _dense_expert(h[t:t + 1], *experts[int(idx[t, s])])[0]
        ref[t] += _dense_expert(h[t:t + 1], *shared)[0]
    return ref


def _pins_hold(block_fn, seed=0, k=3):
    h, wr, experts, shared = _block_inputs(seed)
    out, idx, w = block_fn(h, wr, experts, shared, k)
    tok = _per_token_moe(h, wr, experts, shared, k, idx, w)
    ref = _dense_moe(h, experts, shared, k, idx, w)
    return np.array_equal(out, tok), _rel_rms(out, ref) <= REL_RMS


# ------------------------------------------------------------------ pins ----
def test_expert_near_float64_within_e4m3_rounding():
    g = np.random.default_rng(1)
    for d, I in [(256, 256), (384, 200)]:
        x = bf16_round(g.standard_normal((5, d)).astype(F32))
        ex = _expert(g, d, I)
        got = om.expert_mlp_fp8(x, *ex)
        assert _rel_rms(got, _dense_expert(x, *ex)) <= REL_RMS


def test_first_activation_quantisation_point_zeroes_sub_step_values():
    """Each 128-group of the input: one element 448 over a zero gate_up
    column; the rest below half the smallest e4m3 step of that group's scale
    (scale 1: step 2^-9), so they quantise to 0.  gate_up is then exactly 0,
    and so is everything after it."""
    g = np.random.default_rng(2)
    d, I = 256, 256
    wgu_c, sgu, wd_c, sd = _expert(g, d, I)
    x = (g.choice([-1, 1], size=(3, d)) * 2.0 ** -11).astype(F32)
    big = [5, 128 + 77]
    x[:, big] = 448.0
    wgu_c[:, big] = 0
    got = om.expert_mlp_fp8(bf16_round(x), wgu_c, sgu, wd_c, sd)
    assert np.array_equal(got, np.zeros_like(got))
    # without the quantisation the small values would have contributed
    assert np.max(np.abs(_dense_expert(x, wgu_c, sgu, wd_c, sd))) > 0


def test_second_activation_quantisation_point_zeroes_sub_step_values():
    """A one-hot input (exactly representable) makes gate_up a copy of one
    weight column.  Gate and up are chosen so that each 128-group of the
    activation holds one large value over a zero down-projection column and
    otherwise values far below half the group's smallest e4m3 step: the down
    projection then sees only zeros and returns exactly 0."""
    d, I, k0 = 256, 256, 17
    x = np.zeros((1, d), F32)
    x[0, k0] = 448.0
    gate = np.full(I, 2.0 ** -9, F32)
    up = np.full(I, 2.0 ** -9, F32)
    big = [3, 128 + 40]
    gate[big] = 448.0
    up[big] = 1.0
    wgu = np.zeros((2 * I, d), F32)
    wgu[:I, k0] = gate
    wgu[I:, k0] = up
    sgu = np.full((2 * I // 128, d // 128), 2.0 ** -10, F32)
    g = np.random.default_rng(3)
    wd_c = _codes(g, (d, I))
    wd_c[:, big] = 0
    sd = np.full((d // 128, I // 128), 2.0 ** -10, F32)
    got = om.expert_mlp_fp8(x, f32_to_e4m3(wgu), sgu, wd_c, sd)
    assert np.array_equal(got, np.zeros_like(got))
    assert np.max(np.abs(_dense_expert(x, f32_to_e4m3(wgu), sgu, wd_c, sd))) > 0


def test_moe_block_equals_per_token_restatement_and_near_float64():
    for seed in (0, 1):
        same, within = _pins_hold(om.moe_block, seed=seed)
        assert same and within


def test_moe_block_shapes_routing_and_empty_experts():
    h, wr, experts, shared = _block_inputs(4, T=5, E=8)
    out, idx, w = om.moe_block(h, wr, experts, shared, 2)
    assert out.shape == h.shape and idx.shape == (5, 2) and w.shape == (5, 2)
    ri, rw = ops.router_topk(ops.gemm(h, wr, out="f32"), 2)
    assert np.array_equal(idx, ri) and np.array_equal(w, rw)
    # with five tokens and two slots, some of the eight experts get no rows
    assert len(set(idx.ravel().tolist())) < 8


# ------------------------------------------------------ planted mistakes ----
def _moe_slots_rotated(h, router_w, experts, shared, top_k):
    logits = ops.gemm(h, router_w, out="f32")
    idx, w = ops.router_topk(logits, top_k)
    T, d = h.shape
    y = np.zeros((T, top_k, d), F32)
    for e in range(len(experts)):
        rows, slots = np.nonzero(idx == e)
        if rows.size:
            y[rows, (slots + 1) % top_k] = om.expert_mlp_fp8(h[rows], *experts[e])
    sh = om.expert_mlp_fp8(h, *shared)
    return ops.moe_combine(y, w, sh), idx, w


def _moe_shared_weighted(h, router_w, experts, shared, top_k):
    logits = ops.gemm(h, router_w, out="f32")
    idx, w = ops.router_topk(logits, top_k)
    T, d = h.shape
    y = np.zeros((T, top_k, d), F32)
    for e in range(len(experts)):
        rows, slots = np.nonzero(idx == e)
        if rows.size:
            y[rows, slots] = om.expert_mlp_fp8(h[rows], *experts[e])
    sh = om.expert_mlp_fp8(h, *shared)
    return ops.moe_combine(y, w, w[:, :1] * sh), idx, w


@pytest.mark.parametrize("bad", [_moe_slots_rotated, _moe_shared_weighted])
def test_planted_block_mistakes_are_caught(bad):
    same, within = _pins_hold(bad)
    assert not (same and within)


def test_planted_gate_up_swap_is_caught(monkeypatch):
    real = om.expert_mlp_fp8

    def swapped(x, wgu_codes, wgu_scale, wd_codes, wd_scale):
        I = wgu_codes.shape[0] // 2
        return real(x, np.concatenate([wgu_codes[I:], wgu_codes[:I]]),
                    np.concatenate([wgu_scale[wgu_scale.shape[0] // 2:], wgu_scale[:wgu_scale.shape[0] // 2]]),
                    wd_codes, wd_scale)

    monkeypatch.setattr(om, "expert_mlp_fp8", swapped)
    h, wr, experts, shared = _block_inputs(0)
    out, idx, w = om.moe_block(h, wr, experts, shared, 3)
    ref = _dense_moe(h, experts, shared, 3, idx, w)      # the float64 side is not patched
    assert _rel_rms(out, ref) > REL_RMS


def test_planted_skipped_activation_quantisation_is_caught(monkeypatch):
    """An expert that skips its first activation quantisation (codes = the
    bf16 input itself) no longer returns 0 on the sub-step construction."""
    real_q = ops.act_quant_fp8
    calls = []

    def first_call_identity(x, group=128):
        calls.append(1)
        if len(calls) == 1:
            x = np.asarray(x, F32)
            G = (x.shape[1] + 127) // 128
            return x, np.ones((x.shape[0], G), F32)
        return real_q(x, group)

    monkeypatch.setattr(ops, "act_quant_fp8", first_call_identity)
    # the planted "codes" are plain values: decode them as themselves
    monkeypatch.setattr(ops, "e4m3_to_f32", lambda c: e4m3_to_f32(c) if c.dtype == np.uint8
                        else np.asarray(c, F32))
    g = np.random.default_rng(2)
    d, I = 256, 256
    wgu_c, sgu, wd_c, sd = _expert(g, d, I)
    x = (g.choice([-1, 1], size=(3, d)) * 2.0 ** -11).astype(F32)
    x[:, [5, 128 + 77]] = 448.0
    wgu_c[:, [5, 128 + 77]] = 0
    got = om.expert_mlp_fp8(bf16_round(x), wgu_c, sgu, wd_c, sd)
    assert np.max(np.abs(got)) > 0
