"""Model-level invariance and oracle parity of the dense decoder.

Invariance (every statistic of the logprob diff, max/mean/std and k3, must be
exactly 0): batch 1 vs batch 8, whole prefill vs chunked prefill, rollout
(prompt prefill + token-by-token decode) vs trainer recompute (private cache),
eager vs CUDA-Graph decode, graph replay after an in-place weight update vs
eager at the new weights.

Parity, free-running (each side feeds its own outputs forward):
|lp_gpu - lp_oracle| <= max(2e-2, envelope), where the envelope is how far
correct FP32 evaluation orders of the oracle itself drift from its default
on the same case (ascending, descending, round-toward-zero and blocked
library orders against float64-then-rounded dot products), widened by the
variability of that maximum among the orders; the measurements are stored in
tests/golden/accumulation_spread.json by the script beside it.  Where bf16
rounding flips are amplified (a x10 LM head, 28 layers of QK-norm attention,
FP8 KV codes) the envelope exceeds 2e-2, and no implementation that does not
reproduce the oracle's exact roundings can promise less.
"""
import json
import os

import numpy as np
import pytest
import torch

import synth
from oracle import ops
from oracle.model import DenseOracle, decode_weights

pytestmark = pytest.mark.gpu
TOL_LP = 2e-2
ZERO = {"max": 0.0, "mean": 0.0, "std": 0.0, "k3": 0.0}
with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                       "accumulation_spread.json")) as _f:
    SPREAD = json.load(_f)


def lp_bound(case):
    """2e-2, or, where larger, the envelope of correct FP32 evaluation orders
    of the oracle on this case widened by how much that statistic varies
    among them: the largest max |dlogprob| any order shows, times the ratio
    of the largest to the smallest order's maximum (a maximum over positions
    is heavy-tailed; the orders' own maxima differ by up to about 1.6x)."""
    m = [o["max"] for o in SPREAD[case]["orders"].values()]
    return max(TOL_LP, max(m) * max(m) / min(m))


def flat(lps):
    return np.concatenate([np.asarray(x, np.float32) for x in lps])


def stats(a, b):
    return ops.diff_stats(flat(a), flat(b))


def make(cfg, seed=0, lm_scale=10.0, max_rows=1024, max_pos=512, pages=256, max_seqs=32, mode=0):
    from invariant_forward_bitwise_gb300 import build
    from invariant_forward_bitwise_gb300.model import DenseModel, PagedKV
    build.build()
    W = synth.dense_weights(cfg, seed=seed, random_gains=True, lm_scale=lm_scale)
    m = DenseModel(cfg, W, max_rows=max_rows, max_pos=max_pos, mode=mode)
    kv = PagedKV(cfg, pages=pages, max_seqs=max_seqs, max_pages=(max_pos + 63) // 64)
    return W, m, kv


def oracle_for(cfg, W):
    return DenseOracle(cfg, decode_weights({k: synth.bf16_bits(v) for k, v in W.items()}))


@pytest.fixture(scope="module", params=[False, True], ids=["bf16kv", "fp8kv"])
def tiny(request):
    cfg = synth.replace(synth.TINY, kv_fp8=request.param)
    W, m, kv = make(cfg)
    seqs = synth.tiny_sequences(cfg, n=8, seed=1)
    return cfg, W, m, kv, seqs


@pytest.mark.parametrize("lm_scale", [1.0, 10.0], ids=["flat", "peaked"])
@pytest.mark.parametrize("kv_fp8", [False, True], ids=["bf16kv", "fp8kv"])
def test_recompute_matches_oracle(kv_fp8, lm_scale, capsys):
    """Free-running parity at the config's own initialisation (N(0, 0.02)),
    and with the x10 "peaked" LM head whose logprobs spread far from -log V
    (the variant that exercises log-softmax)."""
    from invariant_forward_bitwise_gb300.model import recompute
    cfg = synth.replace(synth.TINY, kv_fp8=kv_fp8)
    W, m, kv = make(cfg, lm_scale=lm_scale)
    seqs = synth.tiny_sequences(cfg, n=8, seed=1)
    got = recompute(m, kv, seqs, max_tokens=1024)
    orc = oracle_for(cfg, W)
    refs = [orc.prefill_logprobs(s.tokens)[s.prompt_len - 1:] for s in seqs]
    if lm_scale > 1.0:
        assert np.std(np.concatenate(refs)) > 1.0        # really peaked
        bound = lp_bound("tiny_peaked_fp8kv" if kv_fp8 else "tiny_peaked_bf16kv")
    else:
        bound = TOL_LP
    worst = max(float(np.max(np.abs(g - r))) for g, r in zip(got, refs))
    with capsys.disabled():
        print(f"\n[tiny lm x{lm_scale:g} kv_fp8={kv_fp8}] |dlp| max {worst:.4f} (bound {bound:.4f})")
    assert worst <= bound


def test_batch1_vs_batch8_and_chunked(tiny):
    from invariant_forward_bitwise_gb300.model import recompute
    cfg, W, m, kv, seqs = tiny
    full = recompute(m, kv, seqs, max_tokens=1024)
    alone = [recompute(m, kv, [s], max_tokens=1024)[0] for s in seqs]
    assert stats(full, alone) == ZERO
    chunked = recompute(m, kv, seqs, max_tokens=1024, chunk=16)
    assert stats(full, chunked) == ZERO
    small_steps = recompute(m, kv, seqs, max_tokens=37)          # ragged step boundaries
    assert stats(full, small_steps) == ZERO


def test_rollout_equals_recompute_eager_and_graph(tiny):
    from invariant_forward_bitwise_gb300.model import recompute, rollout
    cfg, W, m, kv, seqs = tiny
    rec = recompute(m, kv, seqs, max_tokens=1024)
    eager = rollout(m, kv, seqs, max_tokens=1024, use_graphs=False)
    assert stats(rec, eager) == ZERO
    graph = rollout(m, kv, seqs, max_tokens=1024, use_graphs=True)
    assert stats(rec, graph) == ZERO


def test_inplace_weight_update_under_graph():
    from invariant_forward_bitwise_gb300.model import DecodeGraphs, recompute, rollout
    cfg = synth.TINY
    W, m, kv = make(cfg, seed=3)
    seqs = synth.tiny_sequences(cfg, n=4, seed=2)
    dg = DecodeGraphs(m, kv, use_graphs=True)
    before = rollout(m, kv, seqs, max_tokens=1024, graphs=dg)
    # in-place update of every weight (same storages the graphs captured)
    W2 = synth.dense_weights(cfg, seed=4, random_gains=True, lm_scale=10.0)
    for k, v in m.W.items():
        v.copy_(W2[k].to(v.device))
    after = rollout(m, kv, seqs, max_tokens=1024, graphs=dg)       # replays old graphs
    rec2 = recompute(m, kv, seqs, max_tokens=1024)                  # eager at new weights
    assert stats(after, rec2) == ZERO
    assert stats(before, after)["max"] > 0
    # and the replayed graphs computed the model at the new weights
    orc = oracle_for(cfg, W2)
    for s, g in zip(seqs, after):
        ref = orc.prefill_logprobs(s.tokens)[s.prompt_len - 1:]
        assert np.max(np.abs(g - ref)) <= lp_bound("tiny_peaked_seed4")


def test_reload_then_first_step():
    """Weights and KV saved to host, reloaded into new allocations: the next
    decode step's logprobs equal those of the original objects."""
    from invariant_forward_bitwise_gb300.model import DenseModel, recompute
    cfg = synth.TINY
    W, m, kv = make(cfg, seed=5)
    seqs = synth.tiny_sequences(cfg, n=3, seed=6)
    a = recompute(m, kv, seqs, max_tokens=1024)
    host = {k: v.cpu().clone() for k, v in m.W.items()}
    m2 = DenseModel(cfg, host, max_rows=1024, max_pos=512)
    b = recompute(m2, kv, seqs, max_tokens=1024)
    assert stats(a, b) == ZERO


def test_qwen3_shape_two_layers_invariance_and_parity():
    from invariant_forward_bitwise_gb300.model import recompute, rollout
    cfg = synth.scaled_dense(synth.QWEN3_1P7B, 2)
    W, m, kv = make(cfg, lm_scale=1.0, max_rows=512, max_pos=256, pages=64, max_seqs=8)
    seqs = synth.tiny_sequences(cfg, n=3, lo=40, hi=70, seed=7)
    rec = recompute(m, kv, seqs, max_tokens=512)
    rol = rollout(m, kv, seqs, max_tokens=512)
    assert stats(rec, rol) == ZERO
    orc = oracle_for(cfg, W)
    worst = max(float(np.max(np.abs(g - orc.prefill_logprobs(s.tokens)[s.prompt_len - 1:])))
                for s, g in zip(seqs, rec))
    assert worst <= lp_bound("qwen3_2L"), worst


@pytest.mark.parametrize("kv_fp8", [False, True], ids=["bf16kv", "fp8kv"])
def test_qwen3_full_depth_per_layer_parity(kv_fp8, capsys):
    """All 28 layers of the Qwen3-1.7B shape at full size, each checked against
    the oracle computing that layer from the GPU's own input residual (1e-2
    relative per layer output), plus the head from the GPU's last residual
    (|dlp| <= 2e-2), plus free-running parity on three sequences within the
    oracle's own order spread at this depth (bf16 flips compound over 28
    layers for any two correct evaluation orders)."""
    from invariant_forward_bitwise_gb300.model import PagedKV, Runner, prefill_rows, DenseModel
    from oracle.codecs import bf16_to_f32
    cfg = synth.replace(synth.QWEN3_1P7B, kv_fp8=kv_fp8)
    W = synth.dense_weights(cfg, seed=0)
    m = DenseModel(cfg, W, max_rows=256, max_pos=256)
    kv = PagedKV(cfg, pages=8, max_seqs=2, max_pages=4)
    s = synth.tiny_sequences(cfg, n=1, lo=48, hi=48, seed=11)[0]
    kv.admit(0, s.length)
    kv.sync_table()
    run = Runner(m)
    rows = prefill_rows([s], [0], [0], [s.length - 1], [0])
    spec = run.load_rows(kv, *rows[:5])
    m.reserve(kv, [spec])
    m.audit = []
    m.step(kv, spec)
    lp = m.lp[:spec.T_lm].cpu().numpy()
    m.audit, audit = None, m.audit
    res = [x for t, l, x in audit if t == "layer"]
    assert len(res) == cfg.layers
    # without the audit the GEMMs leave their chunk partials to the next op
    # (fold fused into QKV finalize and add+RMSNorm): the same bits
    m.step(kv, spec)
    assert np.array_equal(m.lp[:spec.T_lm].cpu().numpy().view(np.uint32), lp.view(np.uint32))

    def h32(t):
        return bf16_to_f32(t.cpu().view(torch.int16).numpy().view(np.uint16))

    orc = oracle_for(cfg, W)
    pos = np.arange(s.length - 1)
    r_prev = orc.W["embed"][s.tokens[:-1]]
    worst = 0.0
    for l in range(cfg.layers):
        ref = orc.layer_from(l, r_prev, pos)
        got = h32(res[l])
        err = float(np.max(np.abs(got - ref)) / np.max(np.abs(ref)))
        worst = max(worst, err)
        assert err <= 1e-2, (l, err)
        r_prev = got                       # next layer starts from the GPU's residual
    head = orc.head_from(r_prev, s.tokens[1:])
    assert np.max(np.abs(lp - head)) <= TOL_LP
    # free-running: the three sequences of the spread measurement, all positions
    seqs = synth.tiny_sequences(cfg, n=3, lo=48, hi=48, seed=11)
    assert np.array_equal(seqs[0].tokens, s.tokens)
    kv2 = PagedKV(cfg, pages=8, max_seqs=3, max_pages=4)
    for i, q in enumerate(seqs):
        kv2.admit(i, q.length)
    kv2.sync_table()
    rows = prefill_rows(seqs, [0, 1, 2], [0, 0, 0], [q.length - 1 for q in seqs], [0, 0, 0])
    spec2 = run.load_rows(kv2, *rows[:5])
    m.reserve(kv2, [spec2])
    m.step(kv2, spec2)
    lp3 = m.lp[:spec2.T_lm].cpu().numpy().reshape(3, -1)
    assert np.array_equal(lp3[0].view(np.uint32), lp.view(np.uint32))   # batch of 3 = alone
    gaps = [np.abs(lp3[i] - orc.prefill_logprobs(q.tokens)) for i, q in enumerate(seqs)]
    case = "qwen3_28L_fp8kv" if kv_fp8 else "qwen3_28L_bf16kv"
    fmax, fmean = max(float(g.max()) for g in gaps), float(np.mean([g.mean() for g in gaps]))
    with capsys.disabled():
        print(f"\n[qwen3 28L kv_fp8={kv_fp8}] worst per-layer rel err {worst:.2e}; "
              f"teacher-forced head |dlp| max {np.max(np.abs(lp - head)):.2e}; "
              f"free-running |dlp| max {fmax:.3f} mean {fmean:.4f}; oracle order spread "
              f"max {SPREAD[case]['max']:.3f} mean {SPREAD[case]['mean']:.4f}")
    assert fmax <= lp_bound(case)
    means = [o["mean"] for o in SPREAD[case]["orders"].values()]
    assert fmean <= max(means) * max(means) / min(means)


def test_fast_mode_differs_but_stays_close():
    """The non-invariant comparator (batch-dependent split-K / split-KV) stays
    within tolerance of the invariant path; it is not required to be bitwise."""
    from invariant_forward_bitwise_gb300.model import recompute, rollout
    cfg = synth.TINY
    W, m_inv, kv = make(cfg, seed=8, lm_scale=1.0)
    _, m_fast, kv2 = make(cfg, seed=8, mode=1, lm_scale=1.0)
    seqs = synth.tiny_sequences(cfg, n=4, seed=9)
    a = rollout(m_inv, kv, seqs, max_tokens=1024)
    b = rollout(m_fast, kv2, seqs, max_tokens=1024)
    assert stats(a, b)["max"] <= TOL_LP


@pytest.mark.parametrize("kv_fp8", [False, True], ids=["bf16kv", "fp8kv"])
def test_continuous_batching_equals_recompute(kv_fp8):
    """Mixed steps (a prefill chunk of one sequence next to decode rows of the
    others, sequences arriving and leaving) give the recompute's bits."""
    from invariant_forward_bitwise_gb300.model import recompute, serve_mixed
    cfg = synth.replace(synth.TINY, kv_fp8=kv_fp8)
    W, m, kv = make(cfg)
    seqs = synth.tiny_sequences(cfg, n=8, lo=40, hi=128, seed=21)
    rec = recompute(m, kv, seqs, max_tokens=1024)
    mixed = serve_mixed(m, kv, seqs, chunk=16, max_decode=3)
    assert stats(rec, mixed) == ZERO


def _decode_steps(dg, kv, seqs, cur, nsteps):
    """nsteps teacher-forced decode steps of the live sequences (slot i =
    sequence i), advancing cur; returns the logprobs of each step."""
    out = []
    for _ in range(nsteps):
        live = [i for i, s in enumerate(seqs) if cur[i] < s.length - 1]
        if not live:
            break
        lp = dg.run(live, [cur[i] for i in live], [int(seqs[i].tokens[cur[i]]) for i in live],
                    [int(seqs[i].tokens[cur[i] + 1]) for i in live])
        out.append(lp.cpu().numpy().copy())
        for i in live:
            cur[i] += 1
    return out


@pytest.mark.parametrize("kv_fp8", [False, True], ids=["bf16kv", "fp8kv"])
def test_save_reload_then_next_decode_step(kv_fp8):
    """Mid-rollout, weights, KV pages (codes and scales), the block table and
    the page ownership go to host memory; a new model and a new cache are
    built from those copies in fresh allocations and their decode graphs are
    captured anew.  The next decode steps give the original objects' bits."""
    from invariant_forward_bitwise_gb300.model import (DecodeGraphs, DenseModel, PagedKV, Runner,
                                                      _run_rows, prefill_rows)
    cfg = synth.replace(synth.TINY, kv_fp8=kv_fp8)
    W, m, kv = make(cfg, seed=5)
    seqs = synth.tiny_sequences(cfg, n=3, lo=60, hi=90, seed=6)
    for i, s in enumerate(seqs):
        kv.admit(i, s.length)
    kv.sync_table()
    rows = prefill_rows(seqs, [0, 1, 2], [0] * 3, [s.prompt_len for s in seqs], [10 ** 9] * 3)
    _run_rows(m, Runner(m), kv, rows, 1024, lambda k, v: None)
    dg = DecodeGraphs(m, kv, use_graphs=True)
    cur = [s.prompt_len for s in seqs]
    _decode_steps(dg, kv, seqs, cur, 5)
    torch.cuda.synchronize()
    # snapshot to host
    host_w = {k: v.cpu().clone() for k, v in m.W.items()}
    host_kv = {n: getattr(kv, n).cpu().clone() for n in ("k", "v", "ks", "vs") if getattr(kv, n) is not None}
    bt, owned, free = kv.bt_host.copy(), {k: list(v) for k, v in kv.owned.items()}, list(kv.free)
    cur2 = list(cur)
    # the original objects go on
    a = _decode_steps(dg, kv, seqs, cur, 6)
    # new allocations from the host copies, graphs captured again
    m2 = DenseModel(cfg, host_w, max_rows=1024, max_pos=512)
    kv2 = PagedKV(cfg, pages=kv.pages, max_seqs=kv.block_table.shape[0], max_pages=kv.max_pages)
    for n, t in host_kv.items():
        getattr(kv2, n).copy_(t)
    kv2.bt_host[:], kv2.owned, kv2.free = bt, owned, free
    kv2.sync_table()
    dg2 = DecodeGraphs(m2, kv2, use_graphs=True)
    b = _decode_steps(dg2, kv2, seqs, cur2, 6)
    assert len(a) == len(b) == 6
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
