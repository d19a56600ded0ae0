"""Writes ``accumulation_spread.json``: how far two correct FP32 evaluations of
the oracle drift apart in free-running logprobs, per model-level parity case.

The pages fix what must be identical between the compared runs (computation
path, quantisation, tie-break, accumulation order: "Finish RL Training
Faster", section "零差异需要一个精确的比较对象") but give no precision for the
reference itself.  Two evaluations of the same forward that differ only in
how each FP32 dot product is summed -- float64 then rounded once (the
oracle's default) against plain FP32 in ascending k, in descending k,
ascending with IEEE round-toward-zero (as tensor-core accumulators truncate),
or in the FP32 library matmul's blocked order -- are all correct, yet
their bf16 roundings part ways now and then, and a deep stack (QK-norm
attention, residual stream rounded to bf16 at every layer) carries those
flips forward.  The largest gap between the default and any of these orders
(over the case's sequences: the envelope of correct evaluations) is
therefore what an implementation that does not reproduce the oracle's exact
roundings can be held to, and the GPU parity tests assert against
max(2e-2, that envelope) where it exceeds 2e-2.

Only ``oracle/`` and the seeded input generators are called.  Run from the
repository root:  python tests/golden/make_accumulation_spread.py
(the sequential FP32 orders are Python loops: the 28-layer cases take about
half an hour with four worker processes).
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from oracle import ops  # noqa: E402
from oracle.mamba import HybridOracle, decode_hybrid_weights  # noqa: E402
from oracle.model import DenseOracle, decode_weights  # noqa: E402

# the correct FP32 orders compared with the oracle's default (float64 then
# rounded); a case's bound is the largest gap any of them shows
ALTERNATIVES = ("f32", "f32_desc", "f32_rz", "f32_blas")

# name -> (config, weight kwargs, sequence kwargs, first scored position).
# The recipes are those of the GPU parity tests that read this file.
CASES = {
    "qwen3_28L_bf16kv": (synth.QWEN3_1P7B, dict(seed=0), dict(n=3, lo=48, hi=48, seed=11), 0),
    "qwen3_28L_fp8kv": (synth.QWEN3_1P7B_FP8KV, dict(seed=0), dict(n=3, lo=48, hi=48, seed=11), 0),
    "qwen3_2L": (synth.scaled_dense(synth.QWEN3_1P7B, 2), dict(seed=0),
                 dict(n=3, lo=40, hi=70, seed=7), None),
    "tiny_peaked_bf16kv": (synth.TINY, dict(seed=0, random_gains=True, lm_scale=10.0),
                           dict(n=8, seed=1), None),
    "tiny_peaked_fp8kv": (synth.replace(synth.TINY, kv_fp8=True),
                          dict(seed=0, random_gains=True, lm_scale=10.0), dict(n=8, seed=1), None),
    "tiny_peaked_seed4": (synth.TINY, dict(seed=4, random_gains=True, lm_scale=10.0),
                          dict(n=4, seed=2), None),
    "hybrid_tiny_peaked": (synth.HYBRID_TINY, dict(seed=0, random_gains=True, lm_scale=8.0),
                           dict(n=2, lo=280, hi=300, seed=5), None),
    "hybrid_tiny_flat": (synth.HYBRID_TINY, dict(seed=0, random_gains=True, lm_scale=1.0),
                         dict(n=2, lo=280, hi=300, seed=5), None),
}


def _oracle_and_sequences(name):
    cfg, wkw, skw, first = CASES[name]
    if isinstance(cfg, synth.HybridConfig):
        W = synth.hybrid_weights(cfg, **wkw)
        orc = HybridOracle(cfg, decode_hybrid_weights(synth.host_payload(W)), max_pos=512)
        seqs = synth.hybrid_sequences(cfg, **skw)
    else:
        W = synth.dense_weights(cfg, **wkw)
        orc = DenseOracle(cfg, decode_weights({k: synth.bf16_bits(v) for k, v in W.items()}),
                          max_pos=256)
        seqs = synth.tiny_sequences(cfg, **skw)
    return orc, seqs, first


def _task(args):
    """max and mean |dlogprob| between the default order and ``kind`` on
    every sequence of case ``name``."""
    name, kind = args
    orc, seqs, first = _oracle_and_sequences(name)
    per_max, per_mean = [], []
    for s in seqs:
        lo = s.prompt_len - 1 if first is None else first
        a = orc.prefill_logprobs(s.tokens)[lo:]
        with ops.accumulation(kind):
            b = orc.prefill_logprobs(s.tokens)[lo:]
        d = np.abs(a.astype(np.float64) - b)
        per_max.append(float(d.max()))
        per_mean.append(float(d.mean()))
    return name, kind, {"max": max(per_max), "mean": float(np.mean(per_mean)),
                        "per_sequence_max": per_max}


def main(names=None, workers=4):
    import multiprocessing as mp
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "accumulation_spread.json")
    out = json.load(open(path)) if os.path.exists(path) else {}
    names = [n for n in CASES if not names or n in names]
    tasks = [(n, k) for n in names for k in ALTERNATIVES]
    res = {n: {} for n in names}
    with mp.get_context("spawn").Pool(workers) as pool:
        for name, kind, r in pool.imap_unordered(_task, tasks):
            res[name][kind] = r
            print(name, kind, r["max"], r["mean"], flush=True)
    for name in names:
        cfg, wkw, skw, first = CASES[name]
        orders = res[name]
        out[name] = {"max": max(o["max"] for o in orders.values()),
                     "mean": max(o["mean"] for o in orders.values()), "orders": orders,
                     "weights": wkw, "sequences": skw, "config": cfg.name, "kv_fp8": cfg.kv_fp8,
                     "scored": "all positions" if first == 0 else "response positions"}
    with open(path, "w") as f:
        json.dump(out, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main(sys.argv[1:] or None)
