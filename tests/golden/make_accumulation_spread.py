"""Writes ``accumulation_spread.json``: how far two correct FP32 evaluations of
the oracle drift apart in free-running logprobs, per model-level parity case.

The pages fix what must be identical between the compared runs (computation
path, quantisation, tie-break, accumulation order: "Finish RL Training
Faster", section "零差异需要一个精确的比较对象") but give no precision for the
reference itself.  Two evaluations of the same forward that differ only in
how each FP32 dot product is summed -- float64 then rounded once (the
oracle's default) and plain FP32 in ascending k -- are both correct, yet
their bf16 roundings part ways now and then, and a deep stack (QK-norm
attention, residual stream rounded to bf16 at every layer) carries those
flips forward.  The spread between them is therefore a floor on what any
implementation that does not reproduce the oracle's exact rounding can
promise against it, and the GPU parity tests assert against
max(2e-2, that spread) for the cases where it exceeds 2e-2.

Only ``oracle/`` and the seeded input generators are called.  Run from the
repository root:  python tests/golden/make_accumulation_spread.py
(about ten minutes on one core; the FP32 ascending-k path is a Python loop).
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from oracle import ops  # noqa: E402
from oracle.model import DenseOracle, decode_weights  # noqa: E402

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
}


def spread(cfg, wkw, skw, first):
    W = synth.dense_weights(cfg, **wkw)
    orc = DenseOracle(cfg, decode_weights({k: synth.bf16_bits(v) for k, v in W.items()}),
                      max_pos=256)
    per_max, per_mean = [], []
    for s in synth.tiny_sequences(cfg, **skw):
        lo = s.prompt_len - 1 if first is None else first
        a = orc.prefill_logprobs(s.tokens)[lo:]
        with ops.accumulation("f32"):
            b = orc.prefill_logprobs(s.tokens)[lo:]
        d = np.abs(a.astype(np.float64) - b)
        per_max.append(float(d.max()))
        per_mean.append(float(d.mean()))
    return {"max": max(per_max), "mean": float(np.mean(per_mean)),
            "per_sequence_max": per_max, "per_sequence_mean": per_mean}


def main(names=None):
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "accumulation_spread.json")
    out = json.load(open(path)) if os.path.exists(path) else {}
    for name, (cfg, wkw, skw, first) in CASES.items():
        if names and name not in names:
            continue
        out[name] = dict(spread(cfg, wkw, skw, first), weights=wkw, sequences=skw,
                         config=cfg.name, kv_fp8=cfg.kv_fp8,
                         scored="all positions" if first == 0 else "response positions")
        print(name, out[name]["max"], out[name]["mean"], flush=True)
        with open(path, "w") as f:
            json.dump(out, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main(sys.argv[1:] or None)
