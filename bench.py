#!/usr/bin/env python
"""Benchmark of the batch-invariant logprob forward on one GB300 (or N, as
independent replicas).

Workload (Qwen3-1.7B-shaped dense decoder, random-init bf16 weights, synthetic
token ids): 64 prompts x 8 responses, prompt length U[64,512], response length
U[128,1024].  One step = the rollout of all 512 sequences (prompt prefill,
then teacher-forced decode of every response token with CUDA-graph replay and
continuous batching as sequences finish) followed by the trainer recompute of
all 512 full sequences (prefill into a private KV cache).  Each step emits the
logprob of every response token twice (rollout and recompute); the metric
counts those logprob tokens per second.  Weights (3.4 GB) exceed L2, so no
explicit flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "invariant logprob tokens/s (rollout decode + trainer recompute)"
UNIT = "tokens/s"
WORKLOAD = "qwen3-1.7b-shape rollout+recompute, 64 prompts x 8 responses, prompt U[64,512], response U[128,1024], bf16 KV"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--prompts", type=int, default=64)
    ap.add_argument("--responses", type=int, default=8)
    ap.add_argument("--layers", type=int, default=28)
    ap.add_argument("--max-tokens", type=int, default=16384, help="rows per prefill step")
    ap.add_argument("--no-fast", action="store_true", help="skip the non-invariant comparator")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="decode without CUDA-graph replay (for per-launch profilers)")
    ap.add_argument("--prompt-max", type=int, default=512, help="cap prompt length (profiling runs)")
    ap.add_argument("--resp-max", type=int, default=1024, help="cap response length (profiling runs)")
    return ap.parse_args()


# ----------------------------------------------------------------- clocks --
class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during timing."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    mx.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- oracle ---
def oracle_sample(layers: int, n_seq: int = 1, prompt: int = 48, resp: int = 48, seed: int = 11):
    """Time the CPU oracle (as it stands) on a bounded sample of the same
    workload: n_seq sequences of the Qwen3-1.7B shape, rollout (prompt prefill +
    token-by-token decode) and recompute (one prefill).  Returns tokens/s."""
    import synth
    from oracle.model import DenseOracle, decode_weights
    cfg = synth.scaled_dense(synth.QWEN3_1P7B, layers) if layers != 28 else synth.QWEN3_1P7B
    W = synth.dense_weights(cfg, seed=0)
    orc = DenseOracle(cfg, decode_weights({k: synth.bf16_bits(v) for k, v in W.items()}),
                      max_pos=prompt + resp + 1)
    seqs = synth.rollout_sequences(cfg, prompts=n_seq, responses=1, prompt_lo=prompt, prompt_hi=prompt,
                                   resp_lo=resp, resp_hi=resp, seed=seed)
    t0 = time.perf_counter()
    ntok = 0
    for s in seqs:
        a = orc.decode_logprobs(s.tokens, s.prompt_len)[s.prompt_len - 1:]
        b = orc.prefill_logprobs(s.tokens)[s.prompt_len - 1:]
        ntok += a.size + b.size
    dt = time.perf_counter() - t0
    return ntok / dt, dt, ntok


def threads_used():
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 0) for i in threadpool_info()), default=0)
        if n:
            return n
    except Exception:
        pass
    return os.cpu_count()


def run_reference(args, rank):
    """The reference arm: the CPU oracle, timed on the host's cores."""
    if rank != 0:
        return
    sample = "1 sequence (prompt 48, response 48) of the full 28-layer shape: oracle rollout + recompute per step"
    for _ in range(args.warmup):
        oracle_sample(args.layers)
    times, toks = [], 0
    for _ in range(args.steps):
        v, dt, n = oracle_sample(args.layers)
        times.append(dt)
        toks = n
    value = toks / statistics.mean(times)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"kind": "oracle", "value": value, "unit": UNIT, "cores": threads_used(),
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ ours ---
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained", j["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    import torch
    import synth
    from invariant_forward_bitwise_gb300 import biv, build
    from invariant_forward_bitwise_gb300.model import DecodeGraphs, DenseModel, PagedKV, recompute, rollout

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    if local == 0:
        build.build()
    if world > 1:
        dist.barrier()
    biv.load()

    cfg = synth.QWEN3_1P7B if args.layers == 28 else synth.scaled_dense(synth.QWEN3_1P7B, args.layers)
    seqs = synth.rollout_sequences(cfg, prompts=args.prompts, responses=args.responses,
                                   prompt_lo=min(64, args.prompt_max), prompt_hi=args.prompt_max,
                                   resp_lo=min(128, args.resp_max), resp_hi=args.resp_max, seed=1 + rank)
    W = synth.dense_weights(cfg, seed=0)
    max_len = max(s.length for s in seqs)
    max_pos = (max_len + 63) // 64 * 64
    resp_tokens = sum(s.length - s.prompt_len for s in seqs)

    def build_arm(mode):
        m = DenseModel(cfg, W, max_rows=args.max_tokens, max_pos=max_pos, mode=mode)
        pages_roll = sum((s.length + 63) // 64 for s in seqs) + 8
        kv_roll = PagedKV(cfg, pages=pages_roll, max_seqs=len(seqs), max_pages=max_pos // 64)
        group_pages = (args.max_tokens // 64 + 64) * 2
        kv_rec = PagedKV(cfg, pages=group_pages, max_seqs=len(seqs), max_pages=max_pos // 64)
        dg = DecodeGraphs(m, kv_roll, use_graphs=not args.eager)
        return m, kv_roll, kv_rec, dg

    def one_step(arm, collect=False, mid=None):
        m, kv_roll, kv_rec, dg = arm
        a = rollout(m, kv_roll, seqs, args.max_tokens, graphs=dg, collect=collect)
        if mid is not None:
            mid.record(torch.cuda.current_stream())
        b = recompute(m, kv_rec, seqs, args.max_tokens)
        return a, b

    def timed(arm, steps, warmup, clocks=None):
        for _ in range(warmup):
            one_step(arm)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        if clocks:
            clocks.start()
        st = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        arm[0].kernel_timer = timer = KernelTimer()
        # step boundaries and the rollout/recompute boundary of each step
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * steps)]
        e0.record(st)
        for i in range(steps):
            one_step(arm, mid=ev[2 * i])
            ev[2 * i + 1].record(st)
        e1.record(st)
        torch.cuda.synchronize()
        arm[0].kernel_timer = None
        if world > 1:
            dist.barrier()
        ck = clocks.stop() if clocks else None
        ms = e0.elapsed_time(e1) / steps
        starts = [e0] + ev[1::2][:-1]
        roll = sum(a.elapsed_time(b) for a, b in zip(starts, ev[0::2])) / steps
        timer.phases = {"rollout_ms": roll, "recompute_ms": ms - roll}
        return ms, ck, timer

    inv = build_arm(biv.MODE_INVARIANT)
    # invariance check of this very workload: rollout vs recompute, bitwise
    a, b = one_step(inv, collect=True)
    la, lb = np.concatenate(a), np.concatenate(b)
    diff_max = float(np.max(np.abs(la - lb)))
    clocks = Clocks(local)
    ms, ck, timer = timed(inv, args.steps, args.warmup, clocks)
    tokens_per_step = 2 * resp_tokens
    ms, value = reduce_over_ranks(ms, tokens_per_step, world, device="cuda")

    peaks = load_peaks()
    roof = timer.roofline(peaks)
    fast = None
    if not args.no_fast:
        del inv
        torch.cuda.empty_cache()
        fast_arm = build_arm(biv.MODE_FAST)
        ms_f, _, t_f = timed(fast_arm, max(1, args.steps), 1)
        fast = {"value": tokens_per_step / (ms_f / 1e3), "ms_per_step": ms_f, "phases": t_f.phases,
                "invariant_over_fast": (tokens_per_step / (ms / 1e3)) / (tokens_per_step / (ms_f / 1e3))}
        del fast_arm
        torch.cuda.empty_cache()
        inv = build_arm(biv.MODE_INVARIANT)

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(inv if not args.no_fast else inv, one_step, seqs, tokens_per_step, world)

    cpu = None
    if rank == 0 and not args.no_cpu:
        v, dt, n = oracle_sample(args.layers)
        cpu = {"value": v, "unit": UNIT, "cores": threads_used(), "kind": "oracle",
               "sample": f"1 sequence (prompt 48, response 48) of the {args.layers}-layer shape, oracle rollout + recompute ({n} logprob tokens, {dt:.1f} s)"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": WORKLOAD, "sequences": len(seqs), "response_tokens": resp_tokens,
                           "layers": args.layers, "prefill_rows_per_step": args.max_tokens,
                           "l2": "inputs larger than L2 (3.4 GB of weights streamed per pass)",
                           "parallelism": f"replicas x{world}"},
                "logprob_diff_rollout_vs_recompute": diff_max,
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": ck,
                "gpu_launches": timer.launches, "fast_comparator": fast,
                "kernels": timer.summary(peaks), "phases": timer.phases}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def reduce_over_ranks(ms: float, tokens_per_step: int, world: int, device=None):
    """Replicas: every rank runs its own sequences (weak scaling).  The step
    time is the max over ranks; whole-job throughput counts all ranks' tokens
    over that time."""
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms = float(t.item())
    return ms, tokens_per_step * world / (ms / 1e3)


class KernelTimer:
    """CUDA-event brackets around eager launches of the hot kernels (GEMM and
    attention) inside the timed region, plus a count of every libbiv launch."""

    def __init__(self):
        import torch
        self.torch = torch
        self.open = []
        self.launches = 0

    def bracket(self, kind, work, unit):
        t = self.torch
        e0, e1 = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
        e0.record(t.cuda.current_stream())
        return e0, e1, kind, work, unit

    def close(self, tok):
        e0, e1, kind, work, unit = tok
        e1.record(self.torch.cuda.current_stream())
        self.open.append((e0, e1, kind, work, unit))

    def totals(self):
        agg = {}
        for e0, e1, kind, work, unit in self.open:
            ms = e0.elapsed_time(e1)
            a = agg.setdefault(kind, {"ms": 0.0, "work": 0.0, "n": 0, "unit": unit})
            a["ms"] += ms
            a["work"] += work
            a["n"] += 1
        return agg

    def summary(self, peaks):
        out = {}
        for k, a in self.totals().items():
            rate = a["work"] / (a["ms"] / 1e3)
            out[k] = {"launches": a["n"], "ms_total": a["ms"],
                      "achieved": rate / 1e12 if a["unit"] == "flop" else rate / 1e9,
                      "unit": "TFLOP/s" if a["unit"] == "flop" else "GB/s"}
        return out

    def roofline(self, peaks):
        tot = self.totals()
        if not tot:
            return None
        k = max(tot, key=lambda x: tot[x]["ms"])
        a = tot[k]
        if a["unit"] == "flop":
            ach = a["work"] / (a["ms"] / 1e3) / 1e12
            peak = peaks["bf16_tflops_sustained"]
            return {"kernel": k, "bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                    "frac": ach / peak, "traffic": None, "peak_source": peaks["source"] + " sustained bf16"}
        ach = a["work"] / (a["ms"] / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        return {"kernel": k, "bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
                "frac": ach / peak, "traffic": None, "peak_source": peaks["source"] + " hbm"}


def measure_e2e(arm, one_step, seqs, tokens_per_step, world):
    """Same step through the public path with host buffers: every step starts
    by copying all token ids from pinned host memory to the device and ends
    with the device->host copy of every logprob."""
    import torch
    m = arm[0]
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    h0 = m.h2d_bytes
    e0.record(st)
    a, b = one_step(arm, collect=True)
    out = np.concatenate(a + b)
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    return {"value": tokens_per_step * world / (ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": int(m.h2d_bytes - h0), "d2h_bytes_per_step": int(out.size * 4),
            "ms_per_step": ms,
            "path": "token ids and row metadata copied host->device by the scheduler each step; "
                    "every logprob copied device->host"}


if __name__ == "__main__":
    main()
