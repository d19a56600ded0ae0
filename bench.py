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
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the FP8-KV serving and MoE + sparse-attention measurements")
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
    shape = "the full 28-layer shape" if args.layers == 28 else f"the shape cut to {args.layers} layers"
    sample = f"1 sequence (prompt 48, response 48) of {shape}: oracle rollout + recompute per step"
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

    def one_step(arm, collect=False, mid=None, pre=None):
        m, kv_roll, kv_rec, dg = arm
        after = (lambda: pre.record(torch.cuda.current_stream())) if pre is not None else None
        a = rollout(m, kv_roll, seqs, args.max_tokens, graphs=dg, collect=collect, after_prefill=after)
        if mid is not None:
            mid.record(torch.cuda.current_stream())
        b = recompute(m, kv_rec, seqs, args.max_tokens)
        return a, b

    decode_work = decode_step_bytes(cfg, W)

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
        arm[0].kernel_timer = timer = KernelTimer(decode_work)
        # per step: end of the prompt prefill, end of the rollout, end of the step
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3 * steps)]
        e0.record(st)
        for i in range(steps):
            one_step(arm, pre=ev[3 * i], mid=ev[3 * i + 1])
            ev[3 * i + 2].record(st)
        e1.record(st)
        torch.cuda.synchronize()
        arm[0].kernel_timer = None
        if world > 1:
            dist.barrier()
        ck = clocks.stop() if clocks else None
        ms = e0.elapsed_time(e1) / steps
        starts = [e0] + ev[2::3][:-1]
        pre = sum(a.elapsed_time(b) for a, b in zip(starts, ev[0::3])) / steps
        roll = sum(a.elapsed_time(b) for a, b in zip(starts, ev[1::3])) / steps
        timer.phases = {"rollout_ms": roll, "rollout_prompt_prefill_ms": pre,
                        "rollout_decode_ms": roll - pre, "recompute_ms": ms - roll}
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

    configs = None
    if not args.no_configs:
        del inv
        torch.cuda.empty_cache()
        configs = {"fp8_kv_continuous_batching": fp8_serving(W, peaks),
                   "moe_sparse_attention_block": moe_sparse_block(peaks)}
        torch.cuda.empty_cache()
        configs["mamba2_hybrid_unit"] = hybrid_unit(peaks)
        torch.cuda.empty_cache()

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
                "kernels": timer.summary(peaks), "phases": timer.phases, "configs": configs}
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


def decode_step_bytes(cfg, W):
    """Algorithmic HBM bytes of one decode step whose rows sit at positions
    ``pos``: every weight once (the tied LM head streams the embedding table
    once per step; the embedding gather reads only the rows' own entries), the
    cached K/V of positions 0..p of each row's sequence over all layers, the
    row's own K/V write, and the (max, sum exp) pairs of its 128-logit groups
    that the LM head's epilogue writes and the combine reads (the FP32 logits
    never reach memory)."""
    seen, wbytes = set(), 0
    for t in W.values():
        if id(t) not in seen:
            seen.add(id(t))
            wbytes += t.numel() * t.element_size()
    per_tok = cfg.kv_heads * cfg.head_dim * (1 if cfg.kv_fp8 else 2) + (4 * cfg.kv_heads if cfg.kv_fp8 else 0)
    kv_tok = 2 * cfg.layers * per_tok
    extra = kv_tok + 2 * ((cfg.vocab + 127) // 128) * 8

    def work(pos):
        return float(wbytes + sum(int(p) + 1 for p in pos) * kv_tok + len(pos) * extra)

    work.weight_bytes, work.kv_bytes_per_token = wbytes, kv_tok
    return work


class KernelTimer:
    """CUDA-event brackets inside the timed region: around eager launches of
    the hot prefill kernels (GEMM and attention) and around every decode-step
    graph replay, plus a count of every libbiv launch."""

    def __init__(self, decode_work=None):
        import torch
        self.torch = torch
        self.open = []
        self.launches = 0
        self.decode_work = decode_work

    def bracket_decode(self, pos):
        if self.decode_work is None:
            return None
        return self.bracket("decode_step", self.decode_work(pos), "byte")

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

    NAMES = {"decode_step": "decode step (one CUDA-graph replay: 28 layers, LM head, logprob)",
             "gemm_bf16": "prefill bf16 GEMMs (tcgen05)", "attention_prefill": "prefill attention"}

    # DRAM bytes per algorithmic byte of a decode step, from ncu captures of one
    # eager step with every sequence at position 700 (kernel_bench decode_step):
    # 9.337 GB against 8.59 GB at batch 64, 25.77 GB against 23.99 GB at batch
    # 256; the excess is the decode GEMMs' FP32 chunk partials.  The bench's
    # steps mix batch sizes and contexts, so their traffic is this ratio times
    # their own algorithmic bytes.
    DECODE_DRAM_RATIO = (9.337 / 8.59 + 25.77 / 23.99) / 2

    def entry(self, k, a, peaks):
        if a["unit"] == "flop":
            ach = a["work"] / (a["ms"] / 1e3) / 1e12
            peak = peaks["bf16_tflops_sustained"]
            return {"kernel": self.NAMES.get(k, k), "bound": "tensor", "achieved": ach, "peak": peak,
                    "unit": "TFLOP/s", "frac": ach / peak, "traffic": None, "launches": a["n"],
                    "ms_total": a["ms"], "algorithmic_per_launch": a["work"] / a["n"],
                    "peak_source": peaks["source"] + " sustained bf16"}
        ach = a["work"] / (a["ms"] / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        out = {"kernel": self.NAMES.get(k, k), "bound": "hbm", "achieved": ach, "peak": peak,
               "unit": "GB/s", "frac": ach / peak, "traffic": None, "launches": a["n"],
               "ms_total": a["ms"], "algorithmic_per_launch": a["work"] / a["n"],
               "peak_source": peaks["source"] + " hbm"}
        if k == "decode_step":
            out["traffic"] = self.DECODE_DRAM_RATIO * a["work"] / a["n"]
            out["traffic_source"] = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one eager decode "
                                     "step at batch 64 and 256 (position 700), per algorithmic byte "
                                     f"({self.DECODE_DRAM_RATIO:.3f}), times this run's algorithmic "
                                     "bytes per replay")
        return out

    def summary(self, peaks):
        return {k: self.entry(k, a, peaks) for k, a in self.totals().items()}

    def roofline(self, peaks):
        """The entry of the family that takes the most time in the step."""
        tot = self.totals()
        if not tot:
            return None
        k = max(tot, key=lambda x: tot[x]["ms"])
        return self.entry(k, tot[k], peaks)


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


# ----------------------------------------------------- further workloads ----
def fp8_serving(W, peaks, steps=24, pool=256, chunk=512, seed=5):
    """Continuous batching on the FP8 KV cache (Qwen3-1.7B shape, e4m3 pages
    of 64 tokens with one fp32 scale per token and kv head).  A pool of 256
    sequences holds contexts drawn U[1024, 16384]; every step carries one
    prefill chunk of 512 tokens (of a sequence whose chunk starts at a
    position drawn U[0, 15872] in steps of 512) plus one decode row for each
    of N sequences, N drawn U[1, 256] per step from a rotating window of the
    pool.  Every row produces a logprob.  The caches are filled by the FP8
    quantiser from device-drawn N(0, 1) K/V (the values do not change the
    work).  Returns tokens/s and the step roofline: per step the larger of
    FLOPs / bf16 peak and bytes / HBM peak, summed, over the measured time."""
    import torch
    import synth
    from invariant_forward_bitwise_gb300 import biv
    from invariant_forward_bitwise_gb300.model import DenseModel, PagedKV, Runner

    cfg = synth.QWEN3_1P7B_FP8KV
    rng = np.random.Generator(np.random.Philox(seed))
    ctx0 = rng.integers(1024, 16384 + 1, size=pool)
    nmax = 16384 + chunk
    sched = []
    dec = np.zeros(pool, np.int64)               # tokens decoded so far per pool sequence
    start = 0
    for _ in range(steps + 1):                   # one warm-up step, then the timed ones
        n = int(rng.integers(1, pool + 1))
        live = [(start + j) % pool for j in range(n)]
        start = (start + n) % pool
        pos = [int(ctx0[i] + dec[i]) for i in live]
        dec[live] += 1
        sched.append((live, pos, int(rng.integers(0, (16384 - chunk) // chunk + 1)) * chunk))
    max_pos = (int(max(ctx0 + dec)) + 1 + 63) // 64 * 64
    max_pos = max(max_pos, nmax)
    m = DenseModel(cfg, W, max_rows=pool + chunk, max_pos=max_pos)
    pages = sum((int(c + dec[i]) + 1 + 63) // 64 for i, c in enumerate(ctx0)) + nmax // 64 + 8
    kv = PagedKV(cfg, pages=pages, max_seqs=pool + 1, max_pages=max_pos // 64)
    for i in range(pool):
        kv.admit(i, int(ctx0[i] + dec[i]) + 1)
    kv.admit(pool, nmax)
    kv.sync_table()
    # fill every cached position of every layer through the FP8 quantiser
    gen = synth.device_generator(seed)
    Hkv, D = cfg.kv_heads, cfg.head_dim
    blk = 65536
    kd = synth.device_normal(gen, (blk, Hkv * D))
    vd = synth.device_normal(gen, (blk, Hkv * D))
    lens = [int(ctx0[i]) for i in range(pool)] + [nmax]
    slots = np.concatenate([kv.slots(np.full(L, i, np.int32), np.arange(L, dtype=np.int32))
                            for i, L in enumerate(lens)])
    slots_d = torch.from_numpy(slots).cuda()
    for l in range(cfg.layers):
        for a in range(0, slots.size, blk):
            nn = min(blk, slots.size - a)
            biv.biv_kv_fp8_quant(kd[:nn], vd[:nn], Hkv * D, slots_d[a:a + nn], nn, Hkv, D,
                                 kv.k[l], kv.v[l], kv.ks[l], kv.vs[l])
    del kd, vd, slots_d
    run = Runner(m)
    tok = rng.integers(0, cfg.vocab, size=pool + chunk + 1).astype(np.int32)

    def rows_of(live, pos, c0):
        seq = list(live) + [pool] * chunk
        ps = list(pos) + list(range(c0, c0 + chunk))
        ids = [int(tok[j % tok.size]) for j in range(len(ps))]
        tg = [int(tok[(j + 1) % tok.size]) for j in range(len(ps))]
        return seq, ps, ids, list(range(len(ps))), tg

    specs = []
    for live, pos, c0 in sched:                  # size the workspaces before timing
        spec = run.load_rows(kv, *rows_of(live, pos, c0))
        m.reserve(kv, [spec])
        specs.append(spec)
    m.step(kv, specs[0])
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    ntok = 0
    for live, pos, c0 in sched[1:]:
        spec = run.load_rows(kv, *rows_of(live, pos, c0))
        m.step(kv, spec)
        ntok += spec.T
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    # roofline: per step max(FLOPs / tensor peak, bytes / HBM peak)
    wbytes = sum(t.numel() * t.element_size() for t in {id(t): t for t in m.W.values()}.values())
    nonemb = wbytes / 2 - cfg.vocab * cfg.hidden
    kv_tok = 2 * cfg.layers * (Hkv * D + 4 * Hkv)
    lb = 0.0
    byt = 0.0
    for live, pos, c0 in sched[1:]:
        T = len(live) + chunk
        fl = 2.0 * T * (nonemb + cfg.vocab * cfg.hidden)
        fl += 4.0 * cfg.layers * cfg.q_heads * D * (sum(p + 1 for p in pos) + sum(range(c0 + 1, c0 + chunk + 1)))
        b = wbytes + kv_tok * (sum(p + 1 for p in pos) + c0 + chunk + T) + 2 * cfg.vocab * 4 * T
        byt += b
        lb += max(fl / (peaks["bf16_tflops_sustained"] * 1e12), b / (peaks["hbm_gbs"] * 1e9))
    decode_rows = sum(len(x[0]) for x in sched[1:])
    return {"workload": "qwen3-1.7b-shape, FP8 e4m3 KV (pages of 64, fp32 scale per token and kv head); "
                        f"{steps} continuous-batching steps, each a 512-token prefill chunk at a context "
                        "U[0,16K) plus decode rows of N~U[1,256] sequences with contexts U[1K,16K]",
            "value": ntok / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms / steps,
            "tokens": ntok, "decode_rows": decode_rows, "prefill_rows": steps * chunk,
            "roofline": {"bound": "hbm", "achieved": byt / (ms / 1e3) / 1e9, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": lb / (ms / 1e3), "traffic": None,
                         "frac_is": "sum over steps of max(FLOPs / sustained bf16, bytes / HBM) over measured time",
                         "peak_source": peaks["source"]}}


def moe_sparse_block(peaks, steps=5, warmup=3, seed=7, profile_step=False):
    """The MoE + sparse-attention block, 4096 tokens per step: indexer scores of
    4096 queries (positions 28672..32767) against a 32768-token context (one
    128-d head, FP32 out), top 2048 positions per query (lowest position wins
    ties, ascending), bf16 MQA attention (32 heads, D 128) over the selected
    keys, then the MoE (hidden 4096, router over 64 experts, top-6 + 1 shared,
    expert intermediate 1408, FP8 e4m3 weights with 128x128 scales) and the
    FP32 fixed-slot combine.  Inputs drawn on the device from a seeded
    generator.  Roofline: the sum of each part's lower bound over the
    measured time.  profile_step: one more step after the timed ones, inside
    cudaProfilerStart/Stop (for an ncu launch list)."""
    import math
    import torch
    import synth
    from invariant_forward_bitwise_gb300 import biv
    from invariant_forward_bitwise_gb300.moe import MoEBlock

    c = synth.MOE_BLOCK
    T, E, k, d, I = c.tokens, c.experts, c.top_k, c.hidden, c.expert_inter
    ctx, K, Di, Hq, D = c.context, c.index_topk, c.index_dim, c.attn_heads, c.head_dim
    gen = synth.device_generator(seed)
    wr = synth.device_normal(gen, (E, d), 0.05)
    wgu, sgu = synth.device_fp8_block_weights(gen, E, 2 * I, d)
    wd, sd = synth.device_fp8_block_weights(gen, E, d, I)
    shgu, shsgu = synth.device_fp8_block_weights(gen, 1, 2 * I, d)
    shd, shsd = synth.device_fp8_block_weights(gen, 1, d, I)
    blk = MoEBlock(wr, wgu, sgu, wd, sd, shgu[0], shsgu[0], shd[0], shsd[0], top_k=k, max_tokens=T)
    h = synth.device_normal(gen, (T, d))
    q_idx = synth.device_normal(gen, (T, Di))
    k_idx = synth.device_normal(gen, (ctx, Di))
    qpos = torch.arange(ctx - T, ctx, dtype=torch.int32, device="cuda")
    valid = qpos + 1
    scores = torch.empty(T, ctx, dtype=torch.float32, device="cuda")
    idx = torch.empty(T, K, dtype=torch.int32, device="cuda")
    pages = ctx // 64
    kc = synth.device_normal(gen, (pages, 64, 1, D))
    vc = synth.device_normal(gen, (pages, 64, 1, D))
    bt = torch.arange(pages, dtype=torch.int32, device="cuda").view(1, pages)
    q = synth.device_normal(gen, (T, Hq * D))
    out = torch.empty_like(q)
    seq = torch.zeros(T, dtype=torch.int32, device="cuda")
    qb = torch.stack([torch.arange(T, dtype=torch.int32), torch.ones(T, dtype=torch.int32)], 1).cuda()
    ad = biv.AttnDesc()
    ad.q, ad.q_stride, ad.out, ad.out_stride = q.data_ptr(), q.stride(0), out.data_ptr(), out.stride(0)
    ad.T, ad.Hq, ad.Hkv, ad.D = T, Hq, 1, D
    ad.row_seq, ad.row_pos, ad.qblocks, ad.nqblocks, ad.max_rows_per_block = (
        seq.data_ptr(), qpos.data_ptr(), qb.data_ptr(), T, 1)
    ad.kv_dtype = biv.BF16
    ad.k_cache, ad.v_cache, ad.block_table, ad.max_pages, ad.page = (
        kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), pages, 64)
    ad.kv_split, ad.max_ctx, ad.scale = 1024, ctx, 1 / math.sqrt(D)
    ad.topk_idx, ad.topk_stride, ad.topk = idx.data_ptr(), idx.stride(0), K
    ws = torch.empty(max(biv.biv_attention_workspace(ad), 16), dtype=torch.uint8, device="cuda")
    gd = biv.gemm_desc(q_idx, k_idx, scores)
    gws = torch.empty(max(biv.biv_gemm_workspace(gd), 16), dtype=torch.uint8, device="cuda")

    def step():
        biv.biv_gemm(gd, gws)
        biv.biv_topk(scores, valid, K, idx)
        biv.biv_attention(ad, ws)
        blk.forward(h)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(steps):
        step()
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    if profile_step:
        torch.cuda.cudart().cudaProfilerStart()
        step()
        torch.cuda.synchronize()
        torch.cuda.cudart().cudaProfilerStop()
    bw, tf = peaks["hbm_gbs"] * 1e9, peaks["bf16_tflops_sustained"] * 1e12
    fp8 = 2.0 * tf          # FP8 dense rate: the nominal 2x of bf16
    parts = {
        "indexer_gemm": max(2.0 * T * ctx * Di / tf, (T * ctx * 4 + (T + ctx) * Di * 2) / bw),
        "topk": (T * ctx * 4 + T * K * 4) / bw,
        "sparse_attention": max(4.0 * Hq * D * K * T / tf, (2 * ctx * D * 2 + 2 * T * Hq * D * 2 + T * K * 4) / bw),
        "moe_experts": max(2.0 * T * (k + 1) * 3 * d * I / fp8, (E + 1) * 3 * d * I / bw),
        "moe_combine": (T * k * d * 2 + T * d * 2 * 2) / bw,
    }
    lb = sum(parts.values())
    return {"workload": "MoE + sparse-attention block: 4096 tokens, hidden 4096, 64 experts top-6 + 1 shared, "
                        "expert I 1408, FP8 128x128 block-scaled weights; indexer over 32768 positions, "
                        "top 2048; MQA attention 32 heads D 128",
            "value": T / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
            "warmup": warmup,
            "roofline": {"bound": "tensor (FP8 experts) + hbm (scores, top-K)", "frac": lb / (ms / 1e3),
                         "lower_bound_ms": lb * 1e3,
                         "parts_lower_bound_us": {k2: v * 1e6 for k2, v in parts.items()},
                         "frac_is": "sum of the parts' lower bounds over the measured step time",
                         "peak_source": peaks["source"] + " (FP8 = 2 x sustained bf16)"}}


def hybrid_unit(peaks, lengths=(16384, 32768, 57344), decode_steps=256, seed=9):
    """One Mamba-2 hybrid unit (d_model 2560: four Mamba-2 mixers with 64 SSD
    heads of 64, state 128, chunk 256, and one GQA attention with 32 q / 4 kv
    heads of 80, each followed by a SiLU MLP of 6912; NVFP4 weights used
    through their exact bf16 values; vocabulary 131072) on three sequences of
    16K, 32K and 57K tokens: their prefill in steps of up to 16384 rows, then
    256 decode steps of all three.  Returns prefill and decode tokens/s with
    their rooflines (each part's lower bound over the measured time)."""
    import torch
    import synth
    from invariant_forward_bitwise_gb300.hybrid import HybridModel, new_kv

    cfg = synth.HYBRID
    W = synth.device_hybrid_weights(cfg, seed)
    S, max_rows = len(lengths), 16384
    max_pos = (max(lengths) + decode_steps + 1 + 63) // 64 * 64
    m = HybridModel(cfg, W, max_rows=max_rows, max_seqs=S, max_pos=max_pos)
    kv = new_kv(cfg, S, max_pos)
    rng = np.random.Generator(np.random.Philox(seed))
    toks = [rng.integers(0, cfg.vocab, size=L + decode_steps + 1).astype(np.int32) for L in lengths]
    for i, L in enumerate(lengths):
        kv.admit(i, L + decode_steps + 1)
        m.reset_slot(i)
    kv.sync_table()
    # prefill schedule: sequences in order, rows in steps of up to max_rows
    steps, cur = [], [0] * S
    for i, L in enumerate(lengths):
        while cur[i] < L:
            n = min(max_rows, L - cur[i])
            steps.append([(i, cur[i], n)])
            cur[i] += n

    def rows(parts, lm_all):
        seq, pos, ids, lm, tg = [], [], [], [], []
        for i, p0, n in parts:
            for p in range(p0, p0 + n):
                if lm_all:
                    lm.append(len(ids))
                    tg.append(int(toks[i][p + 1]))
                seq.append(i)
                pos.append(p)
                ids.append(int(toks[i][p]))
        return seq, pos, ids, lm, tg

    pre_rows = [rows(parts, True) for parts in steps]
    dec_rows = [rows([(i, L + k, 1) for i, L in enumerate(lengths)], True) for k in range(decode_steps)]
    # the decode step replays from a CUDA graph (fixed shape: one row per
    # sequence, attention splits sized for max_pos); it is captured on a copy
    # of the state after a warm-up step, and the state is then restored
    dspec = dict(T=S, nqblocks=S, max_rows_per_block=1, max_ctx=max_pos, T_lm=S, max_n=1)
    st = torch.cuda.current_stream()
    e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    e[0].record(st)
    for r in pre_rows:
        spec = m.load(kv, *r)
        m.step(kv, spec)
    e[1].record(st)
    torch.cuda.synchronize()
    pre_ms = e[0].elapsed_time(e[1])
    saved = {l: {k: t.clone() for k, t in x.items()} for l, x in m.mstate.items()}
    kv_saved = (kv.k.clone(), kv.v.clone())
    m.load(kv, *dec_rows[0])
    m.step(kv, dspec)                                   # warm-up: sizes every workspace
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(st)
    with torch.cuda.stream(side):
        with torch.cuda.graph(g):
            m.step(kv, dspec)
    st.wait_stream(side)
    for l, x in saved.items():
        for k, t in x.items():
            m.mstate[l][k].copy_(t)
    kv.k.copy_(kv_saved[0])
    kv.v.copy_(kv_saved[1])
    del saved, kv_saved
    torch.cuda.synchronize()
    e[1].record(st)
    for r in dec_rows:
        m.load(kv, *r)
        g.replay()
    e[2].record(st)
    torch.cuda.synchronize()
    dec_ms = e[1].elapsed_time(e[2])
    ntok = sum(lengths)
    # lower bounds.  Parameters per token: every linear layer's N*K plus the LM head
    lin = sum(2 * v[0].numel() for v in W.values() if isinstance(v, tuple))   # codes packed two per byte
    nvfp4_bytes = sum(v[0].numel() + v[1].numel() for v in W.values() if isinstance(v, tuple))
    tf, bw = peaks["bf16_tflops_sustained"] * 1e12, peaks["hbm_gbs"] * 1e9
    alu = 152 * 128 * 2 * 2.07e9            # FP32 FMA rate from unit counts and the max clock
    H, P, N, Q = cfg.ssd_heads, cfg.ssd_head_dim, cfg.state, cfg.chunk
    nm, na = cfg.pattern.count("M"), cfg.pattern.count("A")
    # SSD per token and head: intra-chunk (Q/2 rows x (N + P) MACs), state in/out (2 P N MACs)
    ssd_flops_tok = nm * H * (Q / 2 * (N + P) + 2 * P * N) * 2
    attn_flops = na * sum(4.0 * cfg.q_heads * cfg.head_dim * L * (L + 1) / 2 for L in lengths)
    parts_pre = {"gemm": 2.0 * lin * ntok / tf, "attention": attn_flops / tf,
                 "ssd": ssd_flops_tok * ntok / alu}
    lb_pre = sum(parts_pre.values())
    state_bytes = nm * S * (H * P * N * 4 * 2 + (cfg.conv_width - 1) * cfg.conv_channels * 2 * 2)
    kv_bytes = na * 2 * cfg.kv_heads * cfg.head_dim * 2 * sum(L + decode_steps / 2 for L in lengths)
    dec_bytes = nvfp4_bytes + state_bytes + kv_bytes + S * 2 * cfg.vocab * 4
    lb_dec = decode_steps * dec_bytes / bw
    return {"workload": "Mamba-2 hybrid unit, d_model 2560 (4 x Mamba-2 [64 heads x 64, state 128, chunk 256] "
                        "+ 1 x GQA [32/4 heads, D 80], each + SiLU MLP 6912), NVFP4 weights; sequences "
                        f"of {', '.join(str(L) for L in lengths)} tokens: prefill, then {decode_steps} decode steps",
            "prefill": {"value": ntok / (pre_ms / 1e3), "unit": "tokens/s", "ms": pre_ms,
                        "roofline": {"bound": "tensor (GEMMs, attention) + alu (SSD, FP32)",
                                     "frac": lb_pre / (pre_ms / 1e3),
                                     "parts_lower_bound_ms": {k: v * 1e3 for k, v in parts_pre.items()},
                                     "frac_is": "sum of the parts' lower bounds over the measured time"}},
            "decode": {"value": S * decode_steps / (dec_ms / 1e3), "unit": "tokens/s",
                       "ms_per_step": dec_ms / decode_steps,
                       "roofline": {"bound": "hbm", "achieved": decode_steps * dec_bytes / (dec_ms / 1e3) / 1e9,
                                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                    "frac": lb_dec / (dec_ms / 1e3),
                                    "algorithmic_bytes_per_step": dec_bytes,
                                    "frac_is": "NVFP4 weight bytes (4-bit codes + block scales), SSD and "
                                               "conv state read + write, KV and logits, over the measured time"}}}


if __name__ == "__main__":
    main()
