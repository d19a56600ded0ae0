"""Per-kernel micro-benchmark of libbiv on Qwen3-1.7B-shaped cases.

  python -m invariant_forward_bitwise_gb300.kernel_bench CASE [REPS]

CASE is one of attn_decode (256 sequences x 700 context, one decode row each),
attn_decode4 (the same for 4 sequences), attn_decode_fp8 (128 sequences x 4096
context on the e4m3 cache),
attn_prefill (8 sequences x 1024 tokens), gemm_prefill (M 8192, N 2048,
K 6144), gemm_qkv (M 16384, N 4096, K 2048), gemm_decode (M 64, N 2048, K 6144), lm_head (M 4096, N 151936,
K 2048, with the log-softmax gather in its epilogue), ssd_prefill (16384 tokens, 64 heads), ssd_decode (one token), topk_indexer
(4096 rows x 32768 scores, top 2048), moe_block (4096 tokens through the
64-expert FP8 block), decode_step (one decode step of the 28-layer model
at batch BIV_BENCH_BATCH, default 64, from its CUDA graph and eagerly; the
eager step runs inside cudaProfilerStart/Stop for an ncu launch list) and
fp8_serving (the FP8-KV continuous-batching workload, REPS timed
steps; the third and fourth run inside cudaProfilerStart/Stop),
moe_sparse_step (the MoE + sparse-attention block workload, REPS timed steps
and one more inside cudaProfilerStart/Stop) and
prefill_step (one 16384-row step of the 28-layer model: 16 sequences x 1024
tokens, every row producing a logprob, as in the trainer recompute; one more
step runs inside cudaProfilerStart/Stop) and hybrid_decode_step (one decode step of the
Mamba-2 hybrid unit for 3 sequences, graph-timed, then eagerly inside
cudaProfilerStart/Stop).
Each case times REPS calls with CUDA events after one warm-up call and
prints the time and the rate against the case's algorithmic bytes or FLOPs;
it is also the command that the ncu summaries in profiles/ capture.

Further cases: gemm_nvfp4 (the hybrid unit's linear layers at M = 1, 16, 64
with NVFP4 weights against the same GEMM on bf16 weights), gemm_sweep (the decoder GEMMs over decode batch sizes, weights
rotated through copies larger than L2; BIV_BENCH_MS lists the M values,
BIV_BENCH_SHAPES the GEMMs, BIV_BENCH_DEFER=1 times the GEMM kernel alone
when it leaves chunk partials to the consumer op) and gemm_prefill_layer (the
four GEMMs of a 16384-row prefill step; BIV_BENCH_MODE=fast runs the
batch-dependent comparator).  The library's own tuning switches
(BIV_GEMM_TILE_N, BIV_GEMM_FOLD, BIV_ATTN_DECODE_STAGES,
BIV_ATTN_DECODE_DSPLIT, BIV_ATTN_PREFILL_STAGES, BIV_PDL) apply here too.
"""
import math
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import synth  # noqa: E402
from invariant_forward_bitwise_gb300 import biv, build  # noqa: E402

build.build()
biv.load()
case = sys.argv[1]
reps = int(sys.argv[2]) if len(sys.argv) > 2 else 3
g = synth.rng(0)

def graph_time(fn, n):
    """Device time of one fn() when n calls run back to back from a CUDA graph
    (no host launch cost between them)."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(n):
            fn()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n

def timeit(fn, n=reps):
    fn(); torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n): fn()
    e1.record(); torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n

def fp8_codes(*shape):
    """e4m3 codes of N(0, 64) draws (clipped to the finite range), as uint8."""
    x = (torch.randn(*shape, device="cuda") * 64).clamp(-448, 448)
    return x.to(torch.float8_e4m3fn).view(torch.uint8)

def block_scales(*shape):
    return (0.02 / 64) * torch.exp2(torch.rand(*shape, device="cuda") * 2 - 1)

if case == "decode_step":
    # one decode step of the 28-layer Qwen3-1.7B shape at batch B (every
    # sequence at position 700): prefill fills the caches, then the step is
    # timed replayed from its CUDA graph, and run once eagerly inside
    # cudaProfilerStart/Stop (for ncu --profile-from-start off)
    from invariant_forward_bitwise_gb300.model import DecodeGraphs, DenseModel, PagedKV, Runner, prefill_rows
    Bn = int(os.environ.get("BIV_BENCH_BATCH", "64"))
    cfg = synth.QWEN3_1P7B
    m = DenseModel(cfg, synth.dense_weights(cfg, seed=0), max_rows=16384, max_pos=1536)
    kv = PagedKV(cfg, pages=Bn * 12 + 8, max_seqs=Bn, max_pages=24)
    ctx = 700
    for i in range(Bn):
        kv.admit(i, 768)
    kv.sync_table()
    run = Runner(m)
    toks = g.integers(0, cfg.vocab, size=(Bn, ctx + 1)).astype(np.int32)
    for i0 in range(0, Bn, 16):
        ii = list(range(i0, min(Bn, i0 + 16)))
        seqs = [synth.Sequence(toks[i], 1) for i in ii]
        rows = prefill_rows(seqs, ii, [0] * len(ii), [ctx] * len(ii), [10**9] * len(ii))
        spec = run.load_rows(kv, *rows[:5])
        m.reserve(kv, [spec])
        m.step(kv, spec)
    args = (list(range(Bn)), [ctx] * Bn, [1] * Bn, [2] * Bn)
    for use in (True, False):
        dg = DecodeGraphs(m, kv, use_graphs=use)
        for _ in range(3):
            dg.run(*args)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            dg.run(*args)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        kvb = Bn * ctx * 28 * cfg.kv_heads * cfg.head_dim * 2 * 2
        print(f"decode_step {'graph' if use else 'eager'} batch {Bn}: {ms:.3f} ms  "
              f"(weights 3.44 GB + KV {kvb/1e9:.2f} GB -> {(3.44e9 + kvb)/(ms/1e3)/1e9:.0f} GB/s)", flush=True)
    torch.cuda.cudart().cudaProfilerStart()
    dg.run(*args)
    torch.cuda.synchronize()
    torch.cuda.cudart().cudaProfilerStop()
elif case == "fp8_serving":
    # the FP8-KV continuous-batching workload (bench.py's configs entry) for
    # REPS timed steps over a pool of BIV_BENCH_POOL sequences; its third and
    # fourth model steps run inside cudaProfilerStart/Stop
    import json
    import bench
    from invariant_forward_bitwise_gb300 import model as M
    orig, count = M.DenseModel.step, [0]

    def step(self, *args, **kw):
        count[0] += 1
        if count[0] == 3:
            torch.cuda.synchronize()
            torch.cuda.cudart().cudaProfilerStart()
        r = orig(self, *args, **kw)
        if count[0] == 4:
            torch.cuda.synchronize()
            torch.cuda.cudart().cudaProfilerStop()
        return r

    M.DenseModel.step = step
    W = synth.dense_weights(synth.QWEN3_1P7B_FP8KV, seed=0)
    r = bench.fp8_serving(W, bench.load_peaks(), steps=reps,
                          pool=int(os.environ.get("BIV_BENCH_POOL", "256")))
    print(f"{case}: {r['value']:.0f} tokens/s, {r['ms_per_step']:.2f} ms per step, "
          f"roofline {r['roofline']['frac']:.3f}")
elif case == "moe_sparse_step":
    # the MoE + sparse-attention block workload (bench.py's configs entry):
    # REPS timed steps, then one more inside cudaProfilerStart/Stop
    import bench
    r = bench.moe_sparse_block(bench.load_peaks(), steps=reps, profile_step=True)
    print(f"{case}: {r['value']:.0f} tokens/s, {r['ms_per_step']*1e3:.1f} us per step, "
          f"roofline {r['roofline']['frac']:.3f}")
elif case == "prefill_step":
    from invariant_forward_bitwise_gb300.model import DenseModel, PagedKV, Runner, prefill_rows
    cfg = synth.QWEN3_1P7B
    m = DenseModel(cfg, synth.dense_weights(cfg, seed=0), max_rows=16384, max_pos=1536)
    Bn, ctx = 16, 1024
    kv = PagedKV(cfg, pages=Bn * 17 + 8, max_seqs=Bn, max_pages=24)
    for i in range(Bn):
        kv.admit(i, ctx + 8)
    kv.sync_table()
    run = Runner(m)
    toks = g.integers(0, cfg.vocab, size=(Bn, ctx + 1)).astype(np.int32)
    seqs = [synth.Sequence(toks[i], 1) for i in range(Bn)]
    rows = prefill_rows(seqs, list(range(Bn)), [0] * Bn, [ctx] * Bn, [0] * Bn)
    spec = run.load_rows(kv, *rows[:5])
    m.reserve(kv, [spec])
    m.step(kv, spec)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        m.step(kv, spec)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    fl = 2.0 * Bn * ctx * (28 * 2048 * (4096 + 2048 + 2 * 6144 + 6144) + 2048 * cfg.vocab)
    print(f"prefill_step 16 x 1024 rows: {ms:.2f} ms  ({Bn * ctx / (ms / 1e3):.0f} tokens/s, "
          f"GEMM FLOPs {fl / (ms / 1e3) / 1e12:.0f} TFLOP/s over the whole step)")
    torch.cuda.cudart().cudaProfilerStart()
    m.step(kv, spec)
    torch.cuda.synchronize()
    torch.cuda.cudart().cudaProfilerStop()
elif case == "hybrid_decode_step":
    # one decode step of the Mamba-2 hybrid unit (d 2560, NVFP4 linear layers)
    # for 3 sequences after a 1024-token prefill each; graph-timed, then one
    # eager step inside cudaProfilerStart/Stop
    from invariant_forward_bitwise_gb300.hybrid import HybridModel, new_kv
    cfg = synth.HYBRID
    W = synth.device_hybrid_weights(cfg, 9)
    S, L = 3, 1024
    m = HybridModel(cfg, W, max_rows=4096, max_seqs=S, max_pos=L + 64)
    kv = new_kv(cfg, S, L + 64)
    toks = g.integers(0, cfg.vocab, size=(S, L + 2)).astype(np.int32)
    for i in range(S):
        kv.admit(i, L + 2)
        m.reset_slot(i)
    kv.sync_table()

    def rows(ps, n):
        seq, pos, ids = [], [], []
        for i in range(S):
            for p in range(ps, ps + n):
                seq.append(i)
                pos.append(p)
                ids.append(int(toks[i][p]))
        return seq, pos, ids, list(range(len(ids))), [int(toks[s_][p + 1]) for s_, p in zip(seq, pos)]

    spec = m.load(kv, *rows(0, L))
    m.step(kv, spec)
    dspec = dict(T=S, nqblocks=S, max_rows_per_block=1, max_ctx=L + 64, T_lm=S, max_n=1)
    m.load(kv, *rows(L, 1))
    m.step(kv, dspec)
    gr = torch.cuda.CUDAGraph()
    st = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(st)
    with torch.cuda.stream(side):
        with torch.cuda.graph(gr):
            m.step(kv, dspec)
    st.wait_stream(side)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        gr.replay()
    e1.record()
    torch.cuda.synchronize()
    print(f"hybrid_decode_step graph, 3 sequences: {e0.elapsed_time(e1) / reps * 1e3:.1f} us")
    torch.cuda.cudart().cudaProfilerStart()
    m.step(kv, dspec)
    torch.cuda.synchronize()
    torch.cuda.cudart().cudaProfilerStop()
elif case == "topk_indexer":
    # 4096 query rows over a 32768-key context, top 2048 per row
    R, n, k = 4096, 32768, 2048
    scores = torch.randn(R, n, device="cuda")
    valid = torch.arange(n - R, n, dtype=torch.int32, device="cuda") + 1
    idx = torch.empty(R, k, dtype=torch.int32, device="cuda")
    ms = graph_time(lambda: biv.biv_topk(scores, valid, k, idx), reps)
    rd = R * n * 4
    print(f"topk_indexer {R}x{n} k={k}: {ms*1e3:.1f} us  scores {rd/1e6:.0f} MB -> {rd/(ms/1e3)/1e9:.0f} GB/s")
elif case == "moe_block":
    # 4096 tokens, hidden 4096, 64 routed experts top-6 + 1 shared, expert I 1408
    from invariant_forward_bitwise_gb300.moe import MoEBlock
    T, E, k, d, I = 4096, 64, 6, 4096, 1408
    wr = (torch.randn(E, d, device="cuda") * 0.05).to(torch.bfloat16)
    blk = MoEBlock(wr, fp8_codes(E, 2 * I, d), block_scales(E, 2 * I // 128, d // 128),
                   fp8_codes(E, d, I), block_scales(E, d // 128, I // 128),
                   fp8_codes(2 * I, d), block_scales(2 * I // 128, d // 128),
                   fp8_codes(d, I), block_scales(d // 128, I // 128), top_k=k, max_tokens=T)
    h = torch.randn(T, d, device="cuda").to(torch.bfloat16)
    ms = graph_time(lambda: blk.forward(h), reps)
    flops = 2.0 * T * (k + 1) * 3 * d * I
    wbytes = (E + 1) * 3 * d * I
    print(f"moe_block T={T} E={E} top{k}: {ms*1e3:.1f} us  expert FP8 {flops/(ms/1e3)/1e12:.0f} TFLOP/s  "
          f"weights {wbytes/1e6:.0f} MB")
elif case.startswith("ssd"):
    H, P, N, Q = 64, 64, 128, 256
    T = 16384 if case == "ssd_prefill" else 1
    x, dt, A, Bm, Cm, D = synth.ssd_inputs(g, T)
    st = torch.zeros(1, H, P, N, device="cuda"); bx = torch.zeros(1, Q, H, P, dtype=torch.bfloat16, device="cuda")
    bB = torch.zeros(1, Q, N, dtype=torch.bfloat16, device="cuda"); bC = torch.zeros_like(bB)
    bdt = torch.zeros(1, Q, H, device="cuda")
    xd = x.reshape(T, H * P).cuda(); dtd = torch.from_numpy(dt).cuda(); Ad = torch.from_numpy(A).cuda()
    Bd, Cd, Dd = Bm.cuda(), Cm.cuda(), torch.from_numpy(D).cuda()
    y = torch.empty(T, H * P, dtype=torch.bfloat16, device="cuda")
    keep = [torch.tensor([v], dtype=torch.int32, device="cuda") for v in (0, T, 0 if T > 1 else 200)]
    d = biv.SSDDesc()
    d.x, d.x_stride, d.dt, d.dt_stride, d.A, d.D = xd.data_ptr(), xd.stride(0), dtd.data_ptr(), dtd.stride(0), Ad.data_ptr(), Dd.data_ptr()
    d.B, d.B_stride, d.C, d.C_stride, d.y, d.y_stride = Bd.data_ptr(), Bd.stride(0), Cd.data_ptr(), Cd.stride(0), y.data_ptr(), y.stride(0)
    d.H, d.P, d.N, d.chunk, d.nseq = H, P, N, Q, 1
    d.row0, d.n, d.pos0, d.max_n = keep[0].data_ptr(), keep[1].data_ptr(), keep[2].data_ptr(), T
    d.state, d.buf_x, d.buf_B, d.buf_C, d.buf_dt = st.data_ptr(), bx.data_ptr(), bB.data_ptr(), bC.data_ptr(), bdt.data_ptr()
    ms = timeit(lambda: biv.biv_ssd_scan(d))
    print(f"{case} T={T}: {ms*1e3:.1f} us  ({T/(ms/1e3):.0f} tokens/s per sequence)")
elif case.startswith("attn"):
    Hq, Hkv, D = 16, 8, 128
    B, ctx = {"attn_decode": (256, 700), "attn_decode4": (4, 700),
              "attn_decode_fp8": (128, 4096)}.get(case, (8, 1024))
    fp8 = case.endswith("fp8")
    pages_per = (ctx + 63) // 64
    P = B * pages_per
    if fp8:
        kc = fp8_codes(P, 64, Hkv, D)
        vc = fp8_codes(P, 64, Hkv, D)
        ks = torch.rand(P, 64, Hkv, device="cuda") * 0.01
        vs = torch.rand(P, 64, Hkv, device="cuda") * 0.01
    else:
        kc = (torch.randn(P, 64, Hkv, D, device="cuda") * 0.5).to(torch.bfloat16)
        vc = (torch.randn(P, 64, Hkv, D, device="cuda") * 0.5).to(torch.bfloat16)
    bt = torch.arange(P, dtype=torch.int32, device="cuda").view(B, pages_per)
    if case.startswith("attn_decode"):
        rows = [(i, ctx - 1) for i in range(B)]
        blocks = [(i, 1) for i in range(B)]
    else:
        rows = [(i, p) for i in range(B) for p in range(ctx)]
        # blocks of 128 query vectors, as the model forms them for bf16 pages
        per = int(os.environ.get("BIV_BENCH_BLOCK_ROWS", 128 // (Hq // Hkv)))
        blocks = [(i * ctx + j, min(per, ctx - j)) for i in range(B) for j in range(0, ctx, per)]
    T = len(rows)
    q = torch.randn(T, Hq * D, device="cuda").to(torch.bfloat16)
    out = torch.empty_like(q)
    seq = torch.tensor([r[0] for r in rows], dtype=torch.int32, device="cuda")
    pos = torch.tensor([r[1] for r in rows], dtype=torch.int32, device="cuda")
    qb = torch.tensor(np.array(blocks, np.int32).ravel(), device="cuda")
    d = biv.AttnDesc()
    d.q, d.q_stride, d.out, d.out_stride = q.data_ptr(), q.stride(0), out.data_ptr(), out.stride(0)
    d.T, d.Hq, d.Hkv, d.D = T, Hq, Hkv, D
    d.row_seq, d.row_pos, d.qblocks, d.nqblocks = seq.data_ptr(), pos.data_ptr(), qb.data_ptr(), len(blocks)
    d.max_rows_per_block = max(b[1] for b in blocks)
    d.kv_dtype = biv.E4M3 if fp8 else biv.BF16
    if fp8:
        d.k_scale, d.v_scale = ks.data_ptr(), vs.data_ptr()
    d.k_cache, d.v_cache, d.block_table, d.max_pages = kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), pages_per
    d.page, d.kv_split, d.max_ctx, d.scale, d.num_pages = 64, 1024, ctx, 1 / math.sqrt(D), P
    n = biv.biv_attention_workspace(d)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    ms = graph_time(lambda: biv.biv_attention(d, ws), reps)
    kv_bytes = B * ctx * Hkv * (D * (1 if fp8 else 2) + (4 if fp8 else 0)) * 2
    flops = 4.0 * sum(p + 1 for _, p in rows) * Hq * D
    print(f"{case}: {ms*1e3:.1f} us  KV {kv_bytes/1e6:.0f} MB -> {kv_bytes/(ms/1e3)/1e9:.0f} GB/s;  {flops/(ms/1e3)/1e12:.1f} TFLOP/s")
elif case == "gemm_nvfp4":
    # the hybrid unit's linear layers at decode batch sizes: NVFP4 weights
    # (4-bit codes decoded in shared memory) against the same GEMM on bf16
    # weights; weights rotate through copies larger than L2
    shapes = {"in_proj": (8512, 2560), "out_proj": (2560, 4096), "gate_up": (13824, 2560),
              "down": (2560, 6912), "lm_head": (131072, 2560)}
    if os.environ.get("BIV_BENCH_SHAPES"):
        shapes = {k: shapes[k] for k in os.environ["BIV_BENCH_SHAPES"].split(",")}
    ms_list = [int(x) for x in os.environ.get("BIV_BENCH_MS", "1,16,64").split(",")]
    gg = synth.device_generator(1)
    for name, (N, K) in shapes.items():
        copies = max(1, -(-300_000_000 // (N * K // 2)))
        ws4 = [synth.device_nvfp4_weights(gg, N, K) for _ in range(copies)]
        wb = torch.empty(N, K, dtype=torch.bfloat16, device="cuda")
        biv.biv_nvfp4_dequant(ws4[0][0], ws4[0][1], wb)
        wbs = [wb] + [wb.clone() for _ in range(max(0, -(-300_000_000 // (N * K * 2)) - 1))]
        for M in ms_list:
            a = torch.randn(M, K, device="cuda").to(torch.bfloat16)
            c = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
            n4 = len(ws4) * max(1, 8 // len(ws4))
            t4 = graph_time(lambda: [biv.biv_gemm_nvfp4(a, *ws4[i % len(ws4)], c) for i in range(n4)], 1) / n4
            ds = [biv.gemm_desc(a, w, c) for w in wbs]
            nb = len(ds) * max(1, 8 // len(ds))
            tb = graph_time(lambda: [biv.biv_gemm(ds[i % len(ds)]) for i in range(nb)], 1) / nb
            print(f"{name:8s} M={M:3d} N={N:6d} K={K}: nvfp4 {t4*1e3:7.1f} us "
                  f"({N*K*0.5625/(t4/1e3)/1e9:5.0f} GB/s)  bf16 {tb*1e3:7.1f} us "
                  f"({N*K*2/(tb/1e3)/1e9:5.0f} GB/s)", flush=True)
        del ws4, wbs
elif case == "gemm_prefill_layer":
    # the four decoder-layer GEMMs at a 16384-row prefill step
    M = 16384
    for name, (N, K) in {"qkv": (4096, 2048), "o": (2048, 2048), "gate_up": (12288, 2048),
                         "down": (2048, 6144)}.items():
        a = torch.randn(M, K, device="cuda").to(torch.bfloat16)
        b = (torch.randn(N, K, device="cuda") * 0.02).to(torch.bfloat16)
        c = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
        mode = biv.MODE_FAST if os.environ.get("BIV_BENCH_MODE") == "fast" else biv.MODE_INVARIANT
        d = biv.gemm_desc(a, b, c, mode=mode)
        ms = graph_time(lambda: biv.biv_gemm(d), reps)
        print(f"{name:8s} M={M} N={N:6d} K={K}: {ms*1e3:8.1f} us  {2*M*N*K/(ms/1e3)/1e12:6.0f} TFLOP/s",
              flush=True)
        del a, b, c
elif case == "gemm_sweep":
    # weights rotate through enough copies to exceed L2, as in a decode step
    # where every layer's weights are cold
    # BIV_BENCH_MS: comma-separated M values; BIV_BENCH_DEFER=1 times the GEMM
    # kernel alone when it leaves chunk partials (the consumer op folds them)
    shapes = {"qkv": (4096, 2048), "o": (2048, 2048), "gate_up": (12288, 2048),
              "down": (2048, 6144), "lm_head": (151936, 2048)}
    ms_list = [int(x) for x in os.environ.get("BIV_BENCH_MS", "1,16,64,128,256,512").split(",")]
    defer = os.environ.get("BIV_BENCH_DEFER") == "1"
    if os.environ.get("BIV_BENCH_SHAPES"):
        shapes = {k: shapes[k] for k in os.environ["BIV_BENCH_SHAPES"].split(",")}
    for name, (N, K) in shapes.items():
        copies = max(1, -(-300_000_000 // (N * K * 2)))
        bs = [(torch.randn(N, K, device="cuda") * 0.02).to(torch.bfloat16) for _ in range(copies)]
        for M in ms_list:
            a = torch.randn(M, K, device="cuda").to(torch.bfloat16)
            c = torch.empty(M, N, device="cuda",
                            dtype=torch.float32 if name == "lm_head" else torch.bfloat16)
            ds = [biv.gemm_desc(a, b, c) for b in bs]
            need = biv.biv_gemm_workspace(ds[0])
            for d in ds:
                d.defer_fold = int(defer)
            ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
            n = copies * max(1, 8 // copies)
            ms = graph_time(lambda: [biv.biv_gemm(ds[i % copies], ws) for i in range(n)], 1) / n
            print(f"{name:8s} M={M:4d} N={N:6d} K={K}: {ms*1e3:8.1f} us  weights {N*K*2/(ms/1e3)/1e9:6.0f} GB/s"
                  f"  {2*M*N*K/(ms/1e3)/1e12:6.1f} TFLOP/s  {'partials' if need else 'in-CTA fold'}",
                  flush=True)
        del bs
else:
    M, N, K = {"gemm_prefill": (8192, 2048, 6144), "gemm_qkv": (16384, 4096, 2048),
               "gemm_decode": (64, 2048, 6144), "lm_head": (4096, 151936, 2048)}[case]
    a = torch.randn(M, K, device="cuda").to(torch.bfloat16)
    b = (torch.randn(N, K, device="cuda") * 0.02).to(torch.bfloat16)
    if case == "lm_head":
        # the model's LM head: the log-softmax gather in the GEMM's epilogue
        tgt = torch.randint(0, N, (M,), dtype=torch.int32, device="cuda")
        lp = torch.empty(M, device="cuda")
        ws = torch.empty(biv.biv_lm_head_logprob_workspace(M, N), dtype=torch.uint8, device="cuda")
        ms = timeit(lambda: biv.biv_lm_head_logprob(a, b, tgt, lp, ws))
    else:
        c = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
        d = biv.gemm_desc(a, b, c)
        ms = timeit(lambda: biv.biv_gemm(d))
    print(f"{case} M={M} N={N} K={K}: {ms*1e3:.1f} us  {2*M*N*K/(ms/1e3)/1e12:.0f} TFLOP/s  weights {N*K*2/(ms/1e3)/1e9:.0f} GB/s")
