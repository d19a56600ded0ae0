"""MoE + sparse-attention block: parity with the oracle and row invariance.

Integer outputs (routing, Top-K positions) must be bit-exact given the same
scores; floating outputs within 1e-2 relative; a token's output must not
depend on the other tokens of the step."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import ops
from oracle.codecs import bf16_to_f32
from oracle.model import moe_block

pytestmark = pytest.mark.gpu
REL = 1e-2


def host_f32(t):
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return bf16_to_f32(t.view(torch.int16).numpy().view(np.uint16))
    return t.float().numpy()


def bits(t):
    return t.detach().contiguous().view(torch.uint8).cpu().numpy()


def rel_err(got, ref):
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(np.asarray(got, np.float64) - ref)) / max(np.max(np.abs(ref)), 1e-30))


def _weights(g, E, d, I):
    wr = synth.normal_bf16(g, (E, d), 0.05)
    wgu, sgu = synth.fp8_block_weights(g, E, 2 * I, d)
    wd, sd = synth.fp8_block_weights(g, E, d, I)
    shgu, shsgu = synth.fp8_block_weights(g, 1, 2 * I, d)
    shd, shsd = synth.fp8_block_weights(g, 1, d, I)
    return wr, wgu, sgu, wd, sd, shgu[0], shsgu[0], shd[0], shsd[0]


@pytest.mark.parametrize("T,E,k,d,I", [(64, 8, 2, 512, 256), (200, 64, 6, 1024, 1408),
                                       (256, 64, 6, 4096, 1408)])
def test_moe_block_parity_and_invariance(T, E, k, d, I):
    """The last case is the MoE block's own width (hidden 4096, 64 experts
    top-6 + shared, expert intermediate 1408) on 256 tokens."""
    from invariant_forward_bitwise_gb300 import build
    from invariant_forward_bitwise_gb300.moe import MoEBlock
    build.build()
    g = synth.rng(T + E)
    W = _weights(g, E, d, I)
    blk = MoEBlock(*[torch.from_numpy(x) if isinstance(x, np.ndarray) else x for x in W],
                   top_k=k, max_tokens=T)
    h = synth.normal_bf16(g, (T, d))
    out = blk.forward(h.cuda()).clone()
    logits = blk.logits[:T].cpu().numpy()
    hf = h.float().numpy()
    # router logits: the FP32 GEMM within FP32 rounding of the oracle's
    assert rel_err(logits, ops.gemm(hf, W[0].float().numpy(), out="f32")) < 1e-5
    # routing: bit-exact against the oracle's rule on the same logits
    ri, rw = ops.router_topk(logits, k)
    assert np.array_equal(blk.idx[:T].cpu().numpy(), ri)
    assert np.max(np.abs(blk.w[:T].cpu().numpy() - rw)) < 1e-6
    # block output against the oracle's block (same quantisation rules),
    # routed by the same logits so that every token's experts are compared
    experts = [(synth.fp8_bits(W[1][e]), W[2][e], synth.fp8_bits(W[3][e]), W[4][e]) for e in range(E)]
    shared = (synth.fp8_bits(W[5]), W[6], synth.fp8_bits(W[7]), W[8])
    ref, oi, ow = moe_block(hf, W[0].float().numpy(), experts, shared, k, logits=logits)
    assert np.array_equal(oi, ri)
    assert rel_err(host_f32(out), ref) < REL
    # a token alone gives the bits it had inside the batch
    for t in [0, T // 2, T - 1]:
        one = blk.forward(h[t:t + 1].cuda())
        assert np.array_equal(bits(one), bits(out[t:t + 1])), t


def test_indexer_topk_sparse_attention_block():
    from invariant_forward_bitwise_gb300 import biv, build
    from invariant_forward_bitwise_gb300.moe import indexer_topk
    build.build()
    biv.load()
    g = synth.rng(99)
    ctx, T, Di, topk, Hq, D = 4096, 48, 128, 256, 32, 128
    qpos = np.arange(ctx - T, ctx).astype(np.int32)
    q_idx = synth.normal_bf16(g, (T, Di))
    k_idx = synth.normal_bf16(g, (ctx, Di))
    idx, scores = indexer_topk(q_idx.cuda(), k_idx.cuda(), torch.from_numpy(qpos).cuda(), topk)
    sc = scores.cpu().numpy()
    ref_idx = ops.topk_positions(sc, qpos + 1, topk)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)                  # bit-exact given the scores
    assert rel_err(sc[:4], ops.gemm(q_idx.float().numpy()[:4], k_idx.float().numpy(), out="f32")) < 1e-5
    # sparse attention over the selected positions (MQA: one KV head)
    pages = ctx // 64
    kv_k = synth.normal_bf16(g, (ctx, 1, D))
    kv_v = synth.normal_bf16(g, (ctx, 1, D))
    kc = kv_k.reshape(pages, 64, 1, D).cuda()
    vc = kv_v.reshape(pages, 64, 1, D).cuda()
    bt = torch.arange(pages, dtype=torch.int32, device="cuda").view(1, pages)
    q = synth.normal_bf16(g, (T, Hq * D)).cuda()
    out = torch.empty_like(q)
    seq = torch.zeros(T, dtype=torch.int32, device="cuda")
    pos = torch.from_numpy(qpos).cuda()
    qb = torch.tensor(np.stack([np.arange(T), np.ones(T)], 1).astype(np.int32).ravel(), device="cuda")
    d = biv.AttnDesc()
    d.q, d.q_stride, d.out, d.out_stride = q.data_ptr(), q.stride(0), out.data_ptr(), out.stride(0)
    d.T, d.Hq, d.Hkv, d.D = T, Hq, 1, D
    d.row_seq, d.row_pos, d.qblocks, d.nqblocks, d.max_rows_per_block = (
        seq.data_ptr(), pos.data_ptr(), qb.data_ptr(), T, 1)
    d.kv_dtype = biv.BF16
    d.k_cache, d.v_cache, d.block_table, d.max_pages, d.page = (
        kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), pages, 64)
    d.kv_split, d.max_ctx, d.scale = 128, ctx, 1 / math.sqrt(D)
    d.topk_idx, d.topk_stride, d.topk = idx.data_ptr(), idx.stride(0), topk
    n = biv.biv_attention_workspace(d)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    biv.biv_attention(d, ws)
    torch.cuda.synchronize()
    rows = [0, 17, T - 1]
    ref = ops.sparse_attention(host_f32(q).reshape(T, Hq, D)[rows], kv_k.float().numpy(),
                               kv_v.float().numpy(), ref_idx[rows], qpos[rows], 1 / math.sqrt(D))
    assert rel_err(host_f32(out).reshape(T, Hq, D)[rows], ref) < REL


def test_expert_parallel_path_equals_block_on_one_rank():
    """The expert-parallel path (ExpertRouter bookkeeping and NCCL
    all-to-alls around the same kernels) on a one-rank group gives the
    one-GPU block's bits; the two-rank exchange itself is covered over gloo
    on CPU (tests/test_ep.py)."""
    import socket
    import torch.distributed as dist
    from invariant_forward_bitwise_gb300 import build
    from invariant_forward_bitwise_gb300.ep import ExpertParallelMoE, ExpertRouter
    from invariant_forward_bitwise_gb300.moe import MoEBlock
    build.build()
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        T, E, k, d, I = 96, 16, 4, 512, 256
        g = synth.rng(4242)
        W = _weights(g, E, d, I)
        tw = [torch.from_numpy(x) if isinstance(x, np.ndarray) else x for x in W]
        blk = MoEBlock(*tw, top_k=k, max_tokens=T)
        ep = ExpertParallelMoE(ExpertRouter(E, 1, 0), *tw, top_k=k, max_tokens=T)
        h = synth.normal_bf16(g, (T, d)).cuda()
        a = blk.forward(h).clone()
        b = ep.forward(h).clone()
        torch.cuda.synchronize()
        assert np.array_equal(bits(a), bits(b))
    finally:
        dist.destroy_process_group()
