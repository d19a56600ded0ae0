"""Expert parallelism's host-side path on CPU: two gloo ranks, each owning
half of the experts.  Every rank routes its own tokens, sends each run of
expert-ordered rows to the owner of those experts, the owner regroups and
runs its experts, the outputs come back, and the token's own rank merges its
slots in FP32 in slot order ("Finish RL Training Faster", section
"让训练前向使用推理的数值").  The expert MLP here is the oracle's, so the
distributed result must equal the one-process oracle block bit for bit;
the GPU path (the same ExpertRouter around libbiv kernels) is checked
against the one-GPU block in tests/test_gpu_moe.py."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle.model as om
from oracle import ops
from oracle.codecs import bf16_round, f32_to_e4m3

F32 = np.float32


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _inputs(T=10, E=8, d=256, I=256, seed=5):
    g = np.random.default_rng(seed)
    h = bf16_round(g.standard_normal((2 * T, d)).astype(F32))          # both ranks' tokens
    wr = bf16_round((g.standard_normal((E, d)) * 0.05).astype(F32))

    def expert():
        c = lambda n, k: f32_to_e4m3(np.clip(g.standard_normal((n, k)) * 64, -448, 448).astype(F32))
        s = lambda n, k: (F32(0.02 / 64) * np.exp2(g.uniform(-1, 1, ((n + 127) // 128, (k + 127) // 128)))).astype(F32)
        return c(2 * I, d), s(2 * I, d), c(d, I), s(d, I)
    return h, wr, [expert() for _ in range(E)], expert()


def _dispatch(idx, E):
    """The deterministic dispatch's layout (rows of expert e in ascending
    (token, slot) order), restated for the host test."""
    T, k = idx.shape
    flat = idx.reshape(-1)
    order = np.lexsort((np.arange(T * k), flat))        # expert, then (t, s)
    offsets = np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]).astype(np.int32)
    src_row = np.empty(T * k, np.int32)
    src_row[order] = np.arange(T * k)
    return offsets, order.astype(np.int32), src_row


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from invariant_forward_bitwise_gb300.ep import ExpertRouter
    T, E, k = 10, 8, 3
    h_all, wr, experts, shared = _inputs(T=T, E=E)
    h = h_all[rank * T:(rank + 1) * T]
    r = ExpertRouter(E, world, rank)
    idx, w = ops.router_topk(ops.gemm(h, wr, out="f32"), k)
    offsets, perm, src_row = _dispatch(idx, E)
    aq, sa = ops.act_quant_fp8(h)
    rows_q, rows_s = aq[perm // k], sa[perm // k]                       # expert order
    rows_e = idx.reshape(-1)[perm]
    send_splits, counts = r.send_plan(offsets)
    recv_counts = r.exchange_counts(counts, "cpu")
    recv_splits = recv_counts.sum(1).astype(int).tolist()
    rq = r.exchange_rows(torch.from_numpy(rows_q), send_splits, recv_splits).numpy()
    rs = r.exchange_rows(torch.from_numpy(rows_s), send_splits, recv_splits).numpy()
    re = r.exchange_rows(torch.from_numpy(rows_e.astype(np.int64)), send_splits, recv_splits).numpy()
    loffs, lperm = ExpertRouter.receive_plan(recv_counts)
    # every grouped row belongs to the local expert its group says
    for j in range(r.epr):
        assert np.all(re[lperm[loffs[j]:loffs[j + 1]]] == rank * r.epr + j)
    y_recv = np.zeros((lperm.size, h.shape[1]), F32)
    for j in range(r.epr):
        sel = lperm[loffs[j]:loffs[j + 1]]
        if sel.size:
            wgu_c, sgu, wd_c, sd = experts[rank * r.epr + j]
            gu = ops.gemm_fp8_block(rq[sel], rs[sel], wgu_c, sgu)
            aq2, sa2 = ops.act_quant_fp8(ops.silu_mul(gu))
            y_recv[sel] = ops.gemm_fp8_block(aq2, sa2, wd_c, sd)
    y = r.exchange_rows(torch.from_numpy(y_recv), recv_splits, send_splits).numpy()
    yk = y[src_row].reshape(T, k, -1)                                  # (token, slot)
    sh = om.expert_mlp_fp8(h, *shared)
    out[rank] = (ops.moe_combine(yk, w, sh), recv_counts.sum())
    dist.destroy_process_group()


def test_two_rank_expert_parallel_equals_one_process_block():
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, _free_port(), out), nprocs=2, join=True)
    h_all, wr, experts, shared = _inputs()
    ref, _, _ = om.moe_block(h_all, wr, experts, shared, 3)
    got = np.concatenate([out[0][0], out[1][0]])
    assert np.array_equal(got, ref)
    assert out[0][1] > 0 and out[1][1] > 0            # both ranks ran experts


def test_receive_plan_groups_sources_in_rank_order():
    from invariant_forward_bitwise_gb300.ep import ExpertRouter
    counts = np.array([[2, 0, 1], [1, 3, 0]])          # [source, local expert]
    offs, perm = ExpertRouter.receive_plan(counts)
    # received rows: source 0 = [e0, e0, e2], source 1 = [e0, e1, e1, e1]
    assert offs.tolist() == [0, 3, 6, 7]
    assert perm.tolist() == [0, 1, 3, 4, 5, 6, 2]
    r = ExpertRouter(6, 2, 1)
    sends, c = r.send_plan(np.array([0, 2, 2, 5, 6, 6, 9]))
    assert sends == [5, 4] and c.tolist() == [[2, 0, 3], [1, 0, 3]]
