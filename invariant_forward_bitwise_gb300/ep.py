"""Expert parallelism for the MoE block: experts split over ranks, each token's
expert outputs merged on the token's own GPU in FP32 fixed slot order.

"Finish RL Training Faster" (section "让训练前向使用推理的数值") keeps the
expert outputs' merge on the token's GPU, in FP32 and in slot order, so that
where an expert runs cannot change a bit.  Rank r owns experts
[r * E/W, (r+1) * E/W).  A step:

  1. router logits, Top-k and the deterministic dispatch (rows in expert
     order, offsets [E+1]) on the token's rank, as in the one-GPU block;
  2. per-token FP8 activation codes and scales gathered into that order: the
     rows bound for rank r are one contiguous run;
  3. an all-to-all sends each run, with its per-expert row counts, to the
     rank that owns those experts;
  4. the owner regroups what it received by local expert (sources in rank
     order, rows in the order they came), runs the grouped FP8 expert GEMMs,
     and puts the outputs back in received order;
  5. a second all-to-all returns every output row to its sender, which
     combines its tokens' slots in FP32 in slot order with the shared expert.

A grouped GEMM row's result does not depend on which other rows share its
group or where it sits, so every output bit equals the one-GPU block's.
Collectives are torch.distributed all-to-alls (NCCL between GPUs, gloo on
CPU for the host-side tests); nothing is multicast.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np
import torch
import torch.distributed as dist

from . import biv


class ExpertRouter:
    """The host-side bookkeeping of expert parallelism over ``world`` ranks
    (experts split evenly, contiguous ranges)."""

    def __init__(self, E: int, world: int, rank: int, group=None):
        if E % world:
            raise ValueError("experts must split evenly over the ranks")
        self.E, self.world, self.rank, self.group = E, world, rank, group
        self.epr = E // world

    def owner(self, e: int) -> int:
        return e // self.epr

    def send_plan(self, offsets: np.ndarray) -> Tuple[List[int], np.ndarray]:
        """From the dispatch offsets [E+1] (rows in expert order): rows sent to
        each rank, and the per-expert counts [W, epr] of those runs."""
        counts = np.diff(np.asarray(offsets, np.int64)).reshape(self.world, self.epr)
        return counts.sum(1).astype(int).tolist(), counts

    def exchange_counts(self, counts: np.ndarray, device) -> np.ndarray:
        """All-to-all of the per-expert counts: returns [W (source), epr]."""
        send = torch.as_tensor(np.ascontiguousarray(counts, np.int64), device=device).reshape(-1)
        recv = torch.empty_like(send)
        dist.all_to_all_single(recv, send, group=self.group)
        return recv.cpu().numpy().reshape(self.world, self.epr)

    def exchange_rows(self, t: torch.Tensor, send_splits: Sequence[int],
                      recv_splits: Sequence[int]) -> torch.Tensor:
        """All-to-all of rows: run r of ``t`` goes to rank r; returns the
        received rows, sources in rank order."""
        out = torch.empty((int(sum(recv_splits)),) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
        dist.all_to_all_single(out, t.contiguous(), output_split_sizes=list(recv_splits),
                               input_split_sizes=list(send_splits), group=self.group)
        return out

    @staticmethod
    def receive_plan(recv_counts: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
        """Regrouping of received rows by local expert.  recv_counts [W, epr]:
        rows from source s are its experts' runs, expert-major.  Returns the
        local offsets [epr+1] and perm: grouped row i is received row perm[i]
        (expert j's rows: source 0's first, then source 1's, ...)."""
        W, epr = recv_counts.shape
        src_base = np.concatenate([[0], np.cumsum(recv_counts.sum(1))])[:-1]
        within = np.concatenate([np.zeros((W, 1), np.int64), np.cumsum(recv_counts, 1)[:, :-1]], 1)
        perm, offsets = [], [0]
        for j in range(epr):
            for s in range(W):
                start = src_base[s] + within[s, j]
                perm.extend(range(int(start), int(start + recv_counts[s, j])))
            offsets.append(len(perm))
        return np.asarray(offsets, np.int32), np.asarray(perm, np.int32)


class ExpertParallelMoE:
    """The MoE block with this rank's experts only (FP8 e4m3 weights with
    128x128 scales, as MoEBlock) and the shared expert on every rank."""

    def __init__(self, router: ExpertRouter, w_router, wgu, sgu, wd, sd, sh_gu, sh_sgu, sh_d, sh_sd,
                 top_k: int, max_tokens: int, device="cuda"):
        """wgu/sgu/wd/sd: this rank's experts only, [epr, ...] as in MoEBlock."""
        biv.load()
        self.r = router
        dv = lambda t: t.to(device).contiguous()
        self.wr = dv(w_router)
        self.E, self.d = self.wr.shape
        if self.E != router.E:
            raise ValueError("router and weights disagree on the expert count")
        self.k, self.epr = top_k, router.epr
        self.I2 = wgu.shape[1]
        self.I = self.I2 // 2
        self.wgu = dv(wgu.reshape(self.epr * self.I2, self.d).view(torch.uint8))
        self.sgu = dv(sgu)
        self.wd = dv(wd.reshape(self.epr * self.d, self.I).view(torch.uint8))
        self.sd = dv(sd)
        self.sh_gu, self.sh_sgu = dv(sh_gu.view(torch.uint8)), dv(sh_sgu)
        self.sh_d, self.sh_sd = dv(sh_d.view(torch.uint8)), dv(sh_sd)
        T, R, d, I, I2 = max_tokens, max_tokens * top_k, self.d, self.I, self.I2
        kb = lambda n: (n + 127) // 128
        u8, f32, i32, bf = (dict(dtype=t, device=device) for t in
                            (torch.uint8, torch.float32, torch.int32, torch.bfloat16))
        self.logits = torch.empty(T, self.E, **f32)
        self.idx = torch.empty(T, top_k, **i32)
        self.w = torch.empty(T, top_k, **f32)
        self.offs = torch.empty(self.E + 1, **i32)
        self.perm = torch.empty(R, **i32)
        self.src = torch.empty(R, **i32)
        self.hq = torch.empty(T, d, **u8)
        self.hs = torch.empty(T, kb(d), **f32)
        self.aq = torch.empty(R, d, **u8)
        self.as_ = torch.empty(R, kb(d), **f32)
        self.sgu_out = torch.empty(T, I2, **bf)
        self.sactq = torch.empty(T, I, **u8)
        self.sacts = torch.empty(T, kb(I), **f32)
        self.shared = torch.empty(T, d, **bf)
        self.out = torch.empty(T, d, **bf)

    def _experts(self, aq, as_, offsets_dev, n):
        """Grouped FP8 MLPs of the local experts over n grouped rows."""
        dev = aq.device
        gu = torch.empty(n, self.I2, dtype=torch.bfloat16, device=dev)
        actq = torch.empty(n, self.I, dtype=torch.uint8, device=dev)
        acts = torch.empty(n, (self.I + 127) // 128, dtype=torch.float32, device=dev)
        y = torch.empty(n, self.d, dtype=torch.bfloat16, device=dev)
        if n:
            biv.biv_gemm(biv.gemm_desc(aq, self.wgu, gu, sa=as_, sb=self.sgu, group_offsets=offsets_dev,
                                       groups=self.epr, M=n))
            biv.biv_silu_mul_quant_fp8(gu, actq, acts)
            biv.biv_gemm(biv.gemm_desc(actq, self.wd, y, sa=acts, sb=self.sd, group_offsets=offsets_dev,
                                       groups=self.epr, M=n))
        return y

    def forward(self, h: torch.Tensor) -> torch.Tensor:
        """h bf16 [T, d] (this rank's tokens) -> bf16 [T, d]."""
        T, k, E, dev = h.shape[0], self.k, self.E, h.device
        R = T * k
        biv.biv_gemm(biv.gemm_desc(h, self.wr, self.logits[:T]))
        biv.biv_router_topk(self.logits[:T], k, self.idx[:T], self.w[:T])
        biv.biv_moe_dispatch(self.idx[:T], E, self.offs, self.perm[:R], self.src[:R])
        biv.biv_act_quant_fp8(h, self.hq[:T], self.hs[:T])
        biv.biv_gather_rows(self.hq[:T], self.perm[:R], k, R, self.aq)
        biv.biv_gather_rows(self.hs[:T], self.perm[:R], k, R, self.as_)
        # send each owner its run of rows with the run's per-expert counts
        send_splits, counts = self.r.send_plan(self.offs.cpu().numpy())
        recv_counts = self.r.exchange_counts(counts, dev)
        recv_splits = recv_counts.sum(1).astype(int).tolist()
        rq = self.r.exchange_rows(self.aq[:R], send_splits, recv_splits)
        rs = self.r.exchange_rows(self.as_[:R], send_splits, recv_splits)
        # regroup by local expert, run the experts, back to received order
        loffs, lperm = self.r.receive_plan(recv_counts)
        n = int(lperm.size)
        loffs_d = torch.from_numpy(loffs).to(dev)
        lperm_d = torch.from_numpy(lperm).to(dev)
        gq = torch.empty(n, self.d, dtype=torch.uint8, device=dev)
        gs = torch.empty(n, rs.shape[1], dtype=torch.float32, device=dev)
        y_recv = torch.empty(n, self.d, dtype=torch.bfloat16, device=dev)
        if n:
            biv.biv_gather_rows(rq, lperm_d, 1, n, gq)
            biv.biv_gather_rows(rs, lperm_d, 1, n, gs)
        y_grp = self._experts(gq, gs, loffs_d, n)
        if n:
            inv = np.empty_like(lperm)
            inv[lperm] = np.arange(n, dtype=np.int32)
            biv.biv_gather_rows(y_grp, torch.from_numpy(inv).to(dev), 1, n, y_recv)
        # outputs back to their senders, in the order they were sent
        y = self.r.exchange_rows(y_recv, recv_splits, send_splits)
        # shared expert on this rank's tokens, then the FP32 fixed-slot merge
        biv.biv_gemm(biv.gemm_desc(self.hq[:T], self.sh_gu, self.sgu_out[:T], sa=self.hs[:T], sb=self.sh_sgu))
        biv.biv_silu_mul_quant_fp8(self.sgu_out[:T], self.sactq[:T], self.sacts[:T])
        biv.biv_gemm(biv.gemm_desc(self.sactq[:T], self.sh_d, self.shared[:T], sa=self.sacts[:T], sb=self.sh_sd))
        biv.biv_moe_combine(y, self.src[:R], self.w[:T], self.shared[:T], self.out[:T])
        return self.out[:T]
