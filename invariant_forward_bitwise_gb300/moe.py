"""MoE block and sparse-attention indexer block, as sequences of libbiv calls.

"Finish RL Training Faster" (section "让训练前向使用推理的数值") asks the MoE
path to unify quantisation rounding, per-row computation and the merge of
expert outputs, and sparse attention to resolve Top-K ties one fixed way and
lay the selection out in position order.  Here every token row is routed,
quantised (1x128 e4m3 groups), multiplied by FP8 128x128 block-scaled expert
weights in grouped GEMMs, and merged in FP32 in fixed slot order; nothing a
row computes depends on which other tokens share the step, because the
grouped GEMM's per-row result does not depend on the row's place in its
expert group.
"""
from __future__ import annotations

import math
from typing import Optional

import torch

from . import biv


class MoEBlock:
    """Routed experts (top-k of E) + one shared expert, FP8 weights.

    w_router bf16 [E, d]; wgu codes [E, 2I, d] (uint8) with scales
    [E, 2I/128, d/128]; wd codes [E, d, I] with scales [E, d/128, I/128]; the
    shared expert's four tensors have no leading E."""

    def __init__(self, w_router, wgu, sgu, wd, sd, sh_gu, sh_sgu, sh_d, sh_sd, top_k: int,
                 max_tokens: int, device="cuda"):
        biv.load()
        dv = lambda t: t.to(device).contiguous()
        self.wr = dv(w_router)
        self.E, self.d = self.wr.shape
        self.k = top_k
        self.I2 = wgu.shape[1]
        self.I = self.I2 // 2
        self.wgu = dv(wgu.reshape(self.E * self.I2, self.d).view(torch.uint8))
        self.sgu = dv(sgu)
        self.wd = dv(wd.reshape(self.E * self.d, self.I).view(torch.uint8))
        self.sd = dv(sd)
        self.sh_gu, self.sh_sgu = dv(sh_gu.view(torch.uint8)), dv(sh_sgu)
        self.sh_d, self.sh_sd = dv(sh_d.view(torch.uint8)), dv(sh_sd)
        T, R = max_tokens, max_tokens * top_k
        d, I, I2 = self.d, self.I, self.I2
        u8, f32, i32, bf = (dict(dtype=t, device=device) for t in
                            (torch.uint8, torch.float32, torch.int32, torch.bfloat16))
        self.logits = torch.empty(T, self.E, **f32)
        self.idx = torch.empty(T, top_k, **i32)
        self.w = torch.empty(T, top_k, **f32)
        self.offs = torch.empty(self.E + 1, **i32)
        self.perm = torch.empty(R, **i32)
        self.src = torch.empty(R, **i32)
        self.hq = torch.empty(T, d, **u8)
        self.hs = torch.empty(T, (d + 127) // 128, **f32)
        self.aq = torch.empty(R, d, **u8)
        self.as_ = torch.empty(R, (d + 127) // 128, **f32)
        self.gu = torch.empty(R, I2, **bf)
        self.actq = torch.empty(R, I, **u8)
        self.acts = torch.empty(R, (I + 127) // 128, **f32)
        self.y = torch.empty(R, d, **bf)
        self.sgu_out = torch.empty(T, I2, **bf)
        self.sactq = torch.empty(T, I, **u8)
        self.sacts = torch.empty(T, (I + 127) // 128, **f32)
        self.shared = torch.empty(T, d, **bf)
        self.out = torch.empty(T, d, **bf)

    def forward(self, h: torch.Tensor) -> torch.Tensor:
        """h bf16 [T, d] -> bf16 [T, d] (view of an internal buffer)."""
        T, k, E = h.shape[0], self.k, self.E
        R = T * k
        biv.biv_gemm(biv.gemm_desc(h, self.wr, self.logits[:T]))
        biv.biv_router_topk(self.logits[:T], k, self.idx[:T], self.w[:T])
        biv.biv_moe_dispatch(self.idx[:T], E, self.offs, self.perm[:R], self.src[:R])
        biv.biv_act_quant_fp8(h, self.hq[:T], self.hs[:T])
        biv.biv_gather_rows(self.hq[:T], self.perm[:R], k, R, self.aq)
        biv.biv_gather_rows(self.hs[:T], self.perm[:R], k, R, self.as_)
        # routed experts: grouped FP8 GEMMs over the dispatched rows
        biv.biv_gemm(biv.gemm_desc(self.aq[:R], self.wgu, self.gu[:R], sa=self.as_[:R], sb=self.sgu,
                                   group_offsets=self.offs, groups=E, M=R))
        biv.biv_silu_mul_quant_fp8(self.gu[:R], self.actq[:R], self.acts[:R])
        biv.biv_gemm(biv.gemm_desc(self.actq[:R], self.wd, self.y[:R], sa=self.acts[:R], sb=self.sd,
                                   group_offsets=self.offs, groups=E, M=R))
        # shared expert on every token
        biv.biv_gemm(biv.gemm_desc(self.hq[:T], self.sh_gu, self.sgu_out[:T], sa=self.hs[:T], sb=self.sh_sgu))
        biv.biv_silu_mul_quant_fp8(self.sgu_out[:T], self.sactq[:T], self.sacts[:T])
        biv.biv_gemm(biv.gemm_desc(self.sactq[:T], self.sh_d, self.shared[:T], sa=self.sacts[:T], sb=self.sh_sd))
        # FP32 fixed-slot merge
        biv.biv_moe_combine(self.y, self.src[:R], self.w[:T], self.shared[:T], self.out[:T])
        return self.out[:T]


def indexer_topk(q_idx: torch.Tensor, k_idx: torch.Tensor, q_pos: torch.Tensor, topk: int,
                 scores: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Indexer scores q_idx . k_idx^T (FP32 GEMM) and the Top-K positions per
    query (keys past the query's position excluded through valid_len), in
    ascending order.  q_idx bf16 [T, Di], k_idx bf16 [ctx, Di]."""
    T, ctx = q_idx.shape[0], k_idx.shape[0]
    if scores is None:
        scores = torch.empty(T, ctx, dtype=torch.float32, device=q_idx.device)
    biv.biv_gemm(biv.gemm_desc(q_idx, k_idx, scores))
    idx = torch.empty(T, topk, dtype=torch.int32, device=q_idx.device)
    biv.biv_topk(scores, (q_pos + 1).to(torch.int32), topk, idx)
    return idx, scores
