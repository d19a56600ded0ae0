"""The batch-invariant decoder forward, as a sequence of libbiv calls.

One code path turns rows (token, sequence, absolute position) into next-token
logprobs; rollout (prompt prefill, then teacher-forced decode) and trainer
recompute (full-sequence prefill into a private KV cache) both run it, which
is how "Finish RL Training Faster" (section "让训练前向使用推理的数值") makes
the training forward use the inference numerics.  Every row's result depends
only on its own prefix and the weights: the batch it shares a step with, the
chunking of the prefill and eager vs CUDA-Graph execution do not enter any
reduction.

PyTorch is used for device memory, streams and CUDA-Graph capture only; all
arithmetic runs in libbiv's kernels.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from . import biv

PAGE = 64


# ------------------------------------------------------------------ cache --
class PagedKV:
    """Per-layer paged KV cache ([pages, 64, Hkv, D] per layer), bf16 or FP8
    e4m3 codes with one FP32 scale per (token, kv head), plus a host-side free
    list of pages and a device block table [max_seqs, max_pages]."""

    def __init__(self, cfg, pages: int, max_seqs: int, max_pages: int, device="cuda"):
        self.cfg, self.pages, self.fp8 = cfg, pages, cfg.kv_fp8
        L, Hkv, D = cfg.layers, cfg.kv_heads, cfg.head_dim
        shape = (L, pages, PAGE, Hkv, D)
        if self.fp8:
            self.k = torch.zeros(shape, dtype=torch.uint8, device=device)
            self.v = torch.zeros(shape, dtype=torch.uint8, device=device)
            self.ks = torch.zeros(shape[:4], dtype=torch.float32, device=device)
            self.vs = torch.zeros(shape[:4], dtype=torch.float32, device=device)
        else:
            self.k = torch.zeros(shape, dtype=torch.bfloat16, device=device)
            self.v = torch.zeros(shape, dtype=torch.bfloat16, device=device)
            self.ks = self.vs = None
        self.max_pages = max_pages
        self.block_table = torch.zeros(max_seqs, max_pages, dtype=torch.int32, device=device)
        self.bt_host = np.zeros((max_seqs, max_pages), np.int32)
        self.free = list(range(pages - 1, -1, -1))
        self.owned: Dict[int, List[int]] = {}

    @staticmethod
    def bytes_per_page(cfg) -> int:
        per_tok = cfg.kv_heads * cfg.head_dim * (1 if cfg.kv_fp8 else 2) + (cfg.kv_heads * 4 if cfg.kv_fp8 else 0)
        return 2 * cfg.layers * PAGE * per_tok

    def admit(self, slot: int, length: int):
        """Give sequence slot `slot` pages for `length` tokens."""
        n = (length + PAGE - 1) // PAGE
        if n > self.max_pages or n > len(self.free):
            raise RuntimeError("KV cache out of pages")
        pages = [self.free.pop() for _ in range(n)]
        self.owned[slot] = pages
        self.bt_host[slot, :] = 0
        self.bt_host[slot, :n] = pages

    def release(self, slot: int):
        self.free.extend(reversed(self.owned.pop(slot, [])))

    def sync_table(self):
        self.block_table.copy_(torch.from_numpy(self.bt_host), non_blocking=False)

    def slots(self, seq_slot: np.ndarray, pos: np.ndarray) -> np.ndarray:
        return (self.bt_host[seq_slot, pos // PAGE].astype(np.int64) * PAGE + pos % PAGE)


# ------------------------------------------------------------------ model --
@dataclass
class StepSpec:
    """Host-side shape of one forward step (what a captured graph bakes in)."""
    T: int                  # rows
    nqblocks: int
    max_rows_per_block: int
    max_ctx: int            # bound on row position + 1
    T_lm: int               # rows that produce a logprob
    attn_flops: float = 0.0  # algorithmic attention FLOPs of the step (4 * sum(ctx) * Hq * D)
    # a step that mixes prefill blocks with single-vector (decode) blocks holds
    # the multi-row blocks first: the first n_multi blocks (max_rows_per_block
    # rows at most) and the rest (max_rows_single at most) go to attention as
    # two calls, so that decode rows run the decode-shaped CTA
    n_multi: int = 0
    max_rows_single: int = 1


class DenseModel:
    """Device weights, rope table and static activation buffers for up to
    ``max_rows`` rows per step."""

    def __init__(self, cfg, weights: Dict[str, torch.Tensor], max_rows: int, max_pos: int,
                 mode: int = biv.MODE_INVARIANT, lm_chunk: int = 16384, device="cuda"):
        biv.load()
        self.cfg, self.mode, self.max_rows, self.max_pos = cfg, mode, max_rows, max_pos
        self.lm_chunk = min(lm_chunk, max_rows)
        self.W = {k: v.to(device).contiguous() for k, v in weights.items()}
        if cfg.tied and weights["lm_head"] is weights["embed"]:
            self.W["lm_head"] = self.W["embed"]
        D = cfg.head_dim
        self.rope = torch.empty(2 * max_pos * (D // 2), dtype=torch.float32, device=device)
        biv.biv_rope_table(cfg.rope_theta, D, max_pos, self.rope)
        T, d, I = max_rows, cfg.hidden, cfg.intermediate
        bf = dict(dtype=torch.bfloat16, device=device)
        self.r = torch.empty(T, d, **bf)
        self.y = torch.empty(T, d, **bf)
        self.qkv = torch.empty(T, cfg.qkv_width, **bf)
        self.o = torch.empty(T, cfg.q_heads * D, **bf)
        self.a = torch.empty(T, d, **bf)
        self.gu = torch.empty(T, 2 * I, **bf)
        self.act = torch.empty(T, I, **bf)
        self.ylm = torch.empty(T, d, **bf)
        # LM head + log-softmax: per-row (max, sum exp) pairs of 128-logit groups
        self.lse_ws = torch.empty(biv.biv_lm_head_logprob_workspace(self.lm_chunk, cfg.vocab),
                                  dtype=torch.uint8, device=device)
        self.lp = torch.empty(T, dtype=torch.float32, device=device)
        # step inputs (static, so that captured graphs read fresh values)
        i32 = dict(dtype=torch.int32, device=device)
        self.ids = torch.zeros(T, **i32)
        self.row_seq = torch.zeros(T, **i32)
        self.row_pos = torch.zeros(T, **i32)
        self.slot = torch.full((T,), -1, dtype=torch.int64, device=device)
        self.qblocks = torch.zeros(T, 2, **i32)
        self.lm_rows = torch.zeros(T, **i32)
        self.targets = torch.zeros(T, **i32)
        self.ws = torch.empty(16, dtype=torch.uint8, device=device)     # attention partials
        self.gws = torch.empty(256, dtype=torch.uint8, device=device)   # GEMM chunk partials
        self._old_ws: List[torch.Tensor] = []
        self.audit: Optional[list] = None  # when a list: residual stream copied after each layer
        self.launches = 0        # libbiv launches of the last step()
        self.kernel_timer = None  # optional event brackets around GEMM/attention
        self.h2d_bytes = 0       # host->device bytes of step inputs copied so far

    # -- helpers --------------------------------------------------------------
    def _timer(self):
        t = self.kernel_timer
        if t is None or torch.cuda.is_current_stream_capturing():
            return None
        return t

    def _gemm(self, A, Bw, Cout, M, stream=None, defer=False):
        """Cout = A . Bw^T.  With defer=True a plan that leaves chunk partials
        skips its fold kernel and returns the partials for the consumer op
        (Cout is then not written); otherwise returns None."""
        d = biv.gemm_desc(A, Bw, Cout, mode=self.mode, M=M)
        need = biv.biv_gemm_workspace(d)
        if need > self.gws.numel():
            raise RuntimeError(f"GEMM workspace too small ({need} > {self.gws.numel()}); call reserve()")
        d.defer_fold = 1 if (defer and need) else 0
        t = self._timer()
        tok = t.bracket("gemm_bf16", 2.0 * M * d.N * d.K, "flop") if t else None
        biv.biv_gemm(d, self.gws, stream=stream)
        if tok:
            t.close(tok)
        self.launches += 2 if (need and not d.defer_fold) else 1   # partials add the fold kernel
        return biv.biv_gemm_partials(d, self.gws) if d.defer_fold else None

    @staticmethod
    def _add_rmsnorm(x, xp, r, w, y, T, eps, st):
        """Residual add + RMSNorm of x[:T] (a GEMM output, or its chunk partials xp)."""
        if xp is not None:
            biv.biv_add_rmsnorm_partials(xp, r, w, y, T, eps, stream=st)
        else:
            biv.biv_add_rmsnorm(x[:T], r, w, y, eps, stream=st)

    def _attn_descs(self, kv: PagedKV, layer: int, spec: StepSpec, qblocks=None):
        """Attention call(s) of a layer: one, or two when the step mixes
        prefill blocks with decode blocks (see StepSpec)."""
        qb = self.qblocks if qblocks is None else qblocks
        if 0 < spec.n_multi < spec.nqblocks:
            return [self._attn_desc(kv, layer, spec, qb.data_ptr(), spec.n_multi,
                                    spec.max_rows_per_block),
                    self._attn_desc(kv, layer, spec, qb.data_ptr() + 8 * spec.n_multi,
                                    spec.nqblocks - spec.n_multi, spec.max_rows_single)]
        return [self._attn_desc(kv, layer, spec, qb.data_ptr(), spec.nqblocks,
                                spec.max_rows_per_block)]

    def _attn_desc(self, kv: PagedKV, layer: int, spec: StepSpec, qblocks_ptr: int, nqblocks: int,
                   max_rows: int):
        cfg = self.cfg
        d = biv.AttnDesc()
        d.q, d.q_stride = self.qkv.data_ptr(), self.qkv.stride(0)
        d.out, d.out_stride = self.o.data_ptr(), self.o.stride(0)
        d.T, d.Hq, d.Hkv, d.D = spec.T, cfg.q_heads, cfg.kv_heads, cfg.head_dim
        d.row_seq, d.row_pos = self.row_seq.data_ptr(), self.row_pos.data_ptr()
        d.qblocks = qblocks_ptr
        d.nqblocks = nqblocks
        d.max_rows_per_block = max_rows
        d.kv_dtype = biv.E4M3 if kv.fp8 else biv.BF16
        d.k_cache, d.v_cache = kv.k[layer].data_ptr(), kv.v[layer].data_ptr()
        if kv.fp8:
            d.k_scale, d.v_scale = kv.ks[layer].data_ptr(), kv.vs[layer].data_ptr()
        d.block_table, d.max_pages = kv.block_table.data_ptr(), kv.max_pages
        d.page, d.kv_split, d.max_ctx = PAGE, cfg.kv_split, spec.max_ctx
        d.scale = 1.0 / math.sqrt(cfg.head_dim)
        d.mode = self.mode
        d.num_pages = kv.pages
        return d

    def reserve(self, kv: PagedKV, specs: Sequence[StepSpec]):
        """Size the attention and GEMM workspaces for the given step shapes
        (before capture)."""
        need, gneed = 16, 256
        cfg = self.cfg
        for s in specs:
            for ad in self._attn_descs(kv, 0, s):
                need = max(need, biv.biv_attention_workspace(ad))
            for (N, K) in [(cfg.qkv_width, cfg.hidden), (cfg.hidden, cfg.q_heads * cfg.head_dim),
                           (2 * cfg.intermediate, cfg.hidden), (cfg.hidden, cfg.intermediate)]:
                d = biv.GemmDesc()
                d.M, d.N, d.K = s.T, N, K
                d.a_dtype = d.b_dtype = d.c_dtype = biv.BF16
                d.A = d.B = d.C = self.y.data_ptr()
                d.lda = d.ldb = K
                d.ldc = N
                d.mode = self.mode
                gneed = max(gneed, biv.biv_gemm_workspace(d))
        # captured graphs keep the address they saw: never free a workspace
        if need > self.ws.numel():
            self._old_ws.append(self.ws)
            self.ws = torch.empty(need, dtype=torch.uint8, device=self.ws.device)
        if gneed > self.gws.numel():
            self._old_ws.append(self.gws)
            self.gws = torch.empty(gneed, dtype=torch.uint8, device=self.gws.device)

    # -- the forward ------------------------------------------------------------
    def step(self, kv: PagedKV, spec: StepSpec, qblocks=None, lm_rows=None):
        """Rows [0, spec.T) of the static inputs through the model; logprobs of
        targets[0, T_lm) for rows lm_rows[0, T_lm) land in lp[0, T_lm).
        ``qblocks`` / ``lm_rows`` default to the shared step buffers; captured
        decode graphs pass constant buffers of their own."""
        cfg, W, T = self.cfg, self.W, spec.T
        st = torch.cuda.current_stream()  # fetched once: every call below runs on it
        qblocks = self.qblocks if qblocks is None else qblocks
        lm_rows = self.lm_rows if lm_rows is None else lm_rows
        Hq, Hkv, D = cfg.q_heads, cfg.kv_heads, cfg.head_dim
        eps = cfg.eps
        r, y = self.r[:T], self.y[:T]
        self.launches = 0
        biv.biv_embed(self.ids[:T], W["embed"], r, stream=st)
        biv.biv_add_rmsnorm(r, None, W["l0.attn_norm"], y, eps, stream=st)
        self.launches += 2
        # GEMMs whose plan leaves chunk partials hand them straight to the next
        # op (the same bits, one launch fewer); the per-op audit wants every
        # GEMM output stored, so it keeps the folds
        defer = self.audit is None
        for l in range(cfg.layers):
            p = f"l{l}."
            qp = self._gemm(y, W[p + "wqkv"], self.qkv, T, st, defer=defer)
            # QK-norm + RoPE and the k/v cache store in one pass
            biv.biv_qkv_finalize(self.qkv, T, Hq, Hkv, D, W.get(p + "q_norm") if cfg.qk_norm else None,
                                 W.get(p + "k_norm") if cfg.qk_norm else None, self.rope, self.max_pos,
                                 self.row_pos, eps, self.slot, biv.E4M3 if kv.fp8 else biv.BF16,
                                 kv.k[l], kv.v[l], kv.ks[l] if kv.fp8 else None,
                                 kv.vs[l] if kv.fp8 else None, partials=qp, stream=st)
            t = self._timer()
            tok = t.bracket("attention_prefill", spec.attn_flops, "flop") if t and spec.attn_flops else None
            attn_launches = 0
            for ad in self._attn_descs(kv, l, spec, qblocks):
                need = biv.biv_attention_workspace(ad)
                biv.biv_attention(ad, self.ws if need else None, stream=st)
                attn_launches += 1 + (1 if need else 0)   # + the split merge
            if tok:
                t.close(tok)
            op = self._gemm(self.o, W[p + "wo"], self.a, T, st, defer=defer)
            aud = self.audit is not None and not torch.cuda.is_current_stream_capturing()
            if aud:
                self.audit.append(("qkv", l, self.qkv[:T].clone()))
                self.audit.append(("attn_o", l, self.o[:T].clone()))
                self.audit.append(("attn_proj", l, self.a[:T].clone()))
            self._add_rmsnorm(self.a, op, r, W[p + "mlp_norm"], y, T, eps, st)
            gp = self._gemm(y, W[p + "wgu"], self.gu, T, st, defer=defer)
            if gp is not None:
                biv.biv_silu_mul_partials(gp, self.act[:T], T, stream=st)
            else:
                biv.biv_silu_mul(self.gu[:T], self.act[:T], stream=st)
            dp = self._gemm(self.act, W[p + "wd"], self.a, T, st, defer=defer)
            if self.audit is not None and not torch.cuda.is_current_stream_capturing():
                self.audit.append(("mlp_out", l, self.a[:T].clone()))
            nxt = W[f"l{l + 1}.attn_norm"] if l + 1 < cfg.layers else W["final_norm"]
            self._add_rmsnorm(self.a, dp, r, nxt, y, T, eps, st)
            # qkv finalize, attention (+ split merge), 2 x add_rmsnorm, silu_mul
            self.launches += 4 + attn_launches
            if self.audit is not None and not torch.cuda.is_current_stream_capturing():
                self.audit.append(("layer", l, r.clone()))
        # LM head + logprob over the rows that produce a logprob
        Tl = spec.T_lm
        if Tl == 0:
            return
        biv.biv_gather_rows(y, lm_rows, 1, Tl, self.ylm, stream=st)
        self.launches += 1
        for c0 in range(0, Tl, self.lm_chunk):
            n = min(self.lm_chunk, Tl - c0)
            t = self._timer()
            tok = t.bracket("gemm_bf16", 2.0 * n * cfg.vocab * cfg.hidden, "flop") if t else None
            biv.biv_lm_head_logprob(self.ylm[c0:c0 + n], W["lm_head"], self.targets[c0:c0 + n],
                                    self.lp[c0:c0 + n], self.lse_ws, M=n, mode=self.mode, stream=st)
            if tok:
                t.close(tok)
            self.launches += 2
        t = self._timer()
        if t:
            t.launches += self.launches


# ------------------------------------------------------------- batching ----
def qblocks_for(row_seq: np.ndarray, per: int) -> np.ndarray:
    """Blocks of up to `per` consecutive rows that share a sequence."""
    out = []
    i, T = 0, row_seq.shape[0]
    while i < T:
        j = i
        while j < T and j - i < per and row_seq[j] == row_seq[i]:
            j += 1
        out.append((i, j - i))
        i = j
    return np.array(out, np.int32).reshape(-1, 2)


def split_blocks(qb: np.ndarray, G: int):
    """Order query blocks for attention: returns (blocks, n_multi).  When a
    step holds both multi-row blocks (more than 16 query vectors) and at least
    as many single-vector (decode-shaped) blocks, the multi-row blocks come
    first and n_multi counts them: attention then runs them as two calls, the
    decode-shaped blocks on the decode CTA.  Otherwise the blocks keep their
    order and n_multi is 0 (one call).  A handful of short sequence tails in a
    prefill step cost less inside the prefill call than as a second call after
    it (measured on the rollout + recompute workload: prefill attention 686 ->
    819 ms when split).  Each block is computed on its own, so neither the
    order nor the split changes a result."""
    multi = qb[:, 1] * G > 16
    n_multi = int(multi.sum())
    if not 0 < n_multi <= qb.shape[0] - n_multi:
        return qb, 0
    return np.concatenate([qb[multi], qb[~multi]]), n_multi


class Runner:
    """Feeds host-side row batches into a DenseModel's static inputs."""

    def __init__(self, model: DenseModel):
        self.m = model
        cfg = model.cfg
        G = cfg.q_heads // cfg.kv_heads
        # bf16 pages with D 64 / 128 run prefill blocks on the tcgen05 kernel,
        # whose CTA takes 128 query vectors; other caches take 64 per CTA
        nv = 128 if (not cfg.kv_fp8 and cfg.head_dim % 64 == 0 and 128 % G == 0) else 64
        self.rows_per_block = max(1, nv // G)

    def load_rows(self, kv: PagedKV, seq_slot, pos, ids, lm_rows, targets, write_kv=None):
        m = self.m
        T = len(ids)
        seq_slot = np.asarray(seq_slot, np.int32)
        pos = np.asarray(pos, np.int32)
        qb, n_multi = split_blocks(qblocks_for(seq_slot, self.rows_per_block),
                                   m.cfg.q_heads // m.cfg.kv_heads)
        slots = kv.slots(seq_slot, pos)
        if write_kv is not None:
            slots = np.where(write_kv, slots, -1)
        m.ids[:T].copy_(torch.from_numpy(np.asarray(ids, np.int32)), non_blocking=True)
        m.row_seq[:T].copy_(torch.from_numpy(seq_slot), non_blocking=True)
        m.row_pos[:T].copy_(torch.from_numpy(pos), non_blocking=True)
        m.slot[:T].copy_(torch.from_numpy(slots), non_blocking=True)
        m.qblocks[:qb.shape[0]].copy_(torch.from_numpy(qb), non_blocking=True)
        nl = len(lm_rows)
        if nl:
            m.lm_rows[:nl].copy_(torch.from_numpy(np.asarray(lm_rows, np.int32)), non_blocking=True)
            m.targets[:nl].copy_(torch.from_numpy(np.asarray(targets, np.int32)), non_blocking=True)
        m.h2d_bytes += T * (4 + 4 + 4 + 8) + qb.size * 4 + nl * 8
        cfg = m.cfg
        attn_flops = 4.0 * float(np.sum(pos.astype(np.int64) + 1)) * cfg.q_heads * cfg.head_dim
        mixed = n_multi > 0
        return StepSpec(T=T, nqblocks=int(qb.shape[0]),
                        max_rows_per_block=int(qb[:n_multi if mixed else qb.shape[0], 1].max()),
                        max_ctx=int(pos.max()) + 1, T_lm=nl, attn_flops=attn_flops,
                        n_multi=n_multi if mixed else 0,
                        max_rows_single=int(qb[n_multi:, 1].max()) if mixed else 1)


def prefill_rows(seqs, slots, starts, ends, lm_from):
    """Rows for sequences i: positions [starts[i], ends[i]); a row at position
    p produces the logprob of token p+1 when p >= lm_from[i] and p+1 < len."""
    seq_slot, pos, ids, lm_rows, targets, owner = [], [], [], [], [], []
    for i, s in enumerate(seqs):
        for p in range(starts[i], ends[i]):
            if p >= lm_from[i] and p + 1 < s.length:
                lm_rows.append(len(ids))
                targets.append(int(s.tokens[p + 1]))
                owner.append((i, p))
            seq_slot.append(slots[i])
            pos.append(p)
            ids.append(int(s.tokens[p]))
    return seq_slot, pos, ids, lm_rows, targets, owner


def recompute(model: DenseModel, kv: PagedKV, seqs, max_tokens: int, chunk: Optional[int] = None):
    """Trainer recompute: full-sequence prefill of every sequence into a
    private cache; returns, per sequence, the logprobs of its response tokens
    (positions prompt_len .. len-1).  ``chunk`` splits each sequence's prefill
    into pieces of that many tokens (chunked prefill)."""
    run = Runner(model)
    out = [np.zeros(s.length - s.prompt_len, np.float32) for s in seqs]
    i = 0
    while i < len(seqs):
        # admit as many whole sequences as fit in max_tokens (and the cache)
        group, tok = [], 0
        while i < len(seqs) and (not group or tok + seqs[i].length - 1 <= max_tokens):
            group.append(i)
            tok += seqs[i].length - 1
            i += 1
        slots = list(range(len(group)))
        for j, gi in enumerate(group):
            kv.admit(slots[j], seqs[gi].length)
        kv.sync_table()
        gseqs = [seqs[gi] for gi in group]
        step = chunk or max(s.length for s in gseqs)
        start = [0] * len(gseqs)
        while True:
            live = [j for j, s in enumerate(gseqs) if start[j] < s.length - 1]
            if not live:
                break
            ends = [min(gseqs[j].length - 1, start[j] + step) for j in live]
            rows = prefill_rows([gseqs[j] for j in live], [slots[j] for j in live],
                                [start[j] for j in live], ends,
                                [gseqs[j].prompt_len - 1 for j in live])
            # keep each call under max_tokens rows
            _run_rows(model, run, kv, rows, max_tokens,
                      lambda k, lpv: _scatter(out, [group[live[i_]] for i_ in range(len(live))], seqs, k, lpv))
            for jj, j in enumerate(live):
                start[j] = ends[jj]
        for j in range(len(group)):
            kv.release(slots[j])
    return out


def _scatter(out, gids, seqs, owner_items, lpv):
    for (li, p), v in zip(owner_items, lpv):
        s = seqs[gids[li]]
        out[gids[li]][p + 1 - s.prompt_len] = v


def _run_rows(model, run, kv, rows, max_tokens, sink):
    seq_slot, pos, ids, lm_rows, targets, owner = rows
    T = len(ids)
    a = 0
    while a < T:
        b = min(T, a + max_tokens)
        sel = [k for k, r in enumerate(lm_rows) if a <= r < b]
        spec = run.load_rows(kv, seq_slot[a:b], pos[a:b], ids[a:b], [lm_rows[k] - a for k in sel],
                             [targets[k] for k in sel])
        model.reserve(kv, [spec])
        model.step(kv, spec)
        if sel:
            sink([owner[k] for k in sel], model.lp[:len(sel)].cpu().numpy())
        a = b


# ---------------------------------------------------------------- rollout ----
class DecodeGraphs:
    """One CUDA graph per padded decode batch size.  A decode step is one row
    per live sequence; rows past the live count are padding (no KV write,
    result discarded), which cannot change a live row's bits because no
    reduction crosses rows."""

    # padded batch sizes with a captured graph each (finer steps where the
    # padding would waste most)
    BUCKETS = (1, 2, 4, 8, 16, 24, 32, 48, 64, 80, 96, 112, 128, 160, 192, 224, 256, 288, 320,
               384, 448, 512, 640, 768, 1024)

    def __init__(self, model: DenseModel, kv: PagedKV, use_graphs: bool = True):
        self.m, self.kv, self.use = model, kv, use_graphs
        self.graphs: Dict[int, torch.cuda.CUDAGraph] = {}
        self.launches: Dict[int, int] = {}
        # decode rows are one per block and all produce a logprob: constant
        # buffers owned by the graphs (the eager prefill path reuses the
        # model's shared qblocks / lm_rows buffers between replays)
        nmax = self.BUCKETS[-1]
        dev = model.ids.device
        self.qblocks = torch.stack([torch.arange(nmax, dtype=torch.int32),
                                    torch.ones(nmax, dtype=torch.int32)], 1).to(dev)
        self.lm_rows = torch.arange(nmax, dtype=torch.int32, device=dev)

    def spec(self, Tb: int) -> StepSpec:
        return StepSpec(T=Tb, nqblocks=Tb, max_rows_per_block=1, max_ctx=self.m.max_pos, T_lm=Tb)

    def bucket(self, n: int) -> int:
        for b in self.BUCKETS:
            if b >= n:
                return b
        raise ValueError("decode batch above the largest bucket")

    def run(self, seq_slot, pos, ids, targets):
        m, n = self.m, len(ids)
        Tb = self.bucket(n) if self.use else n
        pad = Tb - n
        seq_slot = np.concatenate([np.asarray(seq_slot, np.int32), np.full(pad, seq_slot[0], np.int32)])
        pos_a = np.concatenate([np.asarray(pos, np.int32), np.zeros(pad, np.int32)])
        slots = np.concatenate([self.kv.slots(seq_slot[:n], pos_a[:n]), np.full(pad, -1, np.int64)])
        ids_a = np.concatenate([np.asarray(ids, np.int32), np.zeros(pad, np.int32)])
        tg = np.concatenate([np.asarray(targets, np.int32), np.zeros(pad, np.int32)])
        m.ids[:Tb].copy_(torch.from_numpy(ids_a), non_blocking=True)
        m.row_seq[:Tb].copy_(torch.from_numpy(seq_slot), non_blocking=True)
        m.row_pos[:Tb].copy_(torch.from_numpy(pos_a), non_blocking=True)
        m.slot[:Tb].copy_(torch.from_numpy(slots), non_blocking=True)
        m.targets[:Tb].copy_(torch.from_numpy(tg), non_blocking=True)
        m.h2d_bytes += Tb * (4 + 4 + 4 + 8 + 4)
        spec = self.spec(Tb)
        if self.use and Tb not in self.graphs:
            m.reserve(self.kv, [spec])
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                m.step(self.kv, spec, self.qblocks, self.lm_rows)   # warm-up: a real step of these rows
            torch.cuda.current_stream().wait_stream(s)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                m.step(self.kv, spec, self.qblocks, self.lm_rows)
            self.graphs[Tb] = g
            self.launches[Tb] = m.launches
        elif not self.use:
            m.reserve(self.kv, [spec])
            m.step(self.kv, spec, self.qblocks, self.lm_rows)
        else:
            t = m._timer()
            tok = t.bracket_decode(pos) if t and hasattr(t, "bracket_decode") else None
            self.graphs[Tb].replay()
            if tok:
                t.close(tok)
            if t:
                t.launches += self.launches[Tb]
        return m.lp[:n]


def rollout(model: DenseModel, kv: PagedKV, seqs, max_tokens: int, use_graphs: bool = True,
            graphs: Optional[DecodeGraphs] = None, collect: bool = True, after_prefill=None):
    """Rollout: prefill every prompt, then decode one teacher-forced token per
    live sequence per step.  Returns per sequence the logprobs of its response
    tokens (the first one comes from the prompt's last row).  ``after_prefill``
    (optional) is called once the prompt prefill has been issued."""
    run = Runner(model)
    out = [np.zeros(s.length - s.prompt_len, np.float32) for s in seqs]
    slots = list(range(len(seqs)))
    for i, s in enumerate(seqs):
        kv.admit(slots[i], s.length)
    kv.sync_table()
    rows = prefill_rows(seqs, slots, [0] * len(seqs), [s.prompt_len for s in seqs],
                        [s.prompt_len - 1 for s in seqs])
    _run_rows(model, run, kv, rows, max_tokens,
              lambda k, lpv: _scatter(out, list(range(len(seqs))), seqs, k, lpv))
    if after_prefill is not None:
        after_prefill()
    dg = graphs or DecodeGraphs(model, kv, use_graphs)
    cur = [s.prompt_len for s in seqs]
    pending = []
    while True:
        live = [i for i, s in enumerate(seqs) if cur[i] < s.length - 1]
        if not live:
            break
        pos = [cur[i] for i in live]
        lp = dg.run([slots[i] for i in live], pos, [int(seqs[i].tokens[cur[i]]) for i in live],
                    [int(seqs[i].tokens[cur[i] + 1]) for i in live])
        if collect:
            pending.append((live, pos, lp.clone()))
        for i in live:
            cur[i] += 1
    for live, pos, lp in pending:
        v = lp.cpu().numpy()
        for j, i in enumerate(live):
            out[i][pos[j] + 1 - seqs[i].prompt_len] = v[j]
    for i in slots:
        kv.release(i)
    return out


# ---------------------------------------------------- continuous batching ----
def serve_mixed(model: DenseModel, kv: PagedKV, seqs, chunk: int = 512, max_decode: int = 256,
                max_tokens: Optional[int] = None):
    """Continuous batching: every step carries one prefill chunk (<= ``chunk``
    tokens) of the next admitted sequence together with one decode row for
    each live sequence whose prompt is done (at most ``max_decode``).  A
    sequence is admitted when a decode slot is free and leaves when its last
    token is consumed.  Returns per sequence the logprobs of its response
    tokens; they are the same bits as a rollout or a recompute of it alone."""
    run = Runner(model)
    out = [np.zeros(s.length - s.prompt_len, np.float32) for s in seqs]
    free = list(range(len(seqs)))[::-1]
    slot_of, cur = {}, {}
    queue = list(range(len(seqs)))
    prefill_next = {}        # seq -> next prompt position to prefill
    decoding = []            # seqs whose prompt is done and that still decode
    while queue or prefill_next or decoding:
        if queue and not prefill_next and len(decoding) < max_decode:
            i = queue.pop(0)
            slot_of[i] = free.pop()
            kv.admit(slot_of[i], seqs[i].length)
            kv.sync_table()
            prefill_next[i] = 0
        seq_slot, pos, ids, lm_rows, targets, owner = [], [], [], [], [], []
        done_after_step = []
        for i in decoding:
            p = cur[i]
            lm_rows.append(len(ids))
            targets.append(int(seqs[i].tokens[p + 1]))
            owner.append((i, p))
            seq_slot.append(slot_of[i]); pos.append(p); ids.append(int(seqs[i].tokens[p]))
        for i, p0 in list(prefill_next.items()):
            s = seqs[i]
            p1 = min(s.prompt_len, p0 + chunk)
            for p in range(p0, p1):
                if p >= s.prompt_len - 1:
                    lm_rows.append(len(ids))
                    targets.append(int(s.tokens[p + 1]))
                    owner.append((i, p))
                seq_slot.append(slot_of[i]); pos.append(p); ids.append(int(s.tokens[p]))
            if p1 == s.prompt_len:
                del prefill_next[i]
                cur[i] = s.prompt_len
                if cur[i] < s.length - 1:
                    decoding.append(i)
                else:
                    done_after_step.append(i)
            else:
                prefill_next[i] = p1
        if not ids:
            continue
        spec = run.load_rows(kv, seq_slot, pos, ids, lm_rows, targets)
        model.reserve(kv, [spec])
        model.step(kv, spec)
        lp = model.lp[:len(lm_rows)].cpu().numpy()
        for (i, p), v in zip(owner, lp):
            out[i][p + 1 - seqs[i].prompt_len] = v
        nxt = []
        for i in decoding:
            if (i, cur[i]) in set(owner):
                cur[i] += 1
            if cur[i] < seqs[i].length - 1:
                nxt.append(i)
            else:
                kv.release(slot_of[i])
                free.append(slot_of[i])
        decoding = nxt
        for i in done_after_step:
            kv.release(slot_of[i])
            free.append(slot_of[i])
    return out
