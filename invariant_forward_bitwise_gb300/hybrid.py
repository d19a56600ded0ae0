"""The Mamba-2 / attention hybrid stack, as a sequence of libbiv calls.

"Finish RL Training Faster" runs its invariance on a Mamba-2 hybrid with
NVFP4 weights (section "两组结果，要连同分母一起读") and requires the Mamba-2
decode to replay the prefill's chunk order so that state and logprobs match
bit for bit (section "一致性有多个层面").  Each Mamba-2 mixer here is
in-projection GEMM -> causal conv1d + SiLU (and dt softplus) -> SSD scan ->
gated RMSNorm -> out-projection GEMM; every step is a row-local kernel or the
chunked SSD whose rows are computed from their chunk's start state and rows
(prefill, chunked prefill and decode take one code path).  The attention
mixers are the dense model's paged attention (RoPE, no QK-norm).  Every
mixer is followed by a SiLU-gated MLP; norms are pre-norm with the residual
add fused.  Linear layers keep their NVFP4 weights (packed e2m1 codes and
e4m3 block scales) on the device and run through ``biv_gemm_nvfp4``, whose
every output bit equals the bf16 GEMM on the decoded weights: decode-sized
steps stream the 4-bit codes, prefill-sized steps decode once per call.

PyTorch holds device memory and streams; every arithmetic step runs in libbiv.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional

import numpy as np
import torch

from . import biv
from .model import PAGE, PagedKV, qblocks_for


class HybridModel:
    """Weights, per-sequence recurrent state and static buffers for up to
    ``max_rows`` rows per step and ``max_seqs`` sequence slots."""

    def __init__(self, cfg, weights: Dict[str, object], max_rows: int, max_seqs: int,
                 max_pos: int, mode: int = biv.MODE_INVARIANT, lm_chunk: int = 4096, device="cuda"):
        biv.load()
        self.cfg, self.mode, self.max_rows, self.max_seqs = cfg, mode, max_rows, max_seqs
        self.max_pos = max_pos
        self.lm_chunk = min(lm_chunk, max_rows)
        bf = dict(dtype=torch.bfloat16, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        i32 = dict(dtype=torch.int32, device=device)
        self.W: Dict[str, object] = {}
        for k, v in weights.items():
            if isinstance(v, tuple):      # NVFP4: (packed codes [N, K/2], scales [N, K/16])
                self.W[k] = (v[0].to(device).contiguous(), v[1].to(device).contiguous())
            else:
                self.W[k] = v.to(device).contiguous()
        D, T = cfg.head_dim, max_rows
        self.rope = torch.empty(2 * max_pos * (D // 2), **f32)
        biv.biv_rope_table(cfg.rope_theta, D, max_pos, self.rope)
        d, di, ch, H = cfg.d_model, cfg.d_inner, cfg.conv_channels, cfg.ssd_heads
        self.r = torch.empty(T, d, **bf)
        self.y = torch.empty(T, d, **bf)
        self.a = torch.empty(T, d, **bf)
        self.u = torch.empty(T, cfg.in_proj_width, **bf)
        self.xbc = torch.empty(T, ch, **bf)
        self.dt = torch.empty(T, H, **f32)
        self.ys = torch.empty(T, di, **bf)
        self.g = torch.empty(T, di, **bf)
        self.qkv = torch.empty(T, cfg.qkv_width, **bf)
        self.o = torch.empty(T, cfg.q_heads * D, **bf)
        self.gu = torch.empty(T, 2 * cfg.intermediate, **bf)
        self.act = torch.empty(T, cfg.intermediate, **bf)
        self.ylm = torch.empty(T, d, **bf)
        self.logits = torch.empty(self.lm_chunk, cfg.vocab, **f32)
        self.lp = torch.empty(T, **f32)
        # per-step row inputs
        self.ids = torch.zeros(T, **i32)
        self.row_seq = torch.zeros(T, **i32)
        self.row_pos = torch.zeros(T, **i32)
        self.slot = torch.full((T,), -1, dtype=torch.int64, device=device)
        self.qblocks = torch.zeros(T, 2, **i32)
        self.lm_rows = torch.zeros(T, **i32)
        self.targets = torch.zeros(T, **i32)
        self.seq_row0 = torch.zeros(max_seqs, **i32)
        self.seq_n = torch.zeros(max_seqs, **i32)
        self.seq_pos0 = torch.zeros(max_seqs, **i32)
        # recurrent state of every Mamba-2 layer, per sequence slot
        self.mstate = {}
        P, N, Q = cfg.ssd_head_dim, cfg.state, cfg.chunk
        for l, kind in enumerate(cfg.pattern):
            if kind == "M":
                self.mstate[l] = dict(
                    conv=torch.zeros(max_seqs, cfg.conv_width - 1, ch, **bf),
                    ssd=torch.zeros(max_seqs, H, P, N, **f32),
                    bx=torch.zeros(max_seqs, Q, H, P, **bf), bB=torch.zeros(max_seqs, Q, N, **bf),
                    bC=torch.zeros(max_seqs, Q, N, **bf), bdt=torch.zeros(max_seqs, Q, H, **f32))
        self.attn_index = {l: i for i, l in enumerate(l for l, k in enumerate(cfg.pattern) if k == "A")}
        self.ws = torch.empty(16, dtype=torch.uint8, device=device)
        self.gws = torch.empty(256, dtype=torch.uint8, device=device)
        self.sws = torch.empty(256, dtype=torch.uint8, device=device)
        self._old: List[torch.Tensor] = []
        self.launches = 0

    # -- state -----------------------------------------------------------------
    def reset_slot(self, slot: int):
        """A new sequence in ``slot``: zero conv and SSD state."""
        for st in self.mstate.values():
            st["conv"][slot].zero_()
            st["ssd"][slot].zero_()

    def _grow(self, name, need):
        t = getattr(self, name)
        if need > t.numel():
            self._old.append(t)
            setattr(self, name, torch.empty(need, dtype=torch.uint8, device=t.device))
        return getattr(self, name)

    # -- rows ------------------------------------------------------------------
    def load(self, kv: PagedKV, seq_slot, pos, ids, lm_rows, targets):
        """Rows of this step (rows of one sequence contiguous, positions
        consecutive); returns the step's host-side shape."""
        cfg = self.cfg
        T = len(ids)
        seq_slot = np.asarray(seq_slot, np.int32)
        pos = np.asarray(pos, np.int32)
        G = cfg.q_heads // cfg.kv_heads
        qb = qblocks_for(seq_slot, max(1, 64 // G))
        row0 = np.zeros(self.max_seqs, np.int32)
        n = np.zeros(self.max_seqs, np.int32)
        pos0 = np.zeros(self.max_seqs, np.int32)
        i = 0
        while i < T:
            j = i
            while j < T and seq_slot[j] == seq_slot[i]:
                j += 1
            s = seq_slot[i]
            if n[s]:
                raise ValueError("rows of a sequence must be contiguous")
            if np.any(np.diff(pos[i:j]) != 1):
                raise ValueError("positions of a sequence must be consecutive")
            row0[s], n[s], pos0[s] = i, j - i, pos[i]
            i = j
        slots = kv.slots(seq_slot, pos) if kv is not None else np.full(T, -1, np.int64)
        cp = lambda dst, a: dst[:len(a)].copy_(torch.from_numpy(np.ascontiguousarray(a)), non_blocking=True)
        cp(self.ids, np.asarray(ids, np.int32))
        cp(self.row_seq, seq_slot)
        cp(self.row_pos, pos)
        cp(self.slot, slots.astype(np.int64))
        cp(self.qblocks, qb)
        cp(self.seq_row0, row0)
        cp(self.seq_n, n)
        cp(self.seq_pos0, pos0)
        if len(lm_rows):
            cp(self.lm_rows, np.asarray(lm_rows, np.int32))
            cp(self.targets, np.asarray(targets, np.int32))
        return dict(T=T, nqblocks=int(qb.shape[0]), max_rows_per_block=int(qb[:, 1].max()),
                    max_ctx=int(pos.max()) + 1, T_lm=len(lm_rows), max_n=int(n.max()))

    # -- ops -------------------------------------------------------------------
    def _gemm(self, A, Bw, Cout, M, st):
        if isinstance(Bw, tuple):
            codes, sc = Bw
            cdt = biv.F32 if Cout.dtype == torch.float32 else biv.BF16
            ws = self._grow("gws", biv.biv_gemm_nvfp4_workspace(M, codes.shape[0], A.shape[1], cdt,
                                                               self.mode))
            biv.biv_gemm_nvfp4(A, codes, sc, Cout, M=M, mode=self.mode, ws=ws, stream=st)
        else:
            d = biv.gemm_desc(A, Bw, Cout, mode=self.mode, M=M)
            ws = self._grow("gws", biv.biv_gemm_workspace(d))
            biv.biv_gemm(d, ws, stream=st)
        self.launches += 1

    def _mamba(self, l, T, spec, st):
        cfg, W, S = self.cfg, self.W, self.mstate[l]
        p = f"l{l}."
        di, N, H = cfg.d_inner, cfg.state, cfg.ssd_heads
        self._gemm(self.y, W[p + "in_proj"], self.u, T, st)
        c = biv.ConvDesc()
        c.u, c.u_stride = self.u.data_ptr(), self.u.stride(0)
        c.col_x, c.col_dt = di, 2 * di + 2 * N
        c.channels, c.heads, c.width = cfg.conv_channels, H, cfg.conv_width
        c.conv_w, c.conv_b, c.dt_bias = W[p + "conv_w"].data_ptr(), W[p + "conv_b"].data_ptr(), W[p + "dt_bias"].data_ptr()
        c.out, c.out_stride = self.xbc.data_ptr(), self.xbc.stride(0)
        c.dt_out, c.dt_stride = self.dt.data_ptr(), self.dt.stride(0)
        c.T = T
        c.row_seq, c.row_pos = self.row_seq.data_ptr(), self.row_pos.data_ptr()
        c.nseq = self.max_seqs
        c.row0, c.n, c.pos0 = self.seq_row0.data_ptr(), self.seq_n.data_ptr(), self.seq_pos0.data_ptr()
        c.state = S["conv"].data_ptr()
        biv.biv_causal_conv1d(c, stream=st)
        d = biv.SSDDesc()
        d.x, d.x_stride = self.xbc.data_ptr(), self.xbc.stride(0)
        d.dt, d.dt_stride = self.dt.data_ptr(), self.dt.stride(0)
        d.A, d.D = W[p + "A"].data_ptr(), W[p + "D"].data_ptr()
        d.B, d.B_stride = self.xbc[:, di:].data_ptr(), self.xbc.stride(0)
        d.C, d.C_stride = self.xbc[:, di + N:].data_ptr(), self.xbc.stride(0)
        d.y, d.y_stride = self.ys.data_ptr(), self.ys.stride(0)
        d.H, d.P, d.N, d.chunk = H, cfg.ssd_head_dim, N, cfg.chunk
        d.nseq = self.max_seqs
        d.row0, d.n, d.pos0 = self.seq_row0.data_ptr(), self.seq_n.data_ptr(), self.seq_pos0.data_ptr()
        d.max_n = spec["max_n"]
        d.state, d.buf_x, d.buf_B = S["ssd"].data_ptr(), S["bx"].data_ptr(), S["bB"].data_ptr()
        d.buf_C, d.buf_dt = S["bC"].data_ptr(), S["bdt"].data_ptr()
        need = biv.biv_ssd_workspace(d)
        if need:
            ws = self._grow("sws", need)
            d.workspace, d.workspace_bytes = ws.data_ptr(), ws.numel()
        biv.biv_ssd_scan(d, stream=st)
        biv.biv_gated_rmsnorm(self.ys[:T], self.u[:T, :di], W[p + "norm_w"], self.g[:T], cfg.eps, stream=st)
        self._gemm(self.g, W[p + "out_proj"], self.a, T, st)
        self.launches += 4

    def _attn(self, l, T, spec, kv, st):
        cfg, W = self.cfg, self.W
        p = f"l{l}."
        li = self.attn_index[l]
        Hq, Hkv, D = cfg.q_heads, cfg.kv_heads, cfg.head_dim
        self._gemm(self.y, W[p + "wqkv"], self.qkv, T, st)
        biv.biv_qkv_finalize(self.qkv, T, Hq, Hkv, D, None, None, self.rope, self.max_pos, self.row_pos,
                             cfg.eps, self.slot, biv.BF16, kv.k[li], kv.v[li], stream=st)
        ad = biv.AttnDesc()
        ad.q, ad.q_stride = self.qkv.data_ptr(), self.qkv.stride(0)
        ad.out, ad.out_stride = self.o.data_ptr(), self.o.stride(0)
        ad.T, ad.Hq, ad.Hkv, ad.D = T, Hq, Hkv, D
        ad.row_seq, ad.row_pos = self.row_seq.data_ptr(), self.row_pos.data_ptr()
        ad.qblocks, ad.nqblocks = self.qblocks.data_ptr(), spec["nqblocks"]
        ad.max_rows_per_block = spec["max_rows_per_block"]
        ad.kv_dtype = biv.BF16
        ad.k_cache, ad.v_cache = kv.k[li].data_ptr(), kv.v[li].data_ptr()
        ad.block_table, ad.max_pages = kv.block_table.data_ptr(), kv.max_pages
        ad.page, ad.kv_split, ad.max_ctx = PAGE, cfg.kv_split, spec["max_ctx"]
        ad.scale = 1.0 / math.sqrt(D)
        ad.mode = self.mode
        ad.num_pages = kv.pages
        ws = self._grow("ws", biv.biv_attention_workspace(ad))
        biv.biv_attention(ad, ws, stream=st)
        self._gemm(self.o, W[p + "wo"], self.a, T, st)
        self.launches += 3

    def step(self, kv: Optional[PagedKV], spec):
        """Rows [0, T) through the stack; logprobs of lm_rows land in lp."""
        cfg, W, T = self.cfg, self.W, spec["T"]
        st = torch.cuda.current_stream()
        eps = cfg.eps
        r, y = self.r[:T], self.y[:T]
        self.launches = 2
        biv.biv_embed(self.ids[:T], W["embed"], r, stream=st)
        biv.biv_add_rmsnorm(r, None, W["l0.norm"], y, eps, stream=st)
        nl = len(cfg.pattern)
        for l, kind in enumerate(cfg.pattern):
            if kind == "M":
                self._mamba(l, T, spec, st)
            else:
                self._attn(l, T, spec, kv, st)
            biv.biv_add_rmsnorm(self.a[:T], r, W[f"l{l}.mlp_norm"], y, eps, stream=st)
            self._gemm(self.y, W[f"l{l}.wgu"], self.gu, T, st)
            biv.biv_silu_mul(self.gu[:T], self.act[:T], stream=st)
            self._gemm(self.act, W[f"l{l}.wd"], self.a, T, st)
            nxt = W[f"l{l + 1}.norm"] if l + 1 < nl else W["final_norm"]
            biv.biv_add_rmsnorm(self.a[:T], r, nxt, y, eps, stream=st)
            self.launches += 3
        Tl = spec["T_lm"]
        if Tl == 0:
            return
        biv.biv_gather_rows(y, self.lm_rows, 1, Tl, self.ylm, stream=st)
        for c0 in range(0, Tl, self.lm_chunk):
            n = min(self.lm_chunk, Tl - c0)
            self._gemm(self.ylm[c0:c0 + n], W["lm_head"], self.logits, n, st)
            biv.biv_logprob(self.logits, self.targets[c0:c0 + n], self.lp[c0:c0 + n], T=n, stream=st)
            self.launches += 1
        self.launches += 1


def new_kv(cfg, max_seqs: int, max_pos: int, device="cuda") -> PagedKV:
    """The paged bf16 K/V cache of the stack's attention layers."""
    max_pages = (max_pos + PAGE - 1) // PAGE
    return PagedKV(cfg, pages=max_seqs * max_pages + 1, max_seqs=max_seqs, max_pages=max_pages,
                   device=device)


def run_sequences(model: HybridModel, kv: PagedKV, seqs, pieces) -> List[np.ndarray]:
    """Logprobs of every sequence's tokens 1..L-1 (position t predicts token
    t+1), computed through a schedule of calls: ``pieces[i]`` lists the row
    counts of sequence i's successive calls (e.g. [L-1] for one prefill,
    [P, 1, 1, ...] for a prompt then token-by-token decode).  Calls of all
    sequences are interleaved: step k carries every sequence's k-th piece."""
    out = [np.zeros(s.length - 1, np.float32) for s in seqs]
    for i, s in enumerate(seqs):
        kv.admit(i, s.length)
        model.reset_slot(i)
    kv.sync_table()
    done = [0] * len(seqs)
    k = 0
    while any(k < len(p) for p in pieces):
        seq_slot, pos, ids, lm_rows, targets, owner = [], [], [], [], [], []
        for i, s in enumerate(seqs):
            if k >= len(pieces[i]):
                continue
            for p_ in range(done[i], done[i] + pieces[i][k]):
                lm_rows.append(len(ids))
                targets.append(int(s.tokens[p_ + 1]))
                owner.append((i, p_))
                seq_slot.append(i)
                pos.append(p_)
                ids.append(int(s.tokens[p_]))
            done[i] += pieces[i][k]
        k += 1
        if not ids:
            continue
        spec = model.load(kv, seq_slot, pos, ids, lm_rows, targets)
        model.step(kv, spec)
        lp = model.lp[:len(lm_rows)].cpu().numpy()
        for (i, p_), v in zip(owner, lp):
            out[i][p_] = v
    for i in range(len(seqs)):
        kv.release(i)
    return out
