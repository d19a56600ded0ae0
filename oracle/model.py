"""Model-level oracle: tokens -> per-token next-token logprobs for the dense
decoder, and the MoE + sparse-attention block.  TEST INFRASTRUCTURE ONLY.

Each sequence is computed alone, as one full causal prefill, so nothing here
can depend on batch composition.  The quantisation rules are those of the
CUDA path (bf16 storage, FP8 e4m3 KV per (token, kv head) when configured,
FP8 128x128 expert weights with 1x128 activation groups); everything else is
FP32.  Model-level logprobs are "parity unpinned" beyond the per-op pins and
the oracle's own decode == prefill check.
"""
from __future__ import annotations

from typing import Dict, List

import numpy as np

from . import ops
from .codecs import bf16_to_f32

F32 = np.float32


def decode_weights(W_bits: Dict[str, np.ndarray]) -> Dict[str, np.ndarray]:
    """bf16 payloads (uint16) -> float32 arrays."""
    return {k: bf16_to_f32(v) for k, v in W_bits.items()}


class DenseOracle:
    """The pre-norm decoder: embed; per layer [RMSNorm, QKV, (QK-norm), RoPE,
    KV store (+FP8 round trip), attention, O, add+RMSNorm, gate_up, SiLU-mul,
    down, add+RMSNorm]; LM head in FP32; log-softmax and gather."""

    def __init__(self, cfg, W: Dict[str, np.ndarray], max_pos: int = 4096):
        self.cfg = cfg
        self.W = W
        self.audit = None  # when a list: residual stream after each layer
        self.cos, self.sin = ops.rope_table(cfg.rope_theta, cfg.head_dim, max_pos)
        self.scale = F32(1.0 / np.sqrt(cfg.head_dim))

    # -- one layer over the rows of one sequence, given the cached K/V --------
    def _attn_block(self, l, y, pos, kv):
        cfg, W = self.cfg, self.W
        p = f"l{l}."
        T = y.shape[0]
        Hq, Hkv, D = cfg.q_heads, cfg.kv_heads, cfg.head_dim
        qkv = ops.gemm(y, W[p + "wqkv"])
        q = qkv[:, :Hq * D].reshape(T, Hq, D)
        k = qkv[:, Hq * D:(Hq + Hkv) * D].reshape(T, Hkv, D)
        v = qkv[:, (Hq + Hkv) * D:].reshape(T, Hkv, D)
        qn = W.get(p + "q_norm") if cfg.qk_norm else None
        kn = W.get(p + "k_norm") if cfg.qk_norm else None
        q = ops.qk_norm_rope(q, pos, qn, cfg.eps, self.cos, self.sin)
        k = ops.qk_norm_rope(k, pos, kn, cfg.eps, self.cos, self.sin)
        if cfg.kv_fp8:
            k, v = ops.kv_roundtrip(k), ops.kv_roundtrip(v)
        kc, vc, kp = kv[l]
        kc = np.concatenate([kc, k]) if kc is not None else k
        vc = np.concatenate([vc, v]) if vc is not None else v
        kp = np.concatenate([kp, pos]) if kp is not None else pos
        kv[l] = (kc, vc, kp)
        o = ops.attention(q, kc, vc, pos, kp, self.scale)
        a = ops.gemm(o.reshape(T, Hq * D), W[p + "wo"])
        if self.audit is not None:
            qk = np.concatenate([q.reshape(T, -1), k.reshape(T, -1), v.reshape(T, -1)], 1)
            self.audit.append(("qkv", l, qk))
            self.audit.append(("attn_o", l, o.reshape(T, Hq * D)))
            self.audit.append(("attn_proj", l, a))
        return a

    def forward_rows(self, tokens: np.ndarray, pos: np.ndarray, kv: list) -> np.ndarray:
        """Run rows (one sequence, consecutive positions) through the model,
        appending their K/V to ``kv``; returns FP32 logits [T, V]."""
        cfg, W = self.cfg, self.W
        r = W["embed"][np.asarray(tokens)]
        y = ops.rmsnorm(r, W["l0.attn_norm"], cfg.eps)
        for l in range(cfg.layers):
            a = self._attn_block(l, y, pos, kv)
            r, y = ops.add_rmsnorm(a, r, W[f"l{l}.mlp_norm"], cfg.eps)
            gu = ops.gemm(y, W[f"l{l}.wgu"])
            m = ops.gemm(ops.silu_mul(gu), W[f"l{l}.wd"])
            if self.audit is not None:
                self.audit.append(("mlp_out", l, m))
            nxt = W[f"l{l + 1}.attn_norm"] if l + 1 < cfg.layers else W["final_norm"]
            r, y = ops.add_rmsnorm(m, r, nxt, cfg.eps)
            if self.audit is not None:
                self.audit.append(("layer", l, r.copy()))
        return ops.gemm(y, W["lm_head"], out="f32")

    def layer_from(self, l: int, r_prev: np.ndarray, pos: np.ndarray) -> np.ndarray:
        """One decoder layer on its own: from the residual stream entering layer
        l (all positions of one sequence, a full prefill), the residual leaving
        it.  Used to check each layer of a long model against its own input."""
        cfg, W = self.cfg, self.W
        kv = self.new_cache()
        y = ops.rmsnorm(r_prev, W[f"l{l}.attn_norm"], cfg.eps)
        a = self._attn_block(l, y, pos, kv)
        r, y = ops.add_rmsnorm(a, r_prev, W[f"l{l}.mlp_norm"], cfg.eps)
        gu = ops.gemm(y, W[f"l{l}.wgu"])
        m = ops.gemm(ops.silu_mul(gu), W[f"l{l}.wd"])
        return ops.bf16_round(m + r)

    def head_from(self, r_last: np.ndarray, targets: np.ndarray) -> np.ndarray:
        """Final norm, LM head and logprob from the last layer's residual."""
        y = ops.rmsnorm(r_last, self.W["final_norm"], self.cfg.eps)
        return ops.logprob(ops.gemm(y, self.W["lm_head"], out="f32"), targets)

    def new_cache(self) -> list:
        return [(None, None, None) for _ in range(self.cfg.layers)]

    def prefill_logprobs(self, tokens: np.ndarray) -> np.ndarray:
        """lp[t] = log p(tokens[t+1] | tokens[..t]) for t < len-1, one prefill."""
        tokens = np.asarray(tokens, np.int64)
        L = tokens.shape[0]
        z = self.forward_rows(tokens[:-1], np.arange(L - 1), self.new_cache())
        return ops.logprob(z, tokens[1:])

    def logprobs_at(self, tokens: np.ndarray, rows: np.ndarray) -> np.ndarray:
        """Logprobs of the next token at selected positions only (same prefill)."""
        tokens = np.asarray(tokens, np.int64)
        rows = np.asarray(rows, np.int64)
        last = int(rows.max()) + 1
        kv = self.new_cache()
        cfg, W = self.cfg, self.W
        # run the prefix through the layers, keep logits only where asked
        r = W["embed"][tokens[:last]]
        pos = np.arange(last)
        y = ops.rmsnorm(r, W["l0.attn_norm"], cfg.eps)
        for l in range(cfg.layers):
            a = self._attn_block(l, y, pos, kv)
            r, y = ops.add_rmsnorm(a, r, W[f"l{l}.mlp_norm"], cfg.eps)
            gu = ops.gemm(y, W[f"l{l}.wgu"])
            m = ops.gemm(ops.silu_mul(gu), W[f"l{l}.wd"])
            nxt = W[f"l{l + 1}.attn_norm"] if l + 1 < cfg.layers else W["final_norm"]
            r, y = ops.add_rmsnorm(m, r, nxt, cfg.eps)
        z = ops.gemm(y[rows], W["lm_head"], out="f32")
        return ops.logprob(z, tokens[rows + 1])

    def decode_logprobs(self, tokens: np.ndarray, prompt_len: int) -> np.ndarray:
        """Prefill the prompt, then feed the remaining tokens one at a time
        through the cache (the rollout's recurrence); returns the logprobs of
        tokens[prompt_len-1+1 ...] in the same indexing as prefill_logprobs."""
        tokens = np.asarray(tokens, np.int64)
        L = tokens.shape[0]
        kv = self.new_cache()
        z0 = self.forward_rows(tokens[:prompt_len], np.arange(prompt_len), kv)
        lps = list(ops.logprob(z0, tokens[1:prompt_len + 1]))
        for t in range(prompt_len, L - 1):
            z = self.forward_rows(tokens[t:t + 1], np.array([t]), kv)
            lps.append(float(ops.logprob(z, tokens[t + 1:t + 2])[0]))
        return np.array(lps[:L - 1], F32)


# ------------------------------------------------------------------ MoE ----
def expert_mlp_fp8(x, wgu_codes, wgu_scale, wd_codes, wd_scale):
    """One FP8 expert: quantise activations (1x128 groups), gate_up GEMM,
    SiLU-mul, quantise, down GEMM; bf16 output."""
    aq, sa = ops.act_quant_fp8(x)
    gu = ops.gemm_fp8_block(aq, sa, wgu_codes, wgu_scale)
    act = ops.silu_mul(gu)
    aq2, sa2 = ops.act_quant_fp8(act)
    return ops.gemm_fp8_block(aq2, sa2, wd_codes, wd_scale)


def moe_block(h, router_w, experts: List[tuple], shared: tuple, top_k: int, logits=None):
    """Router logits (FP32 GEMM), Top-k routing, each selected expert per token
    row, the shared expert, FP32 fixed-slot combine.

    ``logits`` (optional, FP32 [T, E]) routes by given router logits instead
    of computing them: a comparison with another implementation can then route
    both sides identically, so that a near-tie that rounds the other way in
    one of them does not decide which experts the float comparison covers."""
    if logits is None:
        logits = ops.gemm(h, router_w, out="f32")
    idx, w = ops.router_topk(logits, top_k)
    T, d = h.shape
    y = np.zeros((T, top_k, d), F32)
    for e in range(len(experts)):
        rows, slots = np.nonzero(idx == e)
        if rows.size == 0:
            continue
        y[rows, slots] = expert_mlp_fp8(h[rows], *experts[e])
    sh = expert_mlp_fp8(h, *shared)
    return ops.moe_combine(y, w, sh), idx, w
