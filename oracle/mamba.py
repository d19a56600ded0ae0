"""Mamba-2 mixer and the Mamba-2 / attention hybrid stack.  TEST INFRASTRUCTURE ONLY.

The pages name the workload (a Mamba-2 hybrid with NVFP4 weights: "Finish RL
Training Faster", section "两组结果，要连同分母一起读") and its invariance
rule: decode must replay the prefill's chunk order and reach the same bits,
not only a close final state (section "一致性有多个层面").  They print no
formulas; the mixer below is the plainest reading of a Mamba-2 layer, and the
oracle's own recurrence is sequential, so its decode equals its prefill by
construction:

  u = in_proj(x) = [z | xBC | dt_raw]            (bf16 GEMM output)
  xBC' = bf16(silu(conv1d_causal_4(xBC) + bias))  (depthwise, width 4, FP32)
  dt   = softplus(dt_raw + dt_bias)               (FP32, not rounded)
  y    = SSD(x', dt, A, B', C', D)                 (sequential recurrence, bf16 out)
  g    = y * silu(z)                               (FP32, not rounded)
  out  = out_proj(bf16(g / sqrt(mean(g^2) + eps) * w_norm))

Each layer of the stack is pre-norm with a fused residual add: the pattern is
four Mamba-2 mixers and one GQA attention (RoPE, no QK-norm), each followed by
a SiLU-gated MLP.  Weights are NVFP4 (e2m1 codes with one e4m3 scale per 16
elements, global scale 1), used through their exact bf16 values.
"""
from __future__ import annotations

from typing import Dict, List, Optional

import numpy as np

from . import ops
from .codecs import bf16_round, bf16_to_f32, nvfp4_dequant
from .ssd import ssd_sequential

F32 = np.float32
CONV_W = 4


def decode_hybrid_weights(raw: Dict[str, object]) -> Dict[str, np.ndarray]:
    """Payloads -> float32 values: NVFP4 (codes, scale codes) pairs through
    the e2m1 / e4m3 codecs, uint16 arrays as bf16 bits, float32 as is."""
    out = {}
    for k, v in raw.items():
        if isinstance(v, tuple):
            out[k] = nvfp4_dequant(v[0], v[1])
        elif v.dtype == np.uint16:
            out[k] = bf16_to_f32(v)
        else:
            out[k] = np.asarray(v, F32)
    return out


def silu(x):
    x = np.asarray(x, F32)
    return x / (F32(1.0) + np.exp(-x, dtype=F32))


def softplus(x):
    """log(1 + e^x) in FP32; x > 20 returns x (e^-20 is below FP32's
    resolution of x there)."""
    x = np.asarray(x, F32)
    return np.where(x > F32(20.0), x, np.log1p(np.exp(np.minimum(x, F32(20.0)), dtype=F32),
                                                dtype=F32)).astype(F32)


def conv1d_causal_silu(xbc, w, bias, state=None):
    """Depthwise causal convolution of width 4 over the rows of xbc [T, Ch]
    (consecutive positions of one sequence), then SiLU, rounded to bf16:
        out[t, c] = bf16(silu(bias[c] + sum_{j=0..3} w[c, j] * x[t-3+j, c]))
    with the sum taken in FP32 in ascending j.  ``state`` [3, Ch] holds the
    three inputs before the first row (zeros at the start of a sequence).
    Returns (out, new state = the last three inputs)."""
    xbc = np.asarray(xbc, F32)
    T, Ch = xbc.shape
    st = np.zeros((CONV_W - 1, Ch), F32) if state is None else np.asarray(state, F32)
    full = np.concatenate([st, xbc], axis=0)                 # positions -3 .. T-1
    w = np.asarray(w, F32)
    out = np.zeros((T, Ch), F32)
    for t in range(T):
        acc = np.asarray(bias, F32).copy()
        for j in range(CONV_W):
            acc = (acc + w[:, j] * full[t + j]).astype(F32)
        out[t] = acc
    return bf16_round(silu(out)), full[-(CONV_W - 1):].copy()


def gated_rmsnorm(y, z, w, eps):
    """g = y * silu(z) in FP32, then RMSNorm of g with gain w, rounded once."""
    g = (np.asarray(y, F32) * silu(z)).astype(F32)
    return ops.rmsnorm(g, w, eps)


class HybridOracle:
    """The hybrid stack on one sequence at a time.  ``cfg`` carries d_model,
    ssd heads H, head dim P, state N, conv width 4, attention heads, MLP
    width, vocabulary, eps, rope theta and the layer pattern; W holds float32
    values on the bf16 grid."""

    def __init__(self, cfg, W: Dict[str, np.ndarray], max_pos: int = 4096):
        self.cfg, self.W = cfg, W
        self.cos, self.sin = ops.rope_table(cfg.rope_theta, cfg.head_dim, max_pos)
        self.scale = F32(1.0 / np.sqrt(cfg.head_dim))

    def new_state(self):
        """Per layer: conv state and SSD state (Mamba) or K/V so far (attention)."""
        st = []
        for kind in self.cfg.pattern:
            st.append({"conv": None, "ssd": None} if kind == "M" else {"k": None, "v": None, "p": None})
        return st

    def _mamba(self, l, y, st):
        cfg, W = self.cfg, self.W
        p = f"l{l}."
        di, N, H, P = cfg.d_inner, cfg.state, cfg.ssd_heads, cfg.ssd_head_dim
        u = ops.gemm(y, W[p + "in_proj"])
        z, xbc, dtr = u[:, :di], u[:, di:2 * di + 2 * N], u[:, 2 * di + 2 * N:]
        xbc, st["conv"] = conv1d_causal_silu(xbc, W[p + "conv_w"], W[p + "conv_b"], st["conv"])
        dt = softplus(dtr + W[p + "dt_bias"][None, :])
        T = y.shape[0]
        x = xbc[:, :di].reshape(T, H, P)
        B, C = xbc[:, di:di + N], xbc[:, di + N:]
        yo, st["ssd"] = ssd_sequential(x, dt, W[p + "A"], B, C, W[p + "D"], h0=st["ssd"])
        g = gated_rmsnorm(yo.reshape(T, di), z, W[p + "norm_w"], cfg.eps)
        return ops.gemm(g, W[p + "out_proj"])

    def _attn(self, l, y, pos, st):
        cfg, W = self.cfg, self.W
        p = f"l{l}."
        T = y.shape[0]
        Hq, Hkv, D = cfg.q_heads, cfg.kv_heads, cfg.head_dim
        qkv = ops.gemm(y, W[p + "wqkv"])
        q = ops.rope(qkv[:, :Hq * D].reshape(T, Hq, D), pos, self.cos, self.sin)
        k = ops.rope(qkv[:, Hq * D:(Hq + Hkv) * D].reshape(T, Hkv, D), pos, self.cos, self.sin)
        v = qkv[:, (Hq + Hkv) * D:].reshape(T, Hkv, D)
        st["k"] = k if st["k"] is None else np.concatenate([st["k"], k])
        st["v"] = v if st["v"] is None else np.concatenate([st["v"], v])
        st["p"] = pos if st["p"] is None else np.concatenate([st["p"], pos])
        o = ops.attention(q, st["k"], st["v"], pos, st["p"], self.scale)
        return ops.gemm(o.reshape(T, Hq * D), W[p + "wo"])

    def forward_rows(self, tokens, pos, state) -> np.ndarray:
        """Rows of one sequence at consecutive positions ``pos`` through the
        stack, carrying ``state``; returns FP32 logits [T, V]."""
        cfg, W = self.cfg, self.W
        r = W["embed"][np.asarray(tokens)]
        y = ops.rmsnorm(r, W["l0.norm"], cfg.eps)
        nl = len(cfg.pattern)
        for l, kind in enumerate(cfg.pattern):
            a = self._mamba(l, y, state[l]) if kind == "M" else self._attn(l, y, pos, state[l])
            r, y = ops.add_rmsnorm(a, r, W[f"l{l}.mlp_norm"], cfg.eps)
            m = ops.gemm(ops.silu_mul(ops.gemm(y, W[f"l{l}.wgu"])), W[f"l{l}.wd"])
            nxt = W[f"l{l + 1}.norm"] if l + 1 < nl else W["final_norm"]
            r, y = ops.add_rmsnorm(m, r, nxt, cfg.eps)
        return ops.gemm(y, W["lm_head"], out="f32")

    def prefill_logprobs(self, tokens) -> np.ndarray:
        tokens = np.asarray(tokens, np.int64)
        L = tokens.shape[0]
        z = self.forward_rows(tokens[:-1], np.arange(L - 1), self.new_state())
        return ops.logprob(z, tokens[1:])

    def decode_logprobs(self, tokens, prompt_len: int, chunk: Optional[int] = None) -> np.ndarray:
        """Prompt in one call (or in pieces of ``chunk`` rows), then one token
        per call through the carried state; same indexing as prefill."""
        tokens = np.asarray(tokens, np.int64)
        L = tokens.shape[0]
        st = self.new_state()
        lps: List[float] = []
        step = chunk or prompt_len
        for a in range(0, prompt_len, step):
            b = min(prompt_len, a + step)
            z = self.forward_rows(tokens[a:b], np.arange(a, b), st)
            lps.extend(ops.logprob(z, tokens[a + 1:b + 1]).tolist())
        for t in range(prompt_len, L - 1):
            z = self.forward_rows(tokens[t:t + 1], np.array([t]), st)
            lps.append(float(ops.logprob(z, tokens[t + 1:t + 2])[0]))
        return np.array(lps[:L - 1], F32)
