"""Backward of the fused forward ops, in float64.  TEST INFRASTRUCTURE ONLY.

The trainer side of the pages runs the imported inference ops' hand-written
backward ("No More Train-Inference Mismatch", section "方法细节": the fused
vLLM ops enter the training forward and get their own backward), with a
straight-through estimator for the FP8 round trip ("Finish RL Training
Faster", section "让训练前向使用推理的数值": the FP8 KV is kept and its
gradient passes straight through).  Each function is the derivative of the
forward definition, written out:

  RMSNorm    y = x * inv * w, inv = (mean(x^2) + eps)^-1/2
             dx = inv * (w dy) - x * inv^3 * mean(x * w * dy);  dw = sum_rows dy x inv
  SiLU-mul   y = silu(g) u:  dg = dy u silu'(g), du = dy silu(g),
             silu'(g) = sig(g) (1 + g (1 - sig(g)))
  logprob    lp = z[t] - logsumexp(z):  dz = dlp (onehot(t) - softmax(z))
  attention  o = softmax(s) v, s = q.k * scale (causal):  D_i = do_i . o_i,
             dp = do . v^T, ds = p (dp - D), dq = ds k scale, dk = ds^T q scale,
             dv = p^T do;  the FP8 round trip of k and v passes dk, dv through.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


def rmsnorm_backward(x, w, dy, eps):
    """x, dy [R, d]; w [d] -> (dx [R, d], dw [d])."""
    x, w, dy = (np.asarray(a, F64) for a in (x, w, dy))
    inv = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    g = dy * w
    dx = inv * g - x * inv ** 3 * np.mean(g * x, axis=-1, keepdims=True)
    dw = np.sum(dy * x * inv, axis=0)
    return dx, dw


def silu_mul_backward(gate_up, dy):
    """[gate | up] [R, 2I], dy [R, I] -> d[gate | up] [R, 2I]."""
    gu, dy = np.asarray(gate_up, F64), np.asarray(dy, F64)
    I = gu.shape[-1] // 2
    g, u = gu[..., :I], gu[..., I:]
    sig = 1.0 / (1.0 + np.exp(-g))
    silu = g * sig
    return np.concatenate([dy * u * sig * (1.0 + g * (1.0 - sig)), dy * silu], axis=-1)


def logprob_backward(z, target, dlp):
    """z [T, V], target [T], dlp [T] -> dz [T, V]."""
    z, dlp = np.asarray(z, F64), np.asarray(dlp, F64)
    m = np.max(z, axis=-1, keepdims=True)
    p = np.exp(z - m)
    p /= np.sum(p, axis=-1, keepdims=True)
    dz = -p
    dz[np.arange(z.shape[0]), np.asarray(target)] += 1.0
    return dz * dlp[:, None]


def attention_backward(q, k, v, q_pos, k_pos, scale, do):
    """Causal GQA attention of one sequence.  q, do [Tq, Hq, D]; k, v [Tk,
    Hkv, D] -> (dq [Tq, Hq, D], dk [Tk, Hkv, D], dv [Tk, Hkv, D])."""
    q, k, v, do = (np.asarray(a, F64) for a in (q, k, v, do))
    Tq, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    vis = np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in range(Hq):
        kv = h // G
        s = np.where(vis, q[:, h] @ k[:, kv].T * scale, -np.inf)
        m = np.max(s, axis=1, keepdims=True)
        m = np.where(np.isfinite(m), m, 0.0)
        p = np.exp(s - m)
        p /= np.maximum(np.sum(p, axis=1, keepdims=True), 1e-300)
        o = p @ v[:, kv]
        Dr = np.sum(do[:, h] * o, axis=1, keepdims=True)
        ds = p * (do[:, h] @ v[:, kv].T - Dr)
        dq[:, h] = ds @ k[:, kv] * scale
        dk[:, kv] += ds.T @ q[:, h] * scale
        dv[:, kv] += p.T @ do[:, h]
    return dq, dk, dv
