"""Per-operation oracle: plain numpy float32, no blocking or fusion beyond the
definition of each op.  TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Every tensor that the method stores in bf16 is held here as float32 values
lying on the bf16 grid (``bf16_round``); FP8 tensors are uint8 codes plus
float32 scales.
"""
from __future__ import annotations

import contextlib

import numpy as np

from .codecs import bf16_round, e4m3_to_f32, f32_to_e4m3

F32 = np.float32

# How the oracle forms a dot product.  "f64" (the default): in float64, rounded
# once to FP32, so the result does not depend on how a library blocks the sum.
# The others are plain FP32 evaluations of the same sums: "f32" in ascending
# k and "f32_desc" in descending k, every product and every partial sum
# rounded to FP32 (nearest), "f32_rz" in ascending k with every partial sum
# rounded toward zero (IEEE's directed rounding; tensor-core accumulators
# truncate in this way), and "f32_blas" the FP32 library matmul with its own
# blocking.  All are correct FP32 evaluations of the same definition; the
# alternatives exist to measure how far correct evaluations drift apart
# through a deep model (tests/golden/make_accumulation_spread.py), which
# bounds what any implementation can promise against the default.
_ACCUMULATION = ["f64"]
KINDS = ("f64", "f32", "f32_desc", "f32_rz", "f32_blas")


@contextlib.contextmanager
def accumulation(kind: str):
    """Run the enclosed oracle calls with dot products formed as ``kind``
    (one of KINDS)."""
    if kind not in KINDS:
        raise ValueError(kind)
    prev = _ACCUMULATION[0]
    _ACCUMULATION[0] = kind
    try:
        yield
    finally:
        _ACCUMULATION[0] = prev


def _dot_f32_sequential(a: np.ndarray, bt: np.ndarray, descending: bool = False) -> np.ndarray:
    """acc = 0; for k = 0, 1, ... (or K-1, K-2, ...):
    acc = fp32(acc + fp32(a[:, k] * bt[k, :]))."""
    a = np.ascontiguousarray(np.asarray(a, F32).T)
    bt = np.ascontiguousarray(bt, F32)
    acc = np.zeros((a.shape[1], bt.shape[1]), F32)
    ks = range(a.shape[0] - 1, -1, -1) if descending else range(a.shape[0])
    for k in ks:
        acc += a[k][:, None] * bt[k][None, :]
    return acc


def _to_f32_toward_zero(x: np.ndarray) -> np.ndarray:
    """float64 -> float32 rounded toward zero: clear the 29 low mantissa bits
    (exact for normal float32 results, which is all a dot product of bf16
    values produces here)."""
    u = np.ascontiguousarray(x, np.float64).view(np.uint64) & np.uint64(0xFFFFFFFFE0000000)
    return u.view(np.float64).astype(F32)


def _dot_f32_rz(a: np.ndarray, bt: np.ndarray) -> np.ndarray:
    """acc = 0; for k ascending: acc = rz32(acc + fp32(a[:, k] * bt[k, :])),
    the sum formed exactly in float64 (two FP32 values) then truncated."""
    a = np.ascontiguousarray(np.asarray(a, F32).T)
    bt = np.ascontiguousarray(bt, F32)
    acc = np.zeros((a.shape[1], bt.shape[1]), F32)
    for k in range(a.shape[0]):
        prod = a[k][:, None] * bt[k][None, :]
        acc = _to_f32_toward_zero(acc.astype(np.float64) + prod.astype(np.float64))
    return acc


# ----------------------------------------------------------------- GEMM ----
def dot_f32(a: np.ndarray, bt: np.ndarray) -> np.ndarray:
    """a @ bt as FP32 values: float64 accumulation rounded once to FP32, or,
    inside ``accumulation(kind)``, one of the plain FP32 orders."""
    kind = _ACCUMULATION[0]
    if kind == "f32":
        return _dot_f32_sequential(a, bt)
    if kind == "f32_desc":
        return _dot_f32_sequential(a, bt, descending=True)
    if kind == "f32_rz":
        return _dot_f32_rz(a, bt)
    if kind == "f32_blas":
        return np.matmul(np.asarray(a, F32), np.asarray(bt, F32))
    return np.matmul(np.asarray(a, np.float64), np.asarray(bt, np.float64)).astype(F32)


def gemm(a: np.ndarray, b: np.ndarray, out: str = "bf16") -> np.ndarray:
    """C = A . B^T with A [M,K], B [N,K] (bf16 values), FP32 result.

    The batch-invariant dense GEMM of "Finish RL Training Faster", section
    "让训练前向使用推理的数值": one result per (row, column) whatever the batch.
    Each dot product is formed in float64 and rounded once to FP32, so the
    oracle's value does not depend on how the matmul library blocks the sum
    (a 1-row and a T-row call agree).  ``out`` = "bf16" rounds the FP32
    result once more; "f32" returns it as is (LM head, router, indexer).
    """
    c = dot_f32(a, b.T if hasattr(b, "T") else np.asarray(b).T)
    return bf16_round(c) if out == "bf16" else c.astype(F32)


# ------------------------------------------------------------ RMSNorm ----
def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """y = bf16(x * 1/sqrt(mean(x^2) + eps) * w) over the last axis, FP32 inside."""
    x = np.asarray(x, F32)
    ms = np.mean(x * x, axis=-1, dtype=F32, keepdims=True)
    inv = F32(1.0) / np.sqrt(ms + F32(eps), dtype=F32)
    return bf16_round((x * inv) * np.asarray(w, F32))


def add_rmsnorm(x: np.ndarray, r: np.ndarray, w: np.ndarray, eps: float):
    """Fused residual add + RMSNorm ("No More Train-Inference Mismatch", section
    "方法细节": the RMSNorm with an added residual is one imported op).

    r' = bf16(x + r) is the new residual; the bf16-rounded sum is what gets
    normalised: y = rmsnorm(r').  Returns (r', y).
    """
    r2 = bf16_round(np.asarray(x, F32) + np.asarray(r, F32))
    return r2, rmsnorm(r2, w, eps)


# ------------------------------------------------------------- SiLU-mul ----
def silu_mul(gate_up: np.ndarray) -> np.ndarray:
    """SiLU-gated MLP activation: [gate | up] -> bf16(silu(gate) * up),
    silu(g) = g / (1 + exp(-g)) in FP32 ("No More Train-Inference Mismatch",
    section "方法细节": fused SiLU MLP)."""
    gu = np.asarray(gate_up, F32)
    I = gu.shape[-1] // 2
    g, u = gu[..., :I], gu[..., I:]
    s = g / (F32(1.0) + np.exp(-g, dtype=F32))
    return bf16_round(s * u)


# ----------------------------------------------------------------- RoPE ----
def rope_table(theta: float, D: int, max_pos: int):
    """cos/sin tables [max_pos, D/2]: angle = pos * theta^(-2i/D), computed in
    float64 and stored as float32 (rotate-half RoPE)."""
    i = np.arange(D // 2, dtype=np.float64)
    inv_freq = theta ** (-(2.0 * i) / D)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.cos(ang).astype(F32), np.sin(ang).astype(F32)


def rope(x: np.ndarray, pos: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate-half RoPE on x [T, H, D]: pairs (i, i + D/2)."""
    x = np.asarray(x, F32)
    h = x.shape[-1] // 2
    c = cos[pos][:, None, :]
    s = sin[pos][:, None, :]
    x1, x2 = x[..., :h], x[..., h:]
    return bf16_round(np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1))


def qk_norm_rope(x, pos, w, eps, cos, sin):
    """Per-head RMSNorm (skipped when ``w`` is None), then RoPE."""
    if w is not None:
        x = rmsnorm(x, w, eps)
    return rope(x, pos, cos, sin)


# ------------------------------------------------------------- FP8 KV ----
def fp8_quant_rows(x: np.ndarray):
    """Quantise the last axis of x to e4m3 with one FP32 scale per row:
    s = amax / 448 (IEEE division; s = 1 when amax = 0), code = e4m3(x / s).

    The KV cache stays in FP8 ("Finish RL Training Faster", section
    "让训练前向使用推理的数值": FP8 KV kept, every path makes the same round trip).
    """
    x = np.asarray(x, F32)
    amax = np.max(np.abs(x), axis=-1)
    s = np.where(amax == 0, F32(1.0), amax / F32(448.0)).astype(F32)
    codes = f32_to_e4m3(x / s[..., None])
    return codes, s


def fp8_dequant_rows(codes: np.ndarray, s: np.ndarray) -> np.ndarray:
    """x_hat = bf16(float(code) * s): one FP32 multiply and one rounding."""
    return bf16_round(e4m3_to_f32(codes) * np.asarray(s, F32)[..., None])


def kv_roundtrip(x: np.ndarray) -> np.ndarray:
    """Quantise then dequantise [T, H, D] per (token, head)."""
    c, s = fp8_quant_rows(x)
    return fp8_dequant_rows(c, s)


# ----------------------------------------------------------- attention ----
def attention(q, k, v, q_pos, k_pos, scale):
    """Causal GQA attention as a plain softmax over every visible key.

    q [Tq, Hq, D]; k, v [Tk, Hkv, D]; key j is visible to query i iff
    k_pos[j] <= q_pos[i].  FP32 scores and probabilities, bf16 output.
    One attention operator for prefill, decode and training ("Finish RL
    Training Faster", section "让训练前向使用推理的数值").
    """
    q = np.asarray(q, F32)
    k = np.asarray(k, F32)
    v = np.asarray(v, F32)
    Tq, Hq, D = q.shape
    Hkv = k.shape[1]
    grp = Hq // Hkv
    vis = np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None]
    o = np.zeros((Tq, Hq, D), F32)
    for h in range(Hq):
        g = h // grp
        s = dot_f32(q[:, h, :], k[:, g, :].T) * F32(scale)
        s = np.where(vis, s, F32(-np.inf))
        m = np.max(s, axis=1, keepdims=True)
        m = np.where(np.isfinite(m), m, F32(0.0))
        p = np.exp(s - m, dtype=F32)
        l = np.sum(p, axis=1, keepdims=True, dtype=F32)
        l = np.where(l > 0, l, F32(1.0))
        o[:, h, :] = dot_f32(p, v[:, g, :]) / l
    return bf16_round(o)


def sparse_attention(q, k_all, v_all, idx, q_pos, scale):
    """Attention of each query over the key positions listed in idx [Tq, topk]
    (ascending, -1 = padding); positions beyond the query are not visible."""
    q = np.asarray(q, F32)
    Tq, Hq, D = q.shape
    out = np.zeros((Tq, Hq, D), F32)
    for t in range(Tq):
        sel = idx[t][idx[t] >= 0]
        sel = sel[sel <= q_pos[t]]
        if sel.size == 0:
            continue
        out[t:t + 1] = attention(q[t:t + 1], k_all[sel], v_all[sel],
                                 np.array([q_pos[t]]), sel, scale)
    return out


# ---------------------------------------------------------------- Top-K ----
def topk_positions(scores: np.ndarray, valid_len: np.ndarray, k: int) -> np.ndarray:
    """Sparse-attention Top-K: per row, the k largest scores among indices
    < valid_len; equal scores -> the lower index wins; the chosen indices are
    returned in ascending position order, padded with -1.  -inf is never
    chosen ("Finish RL Training Faster", section "让训练前向使用推理的数值":
    fixed tie-break, fixed position order)."""
    scores = np.asarray(scores, F32)
    R, n = scores.shape
    out = np.full((R, k), -1, np.int32)
    for r in range(R):
        nv = int(valid_len[r])
        s = scores[r, :nv]
        cand = np.nonzero(s > F32(-np.inf))[0]
        order = np.lexsort((cand, -s[cand].astype(np.float64)))
        chosen = np.sort(cand[order[:k]])
        out[r, :chosen.size] = chosen
    return out


def router_topk(logits: np.ndarray, k: int):
    """MoE router: top-k experts by logit (ties -> lower expert id), slot order =
    rank (logit descending, id ascending); the gate weight of a slot is the
    full softmax probability of that expert (no renormalisation)."""
    z = np.asarray(logits, F32)
    R, E = z.shape
    idx = np.zeros((R, k), np.int32)
    w = np.zeros((R, k), F32)
    m = np.max(z, axis=1, keepdims=True)
    e = np.exp(z - m, dtype=F32)
    p = e / np.sum(e, axis=1, keepdims=True, dtype=F32)
    for r in range(R):
        order = np.lexsort((np.arange(E), -z[r].astype(np.float64)))[:k]
        idx[r] = order
        w[r] = p[r, order]
    return idx, w


# ------------------------------------------------- FP8 block-scaled GEMM ----
def act_quant_fp8(x: np.ndarray, group: int = 128):
    """Per-token activation quantisation in groups of 128 along K:
    codes uint8 [M, K], scales float32 [M, ceil(K/128)]."""
    x = np.asarray(x, F32)
    M, K = x.shape
    G = (K + group - 1) // group
    xp = np.zeros((M, G * group), F32)
    xp[:, :K] = x
    c, s = fp8_quant_rows(xp.reshape(M, G, group))
    return c.reshape(M, G * group)[:, :K], s


def gemm_fp8_block(a_codes, sa, b_codes, sb, out: str = "bf16"):
    """Block-scaled FP8 GEMM: C[m,n] = sum over 128-wide K blocks kb, in
    ascending order, of (sa[m,kb] * sb[n//128,kb]) * (sum_k a[m,k] b[n,k]),
    FP32 throughout; the MoE "unified quantisation rounding" of
    "Finish RL Training Faster", section "让训练前向使用推理的数值"."""
    a = e4m3_to_f32(a_codes)
    b = e4m3_to_f32(b_codes)
    M, K = a.shape
    N = b.shape[0]
    acc = np.zeros((M, N), F32)
    for kb in range((K + 127) // 128):
        ks = slice(kb * 128, min(K, kb * 128 + 128))
        blk = dot_f32(a[:, ks], b[:, ks].T)
        sbn = np.repeat(np.asarray(sb, F32)[:, kb], 128)[:N]
        acc = acc + (np.asarray(sa, F32)[:, kb][:, None] * sbn[None, :]) * blk
    return bf16_round(acc) if out == "bf16" else acc


def moe_combine(y: np.ndarray, w: np.ndarray, shared=None) -> np.ndarray:
    """out[t] = bf16(sum over slots s = 0..k-1, in order, of w[t,s]*y[t,s]
    (+ shared[t] last)), one FP32 accumulator ("Finish RL Training Faster",
    section "让训练前向使用推理的数值": expert outputs merged in FP32 in fixed
    slot order)."""
    y = np.asarray(y, F32)
    w = np.asarray(w, F32)
    acc = np.zeros((y.shape[0], y.shape[2]), F32)
    for s in range(y.shape[1]):
        acc = acc + w[:, s:s + 1] * y[:, s, :]
    if shared is not None:
        acc = acc + np.asarray(shared, F32)
    return bf16_round(acc)


# ----------------------------------------------------------- log-softmax ----
def log_softmax(z: np.ndarray) -> np.ndarray:
    """lp = z - (m + log sum exp(z - m)) over the last axis, FP32."""
    z = np.asarray(z, F32)
    m = np.max(z, axis=-1, keepdims=True)
    lse = m + np.log(np.sum(np.exp(z - m, dtype=F32), axis=-1, keepdims=True, dtype=F32))
    return (z - lse).astype(F32)


def logprob(z: np.ndarray, target: np.ndarray) -> np.ndarray:
    """Per-token logprob of the target id: the compared quantity of "Finish RL
    Training Faster", section "零差异需要一个精确的比较对象"."""
    z = np.asarray(z, F32)
    m = np.max(z, axis=-1)
    lse = m + np.log(np.sum(np.exp(z - m[:, None], dtype=F32), axis=-1, dtype=F32))
    return (z[np.arange(z.shape[0]), np.asarray(target)] - lse).astype(F32)


# ------------------------------------------------------------- metrics ----
def diff_stats(lp_a: np.ndarray, lp_b: np.ndarray) -> dict:
    """max, mean, std of |lp_a - lp_b| and the k3 KL estimate over tokens.

    k3 with log-ratio d = lp_a - lp_b: mean((exp(-d) - 1) + d); it is exactly
    0 when every d is 0 (the pages' acceptance test, "Finish RL Training
    Faster", section "零差异需要一个精确的比较对象")."""
    a = np.asarray(lp_a, np.float64)
    b = np.asarray(lp_b, np.float64)
    d = a - b
    ad = np.abs(d)
    k3 = np.expm1(-d) + d
    return {"max": float(ad.max(initial=0.0)), "mean": float(ad.mean()) if ad.size else 0.0,
            "std": float(ad.std()) if ad.size else 0.0,
            "k3": float(k3.mean()) if k3.size else 0.0}
