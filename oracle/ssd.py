"""Mamba-2 SSD (state-space dual) oracle.  TEST INFRASTRUCTURE ONLY.

The pages require that the Mamba-2 decode step replays the prefill's chunked
computation order, rather than only reaching an approximately equal state
("Finish RL Training Faster", section "一致性有多个层面").  The oracle itself
uses the plain sequential recurrence of the Mamba-2 SSM, for which decode and
prefill are the same loop by construction:

    h_t = exp(dt_t * A) * h_{t-1} + dt_t * x_t B_t^T      (state [P, N] per head)
    y_t = h_t C_t + D * x_t

with x [T, H, P], dt [T, H] (already through softplus), A [H] (< 0),
B, C [T, N] (one group shared by all heads), D [H].

``ssd_chunked`` is a second, independent form of the same map (intra-chunk
decay-masked products plus carried chunk states) used only to pin the
recurrence and to state the chunk algebra the CUDA kernel follows.
"""
from __future__ import annotations

import numpy as np

from .codecs import bf16_round


def ssd_sequential(x, dt, A, B, C, D, h0=None, dtype=np.float32, round_out=True):
    """Sequential recurrence; returns (y [T,H,P], final state [H,P,N])."""
    x = np.asarray(x, dtype)
    dt = np.asarray(dt, dtype)
    A = np.asarray(A, dtype)
    B = np.asarray(B, dtype)
    C = np.asarray(C, dtype)
    D = np.asarray(D, dtype)
    T, H, P = x.shape
    N = B.shape[1]
    h = np.zeros((H, P, N), dtype) if h0 is None else np.array(h0, dtype)
    y = np.zeros((T, H, P), dtype)
    for t in range(T):
        decay = np.exp(dt[t] * A).astype(dtype)                       # [H]
        upd = (dt[t][:, None] * x[t])[:, :, None] * B[t][None, None, :]
        h = decay[:, None, None] * h + upd.astype(dtype)
        y[t] = np.einsum("hpn,n->hp", h, C[t]).astype(dtype) + D[:, None] * x[t]
    if round_out:
        y = bf16_round(y.astype(np.float32))
    return y, h


def ssd_chunked(x, dt, A, B, C, D, chunk, start_pos=0, h0=None, dtype=np.float64):
    """Chunked SSD with chunks aligned to absolute positions (multiples of
    ``chunk``), the first token of x being at ``start_pos``.

    Inside a chunk with log-decays a_t = dt_t A and inclusive prefix sums
    L_t (from the chunk's first position):
      y_t = sum_{s<=t in chunk} exp(L_t - L_s) (C_t . B_s) dt_s x_s
            + exp(L_t) (h_in C_t) + D x_t
      h_out = exp(L_last) h_in + sum_s exp(L_last - L_s) dt_s x_s B_s^T
    Returns (y, final state) unrounded.
    """
    x = np.asarray(x, dtype)
    dt = np.asarray(dt, dtype)
    A = np.asarray(A, dtype)
    B = np.asarray(B, dtype)
    C = np.asarray(C, dtype)
    D = np.asarray(D, dtype)
    T, H, P = x.shape
    N = B.shape[1]
    h = np.zeros((H, P, N), dtype) if h0 is None else np.array(h0, dtype)
    y = np.zeros((T, H, P), dtype)
    t0 = 0
    while t0 < T:
        pos = start_pos + t0
        end = min(T, t0 + (chunk - pos % chunk))
        sl = slice(t0, end)
        a = dt[sl] * A[None, :]                       # [Q, H]
        L = np.cumsum(a, axis=0)                      # inclusive
        CB = C[sl] @ B[sl].T                          # [Q, Q]
        Q = end - t0
        mask = np.tril(np.ones((Q, Q), bool))
        for hh in range(H):
            dec = np.exp(L[:, hh][:, None] - L[:, hh][None, :])
            M = np.where(mask, dec * CB, 0.0)
            xs = dt[sl][:, hh][:, None] * x[sl][:, hh, :]    # [Q, P]
            y[sl, hh, :] = (M @ xs
                            + np.exp(L[:, hh])[:, None] * (C[sl] @ h[hh].T)
                            + D[hh] * x[sl][:, hh, :])
            wl = np.exp(L[-1, hh] - L[:, hh])                 # [Q]
            h[hh] = np.exp(L[-1, hh]) * h[hh] + (xs * wl[:, None]).T @ B[sl]
        t0 = end
    return y, h
