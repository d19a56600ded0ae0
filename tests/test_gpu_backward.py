"""Backward kernels against the float64 oracle: RMSNorm, SiLU-mul, logprob and
causal GQA attention (FP32 on the GPU: within 1e-3 relative of float64).
Each runs twice with the same bits, and a row's gradient does not depend on
the other rows of the call."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import backward as bw
from oracle.codecs import bf16_to_f32

pytestmark = pytest.mark.gpu
REL = 1e-3


@pytest.fixture(scope="module")
def B():
    from invariant_forward_bitwise_gb300 import biv, build
    build.build()
    biv.load()
    return biv


def h32(t):
    return bf16_to_f32(t.detach().cpu().view(torch.int16).numpy().view(np.uint16))


def rel(got, ref):
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(np.asarray(got, np.float64) - ref)) / max(np.max(np.abs(ref)), 1e-30))


def bits(t):
    return t.detach().contiguous().view(torch.uint8).cpu().numpy()


@pytest.mark.parametrize("d", [256, 2048, 2560])
def test_rmsnorm_backward(B, d):
    g = synth.rng(d)
    R = 37
    x = synth.normal_bf16(g, (R, d)).cuda()
    w = synth.to_bf16(1 + synth.normal_f32(g, (d,), 0.1)).cuda()
    dy = torch.from_numpy(synth.normal_f32(g, (R, d))).cuda()
    dx = torch.empty(R, d, device="cuda")
    dw = torch.empty(d, device="cuda")
    B.biv_rmsnorm_backward(x, w, dy, dx, dw, 1e-6)
    torch.cuda.synchronize()
    rdx, rdw = bw.rmsnorm_backward(h32(x), h32(w), dy.cpu().numpy(), 1e-6)
    assert rel(dx.cpu().numpy(), rdx) < REL and rel(dw.cpu().numpy(), rdw) < REL
    dx2, dw2 = torch.empty_like(dx), torch.empty_like(dw)
    B.biv_rmsnorm_backward(x, w, dy, dx2, dw2, 1e-6)
    one = torch.empty(1, d, device="cuda")
    B.biv_rmsnorm_backward(x[5:6], w, dy[5:6], one, torch.empty(d, device="cuda"), 1e-6)
    torch.cuda.synchronize()
    assert np.array_equal(bits(dx2), bits(dx)) and np.array_equal(bits(dw2), bits(dw))
    assert np.array_equal(bits(one), bits(dx[5:6]))


def test_silu_mul_backward(B):
    g = synth.rng(3)
    R, I = 29, 688
    gu = synth.normal_bf16(g, (R, 2 * I), 2.0).cuda()
    dy = torch.from_numpy(synth.normal_f32(g, (R, I))).cuda()
    out = torch.empty(R, 2 * I, device="cuda")
    B.biv_silu_mul_backward(gu, dy, out)
    torch.cuda.synchronize()
    assert rel(out.cpu().numpy(), bw.silu_mul_backward(h32(gu), dy.cpu().numpy())) < REL


@pytest.mark.parametrize("V", [4096, 151936])
def test_logprob_backward(B, V):
    g = synth.rng(V)
    T = 9
    z = torch.from_numpy(synth.normal_f32(g, (T, V), 3.0)).cuda()
    tg = torch.from_numpy(g.integers(0, V, T).astype(np.int32)).cuda()
    dlp = torch.from_numpy(synth.normal_f32(g, (T,))).cuda()
    dz = torch.empty(T, V, device="cuda")
    B.biv_logprob_backward(z, tg, dlp, dz)
    torch.cuda.synchronize()
    ref = bw.logprob_backward(z.cpu().numpy(), tg.cpu().numpy(), dlp.cpu().numpy())
    assert rel(dz.cpu().numpy(), ref) < REL
    assert B.biv_poll_error() == 0


@pytest.mark.parametrize("D,Hq,Hkv", [(64, 4, 2), (128, 16, 8), (80, 4, 1)])
def test_attention_backward(B, D, Hq, Hkv):
    g = synth.rng(D * Hq)
    Tq, Tk = 150, 180                                    # the last 150 positions of 180 keys
    q = synth.normal_bf16(g, (Tq, Hq, D)).cuda()
    k = synth.normal_bf16(g, (Tk, Hkv, D)).cuda()
    v = synth.normal_bf16(g, (Tk, Hkv, D)).cuda()
    do = synth.normal_bf16(g, (Tq, Hq, D)).cuda()
    qpos = torch.arange(Tk - Tq, Tk, dtype=torch.int32, device="cuda")
    kpos = torch.arange(Tk, dtype=torch.int32, device="cuda")
    scale = 1 / math.sqrt(D)
    dq = torch.empty(Tq, Hq, D, device="cuda")
    dk = torch.empty(Tk, Hkv, D, device="cuda")
    dv = torch.empty(Tk, Hkv, D, device="cuda")
    B.biv_attention_backward(q, k, v, do, qpos, kpos, scale, dq, dk, dv)
    torch.cuda.synchronize()
    rq, rk, rv = bw.attention_backward(h32(q), h32(k), h32(v), qpos.cpu().numpy(), kpos.cpu().numpy(),
                                       scale, h32(do))
    for got, ref in [(dq, rq), (dk, rk), (dv, rv)]:
        assert rel(got.cpu().numpy(), ref) < REL
    # again: the same bits; one query row alone: its dq bits
    dq2, dk2, dv2 = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)
    B.biv_attention_backward(q, k, v, do, qpos, kpos, scale, dq2, dk2, dv2)
    dq1 = torch.empty(1, Hq, D, device="cuda")
    B.biv_attention_backward(q[70:71], k, v, do[70:71], qpos[70:71], kpos, scale, dq1,
                             torch.empty_like(dk), torch.empty_like(dv))
    torch.cuda.synchronize()
    for a, b in [(dq2, dq), (dk2, dk), (dv2, dv)]:
        assert np.array_equal(bits(a), bits(b))
    assert np.array_equal(bits(dq1), bits(dq[70:71]))
