"""Pins for the oracle's backward (CPU only): each gradient against torch
autograd in float64 of the forward definition (a library routine), and the
RMSNorm and attention ones also against central finite differences; a
planted sign error in the RMSNorm gradient is caught."""
import numpy as np
import torch

from oracle import backward as bw

F64 = np.float64


def _fd(f, x, eps=1e-6):
    """Central finite differences of scalar f at x (float64)."""
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        xp, xm = x.copy(), x.copy()
        xp[i] += eps
        xm[i] -= eps
        g[i] = (f(xp) - f(xm)) / (2 * eps)
    return g


def test_rmsnorm_backward_against_autograd_and_fd():
    g = np.random.default_rng(0)
    x, w, dy = g.standard_normal((4, 24)), 1 + 0.1 * g.standard_normal(24), g.standard_normal((4, 24))
    dx, dw = bw.rmsnorm_backward(x, w, dy, 1e-6)
    xt = torch.tensor(x, requires_grad=True)
    wt = torch.tensor(w, requires_grad=True)
    y = xt * torch.rsqrt((xt * xt).mean(-1, keepdim=True) + 1e-6) * wt
    y.backward(torch.tensor(dy))
    assert np.allclose(dx, xt.grad.numpy(), atol=1e-12) and np.allclose(dw, wt.grad.numpy(), atol=1e-12)

    def f(xx):
        inv = 1 / np.sqrt(np.mean(xx * xx, -1, keepdims=True) + 1e-6)
        return np.sum(xx * inv * w * dy)
    assert np.allclose(dx, _fd(f, x), atol=1e-6)
    # a planted sign error in the correction term is caught
    inv = 1 / np.sqrt(np.mean(x * x, -1, keepdims=True) + 1e-6)
    bad = inv * dy * w + x * inv ** 3 * np.mean(dy * w * x, -1, keepdims=True)
    assert not np.allclose(bad, xt.grad.numpy(), atol=1e-6)


def test_silu_mul_backward_against_autograd():
    g = np.random.default_rng(1)
    gu, dy = 3 * g.standard_normal((5, 32)), g.standard_normal((5, 16))
    got = bw.silu_mul_backward(gu, dy)
    t = torch.tensor(gu, requires_grad=True)
    y = torch.nn.functional.silu(t[:, :16]) * t[:, 16:]
    y.backward(torch.tensor(dy))
    assert np.allclose(got, t.grad.numpy(), atol=1e-12)


def test_logprob_backward_against_autograd_and_sums_to_zero():
    g = np.random.default_rng(2)
    z, tgt, dlp = 3 * g.standard_normal((6, 50)), g.integers(0, 50, 6), g.standard_normal(6)
    got = bw.logprob_backward(z, tgt, dlp)
    t = torch.tensor(z, requires_grad=True)
    lp = torch.log_softmax(t, -1)[torch.arange(6), torch.tensor(tgt)]
    lp.backward(torch.tensor(dlp))
    assert np.allclose(got, t.grad.numpy(), atol=1e-12)
    assert np.allclose(got.sum(1), 0.0, atol=1e-12)       # softmax's gradient sums to zero


def test_attention_backward_against_autograd_and_fd():
    g = np.random.default_rng(3)
    Tq, Tk, Hq, Hkv, D = 5, 7, 4, 2, 8
    q, k, v = g.standard_normal((Tq, Hq, D)), g.standard_normal((Tk, Hkv, D)), g.standard_normal((Tk, Hkv, D))
    do = g.standard_normal((Tq, Hq, D))
    qpos, kpos = np.arange(2, 7), np.arange(7)
    dq, dk, dv = bw.attention_backward(q, k, v, qpos, kpos, 0.35, do)
    qt, kt, vt = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    mask = torch.tensor(kpos[None, :] <= qpos[:, None])
    outs = []
    for h in range(Hq):
        s = (qt[:, h] @ kt[:, h // 2].T) * 0.35
        s = s.masked_fill(~mask, float("-inf"))
        outs.append(torch.softmax(s, -1) @ vt[:, h // 2])
    torch.stack(outs, 1).backward(torch.tensor(do))
    for a, b in [(dq, qt), (dk, kt), (dv, vt)]:
        assert np.allclose(a, b.grad.numpy(), atol=1e-10)

    def f(vv):
        o = 0.0
        for h in range(Hq):
            s = np.where(kpos[None, :] <= qpos[:, None], q[:, h] @ k[:, h // 2].T * 0.35, -np.inf)
            p = np.exp(s - s.max(1, keepdims=True))
            p /= p.sum(1, keepdims=True)
            o += np.sum((p @ vv[:, h // 2]) * do[:, h])
        return o
    assert np.allclose(dv, _fd(f, v), atol=1e-6)
