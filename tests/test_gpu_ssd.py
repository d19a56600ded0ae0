"""Mamba-2 SSD scan: parity with the oracle's sequential recurrence, and
bitwise equality of one prefill, a chunked prefill and a token-by-token decode
(decode replays the prefill chunk order)."""
import numpy as np
import pytest
import torch

import synth
from oracle.codecs import bf16_to_f32
from oracle.ssd import ssd_sequential

pytestmark = pytest.mark.gpu
REL = 1e-2


@pytest.fixture(scope="module")
def B():
    from invariant_forward_bitwise_gb300 import biv, build
    build.build()
    biv.load()
    return biv


def bits(t):
    return t.detach().contiguous().view(torch.uint8).cpu().numpy()


class SSDRunner:
    def __init__(self, B, nseq, H, Q):
        self.B, self.H, self.Q = B, H, Q
        P, N = 64, 128
        self.state = torch.zeros(nseq, H, P, N, dtype=torch.float32, device="cuda")
        self.bx = torch.zeros(nseq, Q, H, P, dtype=torch.bfloat16, device="cuda")
        self.bB = torch.zeros(nseq, Q, N, dtype=torch.bfloat16, device="cuda")
        self.bC = torch.zeros(nseq, Q, N, dtype=torch.bfloat16, device="cuda")
        self.bdt = torch.zeros(nseq, Q, H, dtype=torch.float32, device="cuda")

    def run(self, x, dt, A, Bm, Cm, D, row0, n, pos0):
        """x [rows,H,P] bf16 cuda ...; row0/n/pos0 lists per sequence; returns y."""
        B = self.B
        rows = x.shape[0]
        y = torch.full((rows, self.H * 64), float("nan"), dtype=torch.bfloat16, device="cuda")
        keep = [torch.tensor(v, dtype=torch.int32, device="cuda") for v in (row0, n, pos0)]
        d = B.SSDDesc()
        d.x, d.x_stride = x.data_ptr(), x.stride(0)
        d.dt, d.dt_stride = dt.data_ptr(), dt.stride(0)
        d.A, d.D = A.data_ptr(), D.data_ptr()
        d.B, d.B_stride = Bm.data_ptr(), Bm.stride(0)
        d.C, d.C_stride = Cm.data_ptr(), Cm.stride(0)
        d.y, d.y_stride = y.data_ptr(), y.stride(0)
        d.H, d.P, d.N, d.chunk = self.H, 64, 128, self.Q
        d.nseq = len(row0)
        d.row0, d.n, d.pos0 = keep[0].data_ptr(), keep[1].data_ptr(), keep[2].data_ptr()
        d.max_n = max(n)
        d.state, d.buf_x, d.buf_B = self.state.data_ptr(), self.bx.data_ptr(), self.bB.data_ptr()
        d.buf_C, d.buf_dt = self.bC.data_ptr(), self.bdt.data_ptr()
        B.biv_ssd_scan(d)
        torch.cuda.synchronize()
        return y


def inputs(seed, T, H):
    g = synth.rng(seed)
    cfg = synth.SSDConfig(heads=H)
    x, dt, A, Bm, Cm, D = synth.ssd_inputs(g, T, cfg)
    return x, dt, A, Bm, Cm, D


@pytest.mark.parametrize("Q,T", [(64, 150), (256, 600)])
def test_ssd_prefill_parity(B, Q, T):
    H = 4
    x, dt, A, Bm, Cm, D = inputs(Q + T, T, H)
    r = SSDRunner(B, 1, H, Q)
    y = r.run(x.reshape(T, H * 64).cuda(), torch.from_numpy(dt).cuda(), torch.from_numpy(A).cuda(),
              Bm.cuda(), Cm.cuda(), torch.from_numpy(D).cuda(), [0], [T], [0])
    ref, _ = ssd_sequential(x.float().numpy(), dt, A, Bm.float().numpy(), Cm.float().numpy(), D)
    got = bf16_to_f32(y.cpu().view(torch.int16).numpy().view(np.uint16)).reshape(T, H, 64)
    err = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
    assert err < REL, err


@pytest.mark.parametrize("Q", [64, 256])
def test_ssd_decode_replays_prefill_bitwise(B, Q):
    H, T = 3, 2 * Q + 37
    x, dt, A, Bm, Cm, D = inputs(7 + Q, T, H)
    xd = x.reshape(T, H * 64).cuda()
    dtd, Ad, Dd = torch.from_numpy(dt).cuda(), torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    Bd, Cd = Bm.cuda(), Cm.cuda()
    full = SSDRunner(B, 1, H, Q).run(xd, dtd, Ad, Bd, Cd, Dd, [0], [T], [0])
    # chunked prefill: 3 calls with ragged cuts
    rc = SSDRunner(B, 1, H, Q)
    parts, at = [], 0
    for n in [Q // 2 + 3, Q + 1, T - (Q // 2 + 3) - (Q + 1)]:
        parts.append(rc.run(xd[at:at + n], dtd[at:at + n], Ad, Bd[at:at + n], Cd[at:at + n], Dd, [0], [n], [at]))
        at += n
    assert np.array_equal(bits(torch.cat(parts)), bits(full))
    # prompt prefill, then one token at a time
    rd = SSDRunner(B, 1, H, Q)
    P0 = Q - 5
    outs = [rd.run(xd[:P0], dtd[:P0], Ad, Bd[:P0], Cd[:P0], Dd, [0], [P0], [0])]
    for t in range(P0, T):
        outs.append(rd.run(xd[t:t + 1], dtd[t:t + 1], Ad, Bd[t:t + 1], Cd[t:t + 1], Dd, [0], [1], [t]))
    assert np.array_equal(bits(torch.cat(outs)), bits(full))


def test_ssd_batch_of_sequences_matches_alone(B):
    H, Q = 2, 64
    lens = [70, 5, 130]
    xs = [inputs(100 + i, L, H) for i, L in enumerate(lens)]
    A, D = torch.from_numpy(xs[0][2]).cuda(), torch.from_numpy(xs[0][5]).cuda()
    x = torch.cat([v[0].reshape(v[0].shape[0], -1) for v in xs]).cuda()
    dt = torch.cat([torch.from_numpy(v[1]) for v in xs]).cuda()
    Bm = torch.cat([v[3] for v in xs]).cuda()
    Cm = torch.cat([v[4] for v in xs]).cuda()
    row0 = [0, 70, 75]
    yb = SSDRunner(B, 3, H, Q).run(x, dt, A, Bm, Cm, D, row0, lens, [0, 0, 0])
    for i, L in enumerate(lens):
        r0 = row0[i]
        y1 = SSDRunner(B, 1, H, Q).run(x[r0:r0 + L], dt[r0:r0 + L], A, Bm[r0:r0 + L], Cm[r0:r0 + L], D, [0], [L], [0])
        assert np.array_equal(bits(y1), bits(yb[r0:r0 + L])), i


def test_ssd_16k_tokens_parity_across_chunk_boundaries(B):
    """16384 tokens (64 chunks of 256) through the parallel many-row path,
    against the oracle's sequential recurrence carried over every chunk."""
    H, T, Q = 4, 16384, 256
    x, dt, A, Bm, Cm, D = inputs(T, T, H)
    r = SSDRunner(B, 1, H, Q)
    y = r.run(x.reshape(T, H * 64).cuda(), torch.from_numpy(dt).cuda(), torch.from_numpy(A).cuda(),
              Bm.cuda(), Cm.cuda(), torch.from_numpy(D).cuda(), [0], [T], [0])
    ref, h = ssd_sequential(x.float().numpy(), dt, A, Bm.float().numpy(), Cm.float().numpy(), D)
    got = bf16_to_f32(y.cpu().view(torch.int16).numpy().view(np.uint16)).reshape(T, H, 64)
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) < REL
    # the carried state after the last full chunk (= the final state here)
    st = r.state[0].cpu().numpy()
    assert np.max(np.abs(st - h)) / np.max(np.abs(h)) < REL
