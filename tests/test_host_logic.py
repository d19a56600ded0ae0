"""Host-side scheduling logic of the model harness (no GPU): query blocks,
prefill rows and the decode-graph batch buckets."""
import types

import numpy as np
import pytest

import synth


@pytest.fixture(scope="module")
def model_mod():
    from invariant_forward_bitwise_gb300 import model
    return model


def test_qblocks_cover_rows_in_order_within_one_sequence(model_mod):
    g = np.random.default_rng(3)
    row_seq = np.repeat(np.arange(7, dtype=np.int32), g.integers(1, 90, size=7))
    for per in (1, 8, 32, 64):
        qb = model_mod.qblocks_for(row_seq, per)
        # consecutive, gap-free cover of every row, in order
        assert qb[0, 0] == 0 and int(qb[-1].sum()) == row_seq.size
        assert np.array_equal(qb[1:, 0], qb[:-1, 0] + qb[:-1, 1])
        for r0, n in qb:
            assert 1 <= n <= per
            assert np.all(row_seq[r0:r0 + n] == row_seq[r0])   # one sequence per block
        # a block ends early only at a sequence boundary
        for (r0, n), (r1, _) in zip(qb[:-1], qb[1:]):
            if n < per:
                assert row_seq[r1] != row_seq[r0]


def test_prefill_rows_emit_the_logprob_of_the_next_token(model_mod):
    cfg = synth.TINY
    seqs = synth.tiny_sequences(cfg, n=3, lo=10, hi=30, seed=4)
    starts = [0, 3, 5]
    ends = [s.length for s in seqs]
    lm_from = [s.prompt_len - 1 for s in seqs]
    seq_slot, pos, ids, lm_rows, targets, owner = model_mod.prefill_rows(
        seqs, [10, 11, 12], starts, ends, lm_from)
    assert len(pos) == sum(e - b for b, e in zip(starts, ends))
    at = 0
    for i, s in enumerate(seqs):
        for p in range(starts[i], ends[i]):
            assert (seq_slot[at], pos[at], ids[at]) == (10 + i, p, int(s.tokens[p]))
            at += 1
    # every logprob row predicts token p + 1 of its own sequence, from lm_from on
    want = [(i, p) for i, s in enumerate(seqs) for p in range(max(starts[i], lm_from[i]), ends[i])
            if p + 1 < s.length]
    assert owner == want
    for r, t, (i, p) in zip(lm_rows, targets, owner):
        assert pos[r] == p and t == int(seqs[i].tokens[p + 1])


def test_decode_buckets(model_mod):
    DG = model_mod.DecodeGraphs
    b = list(DG.BUCKETS)
    assert b == sorted(set(b)) and b[0] == 1
    fake = types.SimpleNamespace(BUCKETS=DG.BUCKETS)
    for n in range(1, b[-1] + 1):
        k = DG.bucket(fake, n)
        assert k >= n and k in b
        assert k == min(x for x in b if x >= n)                 # the smallest that fits
    with pytest.raises(ValueError):
        DG.bucket(fake, b[-1] + 1)


def test_split_blocks_two_calls_only_when_decode_blocks_dominate(model_mod):
    G = 2
    # a prefill step: 64-row blocks with two short sequence tails -> one call
    qb = np.array([(0, 64), (64, 64), (128, 5), (133, 64), (197, 3)], np.int32)
    out, n = model_mod.split_blocks(qb, G)
    assert n == 0 and np.array_equal(out, qb)
    # a mixed step: one prefill chunk's blocks next to more decode rows -> the
    # multi-row blocks first, their relative order kept, then the rest
    qb = np.array([(0, 1), (1, 32), (33, 1), (34, 32), (66, 1), (67, 8)], np.int32)
    out, n = model_mod.split_blocks(qb, G)
    assert n == 2
    assert np.array_equal(out[:2], qb[[1, 3]])
    assert np.array_equal(out[2:], qb[[0, 2, 4, 5]])
    # a block of 8 rows at G = 2 is 16 vectors: decode-shaped; 9 rows is not
    assert model_mod.split_blocks(np.array([(0, 9), (9, 8)], np.int32), G)[1] == 1
    assert model_mod.split_blocks(np.array([(0, 9), (9, 9)], np.int32), G)[1] == 0
    # pure decode and pure prefill steps stay one call
    for qb in (np.array([(i, 1) for i in range(7)], np.int32),
               np.array([(0, 64), (64, 64)], np.int32)):
        out, n = model_mod.split_blocks(qb, G)
        assert n == 0 and np.array_equal(out, qb)
    # every block appears exactly once, whatever the mix
    g = np.random.default_rng(9)
    for _ in range(50):
        rows = g.integers(1, 65, size=g.integers(1, 40))
        starts = np.concatenate([[0], np.cumsum(rows)[:-1]])
        qb = np.stack([starts, rows], 1).astype(np.int32)
        out, n = model_mod.split_blocks(qb, G)
        assert sorted(map(tuple, out)) == sorted(map(tuple, qb))
        if n:
            assert np.all(out[:n, 1] * G > 16) and np.all(out[n:, 1] * G <= 16)
            assert qb.shape[0] - n >= n


def test_decode_step_bytes_counts_each_weight_once_and_the_kv_it_reads():
    """The decode-step roofline's algorithmic bytes: every distinct weight
    tensor once (a tied LM head shares the embedding), 114,688 B of K/V per
    cached token for the Qwen3-1.7B shape in bf16 (28 layers x K and V x 8 kv
    heads x 128 x 2 B), e4m3 codes plus one fp32 scale per token and kv head
    for the FP8 cache, and per row its own K/V write plus the (max, sum exp)
    pairs of its 128-logit groups."""
    import torch
    import bench
    cfg = synth.QWEN3_1P7B
    emb = torch.empty(cfg.vocab, cfg.hidden, dtype=torch.bfloat16, device="meta")
    other = torch.empty(1000, 10, dtype=torch.bfloat16, device="meta")
    W = {"embed": emb, "lm_head": emb, "w": other}
    work = bench.decode_step_bytes(cfg, W)
    wb = (cfg.vocab * cfg.hidden + 1000 * 10) * 2
    assert work.weight_bytes == wb
    assert work.kv_bytes_per_token == 114_688
    groups = (cfg.vocab + 127) // 128
    pos = [699] * 64 + [5]
    want = wb + (64 * 700 + 6) * 114_688 + 65 * (114_688 + 2 * groups * 8)
    assert work(pos) == float(want)
    fp8 = bench.decode_step_bytes(synth.QWEN3_1P7B_FP8KV, W)
    assert fp8.kv_bytes_per_token == 28 * 2 * (8 * 128 + 8 * 4)
