"""Model-level checks of the oracle (CPU only).

The model-level logprob is "parity unpinned" beyond these: the pages print no
numbers for it.  What the mathematics fixes is checked here: the rollout
recurrence (prompt prefill, then one token at a time through the KV cache)
gives the same logprobs as one full prefill, logprobs are normalised, and a
peaked LM head moves them far from -log V.
"""
import math

import numpy as np
import pytest

import synth
from oracle import ops
from oracle.codecs import bf16_round
from oracle.model import DenseOracle, decode_weights


def _oracle(cfg, seed=0, **kw):
    W = synth.dense_weights(cfg, seed=seed, **kw)
    return DenseOracle(cfg, decode_weights({k: synth.bf16_bits(v) for k, v in W.items()}))


@pytest.mark.parametrize("kv_fp8", [False, True])
def test_tiny_decode_matches_prefill(kv_fp8):
    cfg = synth.TINY if not kv_fp8 else synth.replace(synth.TINY, kv_fp8=True)
    orc = _oracle(cfg, random_gains=True, lm_scale=10.0)
    seqs = synth.tiny_sequences(cfg, n=2, lo=20, hi=40, seed=3)
    for s in seqs:
        a = orc.prefill_logprobs(s.tokens)
        b = orc.decode_logprobs(s.tokens, s.prompt_len)
        assert a.shape == b.shape == (s.length - 1,)
        # the oracle's dot products are exact-then-rounded, so a 1-row decode
        # call and a T-row prefill call give the same logprobs
        assert np.max(np.abs(a - b)) == 0.0


def test_logprobs_normalised_and_peaked():
    cfg = synth.TINY
    orc = _oracle(cfg, lm_scale=10.0)
    s = synth.tiny_sequences(cfg, n=1, lo=24, hi=24, seed=4)[0]
    z = orc.forward_rows(s.tokens, np.arange(s.length), orc.new_cache())
    lp = ops.log_softmax(z)
    assert np.allclose(np.exp(lp.astype(np.float64)).sum(1), 1.0, atol=1e-4)
    # peaked head: logprobs spread well away from uniform
    assert np.std(lp) > 1.0
    flat = _oracle(cfg)
    lpf = flat.prefill_logprobs(s.tokens)
    assert abs(float(np.mean(lpf)) + math.log(cfg.vocab)) < 0.3 and np.std(lpf) < 0.6


def test_logprobs_at_matches_prefill_rows():
    cfg = synth.TINY
    orc = _oracle(cfg, lm_scale=20.0)
    s = synth.tiny_sequences(cfg, n=1, lo=30, hi=30, seed=5)[0]
    full = orc.prefill_logprobs(s.tokens)
    rows = np.array([0, 7, 28])
    np.testing.assert_allclose(orc.logprobs_at(s.tokens, rows), full[rows], atol=1e-5)


def test_planted_rope_sign_error_is_caught(monkeypatch):
    """A flipped sign inside RoPE breaks the relative-position property that
    the RoPE pin checks; the pin therefore guards the model path too."""
    cos, sin = ops.rope_table(1e4, 64, 600)
    g = np.random.default_rng(0)
    q = bf16_round(g.standard_normal((1, 1, 64)).astype(np.float32))
    k = bf16_round(g.standard_normal((1, 1, 64)).astype(np.float32))

    def bad_rope(x, pos, c, s):
        x = np.asarray(x, np.float32)
        h = x.shape[-1] // 2
        cc, ss = c[pos][:, None, :], s[pos][:, None, :]
        return bf16_round(np.concatenate([x[..., :h] * cc + x[..., h:] * ss,
                                              x[..., h:] * cc + x[..., :h] * ss], -1))

    def rel_gap(fn):
        d1 = np.dot(fn(q, np.array([500]), cos, sin).ravel(), fn(k, np.array([490]), cos, sin).ravel())
        d2 = np.dot(fn(q, np.array([12]), cos, sin).ravel(), fn(k, np.array([2]), cos, sin).ravel())
        return abs(d1 - d2)

    assert rel_gap(ops.rope) < 0.05 * np.abs(q).sum() * np.abs(k).max()
    assert rel_gap(bad_rope) > rel_gap(ops.rope) * 10


def test_layer_by_layer_entry_points_chain_to_the_forward():
    """Chaining layer_from from the embedding reproduces the full forward's
    residuals, and head_from reproduces its logprobs."""
    cfg = synth.TINY
    orc = _oracle(cfg, random_gains=True, lm_scale=10.0)
    s = synth.tiny_sequences(cfg, n=1, lo=30, hi=30, seed=8)[0]
    orc.audit = []
    full = orc.prefill_logprobs(s.tokens)
    res = [x for t, l, x in orc.audit if t == "layer"]
    orc.audit = None
    pos = np.arange(s.length - 1)
    r = orc.W["embed"][s.tokens[:-1]]
    for l in range(cfg.layers):
        r = orc.layer_from(l, r, pos)
        assert np.array_equal(r, res[l])
    assert np.array_equal(orc.head_from(r, s.tokens[1:]), full)
