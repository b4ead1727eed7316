"""Pins of the oracle's logit_bias: biasing is the same as adding the values to
the logits beforehand (in list order, before the penalties and the mask), and
its limits (ids in range, at most 64 entries per row)."""
import numpy as np

import oracle
import workloads


def _explicit(b):
    """The batch with the bias folded into fp32 logits (one fp32 add per entry)."""
    x = workloads.bf16_bits_to_f32(b.logits).reshape(b.n_rows, -1).copy() if b.dtype == "bf16" \
        else b.logits.copy()
    for r in range(b.n_rows):
        for j in range(b.bias_offsets[r], b.bias_offsets[r + 1]):
            v = b.bias_ids[j]
            x[r, v] = np.float32(x[r, v] + b.bias_values[j])
    return b.with_(logits=x.astype(np.float32), dtype="f32", bias_offsets=None, bias_ids=None,
                   bias_values=None)


def test_bias_equals_pre_added_logits():
    b = workloads.random_batch(81, 16, 600, "bf16", mix="all", want_probs=True)
    offs, ids, vals = workloads.logit_bias(82, b.n_rows, b.vocab, max_per_row=40)
    b = b.with_(bias_offsets=offs, bias_ids=ids, bias_values=vals)
    ra = oracle.sample(b, want_probs=True)
    rb = oracle.sample(_explicit(b), want_probs=True)
    assert np.array_equal(ra.tokens, rb.tokens) and np.array_equal(ra.status, rb.status)
    assert np.array_equal(ra.probs, rb.probs) and np.array_equal(ra.logprobs, rb.logprobs)


def test_bias_comes_before_penalties_and_mask():
    b = workloads.random_batch(83, 4, 50, "f32", mix="plain", penalties=True, max_hist=20)
    offs = np.array([0, 1, 1, 2, 3], np.int32)
    ids = np.array([5, 7, 9], np.int32)
    vals = np.array([3.0, -2.0, 100.0], np.float32)
    m = np.full((4, 2), 0xFFFFFFFF, np.uint32)
    m[3, 0] &= ~np.uint32(1 << 9)  # row 3 masks the token its bias forces
    b = b.with_(bias_offsets=offs, bias_ids=ids, bias_values=vals, vocab_mask=m)
    plain = b.with_(bias_offsets=None, bias_ids=None, bias_values=None, vocab_mask=None)
    for r, tv in enumerate([(5, 3.0), None, (7, -2.0), (9, 100.0)]):
        _, xb = oracle.penalized_logits(b, r)
        if tv is None:
            continue
        tok, val = tv
        # the penalty acts on the biased logit: compare with a batch whose raw logit
        # carries the bias
        x = b.logits.copy()
        x[r, tok] = np.float32(x[r, tok] + np.float32(val))
        _, xe = oracle.penalized_logits(plain.with_(logits=x), r)
        if r == 3:
            assert np.isneginf(xb[tok])
            xe[tok] = -np.inf
        assert np.array_equal(xb, xe)


def test_bias_limits_are_bad_parameters():
    b = workloads.random_batch(84, 3, 100, "f32", mix="plain")
    offs = np.array([0, 65, 66, 66], np.int32)
    ids = np.concatenate([np.arange(65) % 100, [100]]).astype(np.int32)
    vals = np.ones(66, np.float32)
    res = oracle.sample(b.with_(bias_offsets=offs, bias_ids=ids, bias_values=vals))
    assert res.status.tolist() == [oracle.STATUS_BAD_PARAM, oracle.STATUS_BAD_PARAM, 0]
