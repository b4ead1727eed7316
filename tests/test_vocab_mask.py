"""Pins of the oracle's vocabulary bitmask: a masked token is exactly a -inf
logit, bit order (bit v & 31 of word v >> 5), fully masked rows."""
import numpy as np

import oracle
import workloads


def test_mask_equals_minus_inf_logits():
    b = workloads.random_batch(51, 20, 700, "f32", mix="all", want_probs=True)
    m = workloads.vocab_mask(52, b.n_rows, b.vocab, allowed=0.2)
    masked = b.with_(vocab_mask=m)
    bits = np.unpackbits(m.view(np.uint8), bitorder="little").reshape(b.n_rows, -1)[:, :b.vocab].astype(bool)
    x = b.logits.copy()
    x[~bits] = -np.inf
    explicit = b.with_(logits=x)
    ra = oracle.sample(masked, want_probs=True)
    rb = oracle.sample(explicit, want_probs=True)
    assert np.array_equal(ra.tokens, rb.tokens) and np.array_equal(ra.status, rb.status)
    assert np.array_equal(ra.probs, rb.probs) and np.array_equal(ra.logprobs, rb.logprobs)
    ok = ra.status == 0
    assert bits[np.nonzero(ok)[0], ra.tokens[ok]].all()
    assert (ra.probs[~bits & ok[:, None]] == 0).all()


def test_bit_order_and_fully_masked_rows():
    b = workloads.random_batch(53, 3, 100, "f32", mix="plain")
    words = (100 + 31) // 32
    m = np.zeros((3, words), np.uint32)
    for v in (3, 37, 64):
        m[0, v >> 5] |= np.uint32(1 << (v & 31))
    m[1, :] = 0xFFFFFFFF
    # row 2: nothing allowed
    res = oracle.sample(b.with_(vocab_mask=m), want_probs=True)
    assert res.status[0] == 0 and res.tokens[0] in (3, 37, 64)
    assert set(np.nonzero(res.probs[0])[0].tolist()) <= {3, 37, 64}
    assert res.status[1] == 0
    assert res.status[2] == oracle.STATUS_ALL_NEG_INF
    _, x = oracle.penalized_logits(b.with_(vocab_mask=m), 0)
    assert np.isneginf(np.delete(x, [3, 37, 64])).all() and np.isfinite(x[[3, 37, 64]]).all()
