"""Pins of the oracle's per-row logprob outputs (sampled token + top-n) against
scipy's log_softmax and a brute-force order, and their agreement with the
oracle's own materialised probs."""
import numpy as np
import pytest
from scipy.special import log_softmax

import oracle
import workloads


def _batch(seed, n=12, v=57, **kw):
    return workloads.random_batch(seed, n, v, "f32", want_probs=True, **kw)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_scaled_outputs_match_scipy_over_the_kept_set(seed):
    b = _batch(seed)
    res = oracle.sample(b, want_probs=True)
    lo = oracle.logprob_outputs(b, res, top_n=5)
    for r in range(b.n_rows):
        if res.status[r]:
            assert np.isnan(lo.token_logprob[r]) and (lo.top_ids[r] == -1).all()
            continue
        _, x = oracle.penalized_logits(b, r)
        keep = res.logprobs[r] > -np.inf
        T = float(b.temperature[r]) if b.temperature[r] >= 1e-5 else 1.0
        ref = np.full(b.vocab, -np.inf)
        ref[keep] = log_softmax(x[keep].astype(np.float64) / T)
        assert lo.token_logprob[r] == pytest.approx(ref[res.tokens[r]], abs=1e-12)
        # the oracle's own fp32 probs agree
        assert np.exp(lo.token_logprob[r]) == pytest.approx(float(res.probs[r, res.tokens[r]]), rel=1e-6, abs=1e-7)
        # brute-force order: value desc, index asc, kept tokens only
        order = [v for v in sorted(range(b.vocab), key=lambda v: (-float(x[v]), v)) if keep[v]][:5]
        assert lo.top_ids[r, :len(order)].tolist() == order
        assert (lo.top_ids[r, len(order):] == -1).all()
        assert np.allclose(lo.top_logprobs[r, :len(order)], ref[order], atol=1e-12)
        assert np.all(np.diff(lo.top_logprobs[r, :len(order)]) <= 0)


def test_unscaled_outputs_are_the_full_vocabulary_log_softmax():
    b = _batch(4, mix="topk")
    res = oracle.sample(b, want_probs=True)
    lo = oracle.logprob_outputs(b, res, top_n=7, unscaled=True)
    for r in range(b.n_rows):
        _, x = oracle.penalized_logits(b, r)
        ref = log_softmax(x.astype(np.float64))
        assert lo.token_logprob[r] == pytest.approx(ref[res.tokens[r]], abs=1e-12)
        order = sorted(range(b.vocab), key=lambda v: (-float(x[v]), v))[:7]
        assert lo.top_ids[r].tolist() == order
        assert np.allclose(lo.top_logprobs[r], ref[order], atol=1e-12)


def test_greedy_rows_use_temperature_one_and_top_n_pads():
    b = workloads.random_batch(5, 6, 9, "f32", want_probs=True, mix="topk")
    b = b.with_(temperature=np.zeros(6, np.float32), top_k=np.full(6, 3, np.int32))
    res = oracle.sample(b, want_probs=True)
    lo = oracle.logprob_outputs(b, res, top_n=5)
    for r in range(6):
        _, x = oracle.penalized_logits(b, r)
        order = sorted(range(9), key=lambda v: (-float(x[v]), v))[:3]
        ref = log_softmax(x[order].astype(np.float64))
        assert lo.top_ids[r].tolist() == order + [-1, -1]
        assert np.allclose(lo.top_logprobs[r, :3], ref, atol=1e-12)
        assert np.isneginf(lo.top_logprobs[r, 3:]).all()
        assert res.tokens[r] == order[0]
        assert lo.token_logprob[r] == pytest.approx(ref[0], abs=1e-12)


def test_sampled_token_logprob_is_consistent_with_the_gumbel_frequency():
    """Over many Philox offsets the sampled token's reported probability matches
    its frequency (the pick draws from the distribution the logprobs describe)."""
    b = workloads.random_batch(6, 1, 6, "f32", want_probs=True, mix="plain")
    counts = np.zeros(6)
    lp_of = None
    for off in range(3000):
        bb = b.with_(philox_offset=off)
        res = oracle.sample(bb, want_probs=True)
        lo = oracle.logprob_outputs(bb, res, top_n=6)
        counts[res.tokens[0]] += 1
        lp_of = dict(zip(lo.top_ids[0].tolist(), lo.top_logprobs[0].tolist()))
    p = np.array([np.exp(lp_of[v]) for v in range(6)])
    expected = p * counts.sum()
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    assert chi2 < 25.0, (counts, expected)
