"""Pins of the oracle's min_tokens stage (a row that still owes tokens cannot
pick its stop tokens) and of its NaN-sanitising mode (NaN logits are excluded
instead of failing the row), against closed forms and library routines."""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
import workloads


def _stops(n, lists):
    offs = np.zeros(n + 1, np.int32)
    offs[1:] = np.cumsum([len(x) for x in lists])
    return offs, np.array([i for x in lists for i in x], np.int32)


def test_greedy_skips_stop_tokens_while_owed():
    b = workloads.random_batch(91, 6, 300, "f32", mix="plain")
    x = b.logits.copy()
    lists = []
    for r in range(b.n_rows):
        top = np.argsort(-x[r], kind="stable")[:3]
        lists.append(top[: (r % 3) + 1].tolist())  # the row's 1..3 best tokens are stop tokens
    offs, ids = _stops(b.n_rows, lists)
    left = np.array([1, 0, 5, 1, 0, 2], np.int32)
    g = b.with_(temperature=np.zeros(b.n_rows, np.float32), min_tokens_left=left, stop_offsets=offs,
                stop_ids=ids)
    res = oracle.sample(g)
    for r in range(b.n_rows):
        row = x[r].astype(np.float64)
        if left[r] > 0:
            row[lists[r]] = np.nan
        assert res.status[r] == 0
        assert res.tokens[r] == np.nanargmax(row)  # lowest index among equal maxima


def test_probabilities_renormalise_over_the_other_tokens():
    b = workloads.random_batch(92, 8, 500, "bf16", mix="plain", want_probs=True)
    left, offs, ids = workloads.min_tokens(93, b.n_rows, b.vocab, max_stops=6, owe=1.0)
    full = oracle.sample(b, want_probs=True)
    ban = oracle.sample(b.with_(min_tokens_left=left, stop_offsets=offs, stop_ids=ids), want_probs=True)
    for r in range(b.n_rows):
        s = np.unique(ids[offs[r]:offs[r + 1]])
        p = full.probs[r].astype(np.float64)
        want = p / (1.0 - p[s].sum())
        want[s] = 0.0
        assert np.all(ban.probs[r][s] == 0.0)
        np.testing.assert_allclose(ban.probs[r], want, rtol=2e-5, atol=1e-9)


def test_rows_that_owe_nothing_are_unchanged():
    b = workloads.random_batch(94, 16, 400, "bf16", mix="all", want_probs=True)
    left, offs, ids = workloads.min_tokens(95, b.n_rows, b.vocab)
    left[:] = 0
    a = oracle.sample(b, want_probs=True)
    c = oracle.sample(b.with_(min_tokens_left=left, stop_offsets=offs, stop_ids=ids), want_probs=True)
    assert np.array_equal(a.tokens, c.tokens) and np.array_equal(a.probs, c.probs)


def test_stop_limits_and_all_stopped_rows():
    b = workloads.random_batch(96, 4, 16, "f32", mix="plain")
    lists = [list(range(16)) + [0], [16], list(range(16)), [3]]  # 17 > 16; id out of range; every token
    offs, ids = _stops(4, lists)
    left = np.array([1, 0, 1, 0], np.int32)
    res = oracle.sample(b.with_(min_tokens_left=left, stop_offsets=offs, stop_ids=ids))
    assert res.status.tolist() == [oracle.STATUS_BAD_PARAM, oracle.STATUS_BAD_PARAM,
                                   oracle.STATUS_ALL_NEG_INF, 0]


def test_a_banned_stop_token_may_be_nan():
    b = workloads.random_batch(97, 2, 64, "f32", mix="plain")
    x = b.logits.copy()
    x[:, 7] = np.nan
    offs, ids = _stops(2, [[7], [7]])
    res = oracle.sample(b.with_(logits=x, min_tokens_left=np.array([1, 0], np.int32), stop_offsets=offs,
                                stop_ids=ids))
    assert res.status.tolist() == [0, oracle.STATUS_NONFINITE]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sanitised_nan_rows_match_the_clean_subset(dtype):
    b = workloads.random_batch(98, 6, 700, dtype, mix="plain", want_probs=True)
    rng = np.random.default_rng(99)
    x = workloads.bf16_bits_to_f32(b.logits).reshape(b.n_rows, -1).copy() if dtype == "bf16" \
        else b.logits.copy()
    nan_at = rng.random(x.shape) < 0.1
    x[nan_at] = np.nan
    t = np.full(b.n_rows, 0.7, np.float32)
    t[0] = 0.0
    nb = b.with_(logits=x, dtype="f32", temperature=t)
    assert np.all(oracle.sample(nb).status == oracle.STATUS_NONFINITE)
    res = oracle.sample(nb.with_(sanitize_nan=True), want_probs=True)
    assert np.all(res.status == 0)
    assert res.tokens[0] == np.nanargmax(x[0])
    for r in range(1, b.n_rows):
        want = np.zeros(b.vocab)
        ok = ~nan_at[r]
        want[ok] = softmax(x[r, ok].astype(np.float64) / np.float64(np.float32(0.7)))
        np.testing.assert_allclose(res.probs[r], want, rtol=2e-5, atol=1e-9)
        assert ok[res.tokens[r]]


def test_sanitising_leaves_inf_an_error_and_all_nan_empty():
    b = workloads.random_batch(100, 3, 50, "f32", mix="plain")
    x = b.logits.copy()
    x[0, :] = np.nan
    x[1, 4] = np.inf
    x[2, 4] = -np.inf
    res = oracle.sample(b.with_(logits=x, sanitize_nan=True))
    assert res.status.tolist() == [oracle.STATUS_ALL_NEG_INF, oracle.STATUS_NONFINITE, 0]
