"""Pins of the CPU oracle to things other than itself (no GPU).

Each test checks the oracle against what the pages or the mathematics fix:
published known-answer vectors, an independent library generator, textbook
routines (numpy.argmax, scipy softmax), brute force on tiny inputs, closed
forms, hand-computed cases and statistical agreement with the categorical
distribution.
"""
import itertools
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
import workloads
from workloads import SamplerBatch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _batch(x, t, **kw):
    x = np.atleast_2d(np.asarray(x, np.float32))
    n, v = x.shape
    return SamplerBatch("t", x, "f32", v, n, np.asarray(t, np.float32).reshape(n), **kw)


# --------------------------------------------------------------------------- Philox

def test_philox4x32_known_answers():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        vals = [int(h, 16) for h in r]
        out = oracle.philox4x32_10(vals[0:4], vals[4:6])
        assert list(out) == vals[6:10]


@pytest.mark.parametrize("key", [(0, 0), (123456789, 987654321), (2**64 - 1, 17)])
def test_philox_round_structure_matches_numpy_4x64(key):
    # numpy's Philox bit generator is Philox4x64-10; it advances the counter by one
    # before producing a block, so its first block is the oracle's block at counter + 1.
    for ctr0 in (0, 5, 2**64 - 2):
        bg = np.random.Philox(key=np.array(key, np.uint64),
                              counter=np.array([ctr0, 7, 0, 9], np.uint64))
        expect = bg.random_raw(4)
        got = oracle.philox4x64_10([(ctr0 + 1) % 2**64, 7, 0, 9], key)
        assert list(got) == list(expect)


def test_noise_word_layout():
    # counter = (v >> 2, stream, offset lo, offset hi), word v & 3, key = (lo, hi)
    key, stream, off = 0x1122334455667788, 0x80000005, 0xAABBCCDD00112233
    for v in (0, 1, 2, 3, 4, 1023, 151935):
        block = oracle.philox4x32_10([v >> 2, stream, off & 0xFFFFFFFF, off >> 32],
                                     [key & 0xFFFFFFFF, key >> 32])
        assert oracle.noise_word(key, stream, off, v) == block[v & 3]


def test_uniform_and_exp1_closed_forms():
    assert oracle.uniform(0) == 2.0**-24
    assert oracle.uniform(0xFFFFFFFF) == 1.0 - 2.0**-24
    assert oracle.uniform(0x1FF) == 2.0**-24          # low 9 bits are dropped
    assert oracle.uniform(0x200) == 3 * 2.0**-24
    for w in (0, 0x12345678, 0x80000000, 0xFFFFFFFF):
        assert oracle.exp1(w) == pytest.approx(-np.log(oracle.uniform(w)), rel=1e-15)


def test_philox_uniformity_and_exponential_ks():
    # 2^16 consecutive words of one stream: bucket uniformity and Exp(1) shape
    n = 1 << 16
    words = np.array([oracle.noise_word(7, 3, 11, v) for v in range(n)], np.uint64)
    hist = np.bincount((words >> np.uint64(24)).astype(np.int64), minlength=256)
    chi2 = ((hist - n / 256) ** 2 / (n / 256)).sum()
    assert scipy.stats.chi2.sf(chi2, 255) > 1e-4
    e = np.array([oracle.exp1(int(w)) for w in words[:20000]])
    assert scipy.stats.kstest(e, "expon").pvalue > 1e-4


# --------------------------------------------------------------------------- greedy / softmax

def test_greedy_is_numpy_argmax_with_ties_to_lowest_index():
    rng = np.random.default_rng(0)
    x = np.round(rng.standard_normal((50, 37)) * 2) / 2  # many ties
    b = _batch(x, np.zeros(50))
    res = oracle.sample(b)
    assert (res.status == 0).all()
    np.testing.assert_array_equal(res.tokens, np.argmax(x.astype(np.float32), axis=1))


def test_greedy_threshold_is_1e_5():
    x = np.array([[0.0, 1.0, 5.0, 2.0]] * 6, np.float32)
    t = np.array([0.0, 0.9e-5, 1.1e-5, 1e-4, 0.5, 1.0], np.float32)
    res = oracle.sample(_batch(x, t, global_seed=3))
    assert res.tokens[0] == 2 and res.tokens[1] == 2
    assert np.isinf(res.gumbel_gap[:2]).all()      # greedy rows draw nothing
    assert np.isfinite(res.gumbel_gap[2:]).all()   # sampled rows do


def test_probs_logprobs_match_scipy_softmax_at_temperature():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((6, 300)) * 3).astype(np.float32)
    t = np.array([1.0, 0.7, 1.3, 0.25, 2.0, 0.0], np.float32)
    res = oracle.sample(_batch(x, t), want_probs=True)
    for i in range(6):
        te = 1.0 if t[i] < 1e-5 else float(t[i])  # greedy rows report at T = 1
        y = x[i].astype(np.float64) / te
        np.testing.assert_allclose(res.probs[i], scipy.special.softmax(y), rtol=1e-6, atol=1e-9)
        np.testing.assert_allclose(res.logprobs[i], scipy.special.log_softmax(y), rtol=1e-6,
                                   atol=1e-6)
        assert abs(res.probs[i].astype(np.float64).sum() - 1.0) < 1e-6
        # exp(logprobs) == probs up to the fp32 rounding of each (|logp| ulps of the log)
        lp = res.logprobs[i].astype(np.float64)
        tol = res.probs[i] * (np.abs(lp) * 2.0**-23 + 2e-7)
        assert (np.abs(np.exp(lp) - res.probs[i]) <= tol).all()


def test_logprobs_are_temperature_scaled():
    # SGLang manual, "Logprobs are temperature-scaled": log_softmax(logits / T)
    x = np.array([[1.0, 2.0, 3.0]], np.float32)
    res = oracle.sample(_batch(x, [0.5]), want_probs=True)
    np.testing.assert_allclose(res.logprobs[0], scipy.special.log_softmax(x[0] / 0.5), rtol=1e-6)
    assert not np.allclose(res.logprobs[0], scipy.special.log_softmax(x[0]), rtol=1e-3)


# --------------------------------------------------------------------------- kept sets, brute force

def _order_key(x, i):
    return (-float(x[i]), i)


def _kept_from_probs(res, i):
    return set(np.nonzero(res.probs[i] > 0)[0].tolist())


def _brute_topk(x, k):
    v = len(x)
    if k == -1 or k >= v:
        return set(range(v))
    best = None
    for s in itertools.combinations(range(v), k):
        inside = [_order_key(x, i) for i in s]
        outside = [_order_key(x, i) for i in range(v) if i not in s]
        if not outside or max(inside) < min(outside):
            assert best is None
            best = set(s)
    return best


def _brute_topp(x, t, dom, p):
    # the smallest set that is closed upward in (value desc, index asc) order within
    # `dom` and holds at least mass p of the softmax over `dom`
    dom = sorted(dom)
    y = np.array([x[i] / t for i in dom], np.float64)
    w = np.exp(y - y.max())
    w /= w.sum()
    mass = dict(zip(dom, w))
    best = None
    for r in range(1, len(dom) + 1):
        for s in itertools.combinations(dom, r):
            inside = [_order_key(x, i) for i in s]
            outside = [_order_key(x, i) for i in dom if i not in s]
            if outside and not max(inside) < min(outside):
                continue
            if sum(mass[i] for i in s) >= p - 1e-12:
                best = set(s)
                break
        if best is not None:
            break
    return best


@pytest.mark.parametrize("seed", range(12))
def test_topk_topp_minp_kept_sets_by_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    v = int(rng.integers(2, 10))
    x = (np.round(rng.standard_normal(v) * 2, 1)).astype(np.float32)  # ties happen
    t = float(rng.uniform(0.3, 2.0))
    k = int(rng.choice([-1, 1, 2, 3, v - 1, v, v + 3]))
    k = -1 if k == 0 else k
    p = float(rng.choice([1.0, rng.uniform(0.05, 0.99)]))
    mp = float(rng.choice([0.0, rng.uniform(0.01, 0.9)]))
    b = _batch(x, [t], top_k=np.array([k], np.int32), top_p=np.array([p], np.float32),
               min_p=np.array([mp], np.float32))
    res = oracle.sample(b, want_probs=True)
    assert res.status[0] == 0
    p32 = float(np.float32(p))
    dom = _brute_topk(x, k)
    if p32 < 1.0:
        dom = _brute_topp(x, t, dom, p32)
    if mp > 0:
        y = x.astype(np.float64) / t
        pr = scipy.special.softmax(y[sorted(dom)])
        pmax = pr.max()
        dom = {i for i, q in zip(sorted(dom), pr) if q >= np.float32(mp) * pmax * (1 - 1e-12)}
    assert _kept_from_probs(res, 0) == dom
    assert res.tokens[0] in dom
    # probs / logprobs: the softmax at T renormalised over the kept set, 0 and -inf
    # elsewhere
    kept = sorted(dom)
    yk = x.astype(np.float64)[kept] / t
    np.testing.assert_allclose(res.probs[0][kept], scipy.special.softmax(yk), rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(res.logprobs[0][kept], scipy.special.log_softmax(yk), rtol=1e-6,
                               atol=1e-6)
    out = [i for i in range(v) if i not in dom]
    assert (res.probs[0][out] == 0).all() and np.isneginf(res.logprobs[0][out]).all()


def test_topk_ties_keep_lowest_indices():
    x = np.array([[1.0, 3.0, 3.0, 3.0, 0.0, 3.0]], np.float32)
    res = oracle.sample(_batch(x, [1.0], top_k=np.array([2], np.int32)), want_probs=True)
    assert _kept_from_probs(res, 0) == {1, 2}


def test_topp_keeps_at_least_one_and_uses_exclusive_prefix():
    x = np.array([[10.0, 0.0, 0.0, 0.0]], np.float32)
    res = oracle.sample(_batch(x, [1.0], top_p=np.array([0.01], np.float32)), want_probs=True)
    assert _kept_from_probs(res, 0) == {0}
    # two equal tokens, p = 0.5: the first has exclusive prefix 0 < 0.5, the second 0.5
    x = np.array([[1.0, 1.0]], np.float32)
    res = oracle.sample(_batch(x, [1.0], top_p=np.array([0.5], np.float32)), want_probs=True)
    assert _kept_from_probs(res, 0) == {0}
    res = oracle.sample(_batch(x, [1.0], top_p=np.array([0.5000001], np.float32)),
                        want_probs=True)
    assert _kept_from_probs(res, 0) == {0, 1}


def test_minp_closed_form():
    # keep v iff p_v >= min_p * p_max  <=>  x_v - x_max >= T ln(min_p)
    x = np.array([[0.0, -1.0, -2.0, -3.0, -4.0]], np.float32)
    for mp in (0.5, 0.3, 0.1, 0.04, 0.01):
        res = oracle.sample(_batch(x, [1.0], min_p=np.array([mp], np.float32)), want_probs=True)
        expect = {i for i in range(5) if -i >= np.log(np.float32(mp))}
        assert _kept_from_probs(res, 0) == expect


# --------------------------------------------------------------------------- Gumbel-max == categorical

@pytest.mark.parametrize("v", [2, 5, 16])
def test_gumbel_max_draws_the_categorical_distribution(v):
    # many rows of one logits vector, each with its own Philox stream
    rng = np.random.default_rng(v)
    x = (rng.standard_normal(v) * 1.5).astype(np.float32)
    n = 200_000
    b = SamplerBatch("g", x[None, :], "f32", v, n, np.full(n, 0.8, np.float32),
                     logit_row=np.zeros(n, np.int32), global_seed=99, philox_offset=5)
    res = oracle.sample(b, nthreads=os.cpu_count() or 1)
    counts = np.bincount(res.tokens, minlength=v)
    p = scipy.special.softmax(x.astype(np.float64) / 0.8)
    chi2 = ((counts - n * p) ** 2 / (n * p)).sum()
    assert scipy.stats.chi2.sf(chi2, v - 1) > 1e-4
    tvd = 0.5 * np.abs(counts / n - p).sum()
    assert tvd < 0.01


def test_gumbel_max_over_the_kept_set_draws_the_renormalised_distribution():
    # top-k then top-p then min-p by their textbook definitions, then the draw must
    # follow softmax(x / T) over the kept tokens only
    rng = np.random.default_rng(11)
    v, T, k, p, mp = 12, 0.7, 7, 0.95, 0.15
    x = (rng.standard_normal(v) * 1.5).astype(np.float32)
    order = sorted(range(v), key=lambda i: (-float(x[i]), i))[:k]
    y = x.astype(np.float64)[order] / T
    q = scipy.special.softmax(y)
    excl = np.concatenate([[0.0], np.cumsum(q)[:-1]])
    kept_p = [order[i] for i in range(k) if i == 0 or excl[i] < p]
    keep = [i for i in kept_p if x[i] / T - y.max() >= np.log(mp)]
    # each cut removes something here: 12 -> 7 (top-k) -> 5 (top-p) -> 4 (min-p)
    assert (len(order), len(kept_p), len(keep)) == (7, 5, 4)
    want = scipy.special.softmax(x.astype(np.float64)[keep] / T)
    n = 200_000
    b = SamplerBatch("g", x[None, :], "f32", v, n, np.full(n, T, np.float32),
                     top_k=np.full(n, k, np.int32), top_p=np.full(n, p, np.float32),
                     min_p=np.full(n, mp, np.float32), logit_row=np.zeros(n, np.int32),
                     global_seed=7, philox_offset=1)
    res = oracle.sample(b, nthreads=os.cpu_count() or 1)
    counts = np.bincount(res.tokens, minlength=v)
    assert counts[[i for i in range(v) if i not in keep]].sum() == 0
    got = counts[keep]
    chi2 = ((got - n * want) ** 2 / (n * want)).sum()
    assert scipy.stats.chi2.sf(chi2, len(keep) - 1) > 1e-4


def test_seeded_rows_ignore_batch_position_and_forks_differ():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((1, 500)) * 2).astype(np.float32)
    n = 6
    b = SamplerBatch("s", x, "f32", 500, n, np.ones(n, np.float32),
                     logit_row=np.zeros(n, np.int32),
                     seed=np.full(n, 42, np.uint64), has_seed=np.array([1, 1, 1, 0, 0, 1], np.uint8),
                     stream_id=np.array([0, 0, 1, 0, 1, 2], np.uint32), global_seed=42)
    res = oracle.sample(b)
    # same seed and stream -> same draw regardless of row position
    assert res.tokens[0] == res.tokens[1]
    # seeded and unseeded rows with equal key / stream id still draw differently (bit 31)
    words_seeded = oracle.noise_word(42, 0x80000000, 0, 7)
    words_plain = oracle.noise_word(42, 0, 0, 7)
    assert words_seeded != words_plain


# --------------------------------------------------------------------------- penalties

def test_penalty_hand_cases():
    cases = [list(map(float, l.split())) for l in open(os.path.join(GOLDEN, "penalty_cases.txt"))
             if l.strip() and not l.startswith("#")]
    for xv, rep, freq, pres, cnt, expect in cases:
        x = np.array([[xv, 7.0]], np.float32)
        offs = np.array([0, int(cnt)], np.int32)
        ids = np.zeros(int(cnt), np.int32)
        b = _batch(x, [1.0], presence=np.float32([pres]), frequency=np.float32([freq]),
                   repetition=np.float32([rep]), hist_offsets=offs, hist_ids=ids)
        st, xp = oracle.penalized_logits(b, 0)
        assert st == 0
        assert xp[0] == np.float32(expect), (xv, rep, freq, pres, cnt, xp[0])
        assert xp[1] == np.float32(7.0)


def test_penalty_counts_follow_the_history_multiset():
    # counts come from the whole ragged history of the row (repeats and any order),
    # other rows' histories do not leak in, and unseen tokens are untouched
    rng = np.random.default_rng(5)
    v = 40
    x = (rng.standard_normal((2, v)) * 2).astype(np.float32)
    h0 = rng.integers(0, 10, size=25).astype(np.int32)   # row 0: ids 0..9 with repeats
    h1 = np.array([30, 30, 31], np.int32)                  # row 1
    offs = np.array([0, len(h0), len(h0) + len(h1)], np.int32)
    b = _batch(x, [1.0, 1.0], presence=np.float32([0.5, 0.5]), frequency=np.float32([0.25, 0.25]),
               repetition=np.float32([1.0, 1.0]), hist_offsets=offs,
               hist_ids=np.concatenate([h0, h1]))
    st, xp = oracle.penalized_logits(b, 0)
    assert st == 0
    c = np.bincount(h0, minlength=v)
    # repetition 1: x - 0.25 c - 0.5 [c > 0], up to the rounding of two fp32 steps
    want = x[0].astype(np.float64) - 0.25 * c - 0.5 * (c > 0)
    seen = c > 0
    np.testing.assert_allclose(xp[seen], want[seen], rtol=0, atol=4e-6)
    np.testing.assert_array_equal(xp[~seen], x[0][~seen])
    assert (xp[30:32] == x[0][30:32]).all()  # row 1's ids do not touch row 0


def test_identity_penalties_change_nothing():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((1, 64)) * 3).astype(np.float32)
    x[0, 3] = -0.0
    offs = np.array([0, 40], np.int32)
    ids = rng.integers(0, 64, 40).astype(np.int32)
    b = _batch(x, [1.0], presence=np.float32([0.0]), frequency=np.float32([0.0]),
               repetition=np.float32([1.0]), hist_offsets=offs, hist_ids=ids)
    st, xp = oracle.penalized_logits(b, 0)
    assert st == 0 and np.array_equal(xp.view(np.uint32), x[0].view(np.uint32))


def test_penalised_greedy_pick():
    x = np.array([[3.0, 1.0, 2.5]], np.float32)
    offs = np.array([0, 2], np.int32)
    ids = np.array([0, 0], np.int32)
    # token 0 becomes 3 - 0.25 * 2 - 0.25 = 2.25 < 2.5: token 2 wins
    b = _batch(x, [0.0], presence=np.float32([0.25]), frequency=np.float32([0.25]),
               repetition=np.float32([1.0]), hist_offsets=offs, hist_ids=ids)
    assert oracle.sample(b).tokens[0] == 2
    # with frequency 0.125 token 0 becomes exactly 2.5: the tie goes to index 0
    b = b.with_(frequency=np.float32([0.125]))
    assert oracle.penalized_logits(b, 0)[1][0] == np.float32(2.5)
    assert oracle.sample(b).tokens[0] == 0


# --------------------------------------------------------------------------- statuses

def test_status_codes():
    x = np.zeros((8, 4), np.float32)
    x[2, 1] = np.nan
    x[3, 0] = np.inf
    x[4, :] = -np.inf
    t = np.array([1, -1, 1, 1, 1, 1, 1, np.nan], np.float32)
    offs = np.array([0, 0, 0, 0, 0, 0, 1, 1, 1], np.int32)
    ids = np.array([4], np.int32)  # row 5's history has id 4 >= V
    b = _batch(x, t, hist_offsets=offs, hist_ids=ids)
    res = oracle.sample(b, want_probs=True)
    assert list(res.status) == [0, 3, 1, 1, 2, 4, 0, 3]
    assert list(res.tokens[[1, 2, 3, 4, 5, 7]]) == [-1] * 6
    assert np.isnan(res.probs[1]).all() and np.isnan(res.logprobs[4]).all()
    for bad in (dict(top_k=np.int32([0])), dict(top_k=np.int32([-2])),
                dict(top_p=np.float32([0.0])), dict(top_p=np.float32([1.5])),
                dict(min_p=np.float32([-0.1])), dict(min_p=np.float32([1.1])),
                dict(repetition=np.float32([0.0])), dict(presence=np.float32([np.inf]))):
        res = oracle.sample(_batch(np.zeros((1, 3)), [1.0], **bad))
        assert res.status[0] == 3


def test_neg_inf_logits_are_masked_not_errors():
    x = np.array([[-np.inf, 1.0, -np.inf, 0.5]], np.float32)
    res = oracle.sample(_batch(x, [1.0]), want_probs=True)
    assert res.status[0] == 0 and res.tokens[0] in (1, 3)
    assert res.probs[0, 0] == 0 and res.logprobs[0, 2] == -np.inf


# --------------------------------------------------------------------------- workloads

def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.00390625, 1.005859375, -2.5, 3.0e38, 1e-40], np.float32)
    bits = workloads.to_bf16_bits(vals)
    back = workloads.bf16_bits_to_f32(bits)
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even -> 1.0
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == np.float32(1.0078125)
    assert back[3] == -2.5
    # agrees with an independent bf16 implementation where one is installed
    try:
        import ml_dtypes
    except ImportError:
        return
    ref = vals.astype(ml_dtypes.bfloat16).view(np.uint16)
    np.testing.assert_array_equal(bits, ref)
