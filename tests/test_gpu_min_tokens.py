"""min_tokens and NaN sanitising through sampler_sample_ex vs the oracle (needs
a GB300)."""
import numpy as np
import pytest

import oracle
import workloads
from workloads import device as dev
from parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sampler():
    from decode_step_token_gb300 import build
    build.build_library()
    import decode_step_token_gb300 as d
    s = d.Sampler(max_rows=256, max_vocab=262144)
    yield s
    s.close()


def _with_stops(b, seed, max_stops=8, owe=0.5):
    left, offs, ids = workloads.min_tokens(seed, b.n_rows, b.vocab, max_stops, owe)
    return b.with_(min_tokens_left=left, stop_offsets=offs, stop_ids=ids)


def _with_nans(b, seed, frac=0.01):
    """The batch with a fraction of its logits NaN (positive and negative, several payloads)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = b.logits.copy()
    at = rng.random(x.shape) < frac
    if b.dtype == "bf16":
        x[at] = rng.choice(np.array([0x7FC0, 0xFFC0, 0x7F81, 0xFFFF], np.uint16), size=int(at.sum()))
    else:
        x[at] = rng.choice(np.array([0x7FC00000, 0xFFC00000, 0x7F800001], np.uint32),
                           size=int(at.sum())).view(np.float32)
    return b.with_(logits=x, sanitize_nan=True)


def _check(sampler, batch, **kw):
    g = dev.run(sampler, batch, want_probs=False, **kw)
    o = oracle.sample(batch, want_probs=False, nthreads=16)
    rep = compare(batch, g, o)
    assert rep.ok(), rep
    return rep


@pytest.mark.parametrize("name", ["mixed", "latency32", "tiny"])
def test_named_workloads_with_stop_tokens(sampler, name):
    rep = _check(sampler, _with_stops(workloads.make(name), 111))
    assert rep.gumbel_ties == 0 and rep.excused == 0, rep


@pytest.mark.parametrize("name", ["mixed", "latency32"])
def test_named_workloads_sanitised(sampler, name):
    rep = _check(sampler, _with_nans(workloads.make(name), 112))
    assert rep.gumbel_ties == 0 and rep.excused == 0, rep


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_every_extension_together(sampler, dtype):
    b = workloads.random_batch(113, 48, 21000, dtype, mix="all")
    offs, ids, vals = workloads.logit_bias(114, b.n_rows, b.vocab, 40)
    b = _with_stops(b, 115).with_(bias_offsets=offs, bias_ids=ids, bias_values=vals,
                                  vocab_mask=workloads.vocab_mask(116, b.n_rows, b.vocab, allowed=0.5))
    _check(sampler, b)
    _check(sampler, _with_nans(b, 117, frac=0.05))


def test_greedy_rows_skip_their_best_tokens(sampler):
    """The stop tokens are each row's best tokens (one of them NaN): rows that
    owe tokens take the next one."""
    b = workloads.random_batch(118, 8, 30000, "f32", mix="plain")
    b = b.with_(temperature=np.where(np.arange(8) % 2 == 0, 0.0, 0.6).astype(np.float32))
    x = b.logits.copy()
    lists = [np.argsort(-x[r], kind="stable")[:1 + r % 4].astype(np.int32) for r in range(8)]
    for r in range(8):
        x[r, lists[r][0]] = np.nan
    offs = np.zeros(9, np.int32)
    offs[1:] = np.cumsum([len(t) for t in lists])
    left = np.int32([1, 1, 3, 0, 2, 0, 1, 1])
    b = b.with_(logits=x, min_tokens_left=left, stop_offsets=offs, stop_ids=np.concatenate(lists))
    g = dev.run(sampler, b, want_probs=False)
    assert all(g.status[r] == (0 if left[r] else 1) for r in range(8)), g.status
    _check(sampler, b)


def test_ragged_unaligned_and_exact_path_rows(sampler):
    """NaNs and stop tokens in slices the bulk copy does not stage (an unaligned
    row start, a ragged tail) and on rows the exact path finishes."""
    b = workloads.random_batch(119, 20, 5003, "bf16", mix="all", stride_pad=3)
    _check(sampler, _with_nans(_with_stops(b, 120, owe=1.0), 121, frac=0.03), logits_offset_elems=1)
    t = workloads.random_batch(122, 10, 20000, "bf16", mix="topk")
    t = t.with_(top_k=np.int32([200, 500, 1000, 129, 150, 300, 250, 700, 3000, 180]))
    _check(sampler, _with_nans(_with_stops(t, 123, owe=1.0), 124, frac=0.02))


def test_sanitising_edge_rows(sampler):
    b = workloads.random_batch(125, 4, 3000, "f32", mix="all")
    x = b.logits.copy()
    x[0, :] = np.nan            # nothing left: all -inf
    x[1, 5] = np.inf            # +inf stays an error
    x[2, ::2] = np.nan          # half the row
    x[3, :] = -np.inf
    x[3, 2999] = np.nan         # -inf and NaN only
    b = b.with_(logits=x, sanitize_nan=True)
    g = dev.run(sampler, b, want_probs=False)
    assert g.status.tolist() == [2, 1, 0, 2]
    _check(sampler, b)
    g = dev.run(sampler, b.with_(sanitize_nan=False), want_probs=False)
    assert g.status.tolist() == [1, 1, 1, 1]


def test_stop_limits(sampler):
    b = workloads.random_batch(126, 3, 1000, "f32", mix="plain")
    offs = np.array([0, 17, 18, 19], np.int32)
    ids = np.concatenate([np.arange(17), [1000], [3]]).astype(np.int32)
    b = b.with_(min_tokens_left=np.int32([0, 0, 1]), stop_offsets=offs, stop_ids=ids)
    g = dev.run(sampler, b, want_probs=False)
    assert g.status.tolist() == [3, 3, 0]
    _check(sampler, b)


def test_logprob_outputs_see_the_ban_and_the_sanitising(sampler):
    b = workloads.random_batch(127, 16, 12000, "bf16", mix="all")
    b = _with_nans(_with_stops(b, 128, owe=1.0), 129, frac=0.02)
    for unscaled in (False, True):
        g = dev.run_logprobs(sampler, b, 5, unscaled)
        o = oracle.sample(b, want_probs=True, nthreads=16)
        lo = oracle.logprob_outputs(b, o, 5, unscaled)
        amb = o.ambiguous(1e-6)
        for r in range(b.n_rows):
            assert g.status[r] == o.status[r]
            if amb[r] or o.status[r]:
                continue
            assert g.tokens[r] == o.tokens[r]
            assert np.array_equal(g.top_ids[r], lo.top_ids[r]), (r, g.top_ids[r], lo.top_ids[r])
            np.testing.assert_allclose(g.top_logprobs[r], lo.top_logprobs[r], rtol=1e-5, atol=1e-6)
            assert abs(g.token_logprob[r] - lo.token_logprob[r]) <= 1e-6 + 1e-5 * abs(lo.token_logprob[r])
