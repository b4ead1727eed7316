"""logit_bias through sampler_sample_ex vs the oracle (needs a GB300)."""
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


def _with_bias(b, seed, max_per_row=64, scale=5.0):
    offs, ids, vals = workloads.logit_bias(seed, b.n_rows, b.vocab, max_per_row, scale)
    return b.with_(bias_offsets=offs, bias_ids=ids, bias_values=vals)


def _check(sampler, batch, **kw):
    g = dev.run(sampler, batch, want_probs=False, **kw)
    o = oracle.sample(batch, want_probs=False, nthreads=16)
    rep = compare(batch, g, o)
    assert rep.ok(), rep
    return rep


@pytest.mark.parametrize("name", ["mixed", "latency32", "tiny"])
def test_named_workloads_biased(sampler, name):
    rep = _check(sampler, _with_bias(workloads.make(name), 91))
    assert rep.gumbel_ties == 0 and rep.excused == 0, rep


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_every_stage_biased(sampler, dtype):
    _check(sampler, _with_bias(workloads.random_batch(92, 48, 21000, dtype, mix="all"), 93))


def test_forced_and_banned_tokens(sampler):
    """A +50 bias forces its token; -inf bans the maximum; repeated ids add up."""
    b = workloads.random_batch(94, 8, 30000, "bf16", mix="all")
    x = workloads.bf16_bits_to_f32(b.logits).reshape(b.n_rows, -1)
    top = np.argmax(x, axis=1)
    offs = np.arange(0, 25, 3, dtype=np.int32)
    ids, vals = [], []
    for r in range(8):
        ids += [int(top[r]), (r * 977) % 30000, (r * 977) % 30000]
        vals += [-np.inf, 25.0, 25.0]
    b = b.with_(bias_offsets=offs, bias_ids=np.int32(ids), bias_values=np.float32(vals))
    _check(sampler, b)


def test_bias_with_mask_unaligned_and_logprobs(sampler):
    b = workloads.random_batch(95, 20, 5003, "bf16", mix="all", stride_pad=3)
    b = _with_bias(b, 96).with_(vocab_mask=workloads.vocab_mask(97, 20, 5003, allowed=0.3))
    _check(sampler, b, logits_offset_elems=1)
    for unscaled in (False, True):
        g = dev.run_logprobs(sampler, b, 6, unscaled)
        o = oracle.sample(b, want_probs=True, nthreads=16)
        lo = oracle.logprob_outputs(b, o, 6, unscaled)
        amb = o.ambiguous(1e-6)
        for r in range(b.n_rows):
            assert g.status[r] == o.status[r]
            if amb[r] or o.status[r]:
                continue
            assert g.tokens[r] == o.tokens[r]
            assert np.array_equal(g.top_ids[r], lo.top_ids[r]), (r, g.top_ids[r], lo.top_ids[r])
            assert abs(g.token_logprob[r] - lo.token_logprob[r]) <= 1e-6 + 1e-5 * abs(lo.token_logprob[r])


def test_bias_on_exact_path_rows(sampler):
    """Rows the lists cannot settle (top-k above the cap, flat rows) take the
    exact path, which must see the bias too."""
    b = workloads.random_batch(98, 10, 20000, "bf16", mix="topk")
    b = b.with_(top_k=np.int32([200, 500, 1000, 129, 150, 300, 250, 700, 3000, 180]))
    _check(sampler, _with_bias(b, 99, scale=8.0))
    flat = b.with_(logits=np.zeros_like(b.logits), top_k=np.full(10, 20, np.int32))
    _check(sampler, _with_bias(flat, 100))


def test_bias_limits(sampler):
    b = workloads.random_batch(101, 3, 1000, "f32", mix="plain")
    offs = np.array([0, 65, 66, 66], np.int32)
    ids = np.concatenate([np.arange(65), [1000]]).astype(np.int32)
    b = b.with_(bias_offsets=offs, bias_ids=ids, bias_values=np.ones(66, np.float32))
    g = dev.run(sampler, b, want_probs=False)
    assert g.status.tolist() == [3, 3, 0]
    _check(sampler, b)
