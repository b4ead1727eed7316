"""Per-row logprob outputs (sampled token + top-n, scaled or unscaled) of
sampler_sample_ex vs the oracle, element by element (needs a GB300)."""
import numpy as np
import pytest

import oracle
import workloads
from workloads import device as dev
from parity import ATOL, RTOL, TIE_TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sampler():
    from decode_step_token_gb300 import build
    build.build_library()
    import decode_step_token_gb300 as d
    s = d.Sampler(max_rows=256, max_vocab=262144)
    yield s
    s.close()


def _close(g, o):
    g = np.asarray(g, np.float64)
    o = np.asarray(o, np.float64)
    both_inf = np.isneginf(g) & np.isneginf(o)
    both_nan = np.isnan(g) & np.isnan(o)
    with np.errstate(invalid="ignore"):
        ok = both_inf | both_nan | (np.abs(g - o) <= ATOL + RTOL * np.abs(np.where(np.isfinite(o), o, 0)))
    return ok


def _check(sampler, batch, top_n, unscaled, allow_ambiguous=False):
    g = dev.run_logprobs(sampler, batch, top_n, unscaled)
    o = oracle.sample(batch, want_probs=True, nthreads=16)
    lo = oracle.logprob_outputs(batch, o, top_n, unscaled)
    amb = o.ambiguous(TIE_TOL)
    checked = 0
    for r in range(batch.n_rows):
        assert g.status[r] == o.status[r], (r, g.status[r], o.status[r])
        if amb[r]:
            assert allow_ambiguous, f"row {r} is ambiguous"
            continue
        checked += 1
        assert g.tokens[r] == o.tokens[r], (r, g.tokens[r], o.tokens[r])
        assert _close(g.token_logprob[r], lo.token_logprob[r]), (r, g.token_logprob[r], lo.token_logprob[r])
        assert np.array_equal(g.top_ids[r], lo.top_ids[r]), (r, g.top_ids[r], lo.top_ids[r])
        assert _close(g.top_logprobs[r], lo.top_logprobs[r]).all(), (r, g.top_logprobs[r], lo.top_logprobs[r])
    return checked


@pytest.mark.parametrize("unscaled", [False, True])
@pytest.mark.parametrize("name", ["tiny", "mixed", "latency1", "latency32"])
def test_named_workloads(sampler, name, unscaled):
    b = workloads.make(name)
    assert _check(sampler, b, 5, unscaled) == b.n_rows


@pytest.mark.parametrize("unscaled", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_every_stage_random(sampler, dtype, unscaled):
    b = workloads.random_batch(31 + int(unscaled), 40, 17000, dtype, mix="all")
    _check(sampler, b, 16, unscaled, allow_ambiguous=True)


@pytest.mark.parametrize("unscaled", [False, True])
def test_ties_and_short_rows(sampler, unscaled):
    """Coarse ties (lists overflow: the exact path takes the outputs), top_n past
    the kept set (padding), small vocabularies."""
    b = workloads.random_batch(41, 24, 3000, "bf16", mix="all", ties=True)
    _check(sampler, b, 16, unscaled, allow_ambiguous=True)
    b = workloads.random_batch(42, 16, 9, "f32", mix="topk")
    _check(sampler, b, 16, unscaled, allow_ambiguous=True)
    flat = b.with_(logits=np.zeros_like(b.logits))
    _check(sampler, flat, 7, unscaled, allow_ambiguous=True)


def test_error_rows_and_top_n_zero(sampler):
    b = workloads.random_batch(43, 8, 5000, "f32", mix="plain")
    x = b.logits.copy()
    x[2, 17] = np.nan
    x[5, :] = -np.inf
    b = b.with_(logits=x)
    g = dev.run_logprobs(sampler, b, 4)
    assert g.status[2] == 1 and g.status[5] == 2
    for r in (2, 5):
        assert np.isnan(g.token_logprob[r]) and (g.top_ids[r] == -1).all() and np.isnan(g.top_logprobs[r]).all()
    g0 = dev.run_logprobs(sampler, b, 0)
    assert np.array_equal(g0.tokens, g.tokens)
    assert np.array_equal(g0.token_logprob[[0, 1, 3]], g.token_logprob[[0, 1, 3]])


def test_tokens_match_the_plain_call(sampler):
    b = workloads.mixed()
    g = dev.run_logprobs(sampler, b, 8)
    p = dev.run(sampler, b, want_probs=False)
    assert np.array_equal(g.tokens, p.tokens)


def test_unsupported_calls_are_refused(sampler):
    import torch
    import decode_step_token_gb300 as d
    b = workloads.random_batch(44, 4, 1000, "f32", penalties=True)
    dd = dev.to_device(b)
    args = dev.sample_args(sampler, b, dd)
    out = torch.zeros(4, dtype=torch.float32, device="cuda")
    with pytest.raises(d.SamplerError) as e:
        sampler.sample_ex_args(args, out_token_logprob=out)
    assert e.value.code == -8
    b2 = workloads.random_batch(45, 4, 1000, "f32")
    args2 = dev.sample_args(sampler, b2, dev.to_device(b2))
    ids = torch.zeros((4, 17), dtype=torch.int32, device="cuda")
    lps = torch.zeros((4, 17), dtype=torch.float32, device="cuda")
    with pytest.raises(d.SamplerError) as e:
        sampler.sample_ex_args(args2, top_n=17, out_top_ids=ids, out_top_logprobs=lps)
    assert e.value.code == -8
