"""Vocabulary bitmask through sampler_sample_ex vs the oracle (needs a GB300)."""
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


def _check(sampler, batch, **kw):
    g = dev.run(sampler, batch, want_probs=False, **kw)
    o = oracle.sample(batch, want_probs=False, nthreads=16)
    rep = compare(batch, g, o)
    assert rep.ok(), rep
    ok = g.status == 0
    bits = np.unpackbits(batch.vocab_mask.view(np.uint8), bitorder="little").reshape(batch.n_rows, -1)
    assert bits[np.nonzero(ok)[0], g.tokens[ok]].all(), "a disallowed token was sampled"
    return rep


@pytest.mark.parametrize("name", ["mixed", "latency32", "tiny"])
@pytest.mark.parametrize("allowed", [0.02, 0.3])
def test_named_workloads_masked(sampler, name, allowed):
    b = workloads.make(name)
    b = b.with_(vocab_mask=workloads.vocab_mask(61, b.n_rows, b.vocab, allowed=allowed))
    rep = _check(sampler, b)
    assert rep.gumbel_ties == 0 and rep.excused == 0, rep


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_every_stage_masked(sampler, dtype):
    b = workloads.random_batch(62, 48, 23000, dtype, mix="all")
    b = b.with_(vocab_mask=workloads.vocab_mask(63, b.n_rows, b.vocab, allowed=0.05))
    _check(sampler, b)


def test_unaligned_rows_and_tiny_masks(sampler):
    b = workloads.random_batch(64, 20, 5003, "bf16", mix="all", stride_pad=3)
    b = b.with_(vocab_mask=workloads.vocab_mask(65, b.n_rows, b.vocab, allowed=0.01, full_rows=0))
    _check(sampler, b, logits_offset_elems=1)


def test_fully_masked_and_single_token_rows(sampler):
    b = workloads.random_batch(66, 6, 4000, "f32", mix="all")
    m = np.zeros((6, (4000 + 31) // 32), np.uint32)
    m[0, :] = 0xFFFFFFFF
    m[1, 3] = 1 << 7           # only token 103
    m[3, 124] = 1 << 31        # only token 3999
    b = b.with_(vocab_mask=m)
    g = dev.run(sampler, b, want_probs=False)
    assert g.status[2] == 2 and g.status[4] == 2 and g.status[5] == 2
    assert g.tokens[1] == 103 or g.status[1] != 0
    assert g.tokens[3] == 3999 or g.status[3] != 0
    _check(sampler, b)


def test_mask_with_logprob_outputs(sampler):
    b = workloads.random_batch(67, 24, 9000, "bf16", mix="all")
    b = b.with_(vocab_mask=workloads.vocab_mask(68, b.n_rows, b.vocab, allowed=0.1))
    for unscaled in (False, True):
        g = dev.run_logprobs(sampler, b, 8, unscaled)
        o = oracle.sample(b, want_probs=True, nthreads=16)
        lo = oracle.logprob_outputs(b, o, 8, unscaled)
        amb = o.ambiguous(1e-6)
        for r in range(b.n_rows):
            assert g.status[r] == o.status[r]
            if amb[r] or o.status[r]:
                continue
            assert g.tokens[r] == o.tokens[r]
            assert np.array_equal(g.top_ids[r], lo.top_ids[r]), (r, g.top_ids[r], lo.top_ids[r])
            assert abs(g.token_logprob[r] - lo.token_logprob[r]) <= 1e-6 + 1e-5 * abs(lo.token_logprob[r])


def test_mask_refusals(sampler):
    import torch
    import decode_step_token_gb300 as d
    b = workloads.random_batch(69, 4, 1000, "f32", penalties=True)
    b = b.with_(vocab_mask=workloads.vocab_mask(70, 4, 1000))
    dd = dev.to_device(b)
    with pytest.raises(d.SamplerError) as e:
        sampler.sample_ex_args(dev.sample_args(sampler, b, dd), vocab_mask=dd["vocab_mask"])
    assert e.value.code == -8
    b2 = workloads.random_batch(71, 4, 1000, "f32").with_(vocab_mask=workloads.vocab_mask(72, 4, 1000))
    dd2 = dev.to_device(b2)
    with pytest.raises(d.SamplerError) as e:
        sampler.sample_ex_args(dev.sample_args(sampler, b2, dd2), vocab_mask=dd2["vocab_mask"], mask_stride=30)
    assert e.value.code == -8
