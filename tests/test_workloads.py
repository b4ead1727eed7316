"""The seeded synthetic inputs match the stated recipes (shapes, dtypes, parameter
mixes), and the bf16 rounding is round-to-nearest-even. CPU only."""
import numpy as np
import pytest

import workloads


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2.0**-8, 1.0 + 3 * 2.0**-8, 1.0 + 2.0**-9, -2.5, 65504.0], np.float32)
    got = workloads.bf16_bits_to_f32(workloads.to_bf16_bits(x))
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1.0);
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: ties go to 1 + 2^-6
    want = np.array([1.0, 1.0, 1.0 + 2.0**-6, 1.0, -2.5, 65536.0], np.float32)
    np.testing.assert_array_equal(got, want)


def test_tiny_recipe():
    b = workloads.make("tiny")
    assert (b.n_rows, b.vocab, b.dtype) == (4, 1024, "f32")
    np.testing.assert_array_equal(b.temperature, [1.0, 1.0, 1.0, 0.0])


def test_mixed_recipe():
    b = workloads.make("mixed")
    assert (b.n_rows, b.vocab, b.dtype) == (64, 128000, "bf16")
    kinds = b.notes["kinds"]
    assert [(kinds == k).sum() for k in (0, 1, 2)] == [32, 16, 16]
    plain, trunc, greedy = kinds == 0, kinds == 1, kinds == 2
    np.testing.assert_array_equal(b.temperature[plain], np.float32(0.8))
    np.testing.assert_array_equal(b.temperature[trunc], 1.0)
    np.testing.assert_array_equal(b.temperature[greedy], 0.0)
    np.testing.assert_array_equal(b.top_k[trunc], 50)
    np.testing.assert_array_equal(b.top_k[~trunc], -1)
    np.testing.assert_array_equal(b.top_p[trunc], np.float32(0.9))
    np.testing.assert_array_equal(b.top_p[~trunc], 1.0)
    x = b.logits_f32()
    spike = b.notes["spike"]
    # the spiked token carries 2*N(0,1) + 12 and is the row maximum in most rows
    lift = x[np.arange(64), spike] - 12.0
    assert abs(float(lift.mean())) < 0.75 and 1.4 < float(lift.std()) < 2.6
    assert (np.argmax(x, axis=1) == spike).mean() > 0.8
    rest = np.delete(x[0], spike[0])
    assert abs(float(rest.std()) - 2.0) < 0.05 and abs(float(rest.mean())) < 0.05


@pytest.mark.parametrize("n", [1, 32])
def test_latency_recipe(n):
    b = workloads.make(f"latency{n}")
    assert (b.n_rows, b.vocab, b.dtype) == (n, 151936, "bf16")
    np.testing.assert_allclose(b.temperature, 0.7)
    np.testing.assert_array_equal(b.top_k, 20)
    np.testing.assert_allclose(b.top_p, 0.8)
    np.testing.assert_array_equal(b.min_p, 0.0)
    # Zipf-shaped bias: early token ids are larger on average than late ones
    x = b.logits_f32()
    assert x[:, :100].mean() > x[:, -100:].mean() + 8.0


def test_penalties_recipe():
    b = workloads.make("penalties")
    assert (b.n_rows, b.vocab, b.dtype) == (128, 128000, "f32")
    assert b.want_probs
    lens = np.diff(b.hist_offsets)
    assert lens.min() >= 0 and lens.max() <= 4096
    assert b.hist_offsets[0] == 0 and b.hist_offsets[-1] == len(b.hist_ids)
    assert b.hist_ids.min() >= 0 and b.hist_ids.max() < b.vocab
    # Zipf(1.2) ranks: id 0 is the most frequent, and ids are heavily skewed to the head
    counts = np.bincount(b.hist_ids, minlength=8)
    assert counts[0] == counts.max()
    # Zipf(1.2) redrawn until below V: P(rank 1) = 1 / sum_{k<=V} k^-1.2 (0.1954)
    p1 = 1.0 / np.sum(np.arange(1, b.vocab + 1, dtype=np.float64) ** -1.2)
    assert abs(counts[0] / len(b.hist_ids) - p1) < 0.005
    for name, val in (("presence", 0.5), ("frequency", 0.3), ("repetition", 1.1), ("min_p", 0.05),
                      ("temperature", 1.0)):
        np.testing.assert_allclose(getattr(b, name), val, rtol=1e-7)


def test_forks_recipe():
    b = workloads.make("forks")
    base, nf = b.notes["base_rows"], b.notes["n_forks"]
    assert (base, nf, b.n_rows, b.vocab, b.dtype) == (256, 4, 1024, 256000, "bf16")
    assert b.n_logit_rows == base
    np.testing.assert_array_equal(b.logit_row, np.repeat(np.arange(base), nf))
    # every fork has its own Philox stream (the output row index)
    assert len(np.unique(b.stream_id)) == b.n_rows
    per_base = lambda a: a.reshape(base, nf)
    for a in (b.temperature, b.top_k, b.top_p, b.min_p, b.seed, b.has_seed):
        pb = per_base(a)
        assert (pb == pb[:, :1]).all()  # the forks of a base row share its parameters
    t = per_base(b.temperature)[:, 0]
    assert t.min() >= 0.0 and t.max() < 1.5 and 0.03 < (t == 0.0).mean() < 0.2
    assert set(np.unique(b.top_k).tolist()) == {-1, 20, 50, 1000}
    p = per_base(b.top_p)[:, 0]
    assert p.min() >= 0.5 and p.max() < 1.0
    assert set(np.unique(b.min_p).tolist()) <= {0.0, np.float32(0.05)}
    assert 0.15 < per_base(b.has_seed)[:, 0].mean() < 0.35
