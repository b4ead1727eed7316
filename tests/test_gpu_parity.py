"""CUDA sampler vs the CPU oracle, element by element (needs a GB300)."""
import numpy as np
import pytest

import oracle
import workloads
from workloads import SamplerBatch, device as dev
from parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sampler():
    """One handle: small batches without outputs take the slice kernel, the rest
    the fork-group kernel."""
    from decode_step_token_gb300 import build
    build.build_library()
    import decode_step_token_gb300 as d
    s = d.Sampler(max_rows=2048, max_vocab=262144, host_staging=False)
    yield s
    s.close()


def _check(sampler, batch, rows=None, want_probs=None, nthreads=8, **kw):
    g = dev.run(sampler, batch, want_probs=want_probs, **kw)
    o = oracle.sample(batch, rows=rows, want_probs=want_probs, nthreads=nthreads)
    rep = compare(batch, g, o, rows=rows)
    assert rep.ok(), rep
    return g, o, rep


def _named(sampler, batch, want_probs):
    """Every row of a named workload; no Gumbel tie and no excused difference."""
    _, _, rep = _check(sampler, batch, want_probs=want_probs, nthreads=16)
    print(f"{batch.name} want_probs={want_probs}: {rep}")
    assert rep.rows == batch.n_rows
    assert rep.gumbel_ties == 0 and rep.excused == 0, rep
    return rep


# ----------------------------------------------------------------------------- named workloads

@pytest.mark.parametrize("want", [False, True])
def test_tiny(sampler, want):
    _named(sampler, workloads.tiny(), want)


@pytest.mark.parametrize("want", [False, True])
def test_mixed_full_size(sampler, want):
    _named(sampler, workloads.mixed(), want)


@pytest.mark.parametrize("n", [1, 32])
@pytest.mark.parametrize("want", [False, True])
def test_latency_full_size(sampler, n, want):
    _named(sampler, workloads.latency(n), want)


def test_penalties_full_size(sampler):
    _named(sampler, workloads.penalties(), True)


@pytest.mark.parametrize("want", [False, True])
def test_forks_full_size(sampler, want):
    b = workloads.forks()
    _named(sampler, b, want)
    if not want:
        # forks of one base row with different streams draw independently
        g = dev.run(sampler, b, want_probs=False)
        base = g.tokens.reshape(-1, 4)
        assert (base[:, 0] != base[:, 1]).any()


def test_forks_with_probs_sampled_rows(sampler):
    b = workloads.forks(base_rows=24)
    _check(sampler, b, want_probs=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fork_groups_irregular(sampler, dtype):
    """Runs of forks of every length (longer than one group, split, interleaved),
    each fork with its own parameters and stream."""
    rng = np.random.default_rng(12)
    lrow = np.int32([0, 0, 0, 1, 1, 2] + [3] * 12 + [0, 4, 4, 1, 2, 2, 3, 3])
    n = len(lrow)
    b = workloads.random_batch(77, n, 30000, dtype, want_probs=True)
    base = workloads.random_batch(78, 5, 30000, dtype)
    b = b.with_(logits=base.logits, logit_row=lrow,
                stream_id=rng.integers(0, 2**31, size=n).astype(np.uint32))
    g, _, _ = _check(sampler, b)
    g2, _, _ = _check(sampler, b.with_(want_probs=False))
    assert np.array_equal(g.tokens, g2.tokens)


# ----------------------------------------------------------------------------- randomized small

@pytest.mark.parametrize("v", [1, 3, 4, 5, 8, 1023, 1024, 1025, 4099, 17000, 40000])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_random_rows(sampler, v, dtype):
    for seed in range(3):
        b = workloads.random_batch(1000 * v + seed, 12, v, dtype, want_probs=seed == 1,
                                   penalties=seed == 2, stride_pad=seed * 3)
        _check(sampler, b)


@pytest.mark.parametrize("want", [False, True])
@pytest.mark.parametrize("mix", ["topk", "topp", "minp", "plain"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_each_stage_alone(sampler, mix, dtype, want):
    b = workloads.random_batch(7, 16, 50000, dtype, mix=mix, want_probs=want)
    _check(sampler, b)


@pytest.mark.parametrize("want", [False, True])
@pytest.mark.parametrize("k", [65, 100, 1000, 5000, 60000])
def test_large_topk_radix_path(sampler, k, want):
    b = workloads.random_batch(k, 8, 70000, "bf16", mix="plain", want_probs=want)
    b = b.with_(top_k=np.full(8, k, np.int32), top_p=np.float32(np.linspace(0.3, 1.0, 8)))
    _check(sampler, b)


@pytest.mark.parametrize("want", [False, True])
def test_ties_everywhere(sampler, want):
    for dtype in ("f32", "bf16"):
        b = workloads.random_batch(11, 16, 30000, dtype, ties=True, want_probs=want)
        _check(sampler, b)
    # a flat top: more tied candidates than the candidate buffer holds
    x = np.zeros((4, 20000), np.float32)
    x[:, ::3] = 5.0
    b = SamplerBatch("flat", x, "f32", 20000, 4, np.float32([1.0, 0.5, 0.0, 2.0]),
                     top_k=np.int32([50, 3000, 7, 64]), top_p=np.float32([1.0, 0.2, 0.9, 0.999]),
                     want_probs=want)
    _check(sampler, b)


def test_penalties_random(sampler):
    for dtype in ("f32", "bf16"):
        b = workloads.random_batch(5, 16, 30000, dtype, penalties=True, max_hist=3000,
                                   want_probs=True)
        _check(sampler, b)


# ----------------------------------------------------------------------------- edge cases

def test_status_rows(sampler):
    V = 3000
    x = np.random.default_rng(2).standard_normal((9, V)).astype(np.float32)
    x[2, 17] = np.nan
    x[3, 100] = np.inf
    x[4, :] = -np.inf
    x[6, :] = -np.inf
    x[6, 2999] = 1.0  # one finite token at the end
    t = np.float32([1, -1, 1, 1, 1, 1, 0.5, np.nan, 1])
    offs = np.int32([0, 0, 0, 0, 0, 0, 1, 1, 1, 1])
    ids = np.int32([V])  # out of range for row 5
    b = SamplerBatch("st", x, "f32", V, 9, t, top_k=np.int32([5, 5, 5, 5, 5, 5, 5, 5, 0]),
                     hist_offsets=offs, hist_ids=ids, want_probs=True)
    g, o, _ = _check(sampler, b)
    assert list(g.status) == [0, 3, 1, 1, 2, 4, 0, 3, 3]
    assert g.tokens[6] == 2999


def test_long_history_is_rejected_per_row(sampler):
    V = 1000
    x = np.zeros((2, V), np.float32)
    offs = np.int32([0, 70000, 70001])
    ids = np.zeros(70001, np.int32)
    b = SamplerBatch("h", x, "f32", V, 2, np.float32([1, 1]), hist_offsets=offs, hist_ids=ids)
    g, _, _ = _check(sampler, b)
    assert list(g.status) == [4, 0]


@pytest.mark.parametrize("want", [False, True])
def test_unaligned_rows_and_strides(sampler, want):
    for dtype, off in (("bf16", 1), ("bf16", 3), ("f32", 1), ("f32", 2)):
        b = workloads.random_batch(3, 6, 9001, dtype, stride_pad=5, want_probs=want)
        _check(sampler, b, logits_offset_elems=off)


def test_empty_batch_is_a_noop(sampler):
    import torch
    import decode_step_token_gb300 as d
    out = torch.full((1,), 5, dtype=torch.int32, device="cuda")
    args = d.Sampler.make_args(logits=torch.zeros((1, 10), device="cuda"),
                               temperature=torch.zeros(0, device="cuda"), n_rows=0,
                               out_tokens=out)
    sampler.sample_args(args)
    torch.cuda.synchronize()
    assert out.item() == 5


def test_host_rejections(sampler):
    import torch
    import decode_step_token_gb300 as d
    x = torch.zeros((2, 10), device="cuda")
    t = torch.ones(2, device="cuda")
    out = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(d.SamplerError) as e:
        sampler.sample(logits=x, temperature=t, out_tokens=out, vocab=300000, row_stride=300000)
    assert e.value.code == d._binding.SAMPLER_ERR_TOO_LARGE
    with pytest.raises(d.SamplerError) as e:
        sampler.sample(logits=x, temperature=t, out_tokens=out, dtype=9)
    assert e.value.code == d._binding.SAMPLER_ERR_BAD_DTYPE
    with pytest.raises(d.SamplerError) as e:
        sampler.sample(logits=x, temperature=t, out_tokens=out, row_stride=5)
    assert e.value.code == d._binding.SAMPLER_ERR_BAD_SHAPE


@pytest.mark.parametrize("want", [False, True])
def test_greedy_threshold_and_extreme_params(sampler, want):
    V = 5000
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((8, V)) * 3).astype(np.float32)
    t = np.float32([0.0, 0.9e-5, 1.1e-5, 1e-3, 1.0, 5.0, 1.0, 1.0])
    k = np.int32([-1, -1, -1, -1, V, V - 1, 1, -1])
    p = np.float32([1, 1, 1, 1, 1e-7, 1, 1, 1])
    mp = np.float32([0, 0, 0, 0, 0, 0, 0, 1.0])
    b = SamplerBatch("x", x, "f32", V, 8, t, top_k=k, top_p=p, min_p=mp, global_seed=77,
                     want_probs=want)
    _check(sampler, b)


def test_max_vocab_fp32_with_penalties(sampler):
    b = workloads.random_batch(21, 4, 262144, "f32", penalties=True, max_hist=4096,
                               want_probs=True)
    _check(sampler, b)


# ----------------------------------------------------------------------------- properties

def test_seeded_rows_are_batch_invariant(sampler):
    rng = np.random.default_rng(4)
    V = 50000
    row = (rng.standard_normal(V) * 2).astype(np.float32)
    toks = []
    for n, pos in ((1, 0), (7, 3), (33, 32)):
        x = (rng.standard_normal((n, V)) * 2).astype(np.float32)
        x[pos] = row
        seeded = np.zeros(n, np.uint8)
        seeded[pos] = 1
        others_p = np.float32(rng.uniform(0.5, 1.0, n))
        others_p[pos] = 0.95
        b = SamplerBatch("inv", x, "f32", V, n, np.full(n, 0.9, np.float32),
                         top_p=others_p, seed=np.full(n, 1234, np.uint64), has_seed=seeded,
                         stream_id=np.zeros(n, np.uint32), global_seed=int(rng.integers(1 << 40)))
        g = dev.run(sampler, b, want_probs=False)
        toks.append(int(g.tokens[pos]))
    assert len(set(toks)) == 1


def test_plain_rows_ignore_their_neighbours_parameters(sampler):
    b = workloads.mixed(n=16, v=30000)
    g1 = dev.run(sampler, b)
    plain = b.notes["kinds"] == 0
    k2 = b.top_k.copy()
    p2 = b.top_p.copy()
    k2[~plain] = 1
    p2[~plain] = 0.1
    g2 = dev.run(sampler, b.with_(top_k=k2, top_p=p2))
    assert np.array_equal(g1.tokens[plain], g2.tokens[plain])


@pytest.mark.parametrize("k", [5, 20, 32])
def test_masked_rows_with_few_finite_lanes(sampler, k):
    """Rows masked to -inf except one 8-token vector in 32: each slice then has a
    single finite lane maximum, fewer than the top k its list must hold."""
    b = workloads.random_batch(77 + k, 6, 40000, "bf16", mix="topk")
    x = workloads.bf16_bits_to_f32(b.logits).reshape(b.n_rows, -1).copy()
    vec = np.arange(x.shape[1]) // 8
    x[:, (vec % 32) != 0] = -np.inf
    b = b.with_(logits=workloads.to_bf16_bits(x), top_k=np.full(6, k, np.int32),
                top_p=np.ones(6, np.float32), min_p=np.zeros(6, np.float32))
    _check(sampler, b, want_probs=False)


def test_exact_path_runs_and_matches(sampler):
    """Rows the slice kernel's candidate lists cannot settle (top-k above their
    cap, top-p reaching past the lists, flat rows) take its exact path."""
    sampler.stat(0, reset=True)
    b = workloads.random_batch(91, 12, 30000, "bf16", mix="topp")
    b = b.with_(top_k=np.int32([200, 500, -1, -1, 129, 3000, -1, -1, 1000, -1, 150, -1]),
                top_p=np.float32([1.0, 0.9, 0.95, 0.5, 1.0, 0.99, 0.8, 0.999, 0.7, 0.3, 0.6, 0.9]))
    _check(sampler, b, want_probs=False)
    assert sampler.stat(0, reset=True) > 0


def test_truncated_rows_repeat_without_exact_path(sampler):
    """Back-to-back calls with truncated rows on one handle, batches of different
    sizes interleaved: each truncated unit adds its sketch keys to its row's
    histogram and the finishing warp clears it, so every call gives the same
    tokens and no row falls to the exact path (a histogram left over from an
    earlier call would move the bound past the row's k-th value)."""
    lat, mix = workloads.latency(32), workloads.mixed()
    first = {}
    sampler.stat(0, reset=True)
    for rep in range(3):
        for b in (lat, mix, lat):
            g = dev.run(sampler, b, want_probs=False)
            assert (g.status == 0).all()
            if b.name not in first:
                first[b.name] = g.tokens
            assert np.array_equal(g.tokens, first[b.name]), (rep, b.name)
    assert sampler.stat(0, reset=True) == 0
    o = oracle.sample(lat, want_probs=False, nthreads=16)
    assert np.array_equal(first[lat.name][~o.ambiguous()], o.tokens[~o.ambiguous()])


def test_wait_timeout_status():
    """A handle whose staging waits give up at once reports status 5 on every row
    of a small batch (token -1), and the next call on an ordinary handle is
    unaffected."""
    import decode_step_token_gb300 as d
    b = workloads.random_batch(92, 16, 20000, "bf16")
    with d.Sampler(max_rows=64, max_vocab=20000, short_waits=True) as s:
        g = dev.run(s, b, want_probs=False)
    assert (g.status == 5).all(), g.status
    assert (g.tokens == -1).all()
    with d.Sampler(max_rows=64, max_vocab=20000) as s:
        g = dev.run(s, b, want_probs=False)
    o = oracle.sample(b, want_probs=False)
    rep = compare(b, g, o)
    assert rep.ok(), rep


def test_device_philox_offset(sampler):
    import torch
    b = workloads.random_batch(8, 8, 20000, "bf16", mix="plain")
    d = dev.to_device(b)
    off = torch.tensor([b.philox_offset + 5], dtype=torch.int64, device="cuda")
    sampler.sample_args(dev.sample_args(sampler, b, d, philox_offset=0, philox_offset_dev=off))
    torch.cuda.synchronize()
    t_dev = d["out_tokens"].cpu().numpy()
    o = oracle.sample(b.with_(philox_offset=b.philox_offset + 5))
    assert np.array_equal(t_dev[o.ambiguous() == 0], o.tokens[o.ambiguous() == 0])


def test_host_entry_matches_device_entry():
    import ctypes
    import decode_step_token_gb300 as d
    b = workloads.random_batch(31, 10, 7000, "bf16", want_probs=True, penalties=True)
    s = d.Sampler(max_rows=16, max_vocab=8000, max_history=10000, host_staging=True)
    try:
        N, V = b.n_rows, b.vocab
        tok = np.zeros(N, np.int32)
        st = np.zeros(N, np.int32)
        pr = np.zeros((N, V), np.float32)
        lp = np.zeros((N, V), np.float32)
        keep = {}

        def P(a, dt=None):
            if a is None:
                return None
            arr = np.ascontiguousarray(a if dt is None else a.astype(dt))
            keep[id(arr)] = arr
            return arr.ctypes.data

        args = d.sampler_args_t(
            P(b.logits), 1, N, V, b.row_stride, b.n_logit_rows, None, P(b.temperature),
            P(b.top_k), P(b.top_p), P(b.min_p), P(b.presence), P(b.frequency), P(b.repetition),
            P(b.seed), P(b.has_seed), None, P(b.hist_offsets), P(b.hist_ids), b.global_seed,
            b.philox_offset, None, tok.ctypes.data, pr.ctypes.data, lp.ctypes.data, st.ctypes.data)
        s.sample_host_args(args, 0)
        o = oracle.sample(b)
        from workloads.device import GpuResult
        rep = compare(b, GpuResult(tok, st, pr, lp), o)
        assert rep.ok(), rep
    finally:
        s.close()
