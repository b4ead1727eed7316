"""The LM-head GEMM (tcgen05) chained to the sampler, through
sampler_lm_head_sample, vs the oracle (needs a GB300).

The logits are checked against the double-precision product within the bound
of an fp32 sum of K products followed by one rounding to bf16:
    |gpu - exact| <= 2^-8 |exact| + (1 + 2^-8) K 2^-23 sum_k |h_k w_k|
(2^-8 is bf16's unit roundoff, 8 significant bits; 2^-23 per addition allows
for truncating rather than rounding fp32 adds). The
tokens are checked against the oracle's sampler run on the logits the GPU
wrote, so both sides decide on the same fp32 values."""
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
    s = d.Sampler(max_rows=1024, max_vocab=262144, max_history=1 << 16)
    yield s
    s.close()


def _check_logits(g, hidden, weight, n, V, cols=None):
    L, A = oracle.lm_head_logits(hidden, weight, cols)
    got = workloads.bf16_bits_to_f32(g.logits[:n, :V] if cols is None else g.logits[:n, cols]).reshape(L.shape)
    K = hidden.shape[1]
    bound = 2.0 ** -8 * np.abs(L) + (1 + 2.0 ** -8) * K * 2.0 ** -23 * A
    bad = np.abs(got.astype(np.float64) - L) > bound
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], L[bad][:5])


def _check_tokens(g, batch):
    b = batch.with_(logits=g.logits)
    o = oracle.sample(b, want_probs=False, nthreads=16)
    rep = compare(b, g, o)
    assert rep.ok(), rep
    return rep


@pytest.mark.parametrize("n,V,K,hpad,wpad,vpad", [(1, 1000, 64, 0, 0, 0), (5, 5003, 100, 4, 12, 3),
                                                  (16, 4096, 192, 0, 0, 0), (64, 20000, 512, 8, 0, 0),
                                                  (200, 3000, 256, 0, 64, 5), (256, 1024, 1024, 0, 0, 0)])
def test_shapes(sampler, n, V, K, hpad, wpad, vpad):
    """Rows not a multiple of 16, a ragged last tile, K not a multiple of 64,
    padded strides (the padding holds NaN, which the product must not read)."""
    hidden, weight, b = workloads.lm_head(70 + n, n, V, K)
    b = b.with_(logits=np.zeros((n, V + vpad), np.uint16))
    g = dev.run_lm_head(sampler, hidden, weight, b, hidden_stride=K + hpad, weight_stride=K + wpad)
    _check_logits(g, hidden, weight, n, V)
    assert np.all(g.logits[:, V:] == 0x7F81)  # the row padding is never written
    _check_tokens(g, b)


def test_full_size_step(sampler):
    """64 rows x V = 128000 x K = 4096 (the mixed batch's step behind an LM head):
    sampled vocabulary columns against the oracle, every token against the
    oracle's sampler on the written logits."""
    import torch

    n, V, K = 64, 128000, 4096
    hidden, _, b = workloads.lm_head(6, n, V, K, weight=False)
    gen = torch.Generator(device="cuda:0").manual_seed(6)
    w = (torch.randn((V, K), generator=gen, device="cuda:0") * (2.0 / 64.0)).to(torch.bfloat16).view(torch.int16)
    g = dev.run_lm_head(sampler, hidden, w, b)
    cols = np.random.default_rng(0).choice(V, 4096, replace=False)
    wcols = w[torch.from_numpy(cols).to("cuda:0")].cpu().numpy().view(np.uint16)
    L, A = oracle.lm_head_logits(hidden, wcols)
    got = workloads.bf16_bits_to_f32(g.logits[:, cols]).reshape(L.shape).astype(np.float64)
    bound = 2.0 ** -8 * np.abs(L) + (1 + 2.0 ** -8) * K * 2.0 ** -23 * A
    assert np.all(np.abs(got - L) <= bound)
    rep = _check_tokens(g, b)
    assert rep.gumbel_ties == 0, rep
    del w
    torch.cuda.empty_cache()


def test_group_path_and_forks(sampler):
    """A call the small-batch kernel does not take (history) runs the sampler in
    stream order after the GEMM; forks read their base row's logits."""
    hidden, weight, b = workloads.lm_head(80, 24, 6000, 256)
    b = b.with_(presence=np.full(24, 0.5, np.float32),
                hist_offsets=np.arange(0, 25 * 3, 3, dtype=np.int32)[:25],
                hist_ids=np.random.default_rng(1).integers(0, 6000, 72).astype(np.int32))
    g = dev.run_lm_head(sampler, hidden, weight, b)
    _check_logits(g, hidden, weight, 24, 6000)
    _check_tokens(g, b)
    fk = b.with_(hist_offsets=None, hist_ids=None, presence=None, n_rows=48,
                 temperature=np.tile(b.temperature, 2), top_k=np.tile(b.top_k, 2), top_p=np.tile(b.top_p, 2),
                 logit_row=np.tile(np.arange(24, dtype=np.int32), 2),
                 stream_id=np.repeat(np.arange(2, dtype=np.uint32), 24))
    g = dev.run_lm_head(sampler, hidden, weight, fk)
    _check_logits(g, hidden, weight, 24, 6000)
    _check_tokens(g, fk)


def test_extensions_pass_through(sampler):
    hidden, weight, b = workloads.lm_head(81, 32, 9000, 320)
    offs, ids, vals = workloads.logit_bias(82, 32, 9000, 16)
    b = b.with_(bias_offsets=offs, bias_ids=ids, bias_values=vals,
                vocab_mask=workloads.vocab_mask(83, 32, 9000, allowed=0.5))
    g = dev.run_lm_head(sampler, hidden, weight, b, **dev.ext_kw(dev.to_device(b, "cuda:0", False)))
    _check_logits(g, hidden, weight, 32, 9000)
    _check_tokens(g, b)


def test_graph_replay_matches_eager(sampler):
    import torch

    hidden, weight, b = workloads.lm_head(84, 48, 16000, 512)
    g0 = dev.run_lm_head(sampler, hidden, weight, b)
    h = dev.bf16_device(hidden)
    w = dev.bf16_device(weight)
    d = dev.to_device(b, "cuda:0", False)
    args = dev.sample_args(sampler, b, d)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        sampler.lm_head_sample_args(args, h, w, stream=s.cuda_stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            sampler.lm_head_sample_args(args, h, w, stream=torch.cuda.current_stream().cuda_stream)
    d["logits"][0].zero_()
    d["out_tokens"].fill_(-7)
    graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(d["logits"][0].view(torch.int16).cpu().numpy().view(np.uint16), g0.logits)
    assert np.array_equal(d["out_tokens"].cpu().numpy(), g0.tokens)


def test_refusals(sampler):
    import torch
    import decode_step_token_gb300 as dd

    hidden, weight, b = workloads.lm_head(85, 4, 512, 64)
    h = dev.bf16_device(hidden)
    w = dev.bf16_device(weight)
    d = dev.to_device(b, "cuda:0", False)
    args = dev.sample_args(sampler, b, d)
    with pytest.raises(dd.SamplerError) as e:  # a stride that is not a multiple of 8
        sampler.lm_head_sample_args(args, h, w, hidden_stride=66)
    assert e.value.code == -2
    f = b.with_(logits=np.zeros((4, 512), np.float32), dtype="f32")
    df = dev.to_device(f, "cuda:0", False)
    with pytest.raises(dd.SamplerError) as e:
        sampler.lm_head_sample_args(dev.sample_args(sampler, f, df), h, w)
    assert e.value.code == -4
    big_h, _, big = workloads.lm_head(86, 257, 512, 64, weight=False)
    db = dev.to_device(big, "cuda:0", False)
    with pytest.raises(dd.SamplerError) as e:
        sampler.lm_head_sample_args(dev.sample_args(sampler, big, db), dev.bf16_device(big_h), w)
    assert e.value.code == -3
    assert sampler.stat(dd.SAMPLER_STAT_LM_HEAD_TIMEOUTS) == 0


def test_logits_only_entry(sampler):
    import torch

    hidden, weight, b = workloads.lm_head(87, 40, 7000, 384)
    g = dev.run_lm_head(sampler, hidden, weight, b)
    out = torch.zeros((40, 7008), dtype=torch.int16, device="cuda:0")
    sampler.lm_head(dev.bf16_device(hidden), dev.bf16_device(weight), out, vocab=7000)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16)
    assert np.array_equal(got[:, :7000], g.logits)
    assert np.all(got[:, 7000:] == 0)
