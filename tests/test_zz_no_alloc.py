"""The allocation-free entry point against the handle-based one (needs a GB300).

sampler_sample_noalloc keeps its workspace in the library's own device memory
instead of a handle's buffers; on the same inputs it must give what
sampler_sample gives, call after call (its row counters must come back to zero
after every call). The file name sorts last so that the test also runs after
every other GPU test in one process.
"""
import numpy as np
import pytest

import oracle
import workloads
from workloads import device as dev
from parity import compare

pytestmark = pytest.mark.gpu


def _noalloc(args, stream):
    from decode_step_token_gb300 import _binding as abi
    return abi.sampler_sample_noalloc(args, stream)


@pytest.fixture(scope="module")
def lib():
    from decode_step_token_gb300 import build
    build.build_library()
    import decode_step_token_gb300 as d
    s = d.Sampler(max_rows=256, max_vocab=262144)
    yield d, s
    s.close()


def _batches():
    yield workloads.mixed()                       # the 64-row mixed batch, bf16
    yield workloads.latency(32)                   # top-k / top-p rows, Zipf-shaped logits
    yield workloads.random_batch(71, 48, 20011, "f32")
    yield workloads.random_batch(72, 5, 3001, "bf16", ties=True)


@pytest.mark.parametrize("index", range(4))
def test_noalloc_matches_sample_twice(lib, index):
    import torch
    d, s = lib
    batch = list(_batches())[index]
    stream = torch.cuda.current_stream().cuda_stream
    dd = dev.to_device(batch, want_probs=False)
    args = dev.sample_args(s, batch, dd)
    s.sample_args(args)
    torch.cuda.synchronize()
    ref_tok = dd["out_tokens"].cpu().numpy().copy()
    ref_st = dd["out_status"].cpu().numpy().copy()
    for call in range(2):
        dd["out_tokens"].fill_(-7)
        dd["out_status"].fill_(-7)
        rc = _noalloc(args, stream)
        assert rc == d.SAMPLER_OK, d.sampler_status_string(rc)
        torch.cuda.synchronize()
        tok = dd["out_tokens"].cpu().numpy()
        st = dd["out_status"].cpu().numpy()
        # the same kernel on the same inputs: identical ids and statuses
        np.testing.assert_array_equal(tok, ref_tok, err_msg=f"call {call}")
        np.testing.assert_array_equal(st, ref_st, err_msg=f"call {call}")
    # and both agree with the oracle under the parity rules
    g = dev.GpuResult(tok, st, None, None)
    rep = compare(batch, g, oracle.sample(batch, want_probs=False, nthreads=8))
    assert rep.ok(), rep


def test_noalloc_new_offset_each_call(lib):
    import torch
    d, s = lib
    batch = workloads.random_batch(73, 40, 50000, "bf16")
    stream = torch.cuda.current_stream().cuda_stream
    dd = dev.to_device(batch, want_probs=False)
    for off in (11, 12):
        args = dev.sample_args(s, batch, dd, philox_offset=off)
        s.sample_args(args)
        torch.cuda.synchronize()
        ref = dd["out_tokens"].cpu().numpy().copy()
        dd["out_tokens"].fill_(-7)
        assert _noalloc(args, stream) == d.SAMPLER_OK
        torch.cuda.synchronize()
        np.testing.assert_array_equal(dd["out_tokens"].cpu().numpy(), ref)


def test_noalloc_rejections(lib):
    import torch
    d, s = lib
    stream = torch.cuda.current_stream().cuda_stream
    big = workloads.random_batch(74, d.SAMPLER_NOALLOC_MAX_ROWS + 1, 1000, "f32")
    dd = dev.to_device(big, want_probs=False)
    assert _noalloc(dev.sample_args(s, big, dd), stream) == d._binding.SAMPLER_ERR_TOO_LARGE
    small = workloads.random_batch(75, 4, 1000, "f32")
    dd = dev.to_device(small, want_probs=True)
    assert _noalloc(dev.sample_args(s, small, dd), stream) == d._binding.SAMPLER_ERR_UNSUPPORTED
    pen = workloads.random_batch(76, 4, 1000, "f32", penalties=True)
    dd = dev.to_device(pen, want_probs=False)
    assert _noalloc(dev.sample_args(s, pen, dd), stream) == d._binding.SAMPLER_ERR_UNSUPPORTED
    # a vocabulary above 262144 is refused before anything is read
    dd = dev.to_device(small, want_probs=False)
    wide = dev.sample_args(s, small, dd)
    wide.vocab = wide.row_stride = 262145
    assert _noalloc(wide, stream) == d._binding.SAMPLER_ERR_TOO_LARGE
    empty = workloads.random_batch(78, 0, 100, "f32")
    dd = dev.to_device(empty, want_probs=False)
    assert _noalloc(dev.sample_args(s, empty, dd), stream) == d.SAMPLER_OK
