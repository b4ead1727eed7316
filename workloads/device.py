"""Move a ``SamplerBatch`` to the GPU and run it through the library's Python binding.

Marshalling only (numpy -> torch device tensors -> ``Sampler.sample``); no
sampler arithmetic lives here.
"""
from __future__ import annotations

from typing import Optional

import numpy as np


def to_device(batch, device="cuda:0", want_probs: Optional[bool] = None, copies: int = 1,
              logits_offset_elems: int = 0):
    """Device tensors for `batch`; `copies` distinct logits buffers (for rotating past L2);
    `logits_offset_elems` shifts the logits start (to exercise unaligned rows)."""
    import torch

    want = batch.want_probs if want_probs is None else want_probs
    dev = torch.device(device)

    def t(a, dt=None):
        if a is None:
            return None
        arr = np.ascontiguousarray(a)
        if arr.dtype == np.uint64:
            arr = arr.view(np.int64)
        x = torch.from_numpy(arr)
        return x.to(dev) if dt is None else x.to(dev).view(dt)

    if batch.dtype == "bf16":
        host = torch.from_numpy(np.ascontiguousarray(batch.logits).view(np.int16)).view(torch.bfloat16)
    else:
        host = torch.from_numpy(np.ascontiguousarray(batch.logits))
    logits = []
    for _ in range(copies):
        if logits_offset_elems:
            flat = torch.empty(host.numel() + logits_offset_elems, dtype=host.dtype, device=dev)
            view = flat[logits_offset_elems:].view(host.shape)
            view.copy_(host)
            logits.append(view)
        else:
            logits.append(host.to(dev))
    N, V = batch.n_rows, batch.vocab
    d = {
        "logits": logits,
        "temperature": t(batch.temperature),
        "top_k": t(batch.top_k),
        "top_p": t(batch.top_p),
        "min_p": t(batch.min_p),
        "presence_penalty": t(batch.presence),
        "frequency_penalty": t(batch.frequency),
        "repetition_penalty": t(batch.repetition),
        "seed": t(batch.seed),
        "has_seed": t(batch.has_seed),
        "stream_id": t(batch.stream_id.view(np.int32) if batch.stream_id is not None else None),
        "logit_row": t(batch.logit_row),
        "hist_offsets": t(batch.hist_offsets),
        "hist_ids": t(batch.hist_ids),
        "out_tokens": torch.full((N,), -7, dtype=torch.int32, device=dev),
        "out_status": torch.full((N,), -7, dtype=torch.int32, device=dev),
        "out_probs": torch.empty((N, V), dtype=torch.float32, device=dev) if want else None,
        "out_logprobs": torch.empty((N, V), dtype=torch.float32, device=dev) if want else None,
        "vocab_mask": t(batch.vocab_mask.view(np.int32)) if batch.vocab_mask is not None else None,
        "bias_offsets": t(batch.bias_offsets),
        "bias_ids": t(batch.bias_ids),
        "bias_values": t(batch.bias_values),
        "min_tokens_left": t(batch.min_tokens_left),
        "stop_offsets": t(batch.stop_offsets),
        "stop_ids": t(batch.stop_ids),
        "sanitize_nan": bool(batch.sanitize_nan),
    }
    return d


def sample_args(sampler, batch, d, copy_index: int = 0, philox_offset: Optional[int] = None,
                philox_offset_dev=None):
    """The ctypes argument block for one call on device buffers `d`."""
    return sampler.make_args(
        logits=d["logits"][copy_index], vocab=batch.vocab, n_rows=batch.n_rows,
        row_stride=batch.row_stride, n_logit_rows=batch.n_logit_rows,
        temperature=d["temperature"], top_k=d["top_k"], top_p=d["top_p"], min_p=d["min_p"],
        presence_penalty=d["presence_penalty"], frequency_penalty=d["frequency_penalty"],
        repetition_penalty=d["repetition_penalty"], seed=d["seed"], has_seed=d["has_seed"],
        stream_id=d["stream_id"], logit_row=d["logit_row"], hist_offsets=d["hist_offsets"],
        hist_ids=d["hist_ids"], global_seed=batch.global_seed,
        philox_offset=batch.philox_offset if philox_offset is None else philox_offset,
        philox_offset_dev=philox_offset_dev,
        out_tokens=d["out_tokens"], out_probs=d["out_probs"], out_logprobs=d["out_logprobs"],
        out_status=d["out_status"])


def ext_kw(d):
    """The mask, logit_bias, min_tokens and NaN-sanitising arguments of
    sample_ex_args for device buffers `d`."""
    return dict(vocab_mask=d["vocab_mask"], bias_offsets=d["bias_offsets"], bias_ids=d["bias_ids"],
                bias_values=d["bias_values"], min_tokens_left=d["min_tokens_left"],
                stop_offsets=d["stop_offsets"], stop_ids=d["stop_ids"], sanitize_nan=d["sanitize_nan"])


def wants_ext(d) -> bool:
    """Whether the batch carries an extension only sampler_sample_ex takes."""
    return (d["vocab_mask"] is not None or d["bias_offsets"] is not None or d["stop_offsets"] is not None
            or d["sanitize_nan"])


class GpuResult:
    def __init__(self, tokens, status, probs, logprobs):
        self.tokens, self.status, self.probs, self.logprobs = tokens, status, probs, logprobs


def run(sampler, batch, want_probs: Optional[bool] = None, device="cuda:0",
        logits_offset_elems: int = 0) -> GpuResult:
    """One synchronous call; results back on the host as numpy."""
    import torch

    d = to_device(batch, device, want_probs, logits_offset_elems=logits_offset_elems)
    if wants_ext(d):
        sampler.sample_ex_args(sample_args(sampler, batch, d), **ext_kw(d))
    else:
        sampler.sample_args(sample_args(sampler, batch, d))
    torch.cuda.synchronize()
    get = lambda x: None if x is None else x.cpu().numpy()
    return GpuResult(get(d["out_tokens"]), get(d["out_status"]), get(d["out_probs"]),
                     get(d["out_logprobs"]))


class GpuLogprobResult:
    def __init__(self, tokens, status, token_logprob, top_ids, top_logprobs):
        self.tokens, self.status = tokens, status
        self.token_logprob, self.top_ids, self.top_logprobs = token_logprob, top_ids, top_logprobs


def run_logprobs(sampler, batch, top_n: int, unscaled: bool = False, device="cuda:0",
                 token_logprob: bool = True) -> GpuLogprobResult:
    """One synchronous sampler_sample_ex call with logprob outputs (and the batch's
    vocabulary mask, if any); results back on the host."""
    import torch

    d = to_device(batch, device, False)
    N = batch.n_rows
    tok_lp = torch.full((N,), 7.0, dtype=torch.float32, device=device) if token_logprob else None
    ids = torch.full((N, max(top_n, 1)), -7, dtype=torch.int32, device=device)
    lps = torch.full((N, max(top_n, 1)), 7.0, dtype=torch.float32, device=device)
    sampler.sample_ex_args(sample_args(sampler, batch, d), top_n=top_n, unscaled=unscaled,
                           out_token_logprob=tok_lp, out_top_ids=ids if top_n else None,
                           out_top_logprobs=lps if top_n else None, **ext_kw(d))
    torch.cuda.synchronize()
    return GpuLogprobResult(d["out_tokens"].cpu().numpy(), d["out_status"].cpu().numpy(),
                            tok_lp.cpu().numpy() if tok_lp is not None else None,
                            ids.cpu().numpy()[:, :top_n], lps.cpu().numpy()[:, :top_n])


class GpuLmHeadResult:
    def __init__(self, logits, tokens, status):
        self.logits, self.tokens, self.status = logits, tokens, status
        self.probs = self.logprobs = None


def bf16_device(bits, device="cuda:0", stride: Optional[int] = None):
    """Host bf16 bits [rows, k] -> a device int16 tensor [rows, stride] (k <= stride;
    the padding holds NaN bits, which the product must never read)."""
    import torch

    rows, k = bits.shape
    stride = k if stride is None else stride
    t = torch.full((rows, stride), 0x7FC0, dtype=torch.int16, device=device)
    t[:, :k] = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)
    return t


def run_lm_head(sampler, hidden, weight, batch, device="cuda:0", hidden_stride: Optional[int] = None,
                weight_stride: Optional[int] = None, sentinel: int = 0x7F81, **ext) -> GpuLmHeadResult:
    """One synchronous sampler_lm_head_sample call. `hidden` / `weight`: host bf16
    bits or device int16 tensors; batch.logits (its shape gives the row stride) is
    filled with `sentinel` bits on the device and receives the logits. Results
    (the logits buffer as bf16 bits, tokens, status) back on the host."""
    import torch

    K = int(hidden.shape[1])
    h = hidden if isinstance(hidden, torch.Tensor) else bf16_device(hidden, device, hidden_stride)
    w = weight if isinstance(weight, torch.Tensor) else bf16_device(weight, device, weight_stride)
    d = to_device(batch, device, False)
    d["logits"][0].view(torch.int16).fill_(sentinel - 0x10000 if sentinel >= 0x8000 else sentinel)
    args = sample_args(sampler, batch, d)
    sampler.lm_head_sample_args(args, h, w, hidden_dim=K, hidden_stride=int(h.stride(0)),
                                weight_stride=int(w.stride(0)), **ext)
    torch.cuda.synchronize()
    logits = d["logits"][0].view(torch.int16).cpu().numpy().view(np.uint16)
    return GpuLmHeadResult(logits, d["out_tokens"].cpu().numpy(), d["out_status"].cpu().numpy())
