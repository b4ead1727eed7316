"""GB300-native per-decode-step token sampler.

The sampler itself is the CUDA library ``libsampler.so`` (C ABI in
``include/sampler.h``); this package is its thin Python binding. ``Sampler``
wraps a handle and takes torch tensors that already live on the GPU; PyTorch
provides device memory and streams only.
"""
from __future__ import annotations

import ctypes
from typing import Optional

from . import _binding as abi
from ._binding import (EXPORTED, SAMPLER_CREATE_HOST_STAGING, SAMPLER_CREATE_SHORT_WAITS, SAMPLER_DTYPE_BF16,
                       SAMPLER_DTYPE_F32, SAMPLER_MAX_BIAS, SAMPLER_MAX_STOP, SAMPLER_MAX_TOP_N,
                       SAMPLER_LM_HEAD_MAX_ROWS, SAMPLER_NOALLOC_MAX_ROWS, SAMPLER_OK,
                       SAMPLER_STAT_EXACT_ROWS, SAMPLER_STAT_LM_HEAD_TIMEOUTS, sampler_lm_head_t,
                       sampler_lm_head_sample, sampler_lm_head,
                       load_library, sampler_abi_version, sampler_args_t, sampler_config_t, sampler_create,
                       sampler_destroy, sampler_ext_t, sampler_sample, sampler_sample_host,
                       sampler_sample_ex, sampler_sample_noalloc, sampler_status_string,
                       sampler_get_stat)

__all__ = ["Sampler", "SamplerError", "load_library", "sampler_create", "sampler_sample",
           "sampler_sample_host", "sampler_sample_noalloc", "sampler_sample_ex", "sampler_destroy",
           "sampler_status_string", "SAMPLER_NOALLOC_MAX_ROWS", "SAMPLER_MAX_TOP_N", "SAMPLER_MAX_BIAS",
           "SAMPLER_MAX_STOP", "sampler_ext_t", "sampler_lm_head_t", "sampler_lm_head_sample", "sampler_lm_head",
           "SAMPLER_LM_HEAD_MAX_ROWS", "SAMPLER_STAT_EXACT_ROWS", "SAMPLER_STAT_LM_HEAD_TIMEOUTS",
           "sampler_abi_version", "sampler_args_t", "sampler_config_t", "EXPORTED"]


def _make_ext(top_n: int = 0, unscaled: bool = False, out_token_logprob=None, out_top_ids=None,
              out_top_logprobs=None, vocab_mask=None, mask_stride: Optional[int] = None, bias_offsets=None,
              bias_ids=None, bias_values=None, min_tokens_left=None, stop_offsets=None, stop_ids=None,
              sanitize_nan: bool = False) -> sampler_ext_t:
    if vocab_mask is not None and mask_stride is None:
        mask_stride = int(vocab_mask.shape[-1])
    return sampler_ext_t(int(top_n), 1 if unscaled else 0, _ptr(out_token_logprob), _ptr(out_top_ids),
                         _ptr(out_top_logprobs), _ptr(vocab_mask), int(mask_stride or 0),
                         _ptr(bias_offsets), _ptr(bias_ids), _ptr(bias_values),
                         _ptr(min_tokens_left), _ptr(stop_offsets), _ptr(stop_ids), 1 if sanitize_nan else 0)


class SamplerError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {sampler_status_string(code)} ({code})")
        self.code = code


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    return int(t)


class Sampler:
    """One libsampler handle on a CUDA device.

    ``sample`` takes device tensors: logits ``[rows, >= vocab]`` (bf16 or fp32, unit
    inner stride) and per-row parameter tensors, and writes the caller's output
    tensors. It enqueues on torch's current stream (or ``stream``) and returns
    without synchronising.
    """

    def __init__(self, max_rows: int, max_vocab: int, device: int = 0, max_history: int = 0,
                 host_staging: bool = False, short_waits: bool = False):
        flags = ((SAMPLER_CREATE_HOST_STAGING if host_staging else 0)
                 | (SAMPLER_CREATE_SHORT_WAITS if short_waits else 0))
        cfg = sampler_config_t(device, max_rows, max_vocab, max_history, flags)
        rc, h = sampler_create(cfg)
        if rc != SAMPLER_OK:
            raise SamplerError(rc, "sampler_create")
        self._h = h
        self.device = device
        self.max_rows = max_rows
        self.max_vocab = max_vocab

    def close(self):
        if getattr(self, "_h", None):
            sampler_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @staticmethod
    def make_args(*, logits, vocab=None, n_rows=None, temperature, dtype=None, top_k=None,
                  top_p=None, min_p=None, presence_penalty=None, frequency_penalty=None,
                  repetition_penalty=None, seed=None, has_seed=None, stream_id=None,
                  logit_row=None, hist_offsets=None, hist_ids=None, global_seed=0,
                  philox_offset=0, philox_offset_dev=None, out_tokens, out_probs=None,
                  out_logprobs=None, out_status=None, n_logit_rows=None,
                  row_stride=None) -> sampler_args_t:
        if dtype is None:
            import torch
            if logits.dtype == torch.bfloat16:
                dtype = SAMPLER_DTYPE_BF16
            elif logits.dtype == torch.float32:
                dtype = SAMPLER_DTYPE_F32
            else:
                raise TypeError(f"unsupported logits dtype {logits.dtype}")
        if row_stride is None:
            if logits.stride(-1) != 1:
                raise ValueError("logits rows must be contiguous")
            row_stride = logits.stride(0) if logits.dim() == 2 else logits.shape[-1]
        if vocab is None:
            vocab = logits.shape[-1]
        if n_rows is None:
            n_rows = temperature.shape[0]
        if n_logit_rows is None:
            n_logit_rows = logits.shape[0] if logits.dim() == 2 else 1
        return sampler_args_t(
            _ptr(logits), dtype, n_rows, vocab, row_stride, n_logit_rows, _ptr(logit_row),
            _ptr(temperature), _ptr(top_k), _ptr(top_p), _ptr(min_p), _ptr(presence_penalty),
            _ptr(frequency_penalty), _ptr(repetition_penalty), _ptr(seed), _ptr(has_seed),
            _ptr(stream_id), _ptr(hist_offsets), _ptr(hist_ids), global_seed, philox_offset,
            _ptr(philox_offset_dev), _ptr(out_tokens), _ptr(out_probs), _ptr(out_logprobs),
            _ptr(out_status))

    def sample_args(self, args: sampler_args_t, stream: Optional[int] = None) -> None:
        if stream is None:
            import torch
            stream = torch.cuda.current_stream(self.device).cuda_stream
        rc = sampler_sample(self._h, args, stream)
        if rc != SAMPLER_OK:
            raise SamplerError(rc, "sampler_sample")

    def sample(self, stream: Optional[int] = None, **kw) -> None:
        self.sample_args(self.make_args(**kw), stream)

    def sample_ex_args(self, args: sampler_args_t, top_n: int = 0, unscaled: bool = False,
                       out_token_logprob=None, out_top_ids=None, out_top_logprobs=None,
                       vocab_mask=None, mask_stride: Optional[int] = None,
                       bias_offsets=None, bias_ids=None, bias_values=None,
                       min_tokens_left=None, stop_offsets=None, stop_ids=None,
                       sanitize_nan: bool = False, stream: Optional[int] = None) -> None:
        """sampler_sample_ex: the step plus per-row logprob outputs (device tensors:
        out_token_logprob [N] fp32, out_top_ids / out_top_logprobs [N, top_n]
        int32 / fp32), a vocabulary bitmask (device [N, words] int32/uint32),
        logit_bias lists (device CSR: offsets [N + 1], ids, fp32 values), the
        min_tokens ban (device int32: tokens owed [N], stop-token CSR offsets
        [N + 1] and ids) and NaN sanitising."""
        ext = _make_ext(top_n, unscaled, out_token_logprob, out_top_ids, out_top_logprobs, vocab_mask,
                        mask_stride, bias_offsets, bias_ids, bias_values, min_tokens_left, stop_offsets,
                        stop_ids, sanitize_nan)
        rc = sampler_sample_ex(self._h, args, ext, self._stream(stream))
        if rc != SAMPLER_OK:
            raise SamplerError(rc, "sampler_sample_ex")

    def lm_head_sample_args(self, args: sampler_args_t, hidden, weight, hidden_dim: Optional[int] = None,
                            hidden_stride: Optional[int] = None, weight_stride: Optional[int] = None,
                            stream: Optional[int] = None, **ext_kw) -> None:
        """sampler_lm_head_sample: logits = hidden x weight^T (device bf16 tensors
        hidden [rows, K], weight [V, K]) written to args.logits, then the step on
        them; ext_kw as for sample_ex_args."""
        K = int(hidden_dim if hidden_dim is not None else hidden.shape[-1])
        lm = sampler_lm_head_t(_ptr(hidden), _ptr(weight), K,
                               int(hidden_stride if hidden_stride is not None else hidden.stride(0)),
                               int(weight_stride if weight_stride is not None else weight.stride(0)))
        ext = _make_ext(**ext_kw) if ext_kw else None
        rc = sampler_lm_head_sample(self._h, lm, args, ext, self._stream(stream))
        if rc != SAMPLER_OK:
            raise SamplerError(rc, "sampler_lm_head_sample")

    def lm_head(self, hidden, weight, logits, rows: Optional[int] = None, vocab: Optional[int] = None,
                hidden_dim: Optional[int] = None, hidden_stride: Optional[int] = None,
                weight_stride: Optional[int] = None, logits_stride: Optional[int] = None,
                stream: Optional[int] = None) -> None:
        """sampler_lm_head: logits = hidden x weight^T (device bf16 tensors hidden
        [rows, K], weight [V, K], logits [rows, stride])."""
        K = int(hidden_dim if hidden_dim is not None else hidden.shape[-1])
        lm = sampler_lm_head_t(_ptr(hidden), _ptr(weight), K,
                               int(hidden_stride if hidden_stride is not None else hidden.stride(0)),
                               int(weight_stride if weight_stride is not None else weight.stride(0)))
        rc = sampler_lm_head(self._h, lm, _ptr(logits),
                             int(logits_stride if logits_stride is not None else logits.stride(0)),
                             int(rows if rows is not None else hidden.shape[0]),
                             int(vocab if vocab is not None else weight.shape[0]), self._stream(stream))
        if rc != SAMPLER_OK:
            raise SamplerError(rc, "sampler_lm_head")

    def _stream(self, stream: Optional[int]) -> int:
        if stream is None:
            import torch
            stream = torch.cuda.current_stream(self.device).cuda_stream
        return stream

    def stat(self, which: int = 0, reset: bool = False) -> int:
        """A device diagnostic counter (synchronizes the device)."""
        rc, v = sampler_get_stat(self._h, which, reset)
        if rc != SAMPLER_OK:
            raise SamplerError(rc, "sampler_get_stat")
        return v

    def sample_host_args(self, args: sampler_args_t, stream: int = 0) -> None:
        rc = sampler_sample_host(self._h, args, stream)
        if rc != SAMPLER_OK:
            raise SamplerError(rc, "sampler_sample_host")
