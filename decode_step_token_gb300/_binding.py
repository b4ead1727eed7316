"""ctypes binding of libsampler.so, with the C ABI's names (include/sampler.h).

Argument marshalling only: every step of the sampler runs in the CUDA library.
The library must have been built (``decode_step_token_gb300.build``); loading
fails loudly otherwise.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB

SAMPLER_DTYPE_F32 = 0
SAMPLER_DTYPE_BF16 = 1

SAMPLER_OK = 0
SAMPLER_ERR_NULL_ARG = -1
SAMPLER_ERR_BAD_SHAPE = -2
SAMPLER_ERR_TOO_LARGE = -3
SAMPLER_ERR_BAD_DTYPE = -4
SAMPLER_ERR_CUDA = -5
SAMPLER_ERR_NO_DEVICE = -6
SAMPLER_ERR_NO_STAGING = -7
SAMPLER_ERR_UNSUPPORTED = -8

SAMPLER_ROW_OK = 0
SAMPLER_ROW_NONFINITE = 1
SAMPLER_ROW_ALL_NEG_INF = 2
SAMPLER_ROW_BAD_PARAM = 3
SAMPLER_ROW_BAD_HISTORY = 4
SAMPLER_ROW_TIMEOUT = 5

SAMPLER_CREATE_HOST_STAGING = 1
SAMPLER_CREATE_ROW_KERNEL = 2
SAMPLER_CREATE_SHORT_WAITS = 4

EXPORTED = ("sampler_create", "sampler_sample", "sampler_sample_host", "sampler_destroy",
            "sampler_status_string", "sampler_abi_version", "sampler_get_stat",
            "sampler_sample_noalloc", "sampler_sample_ex", "sampler_lm_head_sample", "sampler_lm_head")
SAMPLER_STAT_EXACT_ROWS = 0
SAMPLER_STAT_LM_HEAD_TIMEOUTS = 1
SAMPLER_LM_HEAD_MAX_ROWS = 256
SAMPLER_NOALLOC_MAX_ROWS = 64
SAMPLER_MAX_TOP_N = 16
SAMPLER_MAX_BIAS = 64
SAMPLER_MAX_STOP = 16


class sampler_config_t(ctypes.Structure):
    _fields_ = [
        ("device", ctypes.c_int),
        ("max_rows", ctypes.c_int64),
        ("max_vocab", ctypes.c_int64),
        ("max_history", ctypes.c_int64),
        ("flags", ctypes.c_uint32),
    ]


_P = ctypes.c_void_p


class sampler_args_t(ctypes.Structure):
    _fields_ = [
        ("logits", _P),
        ("dtype", ctypes.c_int32),
        ("n_rows", ctypes.c_int64),
        ("vocab", ctypes.c_int64),
        ("row_stride", ctypes.c_int64),
        ("n_logit_rows", ctypes.c_int64),
        ("logit_row", _P),
        ("temperature", _P),
        ("top_k", _P),
        ("top_p", _P),
        ("min_p", _P),
        ("presence_penalty", _P),
        ("frequency_penalty", _P),
        ("repetition_penalty", _P),
        ("seed", _P),
        ("has_seed", _P),
        ("stream_id", _P),
        ("hist_offsets", _P),
        ("hist_ids", _P),
        ("global_seed", ctypes.c_uint64),
        ("philox_offset", ctypes.c_uint64),
        ("philox_offset_dev", _P),
        ("out_tokens", _P),
        ("out_probs", _P),
        ("out_logprobs", _P),
        ("out_status", _P),
    ]


class sampler_ext_t(ctypes.Structure):
    _fields_ = [
        ("top_n", ctypes.c_int32),
        ("unscaled", ctypes.c_int32),
        ("out_token_logprob", _P),
        ("out_top_ids", _P),
        ("out_top_logprobs", _P),
        ("vocab_mask", _P),
        ("mask_stride", ctypes.c_int64),
        ("bias_offsets", _P),
        ("bias_ids", _P),
        ("bias_values", _P),
        ("min_tokens_left", _P),
        ("stop_offsets", _P),
        ("stop_ids", _P),
        ("sanitize_nan", ctypes.c_int32),
    ]


class sampler_lm_head_t(ctypes.Structure):
    _fields_ = [
        ("hidden", _P),
        ("weight", _P),
        ("hidden_dim", ctypes.c_int64),
        ("hidden_stride", ctypes.c_int64),
        ("weight_stride", ctypes.c_int64),
    ]


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB):
    """Load libsampler.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with decode_step_token_gb300.build.build_library()")
            lib = ctypes.CDLL(path)
            lib.sampler_create.argtypes = [ctypes.POINTER(_P), ctypes.POINTER(sampler_config_t)]
            lib.sampler_create.restype = ctypes.c_int
            lib.sampler_sample.argtypes = [_P, ctypes.POINTER(sampler_args_t), _P]
            lib.sampler_sample.restype = ctypes.c_int
            lib.sampler_sample_host.argtypes = [_P, ctypes.POINTER(sampler_args_t), _P]
            lib.sampler_sample_host.restype = ctypes.c_int
            lib.sampler_destroy.argtypes = [_P]
            lib.sampler_destroy.restype = None
            lib.sampler_status_string.argtypes = [ctypes.c_int]
            lib.sampler_status_string.restype = ctypes.c_char_p
            lib.sampler_get_stat.argtypes = [_P, ctypes.c_int, ctypes.POINTER(ctypes.c_uint64),
                                             ctypes.c_int]
            lib.sampler_get_stat.restype = ctypes.c_int
            lib.sampler_sample_noalloc.argtypes = [ctypes.POINTER(sampler_args_t), _P]
            lib.sampler_sample_noalloc.restype = ctypes.c_int
            lib.sampler_sample_ex.argtypes = [_P, ctypes.POINTER(sampler_args_t), ctypes.POINTER(sampler_ext_t), _P]
            lib.sampler_sample_ex.restype = ctypes.c_int
            lib.sampler_lm_head_sample.argtypes = [_P, ctypes.POINTER(sampler_lm_head_t), ctypes.POINTER(sampler_args_t),
                                                   ctypes.POINTER(sampler_ext_t), _P]
            lib.sampler_lm_head_sample.restype = ctypes.c_int
            lib.sampler_lm_head.argtypes = [_P, ctypes.POINTER(sampler_lm_head_t), _P, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_int64, _P]
            lib.sampler_lm_head.restype = ctypes.c_int
            lib.sampler_abi_version.argtypes = []
            lib.sampler_abi_version.restype = ctypes.c_uint32
            _lib = lib
    return _lib


def sampler_create(cfg: sampler_config_t):
    """Returns (code, handle)."""
    h = _P()
    rc = load_library().sampler_create(ctypes.byref(h), ctypes.byref(cfg))
    return rc, h


def sampler_sample(h, args: sampler_args_t, stream: int) -> int:
    return load_library().sampler_sample(h, ctypes.byref(args), _P(stream))


def sampler_sample_host(h, args: sampler_args_t, stream: int) -> int:
    return load_library().sampler_sample_host(h, ctypes.byref(args), _P(stream))


def sampler_sample_ex(h, args: sampler_args_t, ext, stream: int) -> int:
    """ext: a sampler_ext_t or None."""
    return load_library().sampler_sample_ex(h, ctypes.byref(args), ctypes.byref(ext) if ext is not None else None,
                                            _P(stream))


def sampler_lm_head_sample(h, lm, args: sampler_args_t, ext, stream: int) -> int:
    return load_library().sampler_lm_head_sample(h, ctypes.byref(lm), ctypes.byref(args),
                                                 ctypes.byref(ext) if ext is not None else None, _P(stream))


def sampler_lm_head(h, lm, logits: int, logits_stride: int, rows: int, vocab: int, stream: int) -> int:
    return load_library().sampler_lm_head(h, ctypes.byref(lm), _P(logits), logits_stride, rows, vocab,
                                          _P(stream))


def sampler_sample_noalloc(args: sampler_args_t, stream: int) -> int:
    return load_library().sampler_sample_noalloc(ctypes.byref(args), _P(stream))


def sampler_destroy(h) -> None:
    load_library().sampler_destroy(h)


def sampler_status_string(code: int) -> str:
    return load_library().sampler_status_string(code).decode()


def sampler_abi_version() -> int:
    return int(load_library().sampler_abi_version())


def sampler_get_stat(h, which: int, reset: bool = False):
    """Returns (code, value)."""
    v = ctypes.c_uint64(0)
    rc = load_library().sampler_get_stat(h, which, ctypes.byref(v), 1 if reset else 0)
    return rc, int(v.value)
