"""CPU oracle for the per-decode-step token sampler.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import this package. The product path
(the CUDA library and its Python binding) never does, and shares no code with
it.

The arithmetic lives in ``sampler_oracle.c`` (plain C, double precision after
the fp32 penalties, full sort per row, explicit cumulative sums, its own
Philox4x32-10). This module compiles it on first use with gcc and marshals
numpy arrays through ctypes. ``batch_paths`` restates the pages' batch-wide
path predicates, which the per-row design does not use. ``lm_head_logits`` is
the LM head's matrix product written out in double precision.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sampler_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

GCC_FLAGS = ["-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-std=c11"]

STATUS_OK, STATUS_NONFINITE, STATUS_ALL_NEG_INF, STATUS_BAD_PARAM, STATUS_BAD_HISTORY = 0, 1, 2, 3, 4


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source when missing or stale."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.oracle_philox4x32_10.argtypes = [P, P, P]
            lib.oracle_philox4x32_10.restype = None
            lib.oracle_philox4x64_10.argtypes = [P, P, P]
            lib.oracle_philox4x64_10.restype = None
            lib.oracle_noise_word.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64,
                                              ctypes.c_int64]
            lib.oracle_noise_word.restype = ctypes.c_uint32
            lib.oracle_uniform.argtypes = [ctypes.c_uint32]
            lib.oracle_uniform.restype = ctypes.c_double
            lib.oracle_exp1.argtypes = [ctypes.c_uint32]
            lib.oracle_exp1.restype = ctypes.c_double
            lib.oracle_sample.argtypes = (
                [P, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, P]
                + [P] * 10 + [P, P, ctypes.c_uint64, ctypes.c_uint64, P, ctypes.c_int64, P, P, P]
                + [P, P, P, ctypes.c_int] + [P, ctypes.c_int64] + [P] * 5 + [ctypes.c_int])
            lib.oracle_sample.restype = ctypes.c_int
            lib.oracle_penalized_logits.argtypes = [
                P, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_float, ctypes.c_float, ctypes.c_float, P, P, P, ctypes.c_int64,
                P, P, P, P, P, P, ctypes.c_int, ctypes.c_int64, P]
            lib.oracle_penalized_logits.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def philox4x32_10(ctr: Sequence[int], key: Sequence[int]) -> np.ndarray:
    lib = _load()
    c = np.asarray(ctr, np.uint32)
    k = np.asarray(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib.oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def philox4x64_10(ctr: Sequence[int], key: Sequence[int]) -> np.ndarray:
    lib = _load()
    c = np.asarray(ctr, np.uint64)
    k = np.asarray(key, np.uint64)
    out = np.zeros(4, np.uint64)
    lib.oracle_philox4x64_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def noise_word(key: int, stream: int, offset: int, v: int) -> int:
    return int(_load().oracle_noise_word(key, stream, offset, v))


def uniform(word: int) -> float:
    return float(_load().oracle_uniform(word))


def exp1(word: int) -> float:
    return float(_load().oracle_exp1(word))


def penalized_logits(batch, row: int):
    """(status, fp32 penalised logits) of output row `row` of a SamplerBatch."""
    lib = _load()
    logits = np.ascontiguousarray(batch.logits)
    lr = row if batch.logit_row is None else int(batch.logit_row[row])
    pick = lambda a, d: d if a is None else float(a[row])
    x = np.zeros(batch.vocab, np.float32)
    hoff = _arr(batch.hist_offsets, np.int32)
    hids = _arr(batch.hist_ids, np.int32)
    mask = _arr(batch.vocab_mask, np.uint32)
    boff = _arr(batch.bias_offsets, np.int32)
    bids = _arr(batch.bias_ids, np.int32)
    bval = _arr(batch.bias_values, np.float32)
    mtl = _arr(batch.min_tokens_left, np.int32)
    soff = _arr(batch.stop_offsets, np.int32)
    sids = _arr(batch.stop_ids, np.int32)
    rc = lib.oracle_penalized_logits(
        _ptr(logits), 1 if batch.dtype == "bf16" else 0, batch.vocab, batch.row_stride, lr,
        pick(batch.presence, 0.0), pick(batch.frequency, 0.0), pick(batch.repetition, 1.0),
        _ptr(hoff), _ptr(hids), _ptr(mask), 0 if mask is None else mask.shape[1],
        _ptr(boff), _ptr(bids), _ptr(bval), _ptr(mtl), _ptr(soff), _ptr(sids),
        1 if batch.sanitize_nan else 0, row, _ptr(x))
    if rc < 0:
        raise RuntimeError("oracle_penalized_logits failed")
    return rc, x


class OracleResult:
    """tokens, status, diag[:, 0..3] = (Gumbel top-2 gap, top-p margin, min-p margin,
    kept count), and probs / logprobs when requested."""

    def __init__(self, tokens, status, diag, probs, logprobs):
        self.tokens = tokens
        self.status = status
        self.diag = diag
        self.probs = probs
        self.logprobs = logprobs

    @property
    def gumbel_gap(self):
        return self.diag[:, 0]

    @property
    def topp_margin(self):
        return self.diag[:, 1]

    @property
    def minp_margin(self):
        return self.diag[:, 2]

    @property
    def kept(self):
        return self.diag[:, 3]

    def gumbel_tie(self, tol: float = 1e-6) -> np.ndarray:
        """Rows whose two best Gumbel scores lie within `tol` of each other: the
        sampled token is then one of two correct answers (greedy rows never are)."""
        return self.gumbel_gap < tol

    def topp_boundary(self, tol: float = 1e-6) -> np.ndarray:
        """Rows whose top-p cut has a prefix mass within `tol` of p."""
        return self.topp_margin < tol

    def minp_boundary(self, tol: float = 1e-6) -> np.ndarray:
        """Rows with a kept-set token whose min-p ratio lies within `tol` of ln(min_p)."""
        return self.minp_margin < tol

    def boundary(self, tol: float = 1e-6) -> np.ndarray:
        """Rows whose kept set sits within `tol` of a top-p or min-p cut."""
        return self.topp_boundary(tol) | self.minp_boundary(tol)

    def ambiguous(self, tol: float = 1e-6) -> np.ndarray:
        """Rows that have any of the near-decisions above (for counting)."""
        return self.gumbel_tie(tol) | self.boundary(tol)


def _arr(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def sample(batch, rows: Optional[Sequence[int]] = None, want_probs: Optional[bool] = None,
           nthreads: int = 1) -> OracleResult:
    """Run the oracle on a ``workloads.SamplerBatch`` (all rows, or ``rows``)."""
    lib = _load()
    want = batch.want_probs if want_probs is None else want_probs
    logits = np.ascontiguousarray(batch.logits)
    dtype = 1 if batch.dtype == "bf16" else 0
    if dtype == 1:
        assert logits.dtype == np.uint16
    else:
        assert logits.dtype == np.float32
    rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n_out = batch.n_rows if rows_arr is None else len(rows_arr)
    V = batch.vocab
    tokens = np.zeros(n_out, np.int32)
    status = np.zeros(n_out, np.int32)
    diag = np.zeros((n_out, 4), np.float64)
    probs = np.zeros((n_out, V), np.float32) if want else None
    logprobs = np.zeros((n_out, V), np.float32) if want else None
    keep = [
        _arr(batch.logit_row, np.int32), _arr(batch.temperature, np.float32),
        _arr(batch.top_k, np.int32), _arr(batch.top_p, np.float32), _arr(batch.min_p, np.float32),
        _arr(batch.presence, np.float32), _arr(batch.frequency, np.float32),
        _arr(batch.repetition, np.float32), _arr(batch.seed, np.uint64),
        _arr(batch.has_seed, np.uint8), _arr(batch.stream_id, np.uint32),
        _arr(batch.hist_offsets, np.int32), _arr(batch.hist_ids, np.int32),
    ]
    (lr, t, k, p, mp, pres, freq, rep, seed, has_seed, sid, hoff, hids) = keep
    mask = _arr(batch.vocab_mask, np.uint32)
    boff = _arr(batch.bias_offsets, np.int32)
    bids = _arr(batch.bias_ids, np.int32)
    bval = _arr(batch.bias_values, np.float32)
    mtl = _arr(batch.min_tokens_left, np.int32)
    soff = _arr(batch.stop_offsets, np.int32)
    sids = _arr(batch.stop_ids, np.int32)
    rc = lib.oracle_sample(
        _ptr(logits), dtype, batch.n_rows, V, batch.row_stride, _ptr(lr),
        _ptr(t), _ptr(k), _ptr(p), _ptr(mp), _ptr(pres), _ptr(freq), _ptr(rep),
        _ptr(seed), _ptr(has_seed), _ptr(sid), _ptr(hoff), _ptr(hids),
        ctypes.c_uint64(batch.global_seed), ctypes.c_uint64(batch.philox_offset),
        _ptr(mask), 0 if mask is None else mask.shape[1],
        _ptr(boff), _ptr(bids), _ptr(bval), _ptr(mtl), _ptr(soff), _ptr(sids),
        1 if batch.sanitize_nan else 0,
        _ptr(rows_arr), n_out, _ptr(tokens), _ptr(status), _ptr(probs), _ptr(logprobs),
        _ptr(diag), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_sample failed ({rc})")
    return OracleResult(tokens, status, diag, probs, logprobs)


class LogprobOutputs:
    """Per-row logprob outputs without the [N, V] tensors: the sampled token's
    logprob, and the top_n tokens with theirs (ids -1 and logprob -inf past the
    tokens the distribution gives any mass; NaN / -1 on error rows)."""

    def __init__(self, token_logprob, top_ids, top_logprobs):
        self.token_logprob = token_logprob
        self.top_ids = top_ids
        self.top_logprobs = top_logprobs


def logprob_outputs(batch, result: OracleResult, top_n: int, unscaled: bool = False,
                    rows: Optional[Sequence[int]] = None) -> LogprobOutputs:
    """The logprobs a request gets back with its token (manual-sglang-101, "Logprobs
    are temperature-scaled"): by default those of the distribution the row was
    sampled from, log_softmax(x / T) over its kept set (T := 1 on greedy rows);
    ``unscaled`` asks for log_softmax(x) over the whole vocabulary instead (the
    page's original-logprob switch). x is the penalised fp32 row; the sums run in
    double. The kept set is the one ``sample(..., want_probs=True)`` returned
    (logprobs > -inf); ``result`` must come from such a call on the same rows.
    The top_n order is (logprob desc, index asc)."""
    idx = np.arange(batch.n_rows) if rows is None else np.asarray(rows)
    n_out = len(idx)
    tok = np.full(n_out, np.nan, np.float64)
    ids = np.full((n_out, top_n), -1, np.int32)
    lps = np.full((n_out, top_n), np.nan, np.float64)
    for j, r in enumerate(idx):
        if int(result.status[j]) != 0:
            continue
        _, x = penalized_logits(batch, int(r))
        x = x.astype(np.float64)
        if unscaled:
            keep = x > -np.inf
            T = 1.0
        else:
            keep = result.logprobs[j] > -np.inf
            T = float(np.float32(batch.temperature[r]))
            if T < 1e-5:
                T = 1.0
        y = np.where(keep, x / T, -np.inf)
        ymax = y[keep].max()
        lse = ymax + np.log(np.exp(y[keep] - ymax).sum())
        lp = np.where(keep, y - lse, -np.inf)
        tok[j] = lp[int(result.tokens[j])]
        order = sorted(np.nonzero(keep)[0].tolist(), key=lambda v: (-x[v], v))[:top_n]
        lps[j, :] = -np.inf
        for q, v in enumerate(order):
            ids[j, q] = v
            lps[j, q] = lp[v]
    return LogprobOutputs(tok, ids, lps)


# ---------------------------------------------------------------- LM head
def _bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (exact: bf16 is the top half of a float32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def lm_head_logits(hidden_bits: np.ndarray, weight_bits: np.ndarray, cols: Optional[np.ndarray] = None):
    """The LM head of the xbrilliance.ai note's decode step (section
    "解码一步里采样做什么": the logits are matmul(hidden_states, embedding.t())):
    logits[i, v] = sum_k hidden[i, k] * weight[v, k], from bf16 inputs, in
    float64 (every product of two bf16 values is exact in double; the sum's
    rounding is ~1e-16 relative). Also returns sum_k |hidden[i, k] * weight[v, k]|,
    the scale of the rounding error a lower-precision sum may make.
    ``cols``: only those vocabulary rows (the returned columns follow its order).
    """
    h = _bf16_to_f64(hidden_bits)
    w = _bf16_to_f64(weight_bits if cols is None else weight_bits[cols])
    return h @ w.T, np.abs(h) @ np.abs(w).T
