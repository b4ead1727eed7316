"""Batch-wide path predicates of the two serving systems the pages describe.

TEST INFRASTRUCTURE ONLY: the per-row CUDA sampler has no batch-wide flags. These
restatements exist so the tests can show what the batch flags would have done
and that the per-row design gives every row the same answer whatever its
neighbours ask for. Both are written from the pages' prose and tables:

* SGLang v0.5.20 (dev.to claim check "SGLang's +75% sampler speedup skips Qwen3
  chat requests", section "One request with top_p takes the whole batch off the
  fast path"). After normalisation a temperature-0 request is a top_k = 1
  request, and top_k = -1 stands for the whole vocabulary (the value 1 << 30).
  The batch flags are "any request" predicates: top-p is needed when some
  top_p differs from 1.0, top-k when some top_k is not the whole vocabulary,
  min-p when some min_p is positive. A batch whose every request has
  top_k <= 1 takes the greedy path before the flags are looked at; a server
  started with deterministic inference takes the seeded path; otherwise any
  raised flag means the filtered path and none means the Gumbel-max fast path
  (the page's four-row table). SGLang's greedy threshold (1e-6) is the value
  the page prints.
* vLLM 0.5.0 (xbrilliance.ai note, section "哪些参数会额外打开一趟全词表计算",
  which parameters open an extra full-vocab pass). Its parameter table groups
  the parameters into three stage families, each with one batch flag; a flag
  is raised for the whole batch as soon as one request moves a parameter of
  its family off the default (top_k = -1 counts as the vocabulary size). The
  tolerance is the note's eps, 1e-5, the same value at which the routing of
  section "采样类型与选路" (sampling type and routing) calls a temperature greedy.
* The per-step size of the fp32 probs + logprobs tensors (same note, section
  "解码一步里采样做什么"): two fp32 tensors of N x V, 8 * N * V bytes.
"""
from __future__ import annotations

from typing import Iterable, Mapping

SGLANG_TOP_K_ALL = 1 << 30
SGLANG_EPS = 1e-6
VLLM_EPS = 1e-5


def sglang_normalized(req: Mapping) -> dict:
    """One request's (temperature, top_k, top_p, min_p) as the scheduler sees them:
    a temperature in [0, eps) becomes a top-1 request at temperature 1, and -1
    ("all tokens") becomes the whole-vocabulary constant."""
    greedy = 0.0 <= req["temperature"] < SGLANG_EPS
    top_k = 1 if greedy else req["top_k"]
    return {
        **req,
        "temperature": 1.0 if greedy else req["temperature"],
        "top_k": SGLANG_TOP_K_ALL if top_k == -1 else top_k,
    }


def _sglang_filters(req: Mapping) -> set:
    """The filter stages one normalised request asks for."""
    wanted = set()
    if req["top_k"] != SGLANG_TOP_K_ALL:
        wanted.add("top_k")
    if req["top_p"] != 1.0:
        wanted.add("top_p")
    if req["min_p"] > 0:
        wanted.add("min_p")
    return wanted


def sglang_batch_path(reqs: Iterable[Mapping], deterministic: bool = False) -> str:
    """"greedy", "gumbel", "deterministic" or "filtered" for a batch of normalised requests."""
    reqs = list(reqs)
    if not reqs:
        raise ValueError("empty batch")
    # (outcome, rule) in the order the page says they are checked
    rules = (
        ("greedy", lambda rs: all(r["top_k"] <= 1 for r in rs)),
        ("filtered", lambda rs: bool(set().union(*map(_sglang_filters, rs)))),
        ("deterministic", lambda rs: deterministic),
        ("gumbel", lambda rs: True),
    )
    return next(name for name, rule in rules if rule(reqs))


# vLLM: parameter -> (stage family flag, default value), from the note's table
VLLM_PARAMETERS = {
    "top_p": ("do_top_p_top_k", 1.0),
    "top_k": ("do_top_p_top_k", -1),
    "min_p": ("do_min_p", 0.0),
    "presence_penalty": ("do_penalties", 0.0),
    "frequency_penalty": ("do_penalties", 0.0),
    "repetition_penalty": ("do_penalties", 1.0),
}


def _vllm_off_default(name: str, value, vocab: int) -> bool:
    _, default = VLLM_PARAMETERS[name]
    if name == "top_k":  # -1 and the vocabulary size both mean "no cut"
        return (vocab if value == -1 else value) != vocab
    return abs(float(value) - float(default)) >= VLLM_EPS


def vllm_batch_flags(reqs: Iterable[Mapping], vocab: int) -> dict:
    """The three batch-wide stage flags of vLLM 0.5.0's sampling metadata."""
    flags = {flag: False for flag, _ in VLLM_PARAMETERS.values()}
    for req in reqs:
        for name, (flag, default) in VLLM_PARAMETERS.items():
            if _vllm_off_default(name, req.get(name, default), vocab):
                flags[flag] = True
    return flags


def vllm_sampling_type(temperature: float, seed=None, beam: bool = False) -> str:
    """GREEDY / RANDOM / RANDOM_SEED / BEAM routing of one request."""
    if beam:
        return "BEAM"
    if temperature < VLLM_EPS:
        return "GREEDY"
    return "RANDOM" if seed is None else "RANDOM_SEED"


def sampling_tensor_bytes(n_rows: int, vocab: int) -> int:
    """fp32 probs + logprobs of one step."""
    return 2 * 4 * n_rows * vocab
