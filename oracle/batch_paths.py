"""Batch-wide path predicates of the two serving systems the pages describe.

TEST INFRASTRUCTURE ONLY: the per-row CUDA sampler has no batch-wide flags. These
restatements exist so the tests can show what the batch flags would have done
and that the per-row design gives every row the same answer whatever its
neighbours ask for.

* SGLang v0.5.20 (dev.to claim check "SGLang's +75% sampler speedup skips Qwen3
  chat requests", section "One request with top_p takes the whole batch off the
  fast path"): a temperature below 1e-6 becomes top_k = 1 with T = 1; top_k = -1
  becomes 1 << 30. The batch is greedy when every request has top_k <= 1;
  otherwise it takes the Gumbel-max path only when no request asks for top_p,
  top_k or min_p (or the seeded path when the server runs deterministic
  inference); everything else is "filtered".
* vLLM 0.5.0 (xbrilliance.ai note, section "哪些参数会额外打开一趟全词表计算",
  which parameters open an extra full-vocab pass): one flag per stage family,
  raised for the whole batch by any request with top_p < 1 - eps or
  top_k != V; min_p > eps; |presence| >= eps, |frequency| >= eps or
  |repetition - 1| >= eps; eps = 1e-5.
* The per-step size of the fp32 probs + logprobs tensors (same note, section
  "解码一步里采样做什么"): 8 * N * V bytes.
"""
from __future__ import annotations

from typing import Iterable, Mapping

SGLANG_TOP_K_ALL = 1 << 30
SGLANG_EPS = 1e-6
VLLM_EPS = 1e-5


def sglang_normalized(req: Mapping) -> dict:
    """One request's (temperature, top_k, top_p, min_p) after SGLang's normalisation."""
    out = dict(req)
    if 0 <= out["temperature"] < SGLANG_EPS:
        out["temperature"], out["top_k"] = 1.0, 1
    if out["top_k"] == -1:
        out["top_k"] = SGLANG_TOP_K_ALL
    return out


def sglang_batch_path(reqs: Iterable[Mapping], deterministic: bool = False) -> str:
    """"greedy", "gumbel", "deterministic" or "filtered" for a batch of normalised requests."""
    reqs = list(reqs)
    if not reqs:
        raise ValueError("empty batch")
    if all(r["top_k"] <= 1 for r in reqs):
        return "greedy"
    filtered = any(r["top_p"] != 1.0 or r["top_k"] != SGLANG_TOP_K_ALL or r["min_p"] > 0
                   for r in reqs)
    if filtered:
        return "filtered"
    return "deterministic" if deterministic else "gumbel"


def vllm_batch_flags(reqs: Iterable[Mapping], vocab: int) -> dict:
    """The three batch-wide stage flags of vLLM 0.5.0's sampling metadata."""
    flags = {"do_top_p_top_k": False, "do_min_p": False, "do_penalties": False}
    for r in reqs:
        k = vocab if r.get("top_k", -1) == -1 else r["top_k"]
        if r.get("top_p", 1.0) < 1.0 - VLLM_EPS or k != vocab:
            flags["do_top_p_top_k"] = True
        if r.get("min_p", 0.0) > VLLM_EPS:
            flags["do_min_p"] = True
        if (abs(r.get("presence_penalty", 0.0)) >= VLLM_EPS
                or abs(r.get("frequency_penalty", 0.0)) >= VLLM_EPS
                or abs(r.get("repetition_penalty", 1.0) - 1.0) >= VLLM_EPS):
            flags["do_penalties"] = True
    return flags


def vllm_sampling_type(temperature: float, seed=None, beam: bool = False) -> str:
    """GREEDY / RANDOM / RANDOM_SEED / BEAM routing of one request."""
    if beam:
        return "BEAM"
    if temperature < VLLM_EPS:
        return "GREEDY"
    return "RANDOM_SEED" if seed is not None else "RANDOM"


def sampling_tensor_bytes(n_rows: int, vocab: int) -> int:
    """fp32 probs + logprobs of one step."""
    return 8 * n_rows * vocab
