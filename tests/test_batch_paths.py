"""The batch-wide predicates the per-row design replaces, pinned to the pages' tables."""
import os

import numpy as np

from oracle import batch_paths as bp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _lines(name):
    return [l.rstrip("\n") for l in open(os.path.join(GOLDEN, name))
            if l.strip() and not l.startswith("#")]


def test_sglang_batch_path_table():
    for line in _lines("sglang_batch_paths.txt"):
        det, reqs, expect = [f.strip() for f in line.split("|")]
        batch = []
        for r in reqs.split(";"):
            t, k, p, mp = r.split(",")
            batch.append(bp.sglang_normalized(
                {"temperature": float(t), "top_k": int(k), "top_p": float(p), "min_p": float(mp)}))
        assert bp.sglang_batch_path(batch, deterministic=det == "1") == expect, line


def test_sglang_greedy_request_is_top_k_one():
    r = bp.sglang_normalized({"temperature": 0.0, "top_k": -1, "top_p": 1.0, "min_p": 0.0})
    assert r["top_k"] == 1 and r["temperature"] == 1.0
    r = bp.sglang_normalized({"temperature": 0.5, "top_k": -1, "top_p": 1.0, "min_p": 0.0})
    assert r["top_k"] == bp.SGLANG_TOP_K_ALL


def test_vllm_flag_defaults_table():
    V = 128000
    base = {"temperature": 1.0, "top_p": 1.0, "top_k": -1, "min_p": 0.0,
            "presence_penalty": 0.0, "frequency_penalty": 0.0, "repetition_penalty": 1.0}
    # all-default requests raise nothing
    assert not any(bp.vllm_batch_flags([base] * 4, V).values())
    for line in _lines("vllm_flag_defaults.txt"):
        name, default, other, flag = line.split()
        req = dict(base)
        assert float(req[name]) == float(default)
        req[name] = float(other) if name != "top_k" else int(other)
        flags = bp.vllm_batch_flags([base, base, req], V)
        raised = {f for f, on in flags.items() if on}
        assert raised == (set() if flag == "none" else {flag}), line


def test_vllm_routing():
    assert bp.vllm_sampling_type(0.0) == "GREEDY"
    assert bp.vllm_sampling_type(0.9e-5) == "GREEDY"
    assert bp.vllm_sampling_type(1.1e-5) == "RANDOM"
    assert bp.vllm_sampling_type(0.7, seed=3) == "RANDOM_SEED"
    assert bp.vllm_sampling_type(0.7, beam=True) == "BEAM"


def test_sampling_tensor_bytes_at_vocab_128k_and_64_rows():
    # "about 65 MB" for V = 128k (128,000) at concurrency 64
    assert bp.sampling_tensor_bytes(64, 128000) == 65_536_000
    n = bp.sampling_tensor_bytes(64, 128000) / 1e6
    assert 64 < n < 66


def test_one_filtered_request_moves_the_whole_batch():
    plain = {"temperature": 0.8, "top_k": -1, "top_p": 1.0, "min_p": 0.0}
    nucleus = {"temperature": 1.0, "top_k": 50, "top_p": 0.9, "min_p": 0.0}
    batch = [bp.sglang_normalized(plain)] * 63 + [bp.sglang_normalized(nucleus)]
    assert bp.sglang_batch_path(batch) == "filtered"
    assert bp.sglang_batch_path(batch[:63]) == "gumbel"
