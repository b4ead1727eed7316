"""Seeded synthetic inputs for the per-decode-step token sampler.

This module only draws inputs: logits, per-row parameters and prior-token
histories. It holds none of the sampler's arithmetic, so both the CUDA path and
the CPU oracle can take their inputs from it.

The five named workloads stand in for the LM-head outputs the pages measured
(no real logits, weights or datasets are used):

* ``tiny``      N=4, V=1024 fp32 logits ~ 2*N(0,1); rows 0-2 at T=1.0 (Gumbel-max
                path), row 3 greedy (T=0); no truncation or penalties.
* ``mixed``     N=64, V=128000 bf16 logits ~ 2*N(0,1) with +12 at one random token
                per row; a seeded shuffle of 32 rows T=0.8 plain, 16 rows top_p=0.9 +
                top_k=50 (T=1.0), 16 greedy; token ids only.
* ``latency``   N in {1, 32}, V=151936 bf16 logits 2.5*N(0,1) - 1.1*ln(v+1) (a
                Zipf(1.1)-shaped bias over the token index); every row T=0.7,
                top_k=20, top_p=0.8, min_p=0.
* ``penalties`` N=128, V=128000 fp32 logits ~ 2*N(0,1); per row 0..4096 prior ids
                drawn Zipf(1.2) over V; presence 0.5, frequency 0.3, repetition 1.1,
                min_p 0.05, T=1.0; fp32 probs and logprobs returned.
* ``ablation_*`` the per-family ablation at N=64, V=128000 bf16 (the mixed
                logits, every row T=1.0): plain, then + top_k=50 and top_p=0.9,
                then + min_p=0.05, then + presence / frequency / repetition
                penalties over Zipf(1.2) histories.
* ``forks``     256 base rows x V=256000 bf16 logits ~ 2*Student-t(3); per base row
                T ~ U[0,1.5] (10% exactly 0), top_k in {-1,20,50,1000}, top_p ~
                U[0.5,1], min_p in {0,0.05}, 25% seeded with a u64 seed; each base row
                sampled by 4 output rows (N=1024) with their own Philox streams.

bf16 values are drawn in fp32 and rounded to nearest-even, so the stored bits
are the ground truth for both sides.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

__all__ = [
    "SamplerBatch",
    "to_bf16_bits",
    "bf16_bits_to_f32",
    "tiny",
    "mixed",
    "latency",
    "penalties",
    "forks",
    "random_batch",
    "vocab_mask",
    "logit_bias",
    "ablation",
    "ABLATION_STAGES",
    "min_tokens",
    "lm_head",
    "WORKLOADS",
    "make",
]


@dataclass
class SamplerBatch:
    """One sampling call's inputs, as host numpy arrays.

    ``logits`` is ``[n_logit_rows, row_stride]``: uint16 bf16 bit patterns when
    ``dtype == "bf16"``, float32 when ``dtype == "f32"``. Per-row arrays have
    ``n_rows`` entries; ``None`` takes the library default.
    """

    name: str
    logits: np.ndarray
    dtype: str
    vocab: int
    n_rows: int
    temperature: np.ndarray
    top_k: Optional[np.ndarray] = None
    top_p: Optional[np.ndarray] = None
    min_p: Optional[np.ndarray] = None
    presence: Optional[np.ndarray] = None
    frequency: Optional[np.ndarray] = None
    repetition: Optional[np.ndarray] = None
    seed: Optional[np.ndarray] = None
    has_seed: Optional[np.ndarray] = None
    stream_id: Optional[np.ndarray] = None
    logit_row: Optional[np.ndarray] = None
    hist_offsets: Optional[np.ndarray] = None
    hist_ids: Optional[np.ndarray] = None
    global_seed: int = 0
    philox_offset: int = 0
    want_probs: bool = False
    vocab_mask: Optional[np.ndarray] = None  # [n_rows, ceil(vocab / 32)] uint32; bit set = allowed
    bias_offsets: Optional[np.ndarray] = None  # [n_rows + 1] int32: logit_bias entries of row r are
    bias_ids: Optional[np.ndarray] = None      # bias_ids / bias_values[bias_offsets[r] .. [r + 1])
    bias_values: Optional[np.ndarray] = None
    min_tokens_left: Optional[np.ndarray] = None  # [n_rows] int32: > 0 bans the row's stop tokens
    stop_offsets: Optional[np.ndarray] = None     # [n_rows + 1] int32 CSR over stop_ids
    stop_ids: Optional[np.ndarray] = None
    sanitize_nan: bool = False                    # NaN logits read as -inf (else status 1)
    notes: dict = field(default_factory=dict)

    @property
    def row_stride(self) -> int:
        return int(self.logits.shape[1])

    @property
    def n_logit_rows(self) -> int:
        return int(self.logits.shape[0])

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def logits_f32(self) -> np.ndarray:
        """The stored logits widened to float32 (exact for bf16)."""
        if self.dtype == "bf16":
            return bf16_bits_to_f32(self.logits)
        return self.logits

    def with_(self, **kw) -> "SamplerBatch":
        return replace(self, **kw)

    def unique_logit_bytes(self) -> int:
        """Bytes of logits the step must read at least once."""
        rows = self.n_logit_rows if self.logit_row is None else len(np.unique(self.logit_row))
        return rows * self.vocab * self.elem_bytes

    def history_bytes(self) -> int:
        if self.hist_offsets is None:
            return 0
        return int(self.hist_offsets.nbytes + self.hist_ids.nbytes)

    def param_bytes(self) -> int:
        n = 0
        for a in (self.temperature, self.top_k, self.top_p, self.min_p, self.presence,
                  self.frequency, self.repetition, self.seed, self.has_seed,
                  self.stream_id, self.logit_row):
            if a is not None:
                n += int(a.nbytes)
        return n


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return ((b + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def tiny(seed: int = 1) -> SamplerBatch:
    rng = np.random.Generator(np.random.PCG64(seed))
    n, v = 4, 1024
    logits = _f32(rng.standard_normal((n, v), dtype=np.float32) * 2.0)
    t = _f32([1.0, 1.0, 1.0, 0.0])
    return SamplerBatch("tiny", logits, "f32", v, n, t, global_seed=0, philox_offset=0)


def mixed(seed: int = 2, n: int = 64, v: int = 128000) -> SamplerBatch:
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((n, v), dtype=np.float32) * np.float32(2.0)
    spike = rng.integers(0, v, size=n)
    x[np.arange(n), spike] += np.float32(12.0)
    kinds = np.array([0] * (n // 2) + [1] * (n // 4) + [2] * (n - n // 2 - n // 4))
    rng.shuffle(kinds)
    t = np.where(kinds == 0, 0.8, np.where(kinds == 1, 1.0, 0.0))
    k = np.where(kinds == 1, 50, -1)
    p = np.where(kinds == 1, 0.9, 1.0)
    return SamplerBatch("mixed", to_bf16_bits(x), "bf16", v, n, _f32(t),
                        top_k=k.astype(np.int32), top_p=_f32(p),
                        notes={"kinds": kinds, "spike": spike})


def latency(n: int = 32, seed: int = 3, v: int = 151936) -> SamplerBatch:
    rng = np.random.Generator(np.random.PCG64(seed))
    bias = (-1.1 * np.log(np.arange(v, dtype=np.float64) + 1.0)).astype(np.float32)
    x = rng.standard_normal((n, v), dtype=np.float32) * np.float32(2.5) + bias[None, :]
    return SamplerBatch(f"latency{n}", to_bf16_bits(x), "bf16", v, n,
                        _f32(np.full(n, 0.7)), top_k=np.full(n, 20, np.int32),
                        top_p=_f32(np.full(n, 0.8)), min_p=_f32(np.zeros(n)))


def _zipf_ids(rng, count: int, a: float, v: int) -> np.ndarray:
    ids = rng.zipf(a, size=count) - 1
    bad = ids >= v
    while bad.any():
        ids[bad] = rng.zipf(a, size=int(bad.sum())) - 1
        bad = ids >= v
    return ids.astype(np.int32)


def penalties(seed: int = 4, n: int = 128, v: int = 128000, max_hist: int = 4096) -> SamplerBatch:
    rng = np.random.Generator(np.random.PCG64(seed))
    logits = _f32(rng.standard_normal((n, v), dtype=np.float32) * 2.0)
    lens = rng.integers(0, max_hist + 1, size=n)
    offs = np.zeros(n + 1, np.int32)
    offs[1:] = np.cumsum(lens)
    ids = _zipf_ids(rng, int(offs[-1]), 1.2, v)
    ones = np.ones(n)
    return SamplerBatch("penalties", logits, "f32", v, n, _f32(ones),
                        min_p=_f32(0.05 * ones), presence=_f32(0.5 * ones),
                        frequency=_f32(0.3 * ones), repetition=_f32(1.1 * ones),
                        hist_offsets=offs, hist_ids=ids, want_probs=True)


def forks(seed: int = 5, base_rows: int = 256, n_forks: int = 4, v: int = 256000) -> SamplerBatch:
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_t(3, size=(base_rows, v)).astype(np.float32) * np.float32(2.0)
    t = rng.uniform(0.0, 1.5, size=base_rows)
    t[rng.random(base_rows) < 0.1] = 0.0
    k = rng.choice(np.array([-1, 20, 50, 1000]), size=base_rows)
    p = rng.uniform(0.5, 1.0, size=base_rows)
    mp = rng.choice(np.array([0.0, 0.05]), size=base_rows)
    seeded = rng.random(base_rows) < 0.25
    seeds = rng.integers(0, 2**63, size=base_rows, dtype=np.int64).astype(np.uint64)
    rep = lambda a: np.repeat(a, n_forks)
    n = base_rows * n_forks
    return SamplerBatch(
        "forks", to_bf16_bits(x), "bf16", v, n, _f32(rep(t)),
        top_k=rep(k).astype(np.int32), top_p=_f32(rep(p)), min_p=_f32(rep(mp)),
        seed=rep(seeds), has_seed=rep(seeded).astype(np.uint8),
        stream_id=np.arange(n, dtype=np.uint32),
        logit_row=np.repeat(np.arange(base_rows, dtype=np.int32), n_forks),
        notes={"base_rows": base_rows, "n_forks": n_forks})


def random_batch(seed: int, n: int, v: int, dtype: str = "f32", *, stride_pad: int = 0,
                 scale: float = 2.0, penalties: bool = False, want_probs: bool = False,
                 max_hist: int = 64, mix: str = "all", ties: bool = False) -> SamplerBatch:
    """A small batch with every per-row parameter family drawn at random.

    ``mix``: "all" draws greedy / plain / top-k / top-p / min-p / seeded rows;
    "plain" only temperature rows; "topk", "topp", "minp" force that stage on.
    ``ties`` quantises the logits to a coarse grid so that equal values abound.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((n, v + stride_pad), dtype=np.float32) * np.float32(scale)
    if ties:
        x = np.round(x * 2.0).astype(np.float32) / np.float32(2.0)
    t = rng.uniform(0.3, 1.5, size=n)
    k = np.full(n, -1, np.int64)
    p = np.ones(n)
    mp = np.zeros(n)
    if mix == "all":
        kind = rng.integers(0, 6, size=n)
        t[kind == 0] = 0.0
        k[kind == 2] = rng.integers(1, max(2, min(v, 80)), size=int((kind == 2).sum()))
        p[kind == 3] = rng.uniform(0.3, 0.99, size=int((kind == 3).sum()))
        mp[kind == 4] = rng.uniform(0.001, 0.3, size=int((kind == 4).sum()))
        both = kind == 5
        k[both] = rng.integers(1, v + 5, size=int(both.sum()))
        p[both] = rng.uniform(0.5, 1.0, size=int(both.sum()))
    elif mix == "topk":
        k[:] = rng.integers(1, v + 2, size=n)
    elif mix == "topp":
        p[:] = rng.uniform(0.05, 0.999, size=n)
    elif mix == "minp":
        mp[:] = rng.uniform(0.0005, 0.5, size=n)
    seeded = rng.random(n) < 0.3
    seeds = rng.integers(0, 2**63, size=n, dtype=np.int64).astype(np.uint64)
    if dtype == "bf16":
        logits = to_bf16_bits(x)
    else:
        logits = _f32(x)
    b = SamplerBatch(f"random{seed}", logits, dtype, v, n, _f32(t),
                     top_k=k.astype(np.int32), top_p=_f32(p), min_p=_f32(mp),
                     seed=seeds, has_seed=seeded.astype(np.uint8),
                     global_seed=int(rng.integers(0, 2**63)),
                     philox_offset=int(rng.integers(0, 2**40)), want_probs=want_probs)
    if penalties:
        lens = rng.integers(0, max_hist + 1, size=n)
        offs = np.zeros(n + 1, np.int32)
        offs[1:] = np.cumsum(lens)
        ids = _zipf_ids(rng, int(offs[-1]), 1.2, v)
        b = b.with_(presence=_f32(rng.uniform(-0.5, 1.0, size=n)),
                    frequency=_f32(rng.uniform(-0.2, 0.5, size=n)),
                    repetition=_f32(rng.uniform(0.8, 1.5, size=n)),
                    hist_offsets=offs, hist_ids=ids)
    return b


def vocab_mask(seed: int, n: int, v: int, allowed: float = 0.1, full_rows: int = 1) -> np.ndarray:
    """A grammar-style vocabulary bitmask [n, ceil(v / 32)] (bit v & 31 of word
    v >> 5 set = token v allowed): runs of allowed tokens covering about
    `allowed` of the vocabulary, plus scattered single tokens; the first
    `full_rows` rows allow everything."""
    rng = np.random.Generator(np.random.PCG64(seed))
    words = (v + 31) // 32
    out = np.zeros((n, words), np.uint32)
    for r in range(n):
        ok = np.zeros(words * 32, bool)
        if r < full_rows:
            ok[:v] = True
        else:
            target = max(1, int(allowed * v))
            while ok[:v].sum() < target:
                start = int(rng.integers(0, v))
                ok[start:min(v, start + int(rng.integers(1, 200)))] = True
                ok[rng.integers(0, v, size=8)] = True
        bits = ok.reshape(words, 32).astype(np.uint64) << np.arange(32, dtype=np.uint64)
        out[r] = bits.sum(axis=1).astype(np.uint32)
    return out


def logit_bias(seed: int, n: int, v: int, max_per_row: int = 64, scale: float = 5.0):
    """Per-row logit_bias lists in CSR form (offsets, ids, values): 0..max_per_row
    entries per row, ids uniform over the vocabulary with a few repeats, values
    ~ scale * N(0,1) with some -inf (banned) and some large (forced) entries."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = rng.integers(0, max_per_row + 1, size=n)
    offs = np.zeros(n + 1, np.int32)
    offs[1:] = np.cumsum(lens)
    ids = rng.integers(0, v, size=int(offs[-1])).astype(np.int32)
    rep_at = rng.random(ids.size) < 0.05
    ids[1:][rep_at[1:]] = ids[:-1][rep_at[1:]]  # repeated ids add up
    vals = (rng.standard_normal(ids.size) * scale).astype(np.float32)
    vals[rng.random(ids.size) < 0.05] = -np.inf
    vals[rng.random(ids.size) < 0.02] = np.float32(50.0)
    return offs, ids, vals


def min_tokens(seed: int, n: int, v: int, max_stops: int = 4, owe: float = 0.5):
    """Per-row min_tokens state (tokens still owed, stop-token lists in CSR
    form): 1..max_stops stop tokens per row (the last ids of the vocabulary,
    where chat models keep their end-of-turn tokens, plus a random one), and a
    fraction ``owe`` of the rows still owing 1..16 tokens (the others 0)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = rng.integers(1, max_stops + 1, size=n)
    offs = np.zeros(n + 1, np.int32)
    offs[1:] = np.cumsum(lens)
    ids = np.empty(int(offs[-1]), np.int32)
    for r in range(n):
        L = int(lens[r])
        ids[offs[r]:offs[r + 1]] = np.concatenate([v - 1 - np.arange(L - 1), rng.integers(0, v, 1)])
    left = np.where(rng.random(n) < owe, rng.integers(1, 17, size=n), 0).astype(np.int32)
    return left, offs, ids


ABLATION_STAGES = ("plain", "topkp", "minp", "penalties")


def ablation(stage: str, seed: int = 2, n: int = 64, v: int = 128000, max_hist: int = 4096) -> SamplerBatch:
    """The per-family ablation at N=64, V=128000 bf16 (the mixed workload's logits):
    every row T=1.0; ``topkp`` adds top_k=50 and top_p=0.9; ``minp`` also
    min_p=0.05; ``penalties`` also presence 0.5, frequency 0.3, repetition 1.1
    over a 0..4096-token Zipf(1.2) history per row."""
    if stage not in ABLATION_STAGES:
        raise ValueError(stage)
    base = mixed(seed, n, v)
    ones = np.ones(n)
    kw = {}
    upto = ABLATION_STAGES.index(stage)
    if upto >= 1:
        kw.update(top_k=np.full(n, 50, np.int32), top_p=_f32(0.9 * ones))
    if upto >= 2:
        kw.update(min_p=_f32(0.05 * ones))
    if upto >= 3:
        rng = np.random.Generator(np.random.PCG64(seed + 100))
        lens = rng.integers(0, max_hist + 1, size=n)
        offs = np.zeros(n + 1, np.int32)
        offs[1:] = np.cumsum(lens)
        kw.update(presence=_f32(0.5 * ones), frequency=_f32(0.3 * ones), repetition=_f32(1.1 * ones),
                  hist_offsets=offs, hist_ids=_zipf_ids(rng, int(offs[-1]), 1.2, v))
    return SamplerBatch(f"ablation_{stage}", base.logits, "bf16", v, n, _f32(ones), notes={"stage": stage},
                        **kw)


WORKLOADS = {
    "tiny": tiny,
    "mixed": mixed,
    "latency1": lambda: latency(1),
    "latency32": lambda: latency(32),
    "penalties": penalties,
    "forks": forks,
    "ablation_plain": lambda: ablation("plain"),
    "ablation_topkp": lambda: ablation("topkp"),
    "ablation_minp": lambda: ablation("minp"),
    "ablation_penalties": lambda: ablation("penalties"),
}


def make(name: str) -> SamplerBatch:
    return WORKLOADS[name]()


def lm_head(seed: int = 6, n: int = 64, v: int = 128000, k: int = 4096, *, weight: bool = True):
    """An LM-head decode step: hidden states [n, k] ~ N(0, 1) and an LM-head
    weight [v, k] ~ N(0, (2 / sqrt(k))^2), both rounded to bf16 (bits), so that
    the logits are ~ N(0, 4) like the mixed batch's; and the sampler parameters
    of the mixed batch (32 rows T=0.8, 16 rows top_k=50 top_p=0.9, 16 greedy at
    n = 64) with a placeholder for the logits the LM head writes.
    ``weight=False`` skips the weight (the caller draws it on the device)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    hidden = to_bf16_bits(rng.standard_normal((n, k), dtype=np.float32))
    w = None
    if weight:
        w = to_bf16_bits(rng.standard_normal((v, k), dtype=np.float32) * np.float32(2.0 / np.sqrt(k)))
    kinds = np.array([0] * (n // 2) + [1] * (n // 4) + [2] * (n - n // 2 - n // 4))
    rng.shuffle(kinds)
    t = np.where(kinds == 0, 0.8, np.where(kinds == 1, 1.0, 0.0))
    b = SamplerBatch("lm_head", np.zeros((n, v), np.uint16), "bf16", v, n, _f32(t),
                     top_k=np.where(kinds == 1, 50, -1).astype(np.int32),
                     top_p=_f32(np.where(kinds == 1, 0.9, 1.0)), notes={"kinds": kinds})
    return hidden, w, b
