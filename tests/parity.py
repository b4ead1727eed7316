"""Element-by-element comparison of the CUDA sampler against the CPU oracle.

Acceptance rules:
* status codes: identical;
* greedy rows and rows with a top-k cut: the token is identical;
* sampled rows: the token is identical unless the oracle marks the row as
  sitting within 1e-6 of a decision (top-2 Gumbel scores, the top-p boundary
  or the min-p threshold); such rows are counted and reported;
* probs / logprobs (fp32): |gpu - oracle| <= 1e-6 + 1e-5 * |oracle|, and the
  kept set (probs > 0, logprobs > -inf) identical outside ambiguous rows.
"""
from __future__ import annotations

import numpy as np

ATOL = 1e-6
RTOL = 1e-5
TIE_TOL = 1e-6


class ParityReport:
    def __init__(self):
        self.rows = 0
        self.ambiguous = 0
        self.token_mismatch_ambiguous = 0
        self.messages = []

    def fail(self, msg):
        self.messages.append(msg)

    def ok(self):
        return not self.messages

    def __repr__(self):
        return (f"rows={self.rows} ambiguous={self.ambiguous} "
                f"ambiguous_mismatch={self.token_mismatch_ambiguous} errors={self.messages[:5]}")


def compare(batch, gpu, ora, rows=None, check_probs=True) -> ParityReport:
    """gpu: results for all rows of `batch`; ora: oracle results for `rows` (or all)."""
    rep = ParityReport()
    idx = np.arange(batch.n_rows) if rows is None else np.asarray(rows)
    amb = ora.ambiguous(TIE_TOL)
    for j, r in enumerate(idx):
        rep.rows += 1
        gs, os_ = int(gpu.status[r]), int(ora.status[j])
        if gs != os_:
            rep.fail(f"row {r}: status gpu={gs} oracle={os_}")
            continue
        if amb[j]:
            rep.ambiguous += 1
        gt, ot = int(gpu.tokens[r]), int(ora.tokens[j])
        if gt != ot:
            if amb[j]:
                rep.token_mismatch_ambiguous += 1
            else:
                rep.fail(f"row {r}: token gpu={gt} oracle={ot} (T={batch.temperature[r]}, "
                         f"diag={ora.diag[j].tolist()})")
        if check_probs and gpu.probs is not None and ora.probs is not None:
            gp, op = gpu.probs[r], ora.probs[j]
            gl, ol = gpu.logprobs[r], ora.logprobs[j]
            if os_ != 0:
                if not (np.isnan(gp).all() and np.isnan(gl).all()):
                    rep.fail(f"row {r}: error row outputs are not NaN")
                continue
            kept_g, kept_o = gp > 0, op > 0
            if not np.array_equal(kept_g, kept_o) or not np.array_equal(gl > -np.inf, ol > -np.inf):
                if not amb[j]:
                    diff = np.nonzero(kept_g != kept_o)[0][:5]
                    rep.fail(f"row {r}: kept sets differ at {diff.tolist()} "
                             f"(gpu {kept_g.sum()} oracle {kept_o.sum()})")
                continue
            bad = np.abs(gp.astype(np.float64) - op) > ATOL + RTOL * np.abs(op)
            if bad.any():
                k = int(np.argmax(bad))
                rep.fail(f"row {r}: probs differ at {k}: {gp[k]} vs {op[k]} ({int(bad.sum())} bad)")
            fin = ol > -np.inf
            badl = np.abs(gl[fin].astype(np.float64) - ol[fin]) > ATOL + RTOL * np.abs(ol[fin])
            if badl.any():
                k = np.nonzero(fin)[0][int(np.argmax(badl))]
                rep.fail(f"row {r}: logprobs differ at {k}: {gl[k]} vs {ol[k]} ({int(badl.sum())} bad)")
    return rep
