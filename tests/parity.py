"""Element-by-element comparison of the CUDA sampler against the CPU oracle.

Acceptance rules (each kind of near-decision excuses only what it can change):
* status codes: identical, always;
* greedy rows: the token is identical, always (the argmax of the penalised
  logits has no tolerance; ties go to the lowest index on both sides);
* sampled rows: the token is identical unless the oracle's two best Gumbel
  scores lie within TIE_TOL (a Gumbel tie), or the row's kept set sits within
  TIE_TOL of its top-p or min-p cut (a boundary row), in which case the kept set
  itself may legitimately differ and the pick with it;
* kept sets (logprobs > -inf; probs are 0 outside): identical, always, for rows without a
  boundary -- in particular every top-k set. On a boundary row the two sets
  must be nested and differ only in tokens that sit at the tail of the kept
  order (no kept token of either side may rank below a token they disagree on);
* probs / logprobs (fp32): |gpu - oracle| <= ATOL + RTOL * |oracle| on rows
  whose kept sets agree; error rows are NaN on both sides.

Rows flagged by either kind of near-decision are counted (``gumbel_ties``,
``boundary_rows``); ``excused`` counts the rows whose token or kept set
actually differed and was accepted for that reason.
"""
from __future__ import annotations

import numpy as np

ATOL = 1e-6
RTOL = 1e-5
TIE_TOL = 1e-6
GREEDY_T = np.float32(1e-5)


class ParityReport:
    def __init__(self):
        self.rows = 0
        self.gumbel_ties = 0
        self.boundary_rows = 0
        self.excused = 0
        self.messages = []

    @property
    def ambiguous(self):
        """Rows with a Gumbel tie or a kept-set boundary (either may excuse a difference)."""
        return self.gumbel_ties + self.boundary_rows

    def fail(self, msg):
        self.messages.append(msg)

    def ok(self):
        return not self.messages

    def __repr__(self):
        return (f"rows={self.rows} gumbel_ties={self.gumbel_ties} boundary_rows={self.boundary_rows} "
                f"excused={self.excused} errors={self.messages[:5]}")


def _tail_only(batch, row, kept_g, kept_o):
    """True when the two kept sets are nested and every token they disagree on
    ranks at or below every token both keep (the order is the penalised logit)."""
    import oracle

    only_g = kept_g & ~kept_o
    only_o = kept_o & ~kept_g
    if only_g.any() and only_o.any():
        return False
    both = kept_g & kept_o
    if not both.any():
        return False
    _, x = oracle.penalized_logits(batch, row)
    diff = only_g | only_o
    return float(x[diff].max()) <= float(x[both].min())


def compare(batch, gpu, ora, rows=None, check_probs=True) -> ParityReport:
    """gpu: results for all rows of `batch`; ora: oracle results for `rows` (or all)."""
    rep = ParityReport()
    idx = np.arange(batch.n_rows) if rows is None else np.asarray(rows)
    tie = ora.gumbel_tie(TIE_TOL)
    bnd = ora.boundary(TIE_TOL)
    for j, r in enumerate(idx):
        rep.rows += 1
        gs, os_ = int(gpu.status[r]), int(ora.status[j])
        if gs != os_:
            rep.fail(f"row {r}: status gpu={gs} oracle={os_}")
            continue
        greedy = bool(np.float32(batch.temperature[r]) < GREEDY_T)
        if os_ == 0 and not greedy and tie[j]:
            rep.gumbel_ties += 1
        if os_ == 0 and bnd[j]:
            rep.boundary_rows += 1
        gt, ot = int(gpu.tokens[r]), int(ora.tokens[j])
        excused = False
        if gt != ot:
            if os_ == 0 and not greedy and (tie[j] or bnd[j]):
                excused = True
            else:
                rep.fail(f"row {r}: token gpu={gt} oracle={ot} (T={batch.temperature[r]}, "
                         f"greedy={greedy}, diag={ora.diag[j].tolist()})")
        if check_probs and gpu.probs is not None and ora.probs is not None:
            gp, op = gpu.probs[r], ora.probs[j]
            gl, ol = gpu.logprobs[r], ora.logprobs[j]
            if os_ != 0:
                if not (np.isnan(gp).all() and np.isnan(gl).all()):
                    rep.fail(f"row {r}: error row outputs are not NaN")
                continue
            # the kept set is where logprobs are finite (a kept token's probability
            # may underflow to 0 in fp32); no token outside it has a probability
            kept_g, kept_o = gl > -np.inf, ol > -np.inf
            if (gp[~kept_g] != 0).any():
                rep.fail(f"row {r}: gpu probability outside its kept set")
                continue
            if not np.array_equal(kept_g, kept_o):
                if bnd[j] and _tail_only(batch, int(r), kept_g, kept_o):
                    excused = True
                    if not kept_g[gt]:
                        rep.fail(f"row {r}: gpu token {gt} is outside its own kept set")
                else:
                    diff = np.nonzero(kept_g != kept_o)[0][:5]
                    rep.fail(f"row {r}: kept sets differ at {diff.tolist()} "
                             f"(gpu {int(kept_g.sum())} oracle {int(kept_o.sum())}, "
                             f"boundary={bool(bnd[j])})")
                rep.excused += int(excused)
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
        rep.excused += int(excused)
    return rep
