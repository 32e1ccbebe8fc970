"""Cut-off margins of a selection, measured on oracle chunk scores.

A kept-list comparison between two implementations is only meaningful when
no floating-point rounding can move the cut-off. For a prompt's chunk scores
(ranked by score descending, index ascending):

* rank gap: (s_j - s_{j+1}) / s_j at the boundary between the last ranked
  chunk kept (j) and the first one dropped (j + 1);
* mass crossing (mass mode only): how far the running sums on either side
  of the crossing chunk sit from theta = mass * total, relative to theta.
"""

import numpy as np

from oracle import specprefill_oracle as so

RANK_GAP = 1e-3        # relative score gap required at the cut-off
CROSSING_GAP = 1e-4    # relative distance of the running sums from theta


def prompt_margins(cs: np.ndarray, mode: str, keep_p: float, mass: float) -> dict:
    cs = np.asarray(cs, dtype=np.float64)
    nc = cs.shape[0]
    order = so.rank_order(cs)
    ranked = cs[order]
    if mode == "fixed":
        j = min(so.fixed_count(nc, keep_p), nc)
        cross = None
    else:
        sel = so.select_mass(cs, mass)
        j = int(sel.sum())
        theta = so.as_f32(mass) * float(np.sum(cs))
        cum_before = float(np.sum(ranked[:j - 1]))
        cum_at = float(np.sum(ranked[:j]))
        cross = min((theta - cum_before) / theta, (cum_at - theta) / theta) if j < nc else None
    gap = None if j >= nc else float((ranked[j - 1] - ranked[j]) / ranked[j - 1])
    return {"selected": j, "n_chunks": nc, "rank_gap": gap, "crossing": cross}


def margins_ok(m: dict) -> bool:
    if m["rank_gap"] is not None and not m["rank_gap"] >= RANK_GAP:
        return False
    if m["crossing"] is not None and not m["crossing"] >= CROSSING_GAP:
        return False
    return True
