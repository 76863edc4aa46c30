"""Comparison rules used by the parity tests (GPU against the oracle).

Bounds:
* layer output: relative L2 <= 1e-2 and cosine >= 0.9997 (the target bounds), plus
* the MoE sum y_shared + y_routed, which the residual would otherwise hide: relative L2
  <= MOE_REL, and the routed sum sum_j w_j y_j alone (so that the shared expert cannot hide
  a routed-expert error either): relative L2 <= MOE_REL, and
* top-k indices equal wherever the oracle's k-th / (k+1)-th probability gap exceeds 1e-4
  (near-ties are the known source of routing flips).
"""
from __future__ import annotations

import numpy as np

from tests.helpers import bf16_f64, cosine, rel_l2

OUT_REL, OUT_COS = 1e-2, 0.9997
MOE_REL = 1e-2
TIE_GAP = 1e-4


def near_tie_rows(probs: np.ndarray, k: int) -> np.ndarray:
    """Rows whose k-th and (k+1)-th largest probabilities are within TIE_GAP."""
    s = -np.sort(-probs, axis=1)
    if s.shape[1] <= k:
        return np.zeros(probs.shape[0], bool)
    return (s[:, k - 1] - s[:, k]) <= TIE_GAP


def topk_agree(gpu_idx, orc_idx, orc_probs, k, valid_rows) -> tuple[bool, np.ndarray]:
    """Same expert sets on every valid row that is not a near-tie.  Returns (ok, tie rows)."""
    ties = near_tie_rows(orc_probs, k)
    ok = True
    for r in np.nonzero(valid_rows)[0]:
        if ties[r]:
            continue
        if sorted(gpu_idx[r].tolist()) != sorted(orc_idx[r].tolist()):
            ok = False
    return ok, ties


def layer_metrics(out_gpu_bits, out_orc_bits, ys_gpu, ys_orc, yr_gpu, yr_orc, rows):
    """Metrics of one layer output: the bf16 output, the MoE sum ys + yr and the routed
    sum yr, each restricted to `rows` (a boolean mask of the non-pad rows)."""
    o_g, o_o = bf16_f64(out_gpu_bits)[rows], bf16_f64(out_orc_bits)[rows]
    s_g, s_o = np.asarray(ys_gpu, np.float64)[rows], np.asarray(ys_orc, np.float64)[rows]
    r_g, r_o = np.asarray(yr_gpu, np.float64)[rows], np.asarray(yr_orc, np.float64)[rows]
    return dict(out_rel=rel_l2(o_g, o_o), out_cos=cosine(o_g, o_o),
                moe_rel=rel_l2(s_g + r_g, s_o + r_o), routed_rel=rel_l2(r_g, r_o))


def layer_ok(m: dict) -> bool:
    return (m["out_rel"] <= OUT_REL and m["out_cos"] >= OUT_COS and m["moe_rel"] <= MOE_REL
            and m["routed_rel"] <= MOE_REL)
