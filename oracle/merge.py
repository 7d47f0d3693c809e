"""LSE merge of partial attention results, fp64 — TEST INFRASTRUCTURE ONLY.

When the keys of a row are split into disjoint sets s = 1..n, each set gives a
normalised partial output O_s = sum_{j in s} p_j v_j / sum_{j in s} p_j and a
log-sum-exp LSE_s = ln sum_{j in s} exp(score_j).  The whole-row result
follows from the running-max / normaliser correction of "Attention softmax
fusion" (section "The tile loop") and "Kernel Fusion and the Memory Wall"
(section "FlashAttention: avoid the full score matrix") applied once per set:

    M = max_s LSE_s,  w_s = exp(LSE_s - M),  L = sum_s w_s,
    O = sum_s w_s O_s / L,  LSE = M + ln L.

Sets without a valid key carry LSE_s = -inf and weight 0; a row where every
set is empty gives O = 0 and LSE = -inf.
"""

from __future__ import annotations

import numpy as np


def lse_merge(o_parts, lse_parts):
    """``o_parts [n, rows, D]``, ``lse_parts [n, rows]`` -> ``(O [rows, D], LSE [rows])`` (float64)."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = np.max(lse_parts, axis=0)
    rows, D = o_parts.shape[1], o_parts.shape[2]
    out = np.zeros((rows, D), dtype=np.float64)
    lse = np.full((rows,), -np.inf, dtype=np.float64)
    has = np.isfinite(m)
    if np.any(has):
        w = np.exp(lse_parts[:, has] - m[has][None, :])  # empty sets: exp(-inf) = 0
        total = np.sum(w, axis=0)
        out[has] = np.einsum("sr,srd->rd", w, o_parts[:, has]) / total[:, None]
        lse[has] = m[has] + np.log(total)
    return out, lse
