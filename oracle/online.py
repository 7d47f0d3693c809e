"""Tiled online-softmax recurrence, fp64 — TEST INFRASTRUCTURE ONLY.

This is the recurrence that "Attention softmax fusion" (section "The tile
loop") and "Kernel Fusion and the Memory Wall" (section "FlashAttention: avoid
the full score matrix") describe for one query: walk the keys in tiles; keep a
running maximum ``m``, a normaliser ``l`` and an unnormalised numerator ``a``;
when a tile has maximum ``m_t`` take ``m' = max(m, m_t)``, multiply ``l`` and
``a`` by ``alpha = exp(m - m')``, then add the tile's ``exp(s - m')`` terms;
after the last tile return ``a / l``.

The equations on the pages are garbled in extraction; this restates them from
the surviving prose (rescale by ``exp(m - m')``, return ``a / l``).  One guard
is added that the prose asks for ("Attention softmax fusion", section "Things
that break": a fully masked tile has maximum -inf and must not poison the
running max with NaN): while ``m`` is still -inf the correction factor is
taken as 0 instead of ``exp(-inf - (-inf))``.

It is not used to produce any expected value for the CUDA path; the tests use
it to pin the materialised oracle (``attention.attention_ref``) against the
pages' own tiled formulation.
"""

from __future__ import annotations

import numpy as np


def online_softmax_attention(scores, v, tile: int):
    """Online softmax-weighted sum of ``v`` rows.

    ``scores [n]`` (already scaled; -inf marks a masked key), ``v [n, Dv]``,
    ``tile`` = keys per tile.  Returns ``(result [Dv], m, l)`` where
    ``result = a / l`` (zeros and ``l = 0`` if every score is -inf)."""
    scores = np.asarray(scores, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    m = -np.inf
    l = 0.0
    a = np.zeros(v.shape[1], dtype=np.float64)
    for start in range(0, scores.shape[0], tile):
        s_t = scores[start:start + tile]
        m_new = max(m, float(np.max(s_t)))
        if m_new == -np.inf:
            continue  # nothing valid seen yet: all accumulators stay zero
        alpha = 0.0 if m == -np.inf else float(np.exp(m - m_new))
        p_t = np.exp(s_t - m_new)
        l = alpha * l + float(np.sum(p_t))
        a = alpha * a + p_t @ v[start:start + tile]
        m = m_new
    if l == 0.0:
        return np.zeros_like(a), m, l
    return a / l, m, l
