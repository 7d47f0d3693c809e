"""Gradients of the exact attention, fp64 — TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline
use this module; the library never does.

The pages mention training ("Fused Multi-Head Attention": fused kernels also
make training with longer sequences more efficient) but give no backward
algorithm.  Plainest reading, used here: the gradients of the forward that
``attention.attention_ref`` defines, with respect to Q, K and V, for an
upstream gradient ``dO`` of the output (the LSE output is not
differentiated).  They are written out from the chain rule on the
materialised softmax of one head:

* ``P_ij = exp(s_ij - LSE_i)`` on valid keys, ``0`` elsewhere (a row without
  a valid key has ``P = 0``), with ``s_ij = scale * <q_i, k_j>``;
* ``dV = P^T dO``;
* ``dP = dO V^T``;
* ``dS_ij = P_ij (dP_ij - Delta_i)`` with ``Delta_i = sum_j P_ij dP_ij``
  (the softmax Jacobian applied to ``dP``; it equals ``sum_d dO_id O_id``);
* ``dQ = scale * dS K`` and ``dK = scale * dS^T Q``.

Delta is computed here as ``sum_j P_ij dP_ij``, straight from the Jacobian;
``<dO_i, O_i>`` is the same number, and the tests pin the two against each
other.  Rows are processed in blocks so that memory stays bounded.
"""

from __future__ import annotations

import numpy as np

from .attention import _as_f64


def _probs(q_rows, row_index, k, scale, causal, kv_len):
    """Exact softmax probabilities of the given query rows over all keys:
    ``P [n, Sk]`` (rows without a valid key are all zero)."""
    Sk = k.shape[0]
    s = (q_rows @ k.T) * np.float64(scale)
    lim = np.full((q_rows.shape[0],), min(max(int(kv_len), 0), Sk), dtype=np.int64)
    if causal:
        lim = np.minimum(lim, row_index.astype(np.int64) + 1)
    valid = np.arange(Sk)[None, :] < lim[:, None]
    sv = np.where(valid, s, -np.inf)
    has_key = lim > 0
    m = np.where(has_key, np.max(sv, axis=1, initial=-np.inf), 0.0)
    e = np.where(valid, np.exp(sv - m[:, None]), 0.0)
    tot = e.sum(axis=1)
    return np.where(has_key[:, None], e / np.where(has_key, tot, 1.0)[:, None], 0.0)


def attention_bwd_head(q, k, v, dout, scale: float, causal: bool = False, kv_len=None, block: int = 256):
    """Gradients for one head: ``q, dout [Sq, D]``, ``k, v [Sk, D]``.
    Returns ``(dQ [Sq, D], dK [Sk, D], dV [Sk, D])`` in float64."""
    q, k, v, dout = (_as_f64(x) for x in (q, k, v, dout))
    Sq, Sk = q.shape[0], k.shape[0]
    kvl = Sk if kv_len is None else kv_len
    dq = np.zeros_like(q)
    dk = np.zeros((Sk, q.shape[1]))
    dv = np.zeros((Sk, v.shape[1]))
    for r0 in range(0, Sq, block):
        rows = np.arange(r0, min(Sq, r0 + block))
        p = _probs(q[rows], rows, k, scale, causal, kvl)
        dv += p.T @ dout[rows]
        dp = dout[rows] @ v.T
        delta = np.sum(p * dp, axis=1)
        ds = p * (dp - delta[:, None])
        dq[rows] = np.float64(scale) * (ds @ k)
        dk += np.float64(scale) * (ds.T @ q[rows])
    return dq, dk, dv


def attention_bwd_ref(q, k, v, dout, scale: float, causal: bool = False, kv_lens=None):
    """Gradients of ``attention_ref``'s O for ``q [B,H,Sq,D]``, ``k, v
    [B,H,Sk,D]`` and ``dout [B,H,Sq,Dv]``.  Returns float64
    ``(dQ, dK, dV)`` shaped like ``q``, ``k`` and ``v``."""
    q, k, v, dout = (_as_f64(x) for x in (q, k, v, dout))
    B, H = q.shape[:2]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        kvl = None if kv_lens is None else int(kv_lens[b])
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = attention_bwd_head(q[b, h], k[b, h], v[b, h], dout[b, h], scale,
                                                              causal, kvl)
    return dq, dk, dv


def attention_bwd_sampled(q, k, v, dout, scale: float, q_rows, k_rows, causal: bool = False, kv_len=None,
                          block: int = 512):
    """One head's dQ for the query rows ``q_rows`` and dK, dV for the key rows
    ``k_rows``, without forming the full gradients (for large heads).
    Returns ``(dQ [len(q_rows), D], dK [len(k_rows), D], dV [len(k_rows), Dv])``."""
    q, k, v, dout = (_as_f64(x) for x in (q, k, v, dout))
    Sq, Sk = q.shape[0], k.shape[0]
    kvl = Sk if kv_len is None else kv_len
    q_rows = np.asarray(q_rows, dtype=np.int64)
    k_rows = np.asarray(k_rows, dtype=np.int64)
    p = _probs(q[q_rows], q_rows, k, scale, causal, kvl)
    dp = dout[q_rows] @ v.T
    ds = p * (dp - np.sum(p * dp, axis=1)[:, None])
    dq = np.float64(scale) * (ds @ k)
    dk = np.zeros((len(k_rows), q.shape[1]))
    dv = np.zeros((len(k_rows), v.shape[1]))
    for r0 in range(0, Sq, block):   # every query row contributes to the chosen keys
        rows = np.arange(r0, min(Sq, r0 + block))
        pf = _probs(q[rows], rows, k, scale, causal, kvl)
        dpf = dout[rows] @ v.T
        delta = np.sum(pf * dpf, axis=1)
        pk = pf[:, k_rows]
        dsk = pk * (dpf[:, k_rows] - delta[:, None])
        dv += pk.T @ dout[rows]
        dk += np.float64(scale) * (dsk.T @ q[rows])
    return dq, dk, dv
