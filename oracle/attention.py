"""Materialised fp64 attention oracle — TEST INFRASTRUCTURE ONLY.

Only tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline legs
may import this module.  It never calls into the CUDA library.

What it computes (one head ``(b, h)``, one query row ``i``):

* scores ``s_ij = scale * sum_d q_id k_jd`` — the dense attention
  ``softmax(Q K^T / sqrt(d)) V`` of "Kernel Fusion and the Memory Wall",
  section "FlashAttention: avoid the full score matrix", with the caller's
  ``scale`` in place of ``1/sqrt(d)``;
* the valid key set ``V_i = {j : j < kv_len[b] and (not causal or j <= i)}``
  (causal masking: "Kernel Fusion and the Memory Wall", the paragraph after
  "A small executable reference"; per-sequence key lengths for the ragged,
  padded batches of "Fused Multi-Head Attention", the continuous-batching
  item);
* the stable softmax over the WHOLE row ("Softmax needs a global row
  statistic": the denominator must include every valid key):
  ``M = max_{j in V_i} s_ij``, ``p_ij = exp(s_ij - M)``, ``L = sum_j p_ij``,
  ``O_i = sum_j p_ij v_j / L`` and ``LSE_i = M + ln L`` (natural log, over the
  scaled scores);
* a row with no valid key ("Attention softmax fusion", section "Things that
  break": a fully masked tile must not poison the result with NaN) has
  ``O_i = +0.0`` in every column and ``LSE_i = -inf``.

Readings where the pages are silent:

* causal alignment is top-left: key ``j`` is masked for query ``i`` when
  ``j > i``, for any ``Sq`` and ``Sk``;
* ``kv_lens`` entries are clamped to ``[0, Sk]``; ``None`` means ``Sk`` for
  every batch entry; causal and key-length masks combine by AND on validity;
* ``LSE`` uses the natural logarithm of the scaled scores.

Implementation: float64 NumPy; query rows are processed in blocks of
``block`` rows so that memory stays bounded at long sequence lengths; within a
block each score row is materialised in full over all ``Sk`` keys (no online
recurrence, no tiling over keys).
"""

from __future__ import annotations

import numpy as np


def _as_f64(x) -> np.ndarray:
    a = np.asarray(x)
    if a.dtype != np.float64:
        a = a.astype(np.float64)
    return a


def valid_key_count(i: int, Sk: int, causal: bool, kv_len: int) -> int:
    """Number of valid keys of query row ``i``: ``|{j : j < kv_len, (not causal or j <= i)}|``.

    ``kv_len`` is clamped to ``[0, Sk]`` first (reading of the pages' silence
    on out-of-range key lengths)."""
    lim = min(max(int(kv_len), 0), Sk)
    if causal:
        lim = min(lim, i + 1)
    return max(lim, 0)


def _head_rows(q_rows: np.ndarray, row_index: np.ndarray, k: np.ndarray, v: np.ndarray,
               scale: float, causal: bool, kv_len: int):
    """Exact attention for the query rows ``q_rows`` (their positions are
    ``row_index``) against all keys ``k`` / values ``v`` of one head.

    Returns ``(O [n, Dv] float64, LSE [n] float64)``."""
    Sk = k.shape[0]
    n = q_rows.shape[0]
    Dv = v.shape[1]
    out = np.zeros((n, Dv), dtype=np.float64)
    lse = np.full((n,), -np.inf, dtype=np.float64)
    if n == 0:
        return out, lse
    # s_ij = scale * <q_i, k_j>, one full row per query
    s = (q_rows @ k.T) * np.float64(scale)
    # validity: j < kv_len (clamped), and j <= i when causal
    lim = np.full((n,), min(max(int(kv_len), 0), Sk), dtype=np.int64)
    if causal:
        lim = np.minimum(lim, row_index.astype(np.int64) + 1)
    cols = np.arange(Sk, dtype=np.int64)
    valid = cols[None, :] < lim[:, None]
    has_key = lim > 0
    if not np.any(has_key):
        return out, lse
    s = np.where(valid, s, -np.inf)
    sv = s[has_key]
    # stable softmax over the whole row: subtract the row maximum of the valid scores
    m = np.max(sv, axis=1)
    p = np.exp(sv - m[:, None])  # masked entries: exp(-inf) = 0
    total = np.sum(p, axis=1)
    out[has_key] = (p @ v) / total[:, None]
    lse[has_key] = m + np.log(total)
    return out, lse


def attention_ref(q, k, v, scale: float, causal: bool = False, kv_lens=None, block: int = 256):
    """Exact attention forward over a padded batch.

    Arguments: ``q [B,H,Sq,D]``, ``k [B,H,Sk,D]``, ``v [B,H,Sk,Dv]`` (any real
    dtype; widened to float64), ``scale`` (the caller's float, widened to
    float64), ``causal`` (top-left aligned), ``kv_lens`` (``None`` or ``B``
    integers, clamped to ``[0, Sk]``).

    Returns ``(O [B,H,Sq,Dv], LSE [B,H,Sq])`` in float64; rows with no valid
    key hold ``O = 0`` and ``LSE = -inf``."""
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    assert k.shape[:2] == (B, H) and k.shape[3] == D
    assert v.shape[:3] == (B, H, Sk)
    Dv = v.shape[3]
    if kv_lens is None:
        kvl = [Sk] * B
    else:
        kvl = [int(x) for x in np.asarray(kv_lens).reshape(-1)]
        assert len(kvl) == B
    out = np.zeros((B, H, Sq, Dv), dtype=np.float64)
    lse = np.full((B, H, Sq), -np.inf, dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for r0 in range(0, Sq, block):
                r1 = min(r0 + block, Sq)
                rows = np.arange(r0, r1)
                o_blk, l_blk = _head_rows(q[b, h, r0:r1], rows, k[b, h], v[b, h],
                                          scale, causal, kvl[b])
                out[b, h, r0:r1] = o_blk
                lse[b, h, r0:r1] = l_blk
    return out, lse


def attention_rows(q_head, k_head, v_head, rows, scale: float, causal: bool = False,
                   kv_len=None):
    """Exact attention for selected query ``rows`` of ONE head.

    ``q_head [Sq,D]``, ``k_head [Sk,D]``, ``v_head [Sk,Dv]``; ``rows`` is a
    sequence of query positions; ``kv_len`` is that head's batch entry's key
    length (``None`` = ``Sk``).  Returns ``(O [len(rows), Dv], LSE [len(rows)])``
    in float64.  Used to check full-size outputs one sampled row at a time."""
    q_head = _as_f64(q_head)
    k_head = _as_f64(k_head)
    v_head = _as_f64(v_head)
    rows = np.asarray(rows, dtype=np.int64)
    Sk = k_head.shape[0]
    return _head_rows(q_head[rows], rows, k_head, v_head, scale, causal,
                      Sk if kv_len is None else kv_len)


def attention_varlen_ref(q, k, v, cu_q, cu_k, scale: float, causal: bool = False):
    """Exact attention over a packed batch of variable-length sequences.

    ``q [total_q, H, D]``, ``k``/``v [total_k, H, D]`` (packed tokens),
    ``cu_q``/``cu_k``: ``batch + 1`` non-decreasing offsets; sequence ``b`` owns
    query tokens ``[cu_q[b], cu_q[b+1])`` and key tokens ``[cu_k[b], cu_k[b+1])``
    (the ragged batches of continuous batching, "Fused Multi-Head Attention",
    section on continuous batching).  Each sequence is exact attention on its
    own tokens; causal masking is top-left within the sequence (query i of the
    sequence sees keys j <= i).

    Returns ``(O [total_q, H, Dv], LSE [H, total_q])`` in float64."""
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    total_q, H, _ = q.shape
    Dv = v.shape[2]
    out = np.zeros((total_q, H, Dv), dtype=np.float64)
    lse = np.full((H, total_q), -np.inf, dtype=np.float64)
    cu_q = [int(x) for x in np.asarray(cu_q).reshape(-1)]
    cu_k = [int(x) for x in np.asarray(cu_k).reshape(-1)]
    for b in range(len(cu_q) - 1):
        qs, qe = cu_q[b], cu_q[b + 1]
        ks, ke = cu_k[b], cu_k[b + 1]
        if qe <= qs:
            continue
        rows = np.arange(qe - qs)
        for h in range(H):
            o_b, l_b = _head_rows(q[qs:qe, h], rows, k[ks:ke, h], v[ks:ke, h], scale, causal, ke - ks)
            out[qs:qe, h] = o_b
            lse[h, qs:qe] = l_b
    return out, lse


def attention_paged_ref(q, k_cache, v_cache, cu_q, seqlens_k, block_table, scale: float, causal: bool = False):
    """Exact attention of packed queries against a paged key/value cache.

    ``q [total_q, H, D]`` with offsets ``cu_q`` (``batch + 1``);
    ``k_cache``/``v_cache [num_pages, page_size, H, D]``; ``seqlens_k [batch]``;
    ``block_table [batch, max_pages]``: key ``j`` of sequence ``b`` is slot
    ``j % page_size`` of page ``block_table[b][j // page_size]`` (the paged
    KV cache that "Fused Multi-Head Attention", section on continuous batching,
    names as PagedAttention).  Each sequence is exact attention of its queries
    on its gathered keys, as ``attention_varlen_ref``; ``seqlens_k`` is
    clamped to ``[0, max_pages * page_size]``.

    Returns ``(O [total_q, H, Dv], LSE [H, total_q])`` in float64."""
    q = _as_f64(q)
    k_cache = _as_f64(k_cache)
    v_cache = _as_f64(v_cache)
    total_q, H, _ = q.shape
    page_size = k_cache.shape[1]
    Dv = v_cache.shape[3]
    table = np.asarray(block_table).reshape(len(seqlens_k), -1)
    out = np.zeros((total_q, H, Dv), dtype=np.float64)
    lse = np.full((H, total_q), -np.inf, dtype=np.float64)
    cu_q = [int(x) for x in np.asarray(cu_q).reshape(-1)]
    for b in range(len(cu_q) - 1):
        qs, qe = cu_q[b], cu_q[b + 1]
        if qe <= qs:
            continue
        n = min(max(int(seqlens_k[b]), 0), table.shape[1] * page_size)
        # gather the sequence's keys in logical order
        pages = [int(table[b, j // page_size]) for j in range(n)]
        slots = [j % page_size for j in range(n)]
        k_seq = k_cache[pages, slots] if n else np.zeros((0, H, k_cache.shape[3]))
        v_seq = v_cache[pages, slots] if n else np.zeros((0, H, Dv))
        rows = np.arange(qe - qs)
        for h in range(H):
            o_b, l_b = _head_rows(q[qs:qe, h], rows, k_seq[:, h], v_seq[:, h], scale, causal, n)
            out[qs:qe, h] = o_b
            lse[h, qs:qe] = l_b
    return out, lse
