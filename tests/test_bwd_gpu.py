"""GPU parity of the backward pass (dQ, dK, dV) against the fp64 oracle.

Tolerance (derived from the arithmetic).  The kernels compute P and dS in
fp32 from fp32 scores, round P (for dV) and dS (for dQ, dK) to bf16 before
the tensor-core products (relative error 2^-9 each), accumulate in fp32 and
round the results to bf16 (2^-9).  Delta = <dO, O> uses the forward's bf16
O, whose own error e_i = |<dO_i, O_gpu_i - O_exact_i>| (plus 2^-16 of
sum_d |dO_id O_id| for the fp32 sum) enters every dS of the row as P_ij e_i.  With all magnitudes from the exact fp64 quantities,
per element (a factor 2 over the rounding terms):

    |ddV| <= 2^-8 (P^T |dO|) + 2^-8 |dV|
    |ddQ| <= |scale| (2^-8 |dS| + P e) |K| + 2^-8 |dQ|
    |ddK| <= |scale| (2^-8 |dS| + P e)^T |Q| + 2^-8 |dK|

plus 1e-5 of the largest reference value of the tensor (fp32 sums and the
hardware exp2).
"""

import math

import numpy as np
import pytest
import torch

from exact_attention_86_gb300 import attn
from exact_attention_86_gb300.build import build
from oracle import attention_bwd_head, attention_bwd_sampled, attention_ref

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    attn.lib()


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _probs(q, k, scale, causal, kv_len, rows):
    Sk = k.shape[0]
    s = (q[rows] @ k.T) * scale
    lim = np.full(len(rows), min(max(kv_len, 0), Sk))
    if causal:
        lim = np.minimum(lim, np.asarray(rows) + 1)
    valid = np.arange(Sk)[None, :] < lim[:, None]
    s = np.where(valid, s, -np.inf)
    m = np.where(lim > 0, s.max(axis=1, initial=-np.inf), 0.0)
    e = np.where(valid, np.exp(s - m[:, None]), 0.0)
    tot = e.sum(axis=1)
    return np.where((lim > 0)[:, None], e / np.where(lim > 0, tot, 1)[:, None], 0.0)


def _delta_err(do, o_gpu, o_exact):
    """Error of the kernel's Delta: the forward's O error, plus an allowance
    for the fp32 sum of D products."""
    return (np.abs(np.sum(do * (o_gpu - o_exact), axis=1))
            + 2.0 ** -16 * np.sum(np.abs(do) * np.abs(o_gpu), axis=1))


def _bounds(q, k, v, do, o_gpu, o_exact, scale, causal, kv_len, q_rows, k_rows, block=512):
    """Per-element bounds for dQ[q_rows], dK[k_rows], dV[k_rows] of one head."""
    Sq = q.shape[0]
    q_rows = np.asarray(q_rows)
    k_rows = np.asarray(k_rows)
    p = _probs(q, k, scale, causal, kv_len, q_rows)
    dp = do[q_rows] @ v.T
    ds = p * (dp - np.sum(p * dp, axis=1)[:, None])
    e = _delta_err(do[q_rows], o_gpu[q_rows], o_exact[q_rows])
    bq = abs(scale) * ((2.0 ** -8 * np.abs(ds) + p * e[:, None]) @ np.abs(k))
    bk = np.zeros((len(k_rows), q.shape[1]))
    bv = np.zeros((len(k_rows), v.shape[1]))
    for r0 in range(0, Sq, block):
        rows = np.arange(r0, min(Sq, r0 + block))
        pf = _probs(q, k, scale, causal, kv_len, rows)
        dpf = do[rows] @ v.T
        dsf = pf * (dpf - np.sum(pf * dpf, axis=1)[:, None])
        ef = _delta_err(do[rows], o_gpu[rows], o_exact[rows])
        bk += abs(scale) * ((2.0 ** -8 * np.abs(dsf[:, k_rows]) + pf[:, k_rows] * ef[:, None]).T @ np.abs(q[rows]))
        bv += 2.0 ** -8 * (pf[:, k_rows].T @ np.abs(do[rows]))
    return bq, bk, bv


def _check(got, ref, bound, what):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite"
    err = np.abs(got - ref)
    tol = bound + 2.0 ** -8 * np.abs(ref) + 1e-5 * (np.abs(ref).max() if ref.size else 0.0)
    bad = err > tol
    assert not np.any(bad), (f"{what}: {int(bad.sum())} of {bad.size} out of bound, max err {err.max():.3e}, "
                             f"max ref {np.abs(ref).max():.3e}")


def _inputs(B, H, Sq, Sk, D, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, H, Sq, D, generator=g) * std).to(torch.bfloat16)
    k = (torch.randn(B, H, Sk, D, generator=g) * std).to(torch.bfloat16)
    v = (torch.randn(B, H, Sk, D, generator=g) * std).to(torch.bfloat16)
    do = torch.randn(B, H, Sq, D, generator=g).to(torch.bfloat16)
    return q, k, v, do


def _run(q, k, v, do, scale, causal, kv):
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    kvd = None if kv is None else torch.tensor(kv, dtype=torch.int32, device=dev)
    o, lse = attn.forward(qd, kd, vd, scale=scale, causal=causal, kv_lens=kvd)
    dq, dk, dv = attn.backward(qd, kd, vd, o, lse, dod, scale=scale, causal=causal, kv_lens=kvd)
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    return o, dq, dk, dv


SHAPES = [
    # B, H, Sq, Sk, D
    (1, 1, 128, 128, 64),
    (1, 2, 1, 130, 128),
    (2, 1, 200, 77, 64),
    (1, 2, 257, 300, 128),
    (2, 2, 384, 384, 128),
    (1, 1, 500, 129, 64),
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_matches_oracle(shape, causal):
    B, H, Sq, Sk, D = shape
    q, k, v, do = _inputs(B, H, Sq, Sk, D, seed=Sq * 3 + Sk + D + int(causal))
    scale = 1.0 / math.sqrt(D)
    kv = [max(Sk - 5 * b, 0) for b in range(B)] if B > 1 else None
    o, dq, dk, dv = _run(q, k, v, do, scale, causal, kv)
    o_exact, _ = attention_ref(_f64(q), _f64(k), _f64(v), scale, causal=causal, kv_lens=kv)
    for b in range(B):
        kvl = Sk if kv is None else kv[b]
        for h in range(H):
            qh, kh, vh, doh = _f64(q[b, h]), _f64(k[b, h]), _f64(v[b, h]), _f64(do[b, h])
            rq, rk, rv = attention_bwd_head(qh, kh, vh, doh, scale, causal, kvl)
            bq, bk, bv = _bounds(qh, kh, vh, doh, _f64(o[b, h]), o_exact[b, h], scale, causal, kvl,
                                 np.arange(Sq), np.arange(Sk))
            what = f"{shape} causal={causal} b{b} h{h}"
            _check(_f64(dq[b, h]), rq, bq, "dQ " + what)
            _check(_f64(dk[b, h]), rk, bk, "dK " + what)
            _check(_f64(dv[b, h]), rv, bv, "dV " + what)


@pytest.mark.parametrize("kv", [[0, 1], [127, 128], [129, 300]])
def test_bwd_key_lengths_and_empty_rows(kv):
    B, H, Sq, Sk, D = 2, 1, 150, 300, 128
    q, k, v, do = _inputs(B, H, Sq, Sk, D, seed=sum(kv))
    o, dq, dk, dv = _run(q, k, v, do, 0.09, False, kv)
    o_exact, _ = attention_ref(_f64(q), _f64(k), _f64(v), 0.09, kv_lens=kv)
    for b in range(B):
        qh, kh, vh, doh = _f64(q[b, 0]), _f64(k[b, 0]), _f64(v[b, 0]), _f64(do[b, 0])
        rq, rk, rv = attention_bwd_head(qh, kh, vh, doh, 0.09, False, kv[b])
        bq, bk, bv = _bounds(qh, kh, vh, doh, _f64(o[b, 0]), o_exact[b, 0], 0.09, False, kv[b], np.arange(Sq),
                             np.arange(Sk))
        _check(_f64(dq[b, 0]), rq, bq, f"dQ kv={kv[b]}")
        _check(_f64(dk[b, 0]), rk, bk, f"dK kv={kv[b]}")
        _check(_f64(dv[b, 0]), rv, bv, f"dV kv={kv[b]}")
        # keys past kv_len get exactly zero gradient; with no key every dQ row is zero
        assert torch.all(dk[b, 0, kv[b]:] == 0) and torch.all(dv[b, 0, kv[b]:] == 0)
        if kv[b] == 0:
            assert torch.all(dq[b, 0] == 0)


def test_bwd_large_scores_and_negative_scale():
    q, k, v, do = _inputs(1, 2, 256, 256, 128, seed=61, std=2.0)
    for scale in (0.3, -0.2):
        o, dq, dk, dv = _run(q, k, v, do, scale, True, None)
        o_exact, _ = attention_ref(_f64(q), _f64(k), _f64(v), scale, causal=True)
        for h in range(2):
            qh, kh, vh, doh = _f64(q[0, h]), _f64(k[0, h]), _f64(v[0, h]), _f64(do[0, h])
            rq, rk, rv = attention_bwd_head(qh, kh, vh, doh, scale, True)
            bq, bk, bv = _bounds(qh, kh, vh, doh, _f64(o[0, h]), o_exact[0, h], scale, True, 256, np.arange(256),
                                 np.arange(256))
            _check(_f64(dq[0, h]), rq, bq, f"dQ scale={scale}")
            _check(_f64(dk[0, h]), rk, bk, f"dK scale={scale}")
            _check(_f64(dv[0, h]), rv, bv, f"dV scale={scale}")


def test_bwd_degenerate_lengths():
    dev = torch.device("cuda:0")
    q, k, v, do = _inputs(1, 2, 0, 64, 64, seed=71)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty(1, 2, 0, device=dev)
    dq, dk, dv = attn.backward(qd, kd, vd, o, lse, do.to(dev))
    torch.cuda.synchronize()
    assert torch.all(dk == 0) and torch.all(dv == 0)
    q, k, v, do = _inputs(1, 2, 70, 0, 64, seed=72)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o, lse = attn.forward(qd, kd, vd)
    dq, dk, dv = attn.backward(qd, kd, vd, o, lse, do.to(dev))
    torch.cuda.synchronize()
    assert torch.all(dq == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_full_size_sampled(causal):
    """The benchmarked backward shape (B2 H16 S8192 D128) in the benchmark's
    launch configuration: sampled dQ rows and dK, dV rows of one head."""
    B, H, S, D = 2, 16, 8192, 128
    q, k, v, do = _inputs(B, H, S, S, D, seed=3)
    scale = 1.0 / math.sqrt(D)
    o, dq, dk, dv = _run(q, k, v, do, scale, causal, None)
    b, h = 1, 7
    qh, kh, vh, doh = _f64(q[b, h]), _f64(k[b, h]), _f64(v[b, h]), _f64(do[b, h])
    rng = np.random.default_rng(11)
    q_rows = sorted(set([0, 1, 127, 128, S - 1] + [int(x) for x in rng.integers(0, S, 19)]))
    k_rows = sorted(set([0, 1, 127, 128, S - 1] + [int(x) for x in rng.integers(0, S, 19)]))
    rq, rk, rv = attention_bwd_sampled(qh, kh, vh, doh, scale, q_rows, k_rows, causal=causal)
    o_rows = np.arange(S)
    o_exact = np.zeros((S, D))
    for r0 in range(0, S, 1024):
        rows = o_rows[r0:r0 + 1024]
        o_exact[rows] = _probs(qh, kh, scale, causal, S, rows) @ vh
    bq, bk, bv = _bounds(qh, kh, vh, doh, _f64(o[b, h]), o_exact, scale, causal, S, q_rows, k_rows)
    _check(_f64(dq[b, h])[q_rows], rq, bq, "dQ full size")
    _check(_f64(dk[b, h])[k_rows], rk, bk, "dK full size")
    _check(_f64(dv[b, h])[k_rows], rv, bv, "dV full size")


def test_bwd_repeated_launches_are_bitwise_identical():
    q, k, v, do = _inputs(2, 4, 1024, 1024, 128, seed=81)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    o, lse = attn.forward(qd, kd, vd, causal=True)
    outs = [attn.backward(qd, kd, vd, o, lse, dod, causal=True) for _ in range(20)]
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    for g in outs[1:]:
        for a, b0 in zip(g, outs[0]):
            assert torch.equal(a.view(torch.int16), b0.view(torch.int16))
