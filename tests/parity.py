"""Comparison helpers shared by the GPU parity tests (no attention arithmetic).

Tolerances: O (bf16) element-wise |gpu - ref| <= 2e-2 + 2e-2 * |ref|; LSE (fp32)
|gpu - ref| <= 1e-3 on rows with a valid key; rows with no valid key must be
exactly O = +0.0 and LSE = -inf; no NaN or Inf anywhere else.
"""

import numpy as np

O_ATOL = 2e-2
O_RTOL = 2e-2
LSE_ATOL = 1e-3


def check(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    assert o_gpu.shape == o_ref.shape and lse_gpu.shape == lse_ref.shape, what
    empty = ~np.isfinite(lse_ref)
    assert np.all(lse_ref[empty] == -np.inf), what
    # rows with no valid key: exact semantics
    assert np.all(lse_gpu[empty] == -np.inf), f"{what}: LSE of rows without keys must be -inf"
    oe = o_gpu[empty]
    assert np.all(oe == 0.0) and not np.any(np.signbit(oe)), f"{what}: O of rows without keys must be +0"
    # every other value finite
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    assert np.all(np.isfinite(lse_gpu[~empty])), f"{what}: non-finite LSE on a row with keys"
    err = np.abs(o_gpu - o_ref)
    bad = err > O_ATOL + O_RTOL * np.abs(o_ref)
    assert not np.any(bad), (f"{what}: {int(bad.sum())} O elements out of tolerance, "
                             f"max abs err {err.max():.3e}")
    lerr = np.abs(lse_gpu[~empty] - lse_ref[~empty])
    assert lerr.size == 0 or lerr.max() <= LSE_ATOL, f"{what}: LSE max abs err {lerr.max():.3e}"
    return float(err.max()) if err.size else 0.0, float(lerr.max()) if lerr.size else 0.0
