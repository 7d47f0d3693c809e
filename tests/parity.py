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


def tile_rows(n_rows, rng, tile=128):
    """Query rows to compare in a full-size output: the first and the last row
    of EVERY 128-row query tile (the kernel's work unit) plus one random row
    inside each tile, so that a unit the schedule skips or runs twice shows up
    in the comparison, not only in a whole-output NaN check."""
    rows = []
    for t0 in range(0, n_rows, tile):
        t1 = min(t0 + tile, n_rows)
        rows.extend({t0, t1 - 1, int(rng.integers(t0, t1))})
    return sorted(rows)


def nan_filled(shape, dtype, device):
    """An output buffer whose every element is NaN before the call: any element
    that the kernel leaves unwritten stays NaN and fails the checks."""
    import torch
    return torch.full(shape, float("nan"), dtype=dtype, device=device)


def assert_no_nan(*tensors, what=""):
    """Every element was written: none of the NaN fill survives."""
    import torch
    for t in tensors:
        n = int(torch.isnan(t.float()).sum())
        assert n == 0, f"{what}: {n} elements still hold the NaN fill (a work unit was not written)"
