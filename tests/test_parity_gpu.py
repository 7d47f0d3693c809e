"""GPU parity: the sm_103a kernel (through the C ABI) against the fp64 oracle on
the same seeded bf16 inputs.

Small cases are compared element by element over the whole output; they span
several 128-row tiles and a ragged tail.  The full-size workloads are run in
exactly the launch configuration the benchmark times, into outputs filled with
NaN before the call (so an element no work unit writes stays NaN and fails),
and compared against the oracle on the first and last row plus one random row
of EVERY (batch entry, head, 128-row query tile): a unit the persistent
schedule skips or runs twice cannot hide in an unsampled head.  Whole-output
properties are checked too (no NaN left, exact empty rows, determinism, no
score-sized allocation)."""

import math

import numpy as np
import pytest
import torch

from exact_attention_86_gb300 import attn, workloads
from exact_attention_86_gb300.build import build
from oracle import attention_ref, attention_rows

from parity import assert_no_nan, check, nan_filled, tile_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    attn.lib()
    torch.cuda.init()


def _run(q, k, v, scale, causal, kv_lens, kernel=attn.ATTN_KERNEL_AUTO):
    dev = torch.device("cuda:0")
    qd, kd, vd = (t.to(dev).contiguous() for t in (q, k, v))
    kvd = kv_lens.to(dev) if kv_lens is not None else None
    # NaN-filled outputs: an element no unit writes cannot pass as a stale
    # result of an earlier call in reused memory
    o = nan_filled(tuple(q.shape), torch.bfloat16, dev)
    lse = nan_filled(tuple(q.shape[:3]), torch.float32, dev)
    attn.forward(qd, kd, vd, scale=scale, causal=causal, kv_lens=kvd, out=o, lse=lse, kernel=kernel)
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    assert_no_nan(o, lse, what="forward")
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _np(t):
    return t.float().numpy().astype(np.float64)


def _inputs(B, H, Sq, Sk, D, seed, std=1.0, kv=None):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, H, Sq, D, generator=g) * std).to(torch.bfloat16)
    k = (torch.randn(B, H, Sk, D, generator=g) * std).to(torch.bfloat16)
    v = (torch.randn(B, H, Sk, D, generator=g) * std).to(torch.bfloat16)
    kvt = None if kv is None else torch.tensor(kv, dtype=torch.int32)
    return q, k, v, kvt


def _full_check(q, k, v, scale, causal, kv_lens, what, kernel=attn.ATTN_KERNEL_AUTO):
    o, lse = _run(q, k, v, scale, causal, kv_lens, kernel)
    o_ref, lse_ref = attention_ref(_np(q), _np(k), _np(v), scale, causal=causal,
                                   kv_lens=None if kv_lens is None else kv_lens.numpy())
    return check(o, lse, o_ref, lse_ref, what)


# ---------------------------------------------------------------- small cases

SMALL = [
    # B, H, Sq, Sk, D, causal
    (1, 2, 300, 300, 64, False),
    (1, 2, 300, 300, 128, False),
    (2, 1, 600, 600, 64, True),
    (2, 1, 600, 600, 128, True),
    (1, 1, 1, 1, 64, False),
    (1, 1, 1, 1, 128, True),
    (1, 2, 127, 129, 128, False),
    (1, 2, 129, 127, 64, False),
    (2, 3, 257, 385, 128, False),
    (1, 1, 200, 700, 64, False),
    (1, 1, 700, 200, 128, False),
    (1, 2, 300, 520, 128, True),   # causal with Sq != Sk: top-left aligned
    (1, 2, 520, 300, 64, True),
    (1, 1, 4097, 130, 64, False),
]


# both padded-forward kernels on every case (the automatic choice takes the
# one-tile kernel for most small batches)
KERNELS = [attn.ATTN_KERNEL_ONE_TILE, attn.ATTN_KERNEL_TWO_TILE]

SMALL_CASES = [(s, kern) for s in SMALL for kern in KERNELS]


@pytest.mark.parametrize("shape,kernel", SMALL_CASES,
                         ids=lambda x: ("B{}H{}q{}k{}d{}{}".format(*x[:5], "c" if x[5] else "")
                                        if isinstance(x, tuple) else ("two" if x else "one")))
def test_small_shapes(shape, kernel):
    B, H, Sq, Sk, D, causal = shape
    q, k, v, _ = _inputs(B, H, Sq, Sk, D, seed=(B * 131 + H * 71 + Sq * 7 + Sk * 13 + D + int(causal)) % 997)
    _full_check(q, k, v, 1.0 / math.sqrt(D), causal, None, f"{shape} kernel {kernel}", kernel)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal,kernel", [(False, 0), (False, 1), (True, 0), (True, 1)])
def test_kv_lens_edges(D, causal, kernel):
    Sk = 400
    kv = [0, 1, 127, 128, 129, Sk, 255, 257]
    q, k, v, kvt = _inputs(len(kv), 2, 384, Sk, D, seed=7 + D, kv=kv)
    _full_check(q, k, v, 1.0 / math.sqrt(D), causal, kvt, f"kv edges D{D} causal{causal} kernel {kernel}", kernel)


def test_kv_lens_out_of_range_are_clamped():
    q, k, v, kvt = _inputs(3, 1, 256, 300, 128, seed=3, kv=[-7, 1000, 300])
    o, lse = _run(q, k, v, 0.1, False, kvt)
    o_ref, lse_ref = attention_ref(_np(q), _np(k), _np(v), 0.1, kv_lens=[0, 300, 300])
    check(o, lse, o_ref, lse_ref, "clamped kv_lens")


@pytest.mark.parametrize("std", [2.0, 4.0])
@pytest.mark.parametrize("causal,kernel", [(False, 0), (False, 1), (True, 0), (True, 1)])
def test_large_scores_stress_rescale(std, causal, kernel):
    # Scores with std ~ std^2 * sqrt(D) * scale: the running max moves often.
    q, k, v, _ = _inputs(1, 2, 512, 1024, 128, seed=11, std=std)
    _full_check(q, k, v, 1.0 / math.sqrt(128), causal, None, f"std {std} kernel {kernel}", kernel)


def test_increasing_scores_force_rescale_every_tile():
    # Keys grow along the sequence so that every K tile raises the row max by
    # more than the lazy-rescale threshold.
    B, H, S, D = 1, 1, 256, 64
    g = torch.Generator().manual_seed(5)
    q = torch.ones(B, H, S, D)
    k = torch.linspace(0, 1, S).view(1, 1, S, 1).expand(B, H, S, D) * 0.5 + torch.randn(B, H, S, D, generator=g) * 0.01
    v = torch.randn(B, H, S, D, generator=g)
    q, k, v = (t.to(torch.bfloat16).contiguous() for t in (q, k, v))
    for kernel in KERNELS:
        _full_check(q, k, v, 2.0, False, None, f"rescale every tile, kernel {kernel}", kernel)
        _full_check(q, k, v, 2.0, True, None, f"rescale every tile, causal, kernel {kernel}", kernel)


@pytest.mark.parametrize("scale", [-0.125, 0.0, 1e-3, 0.5])
@pytest.mark.parametrize("causal,kernel", [(False, 1), (True, 0), (True, 1)])
def test_scale_values(scale, causal, kernel):
    q, k, v, _ = _inputs(1, 2, 300, 300, 64, seed=21)
    _full_check(q, k, v, scale, causal, None, f"scale {scale}", kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_no_keys_at_all(kernel):
    q, k, v, _ = _inputs(2, 2, 200, 1, 128, seed=1)
    k = k[:, :, :0].contiguous()
    v = v[:, :, :0].contiguous()
    dev = torch.device("cuda:0")
    o, lse = attn.forward(q.to(dev), torch.empty(2, 2, 0, 128, dtype=torch.bfloat16, device=dev),
                          torch.empty(2, 2, 0, 128, dtype=torch.bfloat16, device=dev), kernel=kernel)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and not torch.any(torch.signbit(o.float()))
    assert torch.all(lse == float("-inf"))


def test_empty_query_is_a_no_op():
    dev = torch.device("cuda:0")
    q = torch.empty(1, 1, 0, 64, dtype=torch.bfloat16, device=dev)
    k = torch.randn(1, 1, 16, 64, device=dev).to(torch.bfloat16)
    o, lse = attn.forward(q, k, k)
    torch.cuda.synchronize()
    assert o.numel() == 0 and lse.numel() == 0


@pytest.mark.parametrize("causal,kernel", [(False, 1), (True, 0), (True, 1)])
def test_output_guard_bands_untouched(causal, kernel):
    # Canary words around O and LSE catch out-of-bounds writes.
    B, H, Sq, Sk, D = 2, 3, 300, 333, 128
    q, k, v, kvt = _inputs(B, H, Sq, Sk, D, seed=9, kv=[333, 100])
    dev = torch.device("cuda:0")
    pad = 4096
    o_buf = torch.full((2 * pad + B * H * Sq * D,), 12345, dtype=torch.int16, device=dev)
    l_buf = torch.full((2 * pad + B * H * Sq,), 7.25, dtype=torch.float32, device=dev)
    o_view = o_buf[pad:pad + B * H * Sq * D].view(torch.bfloat16).view(B, H, Sq, D)
    l_view = l_buf[pad:pad + B * H * Sq].view(B, H, Sq)
    attn.forward(q.to(dev), k.to(dev), v.to(dev), causal=causal, kv_lens=kvt.to(dev), out=o_view, lse=l_view,
                 kernel=kernel)
    torch.cuda.synchronize()
    assert torch.all(o_buf[:pad] == 12345) and torch.all(o_buf[-pad:] == 12345)
    assert torch.all(l_buf[:pad] == 7.25) and torch.all(l_buf[-pad:] == 7.25)
    o_ref, lse_ref = attention_ref(_np(q), _np(k), _np(v), 1 / math.sqrt(D), causal=causal, kv_lens=[333, 100])
    check(o_view.float().cpu().numpy(), l_view.cpu().numpy(), o_ref, lse_ref, "guard bands")


@pytest.mark.parametrize("causal,kernel", [(False, 1), (True, 0), (True, 1)])
def test_deterministic(causal, kernel):
    q, k, v, _ = _inputs(2, 4, 1000, 1000, 128, seed=13)
    dev = torch.device("cuda:0")
    a = attn.forward(q.to(dev), k.to(dev), v.to(dev), causal=causal, kernel=kernel)
    b = attn.forward(q.to(dev), k.to(dev), v.to(dev), causal=causal, kernel=kernel)
    torch.cuda.synchronize()
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))


def test_wait_timeout_selftest_reports_and_recovers():
    stream = torch.cuda.current_stream().cuda_stream
    assert attn.attn_check_device_status(stream)[0] == attn.ATTN_OK
    assert attn.attn_selftest_wait_timeout(1_000_000, stream) == attn.ATTN_OK
    st, site = attn.attn_check_device_status(stream)
    assert st == attn.ATTN_ERR_DEVICE_TIMEOUT and site == 8
    assert attn.attn_check_device_status(stream)[0] == attn.ATTN_OK  # cleared
    # the context is still healthy: a normal call works and matches the oracle
    q, k, v, _ = _inputs(1, 1, 130, 130, 64, seed=2)
    _full_check(q, k, v, 0.125, False, None, "after selftest")


# every site a bounded wait of the forward kernel can report
WAIT_SITES = set(range(1, 14)) - {8, 12}


@pytest.mark.parametrize("D,causal,kernel,skip", [(128, False, 1, 5), (128, False, 0, 5), (128, True, 0, 0),
                                                  (128, True, 1, 2), (64, False, 1, 3), (64, False, 0, 2),
                                                  (64, True, 0, 10), (64, True, 1, 4)])
def test_forward_kernel_gives_up_drains_and_recovers(D, causal, kernel, skip):
    """The attention kernel's own give-up path: block 0's producer leaves out
    one K fill, so a bounded wait (1 ms) in block 0 runs out; every role of
    that block must drain its copies and products, free Tensor Memory and
    return.  The status reports the timeout and its site, every other block's
    rows are exact, and the context then computes correct results."""
    B, H, S = 1, 2, 2048
    q, k, v, _ = _inputs(B, H, S, S, D, seed=61 + D + int(causal))
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = nan_filled((B, H, S, D), torch.bfloat16, dev)
    lse = nan_filled((B, H, S), torch.float32, dev)
    stream = torch.cuda.current_stream().cuda_stream
    assert attn.attn_check_device_status(stream)[0] == attn.ATTN_OK
    scale = 1.0 / math.sqrt(D)
    st = attn.attn_selftest_fwd_abort(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                      B, H, S, S, D, scale, int(causal), None, kernel, skip, 1_000_000, stream)
    assert st == attn.ATTN_OK
    st, site = attn.attn_check_device_status(stream)
    assert st == attn.ATTN_ERR_DEVICE_TIMEOUT and site in WAIT_SITES, (st, site)
    assert attn.attn_check_device_status(stream)[0] == attn.ATTN_OK  # cleared
    # block 0 handles one unit (fewer units than SMs): only its rows may
    # differ, one 128-row query tile (one-tile kernel) or two adjacent ones of
    # one head (two-tile kernel)
    o_ref, l_ref = attention_ref(_np(q), _np(k), _np(v), scale, causal=causal)
    on, ln = o.float().cpu().numpy(), lse.cpu().numpy()
    bad = []
    for h in range(H):
        for t0 in range(0, S, 128):
            sl = (0, h, slice(t0, t0 + 128))
            try:
                check(on[sl], ln[sl], o_ref[sl], l_ref[sl], "")
            except AssertionError:
                bad.append((h, t0))
    assert len(bad) <= (2 if kernel == attn.ATTN_KERNEL_TWO_TILE else 1), bad
    if len(bad) == 2:
        assert bad[0][0] == bad[1][0] and bad[1][1] - bad[0][1] == 128, bad
    # the context is healthy: a normal call matches the oracle
    _full_check(q, k, v, scale, causal, None, "after the aborted launch", kernel)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mode", [0, 1])
def test_launch_floor_kernel_runs_clean(D, mode):
    # the measurement aid: a full wave of blocks with the forward's launch
    # shape, empty or with the fixed set-up / tear-down only
    stream = torch.cuda.current_stream().cuda_stream
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    for grid in (1, n_sms, 2 * n_sms):
        assert attn.attn_selftest_launch_floor(grid, D, mode, stream) == attn.ATTN_OK
    assert attn.attn_check_device_status(stream)[0] == attn.ATTN_OK
    q, k, v, _ = _inputs(1, 1, 130, 130, D, seed=4)
    _full_check(q, k, v, 0.125, True, None, "after launch floor")


# ------------------------------------------------------ the five workloads

def _device_inputs(w, draw=0):
    q, k, v, kv = workloads.generate(w, draw)
    dev = torch.device("cuda:0")
    return q, k, v, kv, q.to(dev), k.to(dev), v.to(dev), (kv.to(dev) if kv is not None else None)


def _forward_nan_filled(w, qd, kd, vd, kvd):
    """The benchmark's launch of workload w into NaN-filled O and LSE."""
    o = nan_filled((w.B, w.H, w.Sq, w.D), torch.bfloat16, qd.device)
    lse = nan_filled((w.B, w.H, w.Sq), torch.float32, qd.device)
    attn.forward(qd, kd, vd, scale=w.scale, causal=w.causal, kv_lens=kvd, out=o, lse=lse)
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    assert_no_nan(o, lse, what=w.name)
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _every_tile_check(w, q, k, v, kv, o, lse, what):
    """Oracle rows for every (b, h, query tile): first, last and one random row."""
    rng = np.random.default_rng(w.seed)
    for b in range(w.B):
        kvb = None if kv is None else int(kv[b])
        for h in range(w.H):
            rows = tile_rows(w.Sq, rng)
            o_ref, l_ref = attention_rows(_np(q[b, h]), _np(k[b, h]), _np(v[b, h]), rows, w.scale,
                                          causal=w.causal, kv_len=kvb)
            check(o[b, h, rows], lse[b, h, rows], o_ref, l_ref, f"{what} b{b} h{h}")


def _sampled_check(w, draw):
    q, k, v, kv, qd, kd, vd, kvd = _device_inputs(w, draw)
    o, lse = _forward_nan_filled(w, qd, kd, vd, kvd)
    _every_tile_check(w, q, k, v, kv, o, lse, f"{w.name} draw{draw}")
    return o, lse, kv


def test_workload_s128_d64_full():
    w = workloads.WORKLOADS["s128_d64"]
    q, k, v, kv = workloads.generate(w)
    _full_check(q, k, v, w.scale, w.causal, kv, w.name)


def test_workload_s1024_d64_causal_full():
    w = workloads.WORKLOADS["s1024_d64_causal"]
    q, k, v, kv = workloads.generate(w)
    _full_check(q, k, v, w.scale, w.causal, kv, w.name)


def test_workload_s2048_d128_padded():
    w = workloads.WORKLOADS["s2048_d128_padded"]
    q, k, v, kv, qd, kd, vd, kvd = _device_inputs(w)
    assert int(kv[w.kv_zero_index]) == 0
    o, lse = _forward_nan_filled(w, qd, kd, vd, kvd)
    # every batch entry (all key lengths), two heads each, every row
    for b in range(w.B):
        for h in (0, w.H - 1):
            o_ref, l_ref = attention_ref(_np(q[b:b + 1, h:h + 1]), _np(k[b:b + 1, h:h + 1]),
                                         _np(v[b:b + 1, h:h + 1]), w.scale, kv_lens=[int(kv[b])])
            check(o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], o_ref, l_ref, f"{w.name} b{b} h{h}")
    # every other head: three rows of every query tile
    _every_tile_check(w, q, k, v, kv, o, lse, w.name)
    # the sequence with kv_len = 0: every head exactly O = +0, LSE = -inf
    z = w.kv_zero_index
    assert np.all(o[z] == 0.0) and not np.any(np.signbit(o[z])) and np.all(lse[z] == -np.inf)


@pytest.mark.parametrize("name", ["s8192_d128", "s8192_d128_causal"])
@pytest.mark.parametrize("draw", [0, 1])
def test_workload_s8192_every_tile(name, draw):
    w = workloads.WORKLOADS[name]
    _sampled_check(w, draw)


def test_workload_s32768_causal_every_tile_and_memory():
    w = workloads.WORKLOADS["s32768_d128_causal"]
    q, k, v, kv, qd, kd, vd, kvd = _device_inputs(w)
    o = nan_filled((w.B, w.H, w.Sq, w.D), torch.bfloat16, qd.device)
    lse = nan_filled((w.B, w.H, w.Sq), torch.float32, qd.device)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    alloc_before = torch.cuda.max_memory_allocated()
    attn.forward(qd, kd, vd, scale=w.scale, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    # no allocation anywhere near one head's score matrix (2 GiB in bf16)
    assert torch.cuda.max_memory_allocated() == alloc_before
    assert free_before - free_after < (64 << 20)
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    assert_no_nan(o, lse, what=w.name)
    on = o.float().cpu().numpy()
    ln = lse.cpu().numpy()
    assert np.all(np.isfinite(on)) and np.all(np.isfinite(ln))
    _every_tile_check(w, q, k, v, kv, on, ln, w.name)
