"""GPU parity of the FP8 (E4M3) forward against the fp64 oracle.

Tolerance (derived from the arithmetic): the kernel's scores are exact
products of E4M3 values accumulated in fp32, so the LSE keeps the bf16 path's
bound (1e-3).  O differs from the exact result by the rounding of each
probability to E4M3 before the P V product (relative error at most 2^-4 for
normal codes, absolute at most 2^-14 of the row's largest weight for
subnormal ones; the row sums use the unrounded values) and by the final bf16
rounding (2^-8 relative).  Per element:

    |O_gpu - O_ref| <= 2^-4 * A + 2^-8 * |O_ref| + 2^-6 * max|V|

where A = sum_j w_j |v_j| (the oracle's attention of |V|, exact weights w)
bounds the normal-code part and the last term covers subnormal codes and
fp32 accumulation.  Systematic errors that this loose bound could let through
(a descale, a shift) are caught by exact laws below: the V descale scales O
bit for bit, and only the product scale * q_descale * k_descale matters.  An
aggregate check holds the RMS error under 6 % of the RMS of O (the rounding
errors are independent, of RMS 2^-4 / sqrt(3) = 3.6 % of a weight).
"""

import math

import numpy as np
import pytest
import torch

from exact_attention_86_gb300 import attn, workloads
from exact_attention_86_gb300.build import build
from oracle import attention_fp8_ref, attention_rows, decode_e4m3

from parity import assert_no_nan, nan_filled, tile_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    attn.lib()


def _inputs(B, H, Sq, Sk, seed, std=1.0, D=128):
    g = torch.Generator().manual_seed(seed)
    q = workloads.to_e4m3_codes(torch.randn(B, H, Sq, D, generator=g) * std)
    k = workloads.to_e4m3_codes(torch.randn(B, H, Sk, D, generator=g) * std)
    v = workloads.to_e4m3_codes(torch.randn(B, H, Sk, D, generator=g) * std)
    return q, k, v


ROWS, TRANSPOSED = attn.ATTN_V_ROWS, attn.ATTN_V_TRANSPOSED
LAYOUTS = pytest.mark.parametrize("layout", [ROWS, TRANSPOSED], ids=["v_rows", "v_transposed"])
# both padded-forward kernels (small batches take the one-tile kernel unless forced)
KERNELS = pytest.mark.parametrize("kernel", [attn.ATTN_KERNEL_ONE_TILE, attn.ATTN_KERNEL_TWO_TILE],
                                  ids=["one", "two"])


def _run(q, k, v, scale, causal=False, kv=None, qd=1.0, kd=1.0, vd=1.0, layout=TRANSPOSED,
         kernel=attn.ATTN_KERNEL_AUTO):
    """The E4M3 forward with V in the given layout, into NaN-filled outputs."""
    dev = torch.device("cuda:0")
    vl = v if layout == ROWS else v.transpose(-1, -2).contiguous()
    B, H, Sq, D = q.shape
    o = nan_filled((B, H, Sq, D), torch.bfloat16, dev)
    lse = nan_filled((B, H, Sq), torch.float32, dev)
    attn.forward_fp8(q.to(dev), k.to(dev), vl.to(dev), qd, kd, vd, scale=scale, causal=causal,
                     kv_lens=None if kv is None else torch.tensor(kv, dtype=torch.int32, device=dev), out=o, lse=lse,
                     v_layout=layout, kernel=kernel)
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    assert_no_nan(o, lse, what="fp8")
    return o, lse


def check_fp8(o_gpu, lse_gpu, o_ref, l_ref, a_ref, vmax, what=""):
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    empty = ~np.isfinite(l_ref)
    assert np.all(lse_gpu[empty] == -np.inf), what
    oe = o_gpu[empty]
    assert np.all(oe == 0.0) and not np.any(np.signbit(oe)), what
    assert np.all(np.isfinite(o_gpu)) and np.all(np.isfinite(lse_gpu[~empty])), what
    err = np.abs(o_gpu - o_ref)
    bound = 2.0 ** -4 * a_ref + 2.0 ** -8 * np.abs(o_ref) + 2.0 ** -6 * vmax
    bad = err > bound
    assert not np.any(bad), f"{what}: {int(bad.sum())} elements out of bound, max err {err.max():.3e}"
    if o_ref.size:
        rms_err = float(np.sqrt(np.mean(err ** 2)))
        rms_ref = float(np.sqrt(np.mean(o_ref ** 2)))
        assert rms_err <= 0.06 * rms_ref + 1e-6, f"{what}: RMS error {rms_err:.3e} vs RMS {rms_ref:.3e}"
    lerr = np.abs(lse_gpu[~empty] - l_ref[~empty])
    assert lerr.size == 0 or lerr.max() <= 1e-3, f"{what}: LSE err {lerr.max():.3e}"


def _oracle(q, k, v, scale, causal=False, kv=None, qd=1.0, kd=1.0, vd=1.0):
    qn, kn, vn = q.numpy(), k.numpy(), v.numpy()
    o, l = attention_fp8_ref(qn, kn, vn, qd, kd, vd, scale, causal=causal, kv_lens=kv)
    a, _ = attention_fp8_ref(qn, kn, vn & 0x7F, qd, kd, abs(vd), scale, causal=causal, kv_lens=kv)
    vmax = float(np.nanmax(np.abs(decode_e4m3(vn)))) * abs(vd) if vn.size else 0.0
    return o, l, a, vmax


SHAPES = [
    # B, H, Sq, Sk
    (1, 1, 1, 16),
    (1, 2, 100, 144),
    (2, 2, 128, 128),
    (1, 3, 129, 272),
    (2, 1, 300, 400),
    (1, 2, 257, 1024),
    (1, 1, 500, 128),
]


@KERNELS
@LAYOUTS
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_matches_oracle(shape, causal, layout, D, kernel):
    B, H, Sq, Sk = shape
    q, k, v = _inputs(B, H, Sq, Sk, seed=Sq + Sk + int(causal) + D, D=D)
    scale = 1.0 / math.sqrt(D)
    o, lse = _run(q, k, v, scale, causal, layout=layout, kernel=kernel)
    o_ref, l_ref, a_ref, vmax = _oracle(q, k, v, scale, causal)
    check_fp8(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, a_ref, vmax,
              f"fp8 {shape} causal={causal} layout={layout}")


@KERNELS
@LAYOUTS
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("kv", [[0, 1], [16, 143], [128, 129], [255, 256]])
def test_fp8_key_lengths(kv, layout, D, kernel):
    q, k, v = _inputs(2, 2, 200, 256, seed=sum(kv) + D, D=D)
    o, lse = _run(q, k, v, 0.09, kv=kv, layout=layout, kernel=kernel)
    o_ref, l_ref, a_ref, vmax = _oracle(q, k, v, 0.09, kv=kv)
    check_fp8(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, a_ref, vmax, f"fp8 kv={kv} layout={layout}")


@KERNELS
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("shape", [(1, 1, 1, 1), (1, 2, 100, 100), (2, 1, 300, 333), (1, 2, 129, 1000)])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_v_rows_any_key_count(shape, causal, D, kernel):
    """V in rows has no key-count restriction (the transposed layout needs a
    multiple of 16): ragged key counts against the oracle."""
    B, H, Sq, Sk = shape
    q, k, v = _inputs(B, H, Sq, Sk, seed=Sq * 3 + Sk + int(causal) + D, D=D)
    scale = 1.0 / math.sqrt(D)
    o, lse = _run(q, k, v, scale, causal, layout=ROWS, kernel=kernel)
    o_ref, l_ref, a_ref, vmax = _oracle(q, k, v, scale, causal)
    check_fp8(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, a_ref, vmax, f"fp8 rows {shape}")


@KERNELS
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("shape", [(1, 2, 100, 144), (2, 2, 300, 1024), (1, 4, 1000, 2048)])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_v_layouts_bitwise_identical(shape, causal, D, kernel):
    """The two V layouts feed the products the same values in the same order:
    identical bits (on either kernel)."""
    B, H, Sq, Sk = shape
    q, k, v = _inputs(B, H, Sq, Sk, seed=Sq + 7 * Sk + int(causal), std=2.0, D=D)
    o_r, l_r = _run(q, k, v, 0.07, causal, layout=ROWS, kernel=kernel)
    o_t, l_t = _run(q, k, v, 0.07, causal, layout=TRANSPOSED, kernel=kernel)
    assert torch.equal(o_r.view(torch.int16), o_t.view(torch.int16))
    assert torch.equal(l_r.view(torch.int32), l_t.view(torch.int32))


@KERNELS
def test_fp8_descales_and_large_scores(kernel):
    # std 4 inputs (scores std about 16 after scaling by q and k descales) move the max often
    q, k, v = _inputs(1, 2, 256, 512, seed=41, std=4.0)
    for layout in (ROWS, TRANSPOSED):
        o, lse = _run(q, k, v, 0.05, qd=0.5, kd=2.0, vd=0.25, layout=layout, kernel=kernel)
        o_ref, l_ref, a_ref, vmax = _oracle(q, k, v, 0.05, qd=0.5, kd=2.0, vd=0.25)
        check_fp8(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, a_ref, vmax, f"fp8 descales {layout}")


@KERNELS
def test_fp8_descale_laws_bitwise(kernel):
    q, k, v = _inputs(1, 2, 256, 512, seed=43)
    o1, l1 = _run(q, k, v, 0.1, kernel=kernel)
    o2, l2 = _run(q, k, v, 0.1, vd=2.0, kernel=kernel)  # V descale: O doubles exactly, LSE unchanged
    assert torch.equal(o2.view(torch.int16), (2 * o1).view(torch.int16))
    assert torch.equal(l2, l1)
    o3, l3 = _run(q, k, v, 0.05, qd=2.0, kernel=kernel)  # only scale * q_descale * k_descale matters
    o4, l4 = _run(q, k, v, 0.2, kd=0.5, kernel=kernel)
    for o, l in ((o3, l3), (o4, l4)):
        assert torch.equal(o.view(torch.int16), o1.view(torch.int16))
        assert torch.equal(l, l1)


@KERNELS
def test_fp8_negative_scale(kernel):
    q, k, v = _inputs(1, 1, 130, 160, seed=47)
    o, lse = _run(q, k, v, -0.1, kernel=kernel)
    o_ref, l_ref, a_ref, vmax = _oracle(q, k, v, -0.1)
    check_fp8(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, a_ref, vmax, "fp8 negative scale")


@pytest.mark.parametrize("name", sorted(workloads.FP8_WORKLOADS))
def test_fp8_workload_every_tile(name):
    """The benchmarked FP8 workload at full size, in the benchmark's launch
    configuration, into NaN-filled outputs: no NaN may survive, and the first,
    last and one random row of every (batch entry, head, 128-row query tile)
    must match the oracle."""
    w = workloads.FP8_WORKLOADS[name]
    q, k, v, vt, kv = workloads.generate_fp8(w)
    dev = torch.device("cuda:0")
    o = nan_filled((w.B, w.H, w.Sq, w.D), torch.bfloat16, dev)
    lse = nan_filled((w.B, w.H, w.Sq), torch.float32, dev)
    layout = ROWS if w.v_layout == "rows" else TRANSPOSED
    attn.forward_fp8(q.to(dev), k.to(dev), (v if layout == ROWS else vt).to(dev), w.descale, w.descale, w.descale,
                     scale=w.scale, causal=w.causal, out=o, lse=lse, v_layout=layout)
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    assert_no_nan(o, lse, what=name)
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    rng = np.random.default_rng(7)
    for b in range(w.B):
        for h in range(w.H):
            rows = tile_rows(w.Sq, rng)
            qh, kh, vh = (decode_e4m3(t[b, h].numpy()) * w.descale for t in (q, k, v))
            o_ref, l_ref = attention_rows(qh, kh, vh, rows, w.scale, causal=w.causal)
            a_ref, _ = attention_rows(qh, kh, np.abs(vh), rows, w.scale, causal=w.causal)
            check_fp8(o[b, h, rows], lse[b, h, rows], o_ref, l_ref, a_ref, float(np.abs(vh).max()),
                      f"{name} b{b} h{h}")


@LAYOUTS
def test_fp8_repeated_launches_are_bitwise_identical(layout):
    q, k, v = _inputs(2, 8, 1024, 4096, seed=53)
    dev = torch.device("cuda:0")
    qd, kd = q.to(dev), k.to(dev)
    vd = (v if layout == ROWS else v.transpose(-1, -2).contiguous()).to(dev)
    outs = [attn.forward_fp8(qd, kd, vd, causal=True, v_layout=layout) for _ in range(30)]
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    for o, lse in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(lse, outs[0][1])
