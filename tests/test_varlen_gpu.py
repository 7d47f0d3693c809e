"""GPU parity of the packed variable-length forward against the fp64 oracle."""

import math

import numpy as np
import pytest
import torch

from exact_attention_86_gb300 import attn
from exact_attention_86_gb300.build import build
from oracle import attention_ref, attention_varlen_ref

from parity import assert_no_nan, check, nan_filled, tile_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    attn.lib()


def _packed(lens_q, lens_k, H, D, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    tq, tk = int(sum(lens_q)), int(sum(lens_k))
    q = (torch.randn(tq, H, D, generator=g) * std).to(torch.bfloat16)
    k = (torch.randn(tk, H, D, generator=g) * std).to(torch.bfloat16)
    v = (torch.randn(tk, H, D, generator=g) * std).to(torch.bfloat16)
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32)
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32)
    return q, k, v, cu_q, cu_k


def _np(t):
    return t.float().numpy().astype(np.float64)


KERNELS = pytest.mark.parametrize("kernel", [attn.ATTN_KERNEL_ONE_TILE, attn.ATTN_KERNEL_TWO_TILE],
                                  ids=["one", "two"])


def _run(q, k, v, cu_q, cu_k, max_q, scale, causal, kernel=attn.ATTN_KERNEL_AUTO):
    dev = torch.device("cuda:0")
    o, lse = attn.forward_varlen(q.to(dev), k.to(dev), v.to(dev), cu_q.to(dev), cu_k.to(dev), max_q,
                                 scale=scale, causal=causal, kernel=kernel)
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    return o.float().cpu().numpy(), lse.cpu().numpy()


CASES = [
    # lens_q, lens_k
    ([300, 1, 128, 129, 0, 500], [300, 1, 128, 129, 7, 500]),   # self-attention lengths (one empty query set)
    ([127, 64, 260], [400, 0, 200]),                            # Sq != Sk per sequence, one sequence without keys
    ([1, 1, 1, 1], [1000, 5, 130, 256]),                        # decode-like: one query per sequence
]


@KERNELS
@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_varlen_matches_oracle(case, causal, D, kernel):
    lens_q, lens_k = CASES[case]
    H = 3
    q, k, v, cu_q, cu_k = _packed(lens_q, lens_k, H, D, seed=case * 7 + D + int(causal))
    scale = 1.0 / math.sqrt(D)
    o, lse = _run(q, k, v, cu_q, cu_k, max(lens_q), scale, causal, kernel)
    o_ref, l_ref = attention_varlen_ref(_np(q), _np(k), _np(v), cu_q.numpy(), cu_k.numpy(), scale, causal=causal)
    # O [total_q, H, D] against LSE [H, total_q]: compare head-major
    check(o.transpose(1, 0, 2), lse, o_ref.transpose(1, 0, 2), l_ref, f"varlen case {case} causal={causal} D={D}")


@KERNELS
def test_varlen_guard_rows_untouched(kernel):
    # query tiles that run past a sequence end must not write the next sequence's rows,
    # and nothing past total_q may be written
    lens = [130, 3, 250]
    H, D = 2, 128
    q, k, v, cu_q, cu_k = _packed(lens, lens, H, D, seed=3)
    dev = torch.device("cuda:0")
    tq = sum(lens)
    pad = 4 * H * D
    o_buf = torch.full((tq * H * D + pad,), 777, dtype=torch.int16, device=dev)
    l_buf = torch.full((H * tq + 64,), 5.5, dtype=torch.float32, device=dev)
    o_view = o_buf[:tq * H * D].view(torch.bfloat16).view(tq, H, D)
    l_view = l_buf[:H * tq].view(H, tq)
    qd, kd, vd, cqd, ckd = (t.to(dev) for t in (q, k, v, cu_q, cu_k))  # keep alive across the async call
    st = attn.attn_fwd_varlen_variant(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o_view.data_ptr(),
                                      l_view.data_ptr(), cqd.data_ptr(), ckd.data_ptr(), 3, 250, tq, tq, H, D,
                                      1 / math.sqrt(D), 1, None, kernel, torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK
    torch.cuda.synchronize()
    assert torch.all(o_buf[tq * H * D:] == 777) and torch.all(l_buf[H * tq:] == 5.5)
    o_ref, l_ref = attention_varlen_ref(_np(q), _np(k), _np(v), cu_q.numpy(), cu_k.numpy(), 1 / math.sqrt(D),
                                        causal=True)
    check(o_view.float().cpu().numpy().transpose(1, 0, 2), l_view.cpu().numpy(), o_ref.transpose(1, 0, 2), l_ref,
          "varlen guard")


@KERNELS
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_batch_without_any_key(kernel, causal):
    """total_k = 0: no K or V tensor is read (the key maps are never
    dereferenced) and every row gives exactly O = +0, LSE = -inf."""
    lens_q = [130, 5, 300]
    H, D = 2, 128
    q, _, _, cu_q, _ = _packed(lens_q, [1, 1, 1], H, D, seed=29)
    dev = torch.device("cuda:0")
    k = torch.empty(0, H, D, dtype=torch.bfloat16, device=dev)
    v = torch.empty(0, H, D, dtype=torch.bfloat16, device=dev)
    cu_k = torch.zeros(len(lens_q) + 1, dtype=torch.int32, device=dev)
    o, lse = attn.forward_varlen(q.to(dev), k, v, cu_q.to(dev), cu_k, max(lens_q), causal=causal, kernel=kernel)
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    assert torch.all(o.view(torch.int16) == 0)
    assert torch.all(lse == float("-inf"))


@KERNELS
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("max_q", [100, 300, 1000])
def test_varlen_max_seqlen_q_bounds_the_computed_rows(kernel, causal, max_q):
    """max_seqlen_q sizes the launch.  Above the longest sequence the extra
    units are empty; below a sequence's length the rows of the units it
    covers (128 rows a unit on the one-tile kernel, 256 on the two-tile
    kernel) are computed and every later row of O and LSE is left as it was."""
    lens = [600, 50, 257]
    H, D = 2, 64
    q, k, v, cu_q, cu_k = _packed(lens, lens, H, D, seed=17 + max_q + int(causal))
    unit = 128 if kernel == attn.ATTN_KERNEL_ONE_TILE else 256
    covered = -(-max_q // unit) * unit
    dev = torch.device("cuda:0")
    tq = sum(lens)
    o_buf = torch.full((tq, H, D), 777, dtype=torch.int16, device=dev)
    l_buf = torch.full((H, tq), 5.5, dtype=torch.float32, device=dev)
    qd, kd, vd, cqd, ckd = (t.to(dev) for t in (q, k, v, cu_q, cu_k))  # keep alive across the async call
    st = attn.attn_fwd_varlen_variant(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o_buf.data_ptr(),
                                      l_buf.data_ptr(), cqd.data_ptr(), ckd.data_ptr(), len(lens), max_q, tq, tq, H,
                                      D, 1 / math.sqrt(D), int(causal), None, kernel,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    pos = np.concatenate([np.arange(n) for n in lens])  # row of each token within its sequence
    done = pos < covered
    o_raw = o_buf.cpu()
    assert torch.all(o_raw[torch.from_numpy(~done)] == 777)
    assert torch.all(l_buf.cpu()[:, torch.from_numpy(~done)] == 5.5)
    o_ref, l_ref = attention_varlen_ref(_np(q), _np(k), _np(v), cu_q.numpy(), cu_k.numpy(), 1 / math.sqrt(D),
                                        causal=causal)
    o = o_raw.view(torch.bfloat16).float().numpy()
    check(o[done].transpose(1, 0, 2), l_buf.cpu().numpy()[:, done], o_ref[done].transpose(1, 0, 2),
          l_ref[:, done], f"varlen max_seqlen_q={max_q}")


@KERNELS
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equals_padded_forward_for_equal_lengths(kernel, causal):
    """Equal lengths on the same kernel: the packed forward reads the same
    tiles and does the same arithmetic as the padded one, so the bits agree;
    both match the oracle."""
    B, H, S, D = 2, 4, 384, 128
    g = torch.Generator().manual_seed(11)
    q = torch.randn(B, H, S, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, H, S, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, H, S, D, generator=g).to(torch.bfloat16)
    dev = torch.device("cuda:0")
    o_pad, l_pad = attn.forward(q.to(dev), k.to(dev), v.to(dev), causal=causal, kernel=kernel)
    pack = lambda t: t.permute(0, 2, 1, 3).reshape(B * S, H, D).contiguous().to(dev)  # noqa: E731
    cu = torch.arange(0, (B + 1) * S, S, dtype=torch.int32, device=dev)
    o_var, l_var = attn.forward_varlen(pack(q), pack(k), pack(v), cu, cu, S, causal=causal, kernel=kernel)
    torch.cuda.synchronize()
    o_var_p = o_var.view(B, S, H, D).permute(0, 2, 1, 3)
    l_var_p = l_var.view(H, B, S).permute(1, 0, 2)
    assert torch.equal(o_var_p.contiguous().view(torch.int16), o_pad.view(torch.int16))
    assert torch.equal(l_var_p.contiguous(), l_pad)
    o_ref, l_ref = attention_ref(_np(q), _np(k), _np(v), 1 / math.sqrt(D), causal=causal)
    check(o_pad.float().cpu().numpy(), l_pad.cpu().numpy(), o_ref, l_ref, "padded")
    assert float((o_var.float() - pack(o_pad).float()).abs().max()) <= 1e-2
    assert float((l_var - l_pad.permute(1, 0, 2).reshape(H, B * S)).abs().max()) <= 1e-5


@KERNELS
@pytest.mark.parametrize("name", ["varlen_b32_d128_causal", "varlen_b32_d128"])
def test_varlen_benchmark_workload_every_tile(name, kernel):
    """The benchmarked packed batch at full size, in the benchmark's launch
    configuration (dynamic schedule for the non-causal batch), into NaN-filled
    outputs: no NaN may survive, and the first, last and one random row of
    every (sequence, head, 128-row query tile) must match the oracle."""
    from exact_attention_86_gb300 import workloads
    from oracle import attention_rows

    w = workloads.VARLEN_WORKLOADS[name]
    q, k, v, cu = workloads.generate_varlen(w)
    dev = torch.device("cuda:0")
    total = q.shape[0]
    o = nan_filled((total, w.H, w.D), torch.bfloat16, dev)
    lse = nan_filled((w.H, total), torch.float32, dev)
    cud = cu.to(dev)
    attn.forward_varlen(q.to(dev), k.to(dev), v.to(dev), cud, cud, w.max_len, scale=w.scale, causal=w.causal,
                        out=o, lse=lse, kernel=kernel)
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    assert_no_nan(o, lse, what=name)
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    rng = np.random.default_rng(5)
    for b in range(w.batch):
        a, e = int(cu[b]), int(cu[b + 1])
        if e == a:
            continue
        for h in range(w.H):
            rows = tile_rows(e - a, rng)
            o_ref, l_ref = attention_rows(_np(q[a:e, h]), _np(k[a:e, h]), _np(v[a:e, h]), rows, w.scale,
                                          causal=w.causal)
            check(o[a:e, h][rows], lse[h, a:e][rows], o_ref, l_ref, f"{name} seq {b} head {h}")


def test_varlen_repeated_launches_are_bitwise_identical():
    """50 back-to-back launches of the benchmarked causal packed batch: every
    launch must give the same bits and no wait may give up."""
    from exact_attention_86_gb300 import workloads

    w = workloads.VARLEN_WORKLOADS["varlen_b32_d128_causal"]
    q, k, v, cu = workloads.generate_varlen(w)
    dev = torch.device("cuda:0")
    qd, kd, vd, cud = q.to(dev), k.to(dev), v.to(dev), cu.to(dev)
    o0, l0 = attn.forward_varlen(qd, kd, vd, cud, cud, w.max_len, causal=True)
    outs = [attn.forward_varlen(qd, kd, vd, cud, cud, w.max_len, causal=True) for _ in range(49)]
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    for i, (o, lse) in enumerate(outs, 1):
        assert torch.equal(o.view(torch.int16), o0.view(torch.int16)), f"launch {i} differs"
        assert torch.equal(lse, l0), f"launch {i} LSE differs"


@KERNELS
@pytest.mark.parametrize("name", ["varlen_b32_d128_causal", "varlen_b32_d128"])
def test_varlen_dynamic_and_static_scheduling_agree_bitwise(name, kernel):
    """The claimed (dynamic) and dealt (static) schedules run the same units
    with the same arithmetic: identical bits; the counter is zero afterwards
    (on either kernel)."""
    from exact_attention_86_gb300 import workloads

    w = workloads.VARLEN_WORKLOADS[name]
    q, k, v, cu = workloads.generate_varlen(w)
    dev = torch.device("cuda:0")
    qd, kd, vd, cud = q.to(dev), k.to(dev), v.to(dev), cu.to(dev)
    o_s, l_s = attn.forward_varlen(qd, kd, vd, cud, cud, w.max_len, causal=w.causal, dynamic=False, kernel=kernel)
    runs = [attn.forward_varlen(qd, kd, vd, cud, cud, w.max_len, causal=w.causal, dynamic=True, kernel=kernel)
            for _ in range(5)]
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    for o_d, l_d in runs:
        assert torch.equal(o_d.view(torch.int16), o_s.view(torch.int16))
        assert torch.equal(l_d, l_s)
    counter = attn.tile_counter(dev, torch.cuda.current_stream().cuda_stream)
    assert counter.tolist() == [0, 0]
