"""GPU parity of the paged-KV forward against the fp64 oracle."""

import math

import numpy as np
import pytest
import torch

from exact_attention_86_gb300 import attn
from exact_attention_86_gb300.build import build
from oracle import attention_paged_ref

from parity import assert_no_nan, check, nan_filled

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    attn.lib()


def _paged_case(lens_q, lens_k, H, D, page_size, seed, spare_pages=3):
    """Random cache with shuffled pages.  Pages no sequence uses, and every
    64-key half of a last page that lies wholly past the sequence's keys, hold
    NaN: the kernel must never read them."""
    g = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    pages_per = [(n + page_size - 1) // page_size for n in lens_k]
    used = int(sum(pages_per))
    num_pages = used + spare_pages
    max_pages = max(max(pages_per), 1) + 1
    perm = rng.permutation(num_pages)
    table = np.full((len(lens_k), max_pages), -1, dtype=np.int32)
    at = 0
    for b, n in enumerate(pages_per):
        table[b, :n] = perm[at:at + n]
        at += n
    kc = torch.randn(num_pages, page_size, H, D, generator=g)
    vc = torch.randn(num_pages, page_size, H, D, generator=g)
    nan_mask = torch.ones(num_pages, page_size, dtype=torch.bool)
    for b, n in enumerate(lens_k):
        for j in range(0, n, 64):                      # halves that hold a valid key
            pg = table[b, j // page_size]
            nan_mask[pg, j % page_size:j % page_size + 64] = False
    kc[nan_mask] = float("nan")
    vc[nan_mask] = float("nan")
    kc, vc = kc.to(torch.bfloat16), vc.to(torch.bfloat16)
    tq = int(sum(lens_q))
    q = torch.randn(tq, H, D, generator=g).to(torch.bfloat16)
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32)
    seqlens_k = torch.tensor(lens_k, dtype=torch.int32)
    return q, kc, vc, cu_q, seqlens_k, torch.from_numpy(table)


def _np(t):
    return t.float().numpy().astype(np.float64)


KERNELS = pytest.mark.parametrize("kernel", [attn.ATTN_KERNEL_ONE_TILE, attn.ATTN_KERNEL_TWO_TILE],
                                  ids=["one", "two"])


def _run(q, kc, vc, cu_q, sk, table, max_q, scale, causal, kernel=attn.ATTN_KERNEL_AUTO):
    dev = torch.device("cuda:0")
    o, lse = attn.forward_paged(q.to(dev), kc.to(dev), vc.to(dev), cu_q.to(dev), sk.to(dev), table.to(dev), max_q,
                                scale=scale, causal=causal, kernel=kernel)
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    return o.float().cpu().numpy(), lse.cpu().numpy()


CASES = [
    # lens_q, lens_k
    ([300, 1, 128, 129, 0, 64], [300, 1, 128, 129, 7, 65]),    # prefill-like, one empty query set
    ([1, 1, 1, 1, 1], [1000, 0, 63, 64, 257]),                  # decode: one query per sequence
    ([200, 70], [450, 130]),                                    # Sq != Sk per sequence
]


@KERNELS
@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("page_size", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_paged_matches_oracle(case, page_size, causal, D, kernel):
    lens_q, lens_k = CASES[case]
    H = 2
    q, kc, vc, cu_q, sk, table = _paged_case(lens_q, lens_k, H, D, page_size, seed=case * 13 + page_size + D)
    scale = 1.0 / math.sqrt(D)
    o, lse = _run(q, kc, vc, cu_q, sk, table, max(lens_q), scale, causal, kernel)
    o_ref, l_ref = attention_paged_ref(_np(q), _np(kc), _np(vc), cu_q.numpy(), sk.numpy(), table.numpy(), scale,
                                       causal=causal)
    check(o.transpose(1, 0, 2), lse, o_ref.transpose(1, 0, 2), l_ref,
          f"paged case {case} page {page_size} causal={causal} D={D}")


@KERNELS
def test_paged_in_order_pages_equal_varlen_bitwise(kernel):
    """Pages laid out in sequence order turn the cache into the packed keys:
    the paged and variable-length forwards then compute identical bits (on
    the same kernel)."""
    H, D, ps = 4, 128, 128
    lens = [384, 256, 512]
    g = torch.Generator().manual_seed(21)
    dev = torch.device("cuda:0")
    total = sum(lens)
    q = torch.randn(total, H, D, generator=g).to(torch.bfloat16).to(dev)
    k = torch.randn(total, H, D, generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn(total, H, D, generator=g).to(torch.bfloat16).to(dev)
    cu = torch.tensor([0, 384, 640, 1152], dtype=torch.int32, device=dev)
    table = torch.tensor([[0, 1, 2, 0], [3, 4, 0, 0], [5, 6, 7, 8]], dtype=torch.int32, device=dev)
    sk = torch.tensor(lens, dtype=torch.int32, device=dev)
    o_v, l_v = attn.forward_varlen(q, k, v, cu, cu, max(lens), causal=True, kernel=kernel)
    o_p, l_p = attn.forward_paged(q, k.view(total // ps, ps, H, D), v.view(total // ps, ps, H, D), cu, sk, table,
                                  max(lens), causal=True, kernel=kernel)
    torch.cuda.synchronize()
    assert torch.equal(o_v.view(torch.int16), o_p.view(torch.int16))
    assert torch.equal(l_v, l_p)


@KERNELS
def test_paged_benchmark_workload_equals_varlen_bitwise(kernel):
    """The benchmarked paged batch at full size, in the benchmark's launch
    configuration: the shuffled pages hold the same tokens as the packed batch
    (whose parity against the oracle is tested at full size), and the kernel
    stages the same tiles either way, so the bits must agree.  Both outputs
    are NaN-filled before the calls."""
    from exact_attention_86_gb300 import workloads

    w = workloads.PAGED_WORKLOADS["paged_b32_d128_causal"]
    q, kc, vc, cu, sk, table = workloads.generate_paged(w)
    _, k, v, cu2 = workloads.generate_varlen(w)
    assert torch.equal(cu, cu2)
    dev = torch.device("cuda:0")
    qd, cud = q.to(dev), cu.to(dev)
    total = q.shape[0]
    # both outputs start as NaN, so an element that either schedule leaves
    # unwritten cannot compare equal to a stale value
    o_p, o_v = (nan_filled((total, w.H, w.D), torch.bfloat16, dev) for _ in range(2))
    l_p, l_v = (nan_filled((w.H, total), torch.float32, dev) for _ in range(2))
    attn.forward_paged(qd, kc.to(dev), vc.to(dev), cud, sk.to(dev), table.to(dev), w.max_len, causal=w.causal,
                       out=o_p, lse=l_p, kernel=kernel)
    attn.forward_varlen(qd, k.to(dev), v.to(dev), cud, cud, w.max_len, causal=w.causal, out=o_v, lse=l_v,
                        kernel=kernel)
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    assert_no_nan(o_p, l_p, what="paged")
    assert_no_nan(o_v, l_v, what="packed")
    assert torch.equal(o_p.view(torch.int16), o_v.view(torch.int16))
    assert torch.equal(l_p, l_v)


@KERNELS
def test_paged_dynamic_and_static_scheduling_agree_bitwise(kernel):
    from exact_attention_86_gb300 import workloads

    w = workloads.PAGED_WORKLOADS["paged_b32_d128_causal"]
    q, kc, vc, cu, sk, table = workloads.generate_paged(w)
    dev = torch.device("cuda:0")
    args = [t.to(dev) for t in (q, kc, vc, cu, sk, table)]
    o_s, l_s = attn.forward_paged(*args, w.max_len, causal=w.causal, dynamic=False, kernel=kernel)
    o_d, l_d = attn.forward_paged(*args, w.max_len, causal=w.causal, dynamic=True, kernel=kernel)
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    assert torch.equal(o_d.view(torch.int16), o_s.view(torch.int16))
    assert torch.equal(l_d, l_s)
