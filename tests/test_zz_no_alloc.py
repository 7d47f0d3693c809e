"""attn_fwd_splitkv_noalloc: the split-KV forward on the library's fixed
device scratch, for callers that cannot allocate device memory (a plugin in
a framework that owns all device memory, a serving loop under a fixed
budget, code that must not risk the synchronisation of cudaMalloc/cudaFree)
and so cannot hand over a workspace either.

This file is named to be collected last: if the entry point fails, a run that
stops at the first failure has already run every other test.  Its GPU tests
pass in a fresh process too: the first call in the process loads the module
and with it the static scratch."""

import math
import os
import re

import pytest
import torch

from exact_attention_86_gb300 import attn
from exact_attention_86_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_m = re.search(r"#define ATTN_SPLITKV_SCRATCH_BYTES \((\d+)u << (\d+)\)",
               open(os.path.join(ROOT, "include", "attn.h")).read())
SCRATCH = int(_m.group(1)) << int(_m.group(2))
A = 1 << 20  # a 16-byte-aligned dummy address: argument checks never dereference it


@pytest.fixture(scope="module")
def lib():
    build()
    return attn.lib()


def _call(B, H, Sq, Sk, D, ns, q=A, stream=None):
    return attn.attn_fwd_splitkv_noalloc(q, A, A, A, A, B, H, Sq, Sk, D, 0.1, 0, None, ns, stream)


def test_scratch_size_is_what_the_header_says():
    assert SCRATCH == 32 << 20


# Every call below with dummy addresses must end in a host-side check: a call
# that passed them all would launch on a machine with a GPU.

def test_oversize_is_rejected_before_any_cuda_call(lib):
    # 16 ranges x B*H*Sq rows x (D + 1) fp32 values: the first shape above the scratch
    B, H, D, ns = 1, 8, 128, 16
    Sq = 128
    while attn.attn_fwd_splitkv_workspace_size(B, H, Sq, D, ns) <= SCRATCH:
        Sq += 128
    assert attn.attn_fwd_splitkv_workspace_size(B, H, Sq - 128, D, ns) <= SCRATCH
    assert _call(B, H, Sq, 4096, D, ns) == attn.ATTN_ERR_WORKSPACE
    assert _call(2, H, Sq, 4096, D, ns) == attn.ATTN_ERR_WORKSPACE


def test_argument_checks(lib):
    assert _call(1, 8, 128, 4096, 100, 4) == attn.ATTN_ERR_UNSUPPORTED_D
    assert _call(1, 8, 128, 4096, 128, 0) == attn.ATTN_ERR_SHAPE
    assert _call(1, 8, 128, 4096, 128, 4, q=A + 8) == attn.ATTN_ERR_ALIGN
    assert _call(0, 8, 128, 4096, 128, 4) == attn.ATTN_OK


def _noalloc(q, k, v, o, lse, ns, causal, kv):
    B, H, Sq, D = q.shape
    st = attn.attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                       B, H, Sq, k.shape[2], D, 1.0 / math.sqrt(D), int(causal),
                                       None if kv is None else kv.data_ptr(), ns,
                                       torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, st


# (B, H, Sq, Sk, D, num_splits, causal, kv_lens): the decode-like shape the
# split path is for, causal, a padded batch with an empty sequence, D = 64
CASES = [
    (1, 8, 128, 32768, 128, 16, False, None),
    (2, 4, 300, 2000, 128, 7, True, None),
    (3, 2, 256, 1500, 128, 5, False, [1500, 0, 777]),
    (2, 3, 200, 3000, 64, 9, True, [0, 2900]),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", range(len(CASES)))
def test_noalloc_equals_workspace_split_and_allocates_nothing(lib, case):
    """Two calls in a row of the no-allocation entry point give exactly the
    bits of attn_fwd_splitkv with a caller workspace, and device memory stays
    as it was."""
    B, H, Sq, Sk, D, ns, causal, kvl = CASES[case]
    assert attn.attn_fwd_splitkv_workspace_size(B, H, Sq, D, ns) <= SCRATCH
    g = torch.Generator().manual_seed(31 + case)
    dev = torch.device("cuda:0")
    q, k, v = (torch.randn(B, H, n, D, generator=g).to(torch.bfloat16).to(dev) for n in (Sq, Sk, Sk))
    kv = None if kvl is None else torch.tensor(kvl, dtype=torch.int32, device=dev)
    o_ws, l_ws = attn.forward_splitkv(q, k, v, ns, causal=causal, kv_lens=kv)
    outs = [(torch.full_like(q, float("nan")), torch.full((B, H, Sq), float("nan"), device=dev)) for _ in range(2)]
    _noalloc(q, k, v, *outs[0], ns, causal, kv)  # the first call may load the module (and the scratch)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    _noalloc(q, k, v, *outs[1], ns, causal, kv)
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0 and torch.cuda.memory_allocated() == alloc0
    for o, lse in outs:
        assert torch.equal(o.view(torch.int16), o_ws.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), l_ws.view(torch.int32))


@pytest.mark.gpu
def test_noalloc_larger_then_smaller_call_leaves_nothing_stale(lib):
    """A call that fills much of the scratch, then a smaller one of another
    shape: the second result must not pick up anything the first left in the
    shared scratch."""
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(77)
    qb = torch.randn(1, 8, 512, 128, generator=g).to(torch.bfloat16).to(dev)
    kb, vb = (torch.randn(1, 8, 4096, 128, generator=g).to(torch.bfloat16).to(dev) for _ in range(2))
    qs = torch.randn(1, 3, 130, 64, generator=g).to(torch.bfloat16).to(dev)
    ks, vs = (torch.randn(1, 3, 900, 64, generator=g).to(torch.bfloat16).to(dev) for _ in range(2))
    assert 16 << 20 < attn.attn_fwd_splitkv_workspace_size(1, 8, 512, 128, 12) <= SCRATCH
    ob, lb = torch.empty_like(qb), torch.empty(1, 8, 512, device=dev)
    os_, ls = torch.full_like(qs, float("nan")), torch.full((1, 3, 130), float("nan"), device=dev)
    _noalloc(qb, kb, vb, ob, lb, 12, False, None)
    _noalloc(qs, ks, vs, os_, ls, 5, True, None)
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    o_ref, l_ref = attn.forward_splitkv(qs, ks, vs, 5, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(os_.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(ls.view(torch.int32), l_ref.view(torch.int32))


@pytest.mark.gpu
def test_noalloc_oversize_writes_nothing(lib):
    B, H, D, ns = 1, 8, 128, 16
    Sq = 128
    while attn.attn_fwd_splitkv_workspace_size(B, H, Sq, D, ns) <= SCRATCH:
        Sq += 128
    dev = torch.device("cuda:0")
    q = torch.zeros(B, H, Sq, D, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(B, H, 256, D, dtype=torch.bfloat16, device=dev)
    o = torch.full_like(q, 3.0)
    lse = torch.full((B, H, Sq), 7.0, device=dev)
    st = attn.attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), k.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H,
                                       Sq, 256, D, 0.1, 0, None, ns, torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((o == 3.0).all()) and bool((lse == 7.0).all())
