"""attn_fwd_splitkv_noalloc: the split-KV forward on the library's fixed
device scratch (no allocation, no caller workspace)."""

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


@pytest.mark.gpu
def test_noalloc_equals_workspace_split_and_allocates_nothing(lib):
    B, H, Sq, Sk, D, ns = 1, 8, 128, 32768, 128, 16
    assert attn.attn_fwd_splitkv_workspace_size(B, H, Sq, D, ns) <= SCRATCH
    g = torch.Generator().manual_seed(31)
    dev = torch.device("cuda:0")
    q, k, v = (torch.randn(B, H, n, D, generator=g).to(torch.bfloat16).to(dev) for n in (Sq, Sk, Sk))
    o_ws, l_ws = attn.forward_splitkv(q, k, v, ns)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, Sq, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    scale = 1.0 / math.sqrt(D)

    def run():
        st = attn.attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                           B, H, Sq, Sk, D, scale, 0, None, ns, stream)
        assert st == attn.ATTN_OK
    run()  # the first call loads the module (and with it the static scratch)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(20):
        run()
    st, site = attn.attn_check_device_status(stream)
    assert st == attn.ATTN_OK, (st, site)
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0 and torch.cuda.memory_allocated() == alloc0
    assert torch.equal(o.view(torch.int16), o_ws.view(torch.int16))
    assert torch.equal(lse, l_ws)


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
