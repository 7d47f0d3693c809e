"""GPU parity of the split-KV forward and of the LSE merge against the fp64 oracle."""

import math

import numpy as np
import pytest
import torch

from exact_attention_86_gb300 import attn
from exact_attention_86_gb300.build import build
from oracle import attention_ref, attention_rows, lse_merge

from parity import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    attn.lib()


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def _inputs(B, H, Sq, Sk, D, seed, kv=None, std=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, H, Sq, D, generator=g) * std).to(torch.bfloat16)
    k = (torch.randn(B, H, Sk, D, generator=g) * std).to(torch.bfloat16)
    v = (torch.randn(B, H, Sk, D, generator=g) * std).to(torch.bfloat16)
    return q, k, v, (None if kv is None else torch.tensor(kv, dtype=torch.int32))


def _run_split(q, k, v, ns, scale, causal, kv):
    dev = torch.device("cuda:0")
    o, lse = attn.forward_splitkv(q.to(dev), k.to(dev), v.to(dev), ns, scale=scale, causal=causal,
                                  kv_lens=None if kv is None else kv.to(dev))
    st, site = attn.attn_check_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, (st, site)
    return o.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("ns", [1, 2, 3, 7, 16])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_splitkv_matches_oracle(ns, causal, D):
    B, H, Sq, Sk = 2, 2, 300, 900
    q, k, v, kv = _inputs(B, H, Sq, Sk, D, seed=ns * 10 + D + int(causal), kv=[900, 333])
    scale = 1.0 / math.sqrt(D)
    o, lse = _run_split(q, k, v, ns, scale, causal, kv)
    o_ref, l_ref = attention_ref(_np(q), _np(k), _np(v), scale, causal=causal, kv_lens=kv.numpy())
    check(o, lse, o_ref, l_ref, f"splitkv ns={ns} causal={causal} D={D}")


def test_splitkv_more_splits_than_tiles_and_empty_rows():
    # 2 key tiles cut 16 ways: most ranges are empty; one sequence has no key.
    q, k, v, kv = _inputs(3, 1, 200, 250, 128, seed=5, kv=[250, 0, 129])
    o, lse = _run_split(q, k, v, 16, 0.09, False, kv)
    o_ref, l_ref = attention_ref(_np(q), _np(k), _np(v), 0.09, kv_lens=kv.numpy())
    check(o, lse, o_ref, l_ref, "splits > tiles")
    assert np.all(o[1] == 0.0) and np.all(lse[1] == -np.inf)


def test_splitkv_agrees_with_unsplit_forward():
    q, k, v, _ = _inputs(1, 4, 256, 2048, 128, seed=9, std=2.0)
    dev = torch.device("cuda:0")
    o1, l1 = attn.forward(q.to(dev), k.to(dev), v.to(dev), causal=True)
    o2, l2 = attn.forward_splitkv(q.to(dev), k.to(dev), v.to(dev), 8, causal=True)
    torch.cuda.synchronize()
    assert torch.allclose(o1.float(), o2.float(), atol=2e-2, rtol=2e-2)
    assert torch.allclose(l1, l2, atol=1e-3, rtol=0)


def test_splitkv_decode_like_long_context():
    # one 128-row query block per head against 32768 keys: split-KV's use case
    B, H, Sq, Sk, D = 1, 8, 128, 32768, 128
    q, k, v, _ = _inputs(B, H, Sq, Sk, D, seed=17)
    scale = 1.0 / math.sqrt(D)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # 16 ranges, and the suggested count (None: within one wave of the SMs)
    for ns in (16, None):
        o, lse = _run_split(q, k, v, ns, scale, False, None)
        if ns is None:
            assert attn.suggest_num_splits(B, H, Sq, Sk, sms) * H <= sms
        rng = np.random.default_rng(17)
        for h in (0, 5):
            rows = sorted(set([0, 1, 64, 127] + [int(x) for x in rng.integers(0, Sq, 8)]))
            o_ref, l_ref = attention_rows(_np(q[0, h]), _np(k[0, h]), _np(v[0, h]), rows, scale)
            check(o[0, h, rows], lse[0, h, rows], o_ref, l_ref, f"decode-like h{h} splits {ns}")


@pytest.mark.parametrize("D", [64, 128])
def test_lse_merge_kernel_against_oracle_partials(D):
    # partial results from the oracle over 4 key ranges (one empty for some rows)
    rng = np.random.default_rng(D)
    rows, n = 77, 4
    o_parts = rng.normal(size=(n, rows, D))
    lse_parts = rng.normal(size=(n, rows)) * 5
    lse_parts[1, :10] = -np.inf
    lse_parts[:, 20] = -np.inf  # a row with no key anywhere
    o_ref, l_ref = lse_merge(o_parts, lse_parts)
    dev = torch.device("cuda:0")
    o, l = attn.lse_merge(torch.tensor(o_parts, dtype=torch.float32, device=dev),
                          torch.tensor(lse_parts, dtype=torch.float32, device=dev))
    torch.cuda.synchronize()
    # the kernel reads fp32 partials: compare with the oracle merge of the same fp32 values
    o_ref32, l_ref32 = lse_merge(o_parts.astype(np.float32), lse_parts.astype(np.float32))
    check(o.float().cpu().numpy(), l.cpu().numpy(), o_ref32, l_ref32, f"merge D={D}")
    assert np.all(o[20].float().cpu().numpy() == 0.0) and l[20].item() == float("-inf")


def test_splitkv_repeated_launches_are_bitwise_identical():
    """200 back-to-back launches at 16 splits on the decode-like shape (an
    HBM-bound loop in which loads land late and out of order): every launch
    must give the same bits and no wait may give up."""
    B, H, Sq, Sk, D = 1, 8, 128, 32768, 128
    q, k, v, _ = _inputs(B, H, Sq, Sk, D, seed=23)
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    ns = 16
    ws = torch.empty(attn.attn_fwd_splitkv_workspace_size(B, H, Sq, D, ns), dtype=torch.uint8, device=dev)
    outs = []
    stream = torch.cuda.current_stream().cuda_stream
    for i in range(200):
        o = torch.empty_like(qd)
        lse = torch.empty(B, H, Sq, dtype=torch.float32, device=dev)
        st = attn.attn_fwd_splitkv(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H,
                                   Sq, Sk, D, 1 / math.sqrt(D), 0, None, ns, ws.data_ptr(), ws.numel(), stream)
        assert st == attn.ATTN_OK
        outs.append((o, lse))
    st, site = attn.attn_check_device_status(stream)
    assert st == attn.ATTN_OK, (st, site)
    o0, l0 = outs[0]
    for i, (o, lse) in enumerate(outs[1:], 1):
        assert torch.equal(o.view(torch.int16), o0.view(torch.int16)), f"launch {i} differs"
        assert torch.equal(lse, l0), f"launch {i} LSE differs"
