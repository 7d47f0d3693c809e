"""The benchmark's roofline bound (host logic only)."""

import os
import sys

import pytest

sys.path.insert(0, os.path.join(os.path.dirname(__file__), ".."))
import bench  # noqa: E402
from exact_attention_86_gb300 import workloads  # noqa: E402

PEAK, HBM = 1860.3, 6782.4   # TFLOP/s, GB/s


@pytest.mark.parametrize("name,bound", [
    ("s8192_d128", "tensor"), ("s8192_d128_causal", "tensor"), ("s32768_d128_causal", "tensor"),
    ("s2048_d128_padded", "tensor"), ("q128_k32768_d128", "hbm"), ("s1024_d64_causal", "hbm"),
    ("s128_d64", "hbm"),
])
def test_bound_follows_the_ridge(name, bound):
    w = workloads.WORKLOADS[name]
    r = bench.roofline_bound(w.flops, w.min_bytes, 1.0, PEAK, HBM)
    assert r["bound"] == bound
    assert (r["intensity_flop_per_byte"] >= r["ridge_flop_per_byte"]) == (bound == "tensor")


def test_achieved_and_fraction_in_each_unit():
    # 1 TFLOP and 1 GB in 1 ms: 1000 TFLOP/s, or 1000 GB/s
    t = bench.roofline_bound(1e12, 10**8, 1.0, PEAK, HBM)        # 10^4 FLOP/B: tensor
    assert t["unit"] == "TFLOP/s" and t["achieved"] == pytest.approx(1000.0)
    assert t["frac"] == pytest.approx(1000.0 / PEAK)
    h = bench.roofline_bound(1e9, 10**9, 1.0, PEAK, HBM)         # 1 FLOP/B: HBM
    assert h["unit"] == "GB/s" and h["achieved"] == pytest.approx(1000.0)
    assert h["frac"] == pytest.approx(1000.0 / HBM)


def test_backward_is_taken_as_tensor_bound():
    assert bench.roofline_bound(1e9, 10**9, 1.0, PEAK, HBM, backward=True)["bound"] == "tensor"


# ---------------------------------------------------------- split-KV count
from exact_attention_86_gb300 import attn  # noqa: E402
from exact_attention_86_gb300.build import build  # noqa: E402


@pytest.fixture(scope="module")
def _lib():
    build()   # host-only entry point: the library loads and runs without a GPU
    attn.lib()


@pytest.mark.parametrize("B,H,Sq,Sk,sms,expect", [
    (1, 8, 128, 32768, 152, 16),     # 8 units: at most 19 ranges; 16 cut the 256 tiles evenly
    (1, 8, 128, 128 * 19 * 3, 152, 19),  # 57 tiles: 19 even ranges
    (1, 8, 128, 128 * 37, 152, 19),  # 37 tiles (prime): no even cut near 19, so 19
    (1, 8, 128, 1024, 152, 8),       # capped at one range per 128-key tile
    (2, 16, 8192, 8192, 152, 1),     # 2048 units: no split
    (1, 1, 1, 10**6, 152, 128),      # capped at the entry point's limit
    (1, 152, 128, 4096, 152, 1),     # exactly one wave already
    (0, 8, 128, 4096, 152, 1),       # empty batch
])
def test_suggested_splits(_lib, B, H, Sq, Sk, sms, expect):
    s = attn.suggest_num_splits(B, H, Sq, Sk, sms)
    assert s == expect
    units = B * H * ((Sq + 127) // 128)
    assert 1 <= s <= attn.MAX_SPLITS and (units == 0 or units * s <= max(sms, units))


def test_suggested_splits_rejects_negative_sizes(_lib):
    for args in [(-1, 8, 128, 4096, 152), (1, 8, -1, 4096, 152), (1, 8, 128, -5, 152), (1, 8, 128, 4096, 0)]:
        assert attn.attn_fwd_splitkv_suggest_splits(*args) == 0


def test_suggested_splits_against_a_direct_search(_lib):
    # the rule written as a search: among S <= S_max, the largest even cut
    # unless it is below S_max / 2
    import random
    rng = random.Random(3)
    for _ in range(300):
        B, H, Sq, Sk, sms = rng.randint(1, 3), rng.randint(1, 16), rng.randint(1, 600), rng.randint(1, 70000), \
            rng.choice([132, 148, 152, 160])
        units = B * H * -(-Sq // 128)
        tiles = -(-Sk // 128)
        if units >= sms:
            want = 1
        else:
            s_max = max(1, min(sms // units, tiles, 128))
            even = max(s for s in range(1, s_max + 1) if tiles % s == 0)
            want = even if 2 * even >= s_max else s_max
        assert attn.suggest_num_splits(B, H, Sq, Sk, sms) == want, (B, H, Sq, Sk, sms)


# ------------------------------------------- the kernel a bench line names
@pytest.mark.parametrize("name,kernel", [
    ("s8192_d128", "attn_fwd_pair_kernel"),          # 7 pair waves against 14 single-tile waves
    ("s8192_d128_causal", "attn_fwd_pair_kernel"),
    ("s32768_d128_causal", "attn_fwd_pair_kernel"),
    ("s2048_d128_padded", "attn_fwd_pair_kernel"),
    ("s1024_d64_causal", "attn_fwd_kernel"),         # short causal: single tiles
    ("s128_d64", "attn_fwd_kernel"),                 # one query tile
    ("q128_k32768_d128", "attn_fwd_kernel"),         # one query tile per head
    ("varlen_b32_d128_causal", "attn_fwd_pair_kernel"),
    ("paged_b32_d128_causal", "attn_fwd_pair_kernel"),
    ("s8192_d128_fp8", "attn_fwd_pair_kernel"),
    ("s8192_d128_causal_fp8", "attn_fwd_pair_kernel"),
    ("s8192_d64_fp8", "attn_fwd_pair_kernel"),
])
def test_forward_kernel_names_the_routed_kernel(_lib, name, kernel):
    # the kernel the roofline object attributes its launch time to is the one
    # the library's host-only choice functions route the workload to
    assert bench.forward_kernel(bench.lookup(name), 0, 152) == kernel


def test_split_workloads_run_the_one_tile_kernel(_lib):
    assert bench.forward_kernel(bench.lookup("q128_k32768_d128"), 16, 152) == "attn_fwd_kernel"
    assert bench.forward_kernel(bench.lookup("s8192_d128"), 4, 152) == "attn_fwd_kernel"
