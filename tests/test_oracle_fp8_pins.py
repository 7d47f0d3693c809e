"""CPU pins of the FP8 (E4M3) part of the oracle."""

import math

import numpy as np
import pytest
import torch

from oracle import attention_fp8_ref, attention_ref, decode_e4m3

CODES = np.arange(256, dtype=np.uint8)


def test_decode_matches_torch_float8_e4m3fn_for_every_code():
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    want = torch.from_numpy(CODES.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = decode_e4m3(CODES)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x38, 1.0), (0x40, 2.0), (0x3C, 1.5), (0x30, 0.5), (0xB8, -1.0),
    (0x7E, 448.0), (0xFE, -448.0), (0x08, 2.0 ** -6), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9),
    (0x0F, 1.875 * 2.0 ** -6), (0x77, 1.875 * 2.0 ** 7), (0x78, 256.0),
])
def test_decode_closed_forms(code, value):
    assert decode_e4m3(np.array([code], dtype=np.uint8))[0] == value


def test_decode_special_codes_and_order():
    d = decode_e4m3(CODES)
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF]) and np.isnan(d).sum() == 2
    assert d[0x80] == 0.0 and math.copysign(1.0, d[0x80]) == -1.0
    pos = d[:0x7F]
    assert np.all(np.diff(pos) > 0)                      # codes 0..126 strictly increasing
    assert np.array_equal(d[0x80:0xFF], -pos)            # sign bit mirrors
    assert np.all(np.isfinite(d[~np.isnan(d)]))          # no infinities


def _codes(shape, seed, std=1.0):
    # quantise N(0, std^2) draws to E4M3 codes by round-to-nearest on the decoded grid
    grid = decode_e4m3(CODES[:0x7F])
    x = np.random.default_rng(seed).normal(size=shape) * std
    mag = np.minimum(np.abs(x), 448.0)
    idx = np.clip(np.searchsorted(grid, mag), 1, len(grid) - 1)
    lo = grid[idx - 1]
    hi = grid[idx]
    code = np.where(mag - lo <= hi - mag, idx - 1, idx).astype(np.uint8)
    return np.where(x < 0, code | 0x80, code).astype(np.uint8)


def test_fp8_attention_is_attention_of_the_decoded_values():
    B, H, Sq, Sk, D = 2, 2, 5, 9, 4
    q8, k8, v8 = _codes((B, H, Sq, D), 1), _codes((B, H, Sk, D), 2), _codes((B, H, Sk, D), 3)
    for causal in (False, True):
        O, L = attention_fp8_ref(q8, k8, v8, 0.5, 2.0, 0.25, 0.3, causal=causal, kv_lens=[9, 4])
        Ob, Lb = attention_ref(decode_e4m3(q8) * 0.5, decode_e4m3(k8) * 2.0, decode_e4m3(v8) * 0.25, 0.3,
                               causal=causal, kv_lens=[9, 4])
        np.testing.assert_array_equal(O, Ob)
        np.testing.assert_array_equal(L, Lb)


def test_fp8_descale_laws():
    """v_descale scales O and leaves LSE; q and k descales act only through
    their product with scale."""
    B, H, Sq, Sk, D = 1, 2, 6, 7, 8
    q8, k8, v8 = _codes((B, H, Sq, D), 4), _codes((B, H, Sk, D), 5), _codes((B, H, Sk, D), 6)
    O1, L1 = attention_fp8_ref(q8, k8, v8, 1.0, 1.0, 1.0, 0.2)
    O2, L2 = attention_fp8_ref(q8, k8, v8, 1.0, 1.0, 4.0, 0.2)
    np.testing.assert_allclose(O2, 4.0 * O1, rtol=1e-14, atol=0)
    np.testing.assert_array_equal(L2, L1)
    O3, L3 = attention_fp8_ref(q8, k8, v8, 2.0, 0.5, 1.0, 0.2)
    np.testing.assert_allclose(O3, O1, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(L3, L1, rtol=1e-13, atol=1e-15)
    O4, L4 = attention_fp8_ref(q8, k8, v8, 2.0, 1.0, 1.0, 0.1)
    np.testing.assert_allclose(O4, O1, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(L4, L1, rtol=1e-13, atol=1e-15)


def test_fp8_brute_force_small():
    q8, k8, v8 = _codes((1, 1, 3, 2), 7), _codes((1, 1, 4, 2), 8), _codes((1, 1, 4, 2), 9)
    O, L = attention_fp8_ref(q8, k8, v8, 0.5, 1.5, 2.0, 0.7, causal=True)
    q, k, v = decode_e4m3(q8)[0, 0] * 0.5, decode_e4m3(k8)[0, 0] * 1.5, decode_e4m3(v8)[0, 0] * 2.0
    for i in range(3):
        e = [math.exp(0.7 * math.fsum(q[i] * k[j])) for j in range(i + 1)]
        den = math.fsum(e)
        np.testing.assert_allclose(O[0, 0, i], sum(w * v[j] for j, w in enumerate(e)) / den, rtol=1e-12)
        assert abs(L[0, 0, i] - math.log(den)) < 1e-12


FP8_MUTATIONS = {
    "bias_8": ("np.exp2((e - 7).astype(np.float64))", "np.exp2((e - 8).astype(np.float64))"),
    "no_hidden_bit": ("(1.0 + m / 8.0)", "(m / 8.0)"),
    "subnormal_scale": ("(m / 8.0) * 2.0 ** -6", "(m / 8.0) * 2.0 ** -7"),
    "mantissa_4_bits": ("m = (b & 0x7).astype(np.float64)", "m = (b & 0xF).astype(np.float64)"),
    "nan_code_wrong": ("((b & 0x7) == 7)", "((b & 0x7) == 6)"),
    "sign_dropped": ("return sign * val", "return val"),
    "v_descale_dropped": ("decode_e4m3(v8) * vd", "decode_e4m3(v8)"),
}


def _decode_pins_pass(mod) -> bool:
    try:
        d = mod.decode_e4m3(CODES)
        closed = {0x38: 1.0, 0x7E: 448.0, 0x01: 2.0 ** -9, 0x08: 2.0 ** -6, 0xB8: -1.0, 0x3C: 1.5}
        if any(d[c] != v for c, v in closed.items()):
            return False
        if not (np.isnan(d[0x7F]) and np.isnan(d).sum() == 2):
            return False
        q8, k8, v8 = _codes((1, 1, 3, 4), 11), _codes((1, 1, 5, 4), 12), _codes((1, 1, 5, 4), 13)
        O1, _ = mod.attention_fp8_ref(q8, k8, v8, 1.0, 1.0, 1.0, 0.3)
        O2, _ = mod.attention_fp8_ref(q8, k8, v8, 1.0, 1.0, 2.0, 0.3)
        return bool(np.allclose(O2, 2.0 * O1, rtol=1e-14, atol=0))
    except Exception:
        return False


@pytest.mark.parametrize("name", sorted(FP8_MUTATIONS))
def test_fp8_pins_catch_planted_mistake(name):
    import oracle.fp8 as real
    src = open(real.__file__).read().replace("from .attention import attention_ref",
                                             "from oracle.attention import attention_ref")
    assert _decode_pins_pass(_load(src, "real"))
    old, new = FP8_MUTATIONS[name]
    assert src.count(old) == 1, name
    assert not _decode_pins_pass(_load(src.replace(old, new), name)), f"planted mistake {name} went unnoticed"


def _load(src, name):
    import types
    mod = types.ModuleType("oracle_fp8_mutant_" + name)
    exec(compile(src, "<fp8 mutant " + name + ">", "exec"), mod.__dict__)
    return mod
