"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, none of which re-types the oracle's own formula.

* the pages' worked example ("Kernel Fusion and the Memory Wall", section
  "A small executable reference"): the tiled online recurrence agrees with the
  materialised softmax to 1e-12;
* normalisation ("Softmax needs a global row statistic": the denominator covers
  the whole row): with V = identity the output IS the probability matrix, whose
  rows sum to 1, whose masked entries are exactly 0 and whose ratios are
  exp(s_ij - s_ik);
* masking (causal with partially masked tiles, rows with no valid key:
  "Kernel Fusion and the Memory Wall", after the executable reference;
  "Attention softmax fusion", "Things that break"): a brute-force scalar triple
  loop on tiny inputs, and closed forms;
* a library routine: torch's float64 scaled_dot_product_attention;
* invariances: key permutation, score shift, query-block size.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention_ref, attention_rows, online_softmax_attention, valid_key_count

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).normal(size=shape) * std


# --------------------------------------------------------------------------
# The pages' worked example
# --------------------------------------------------------------------------

def test_worked_example_online_matches_materialised():
    fx = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    rng = np.random.default_rng(fx["seed"])
    q = rng.normal(size=fx["d"])
    k = rng.normal(size=(fx["n_keys"], fx["d"]))
    v = rng.normal(size=(fx["n_keys"], fx["dv"]))
    scale = 1.0 / math.sqrt(fx["d"])
    o_ref, lse_ref = attention_ref(q[None, None, None, :], k[None, None], v[None, None], scale)
    scores = (k @ q) * scale
    o_onl, m, l = online_softmax_attention(scores, v, fx["tile"])
    np.testing.assert_allclose(o_onl, o_ref[0, 0, 0], rtol=fx["rtol"], atol=fx["atol"])
    # LSE = m + ln(l) from the recurrence's final state
    assert abs((m + math.log(l)) - lse_ref[0, 0, 0]) < 1e-12


@pytest.mark.parametrize("tile", [1, 2, 3, 4, 5, 7, 11, 64])
@pytest.mark.parametrize("seed", [0, 1])
def test_online_matches_materialised_any_tile(tile, seed):
    rng = np.random.default_rng(100 + seed)
    n, d, dv = 29, 8, 5
    q = rng.normal(size=d) * 3.0
    k = rng.normal(size=(n, d))
    v = rng.normal(size=(n, dv))
    scale = 0.7
    o_ref, _ = attention_ref(q[None, None, None, :], k[None, None], v[None, None], scale)
    o_onl, _, _ = online_softmax_attention((k @ q) * scale, v, tile)
    np.testing.assert_allclose(o_onl, o_ref[0, 0, 0], rtol=1e-12, atol=1e-12)


def test_online_with_masked_leading_tiles_has_no_nan():
    rng = np.random.default_rng(5)
    n, dv = 12, 4
    s = rng.normal(size=n)
    s[:6] = -np.inf          # two fully masked tiles of width 3 come first
    v = rng.normal(size=(n, dv))
    o, m, l = online_softmax_attention(s, v, 3)
    assert np.all(np.isfinite(o))
    p = np.exp(s[6:] - s[6:].max())
    np.testing.assert_allclose(o, (p @ v[6:]) / p.sum(), rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# Normalisation: V = identity turns O into the probability matrix
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows(causal):
    B, H, Sq, Sk, D = 2, 1, 9, 13, 6
    q = _rand((B, H, Sq, D), 1)
    k = _rand((B, H, Sk, D), 2)
    eye = np.broadcast_to(np.eye(Sk), (B, H, Sk, Sk)).copy()
    kv = np.array([13, 7])
    scale = 0.4
    P, lse = attention_ref(q, k, eye, scale, causal=causal, kv_lens=kv)
    for b in range(B):
        for i in range(Sq):
            nv = valid_key_count(i, Sk, causal, kv[b])
            row = P[b, 0, i]
            assert np.all(row >= 0)
            assert np.all(row[nv:] == 0.0)                # masked keys get exactly 0
            assert abs(row.sum() - 1.0) < 1e-14           # the denominator covers the whole row
            s = scale * (k[b, 0] @ q[b, 0, i])
            for j in range(1, nv):                         # ratios are exp(s_ij - s_i0)
                assert abs(row[j] / row[0] - math.exp(s[j] - s[0])) < 1e-12 * max(1.0, math.exp(s[j] - s[0]))
            # LSE = ln(sum_j exp(s_ij)) over the valid keys
            assert abs(lse[b, 0, i] - math.log(math.fsum(math.exp(x) for x in s[:nv]))) < 1e-12


# --------------------------------------------------------------------------
# Brute force on tiny inputs (scalar loops, no BLAS, no max subtraction
# needed at these magnitudes)
# --------------------------------------------------------------------------

def _brute(q, k, v, scale, causal, kv_lens):
    B, H, Sq, D = q.shape
    Sk, Dv = k.shape[2], v.shape[3]
    O = np.zeros((B, H, Sq, Dv))
    L = np.full((B, H, Sq), -np.inf)
    for b in range(B):
        for h in range(H):
            for i in range(Sq):
                w = []
                for j in range(Sk):
                    ok = j < min(max(kv_lens[b], 0), Sk) and (not causal or j <= i)
                    if ok:
                        dot = math.fsum(q[b, h, i, d] * k[b, h, j, d] for d in range(D))
                        w.append((j, math.exp(scale * dot)))
                if not w:
                    continue
                den = math.fsum(e for _, e in w)
                for c in range(Dv):
                    O[b, h, i, c] = math.fsum(e * v[b, h, j, c] for j, e in w) / den
                L[b, h, i] = math.log(den)
    return O, L


@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_tiny(causal):
    B, H, Sq, Sk, D, Dv = 3, 2, 5, 6, 4, 3
    q = _rand((B, H, Sq, D), 11)
    k = _rand((B, H, Sk, D), 12)
    v = _rand((B, H, Sk, Dv), 13)
    kv = [6, 3, 0]
    scale = 0.5
    O, L = attention_ref(q, k, v, scale, causal=causal, kv_lens=kv)
    Ob, Lb = _brute(q, k, v, scale, causal, kv)
    np.testing.assert_allclose(O, Ob, rtol=1e-12, atol=1e-13)
    fin = np.isfinite(Lb)
    assert np.array_equal(fin, np.isfinite(L))
    np.testing.assert_allclose(L[fin], Lb[fin], rtol=1e-12, atol=1e-13)


def test_brute_force_causal_sq_ne_sk_top_left():
    # Reading: causal masking is top-left aligned (key j masked when j > i) for any Sq, Sk.
    B, H, Sq, Sk, D = 1, 1, 4, 9, 3
    q = _rand((B, H, Sq, D), 21)
    k = _rand((B, H, Sk, D), 22)
    v = _rand((B, H, Sk, D), 23)
    O, L = attention_ref(q, k, v, 1.0, causal=True)
    Ob, Lb = _brute(q, k, v, 1.0, True, [Sk])
    np.testing.assert_allclose(O, Ob, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L, Lb, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

def test_causal_row0_is_v0():
    B, H, S, D = 2, 3, 17, 8
    q = _rand((B, H, S, D), 31)
    k = _rand((B, H, S, D), 32)
    v = _rand((B, H, S, D), 33)
    scale = 0.35
    O, L = attention_ref(q, k, v, scale, causal=True)
    np.testing.assert_array_equal(O[:, :, 0], v[:, :, 0])  # p_00 = 1 exactly
    expect = scale * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0])
    np.testing.assert_allclose(L[:, :, 0], expect, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_mean_and_log_count(causal):
    B, H, Sq, Sk, D = 2, 2, 7, 10, 5
    q = np.zeros((B, H, Sq, D))
    k = _rand((B, H, Sk, D), 41)
    v = _rand((B, H, Sk, D), 42)
    kv = [10, 4]
    O, L = attention_ref(q, k, v, 1.3, causal=causal, kv_lens=kv)
    for b in range(B):
        for i in range(Sq):
            n = valid_key_count(i, Sk, causal, kv[b])
            np.testing.assert_allclose(O[b, :, i], v[b, :, :n].mean(axis=1), rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(L[b, :, i], math.log(n), rtol=0, atol=1e-14)


def test_kv_len_one_and_zero():
    B, H, Sq, Sk, D = 3, 2, 6, 8, 4
    q = _rand((B, H, Sq, D), 51)
    k = _rand((B, H, Sk, D), 52)
    v = _rand((B, H, Sk, D), 53)
    scale = 0.9
    kv = [1, 0, 8]
    O, L = attention_ref(q, k, v, scale, kv_lens=kv)
    # kv_len = 1: every row attends to key 0 only
    np.testing.assert_array_equal(O[0], np.broadcast_to(v[0, :, :1], O[0].shape))
    np.testing.assert_allclose(L[0], scale * np.einsum("hid,hd->hi", q[0], k[0, :, 0]), rtol=1e-14, atol=1e-14)
    # kv_len = 0: O = +0.0 exactly, LSE = -inf
    assert np.all(O[1] == 0.0) and not np.any(np.signbit(O[1]))
    assert np.all(L[1] == -np.inf)
    assert np.all(np.isfinite(O[2])) and np.all(np.isfinite(L[2]))


def test_kv_len_clamped():
    B, H, Sq, Sk, D = 2, 1, 3, 5, 4
    q = _rand((B, H, Sq, D), 61)
    k = _rand((B, H, Sk, D), 62)
    v = _rand((B, H, Sk, D), 63)
    O1, L1 = attention_ref(q, k, v, 0.5, kv_lens=[99, -4])
    O2, L2 = attention_ref(q, k, v, 0.5, kv_lens=[5, 0])
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)


def test_scale_zero_is_uniform_average():
    B, H, Sq, Sk, D = 1, 2, 5, 7, 3
    q = _rand((B, H, Sq, D), 71)
    k = _rand((B, H, Sk, D), 72)
    v = _rand((B, H, Sk, D), 73)
    O, L = attention_ref(q, k, v, 0.0, causal=True)
    for i in range(Sq):
        np.testing.assert_allclose(O[0, :, i], v[0, :, :i + 1].mean(axis=1), rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(L[0, :, i], math.log(i + 1), atol=1e-14)


# --------------------------------------------------------------------------
# Invariances
# --------------------------------------------------------------------------

def test_key_permutation_invariance():
    B, H, Sq, Sk, D = 1, 2, 6, 11, 5
    q = _rand((B, H, Sq, D), 81)
    k = _rand((B, H, Sk, D), 82)
    v = _rand((B, H, Sk, D), 83)
    perm = np.random.default_rng(84).permutation(Sk)
    O1, L1 = attention_ref(q, k, v, 0.6)
    O2, L2 = attention_ref(q, k[:, :, perm], v[:, :, perm], 0.6)
    np.testing.assert_allclose(O1, O2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(L1, L2, rtol=1e-13, atol=1e-14)


def test_score_shift_and_large_scores():
    # Adding c_i to every score of row i leaves O unchanged and adds c_i to LSE.
    # The shift is planted through an extra feature: q' = [q, c], k' = [k, 1/scale].
    # With |scores| in the thousands, exp() of an unshifted score would overflow:
    # only a stable (max-subtracted) softmax passes.
    B, H, Sq, Sk, D = 1, 1, 5, 9, 4
    q = _rand((B, H, Sq, D), 91, std=40.0)
    k = _rand((B, H, Sk, D), 92, std=40.0)
    v = _rand((B, H, Sk, D), 93)
    scale = 1.0
    c = np.array([1000.0, -1000.0, 0.0, 500.0, 7.0])
    qp = np.concatenate([q, c.reshape(1, 1, Sq, 1)], axis=-1)
    kp = np.concatenate([k, np.full((B, H, Sk, 1), 1.0 / scale)], axis=-1)
    O1, L1 = attention_ref(q, k, v, scale, causal=True)
    O2, L2 = attention_ref(qp, kp, v, scale, causal=True)
    assert np.all(np.isfinite(O1)) and np.all(np.isfinite(L1))
    np.testing.assert_allclose(O2, O1, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(L2 - c.reshape(1, 1, Sq), L1, rtol=1e-12, atol=1e-9)


def test_query_block_size_does_not_matter():
    B, H, Sq, Sk, D = 1, 1, 37, 29, 6
    q = _rand((B, H, Sq, D), 95)
    k = _rand((B, H, Sk, D), 96)
    v = _rand((B, H, Sk, D), 97)
    O1, L1 = attention_ref(q, k, v, 0.5, causal=True, block=256)
    O2, L2 = attention_ref(q, k, v, 0.5, causal=True, block=5)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)


def test_attention_rows_matches_full():
    B, H, Sq, Sk, D = 2, 2, 40, 33, 8
    q = _rand((B, H, Sq, D), 101)
    k = _rand((B, H, Sk, D), 102)
    v = _rand((B, H, Sk, D), 103)
    kv = [20, 33]
    O, L = attention_ref(q, k, v, 0.3, causal=True, kv_lens=kv)
    rows = [0, 5, 19, 20, 39]
    for b in range(B):
        for h in range(H):
            o, l = attention_rows(q[b, h], k[b, h], v[b, h], rows, 0.3, causal=True, kv_len=kv[b])
            np.testing.assert_array_equal(o, O[b, h, rows])
            np.testing.assert_array_equal(l, L[b, h, rows])


# --------------------------------------------------------------------------
# A library routine: torch float64 SDPA (math backend on the CPU)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(2, 3, 16, 16, 8), (1, 2, 33, 33, 64), (2, 1, 7, 19, 16)])
def test_against_torch_sdpa(causal, shape):
    B, H, Sq, Sk, D = shape
    if causal and Sq != Sk:
        pytest.skip("torch's is_causal aligns the mask differently when Sq != Sk")
    q = _rand((B, H, Sq, D), 111)
    k = _rand((B, H, Sk, D), 112)
    v = _rand((B, H, Sk, D), 113)
    scale = 1.0 / math.sqrt(D)
    O, L = attention_ref(q, k, v, scale, causal=causal)
    t = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), is_causal=causal, scale=scale)
    np.testing.assert_allclose(O, t.numpy(), rtol=1e-12, atol=1e-13)
    s = torch.from_numpy(q) @ torch.from_numpy(k).transpose(-1, -2) * scale
    if causal:
        s = s.masked_fill(torch.ones(Sq, Sk, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(L, torch.logsumexp(s, dim=-1).numpy(), rtol=1e-12, atol=1e-12)


def test_against_torch_sdpa_key_padding():
    B, H, Sq, Sk, D = 3, 2, 12, 12, 16
    q = _rand((B, H, Sq, D), 121)
    k = _rand((B, H, Sk, D), 122)
    v = _rand((B, H, Sk, D), 123)
    kv = [12, 5, 1]
    O, _ = attention_ref(q, k, v, 0.25, kv_lens=kv)
    mask = torch.zeros(B, 1, Sq, Sk, dtype=torch.bool)
    for b in range(B):
        mask[b, :, :, :kv[b]] = True
    t = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), attn_mask=mask, scale=0.25)
    np.testing.assert_allclose(O, t.numpy(), rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# LSE merge of key-range partial results (split-KV / context parallel)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("cuts", [[0, 13, 29], [0, 1, 2, 29], [0, 29], [0, 10, 10, 20, 29]])
def test_merge_of_key_ranges_is_whole_row_attention(causal, cuts):
    from oracle import lse_merge
    B, H, Sq, Sk, D = 1, 2, 17, 29, 6
    q = _rand((B, H, Sq, D), 131)
    k = _rand((B, H, Sk, D), 132)
    v = _rand((B, H, Sk, D), 133)
    scale = 0.45
    O, L = attention_ref(q, k, v, scale, causal=causal)
    parts_o, parts_l = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        # keys outside [a, b) are masked for this range: shift causality by giving
        # the oracle only the range's keys and the row positions relative to it
        o_s = np.zeros((B, H, Sq, D))
        l_s = np.full((B, H, Sq), -np.inf)
        for h in range(H):
            for i in range(Sq):
                valid = [j for j in range(a, b) if (not causal or j <= i)]
                if not valid:
                    continue
                s = scale * (k[0, h, valid] @ q[0, h, i])
                mx = s.max()
                p = np.exp(s - mx)
                o_s[0, h, i] = p @ v[0, h, valid] / p.sum()
                l_s[0, h, i] = mx + math.log(p.sum())
        parts_o.append(o_s.reshape(-1, D))
        parts_l.append(l_s.reshape(-1))
    Om, Lm = lse_merge(np.stack(parts_o), np.stack(parts_l))
    np.testing.assert_allclose(Om, O.reshape(-1, D), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(Lm, L.reshape(-1), rtol=1e-12, atol=1e-12)


def test_merge_of_empty_sets():
    from oracle import lse_merge
    o = np.array([[[1.0, 2.0]], [[5.0, 6.0]]])
    l = np.array([[-np.inf], [-np.inf]])
    Om, Lm = lse_merge(o, l)
    assert np.all(Om == 0.0) and Lm[0] == -np.inf
    l2 = np.array([[-np.inf], [0.3]])
    Om, Lm = lse_merge(o, l2)       # one empty set: the other passes through unchanged
    np.testing.assert_array_equal(Om, o[1])
    assert Lm[0] == 0.3


# --------------------------------------------------------------------------
# Packed variable-length batches
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equal_lengths_is_padded_batch(causal):
    from oracle import attention_varlen_ref
    B, H, S, D = 3, 2, 11, 5
    q = _rand((B, H, S, D), 141)
    k = _rand((B, H, S, D), 142)
    v = _rand((B, H, S, D), 143)
    O, L = attention_ref(q, k, v, 0.6, causal=causal)
    pack = lambda t: t.transpose(0, 2, 1, 3).reshape(B * S, H, D)  # noqa: E731  [B,H,S,D] -> [B*S,H,D]
    cu = np.arange(0, (B + 1) * S, S)
    Ov, Lv = attention_varlen_ref(pack(q), pack(k), pack(v), cu, cu, 0.6, causal=causal)
    np.testing.assert_array_equal(Ov, pack(O))
    np.testing.assert_array_equal(Lv, L.transpose(1, 0, 2).reshape(H, B * S))


def test_varlen_sequences_are_independent_and_match_brute_force():
    from oracle import attention_varlen_ref
    H, D = 2, 4
    lens_q = [3, 0, 5, 1]
    lens_k = [4, 2, 5, 0]
    cu_q = np.concatenate([[0], np.cumsum(lens_q)])
    cu_k = np.concatenate([[0], np.cumsum(lens_k)])
    q = _rand((cu_q[-1], H, D), 151)
    k = _rand((cu_k[-1], H, D), 152)
    v = _rand((cu_k[-1], H, D), 153)
    for causal in (False, True):
        O, L = attention_varlen_ref(q, k, v, cu_q, cu_k, 0.5, causal=causal)
        for b in range(4):
            for i in range(lens_q[b]):
                t = cu_q[b] + i
                for h in range(H):
                    keys = [j for j in range(lens_k[b]) if (not causal or j <= i)]
                    if not keys:
                        assert np.all(O[t, h] == 0) and L[h, t] == -np.inf
                        continue
                    e = [math.exp(0.5 * math.fsum(q[t, h] * k[cu_k[b] + j, h])) for j in keys]
                    den = math.fsum(e)
                    want = sum(w * v[cu_k[b] + j, h] for w, j in zip(e, keys)) / den
                    np.testing.assert_allclose(O[t, h], want, rtol=1e-12, atol=1e-13)
                    assert abs(L[h, t] - math.log(den)) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_paged_with_pages_in_order_is_varlen(causal):
    """Pages laid out back to back in sequence order make the paged cache the
    packed key tensor itself: the paged oracle must then equal the pinned
    variable-length oracle exactly."""
    from oracle import attention_paged_ref, attention_varlen_ref
    H, D, ps = 2, 4, 3
    lens_q = [4, 0, 6, 2]
    lens_k = [6, 3, 5, 0]           # ragged last pages
    pages_per = [(n + ps - 1) // ps for n in lens_k]
    max_pages = max(pages_per)
    num_pages = sum(pages_per)
    # sequence b's keys occupy pages first_page[b] .. first_page[b] + pages_per[b] - 1
    first = np.concatenate([[0], np.cumsum(pages_per)])[:-1]
    table = np.full((4, max_pages), -7, dtype=np.int64)  # unused entries: never read
    for b in range(4):
        table[b, :pages_per[b]] = first[b] + np.arange(pages_per[b])
    k_cache = _rand((num_pages, ps, H, D), 161)
    v_cache = _rand((num_pages, ps, H, D), 162)
    cu_q = np.concatenate([[0], np.cumsum(lens_q)])
    q = _rand((cu_q[-1], H, D), 163)
    # the packed keys of the same sequences, taken from the page rows
    flat_k = k_cache.reshape(num_pages * ps, H, D)
    flat_v = v_cache.reshape(num_pages * ps, H, D)
    idx = np.concatenate([first[b] * ps + np.arange(lens_k[b]) for b in range(4)]).astype(np.int64)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)])
    O, L = attention_paged_ref(q, k_cache, v_cache, cu_q, lens_k, table, 0.7, causal=causal)
    Ov, Lv = attention_varlen_ref(q, flat_k[idx], flat_v[idx], cu_q, cu_k, 0.7, causal=causal)
    np.testing.assert_array_equal(O, Ov)
    np.testing.assert_array_equal(L, Lv)


def test_paged_scattered_pages_match_brute_force():
    """A shuffled page table: every output checked by a loop that looks each
    key up through the table on its own."""
    from oracle import attention_paged_ref
    rng = np.random.default_rng(171)
    H, D, ps = 2, 3, 2
    lens_q = [3, 2, 1]
    lens_k = [5, 0, 3]
    num_pages, max_pages = 9, 3
    perm = rng.permutation(num_pages)
    table = perm[:3 * max_pages].reshape(3, max_pages)
    k_cache = _rand((num_pages, ps, H, D), 172)
    v_cache = _rand((num_pages, ps, H, D), 173)
    cu_q = np.concatenate([[0], np.cumsum(lens_q)])
    q = _rand((cu_q[-1], H, D), 174)
    for causal in (False, True):
        O, L = attention_paged_ref(q, k_cache, v_cache, cu_q, lens_k, table, 0.9, causal=causal)
        for b in range(3):
            for i in range(lens_q[b]):
                t = cu_q[b] + i
                for h in range(H):
                    keys = [j for j in range(lens_k[b]) if (not causal or j <= i)]
                    if not keys:
                        assert np.all(O[t, h] == 0) and L[h, t] == -np.inf
                        continue
                    kv = [(k_cache[table[b][j // ps], j % ps, h], v_cache[table[b][j // ps], j % ps, h])
                          for j in keys]
                    e = [math.exp(0.9 * math.fsum(q[t, h] * kk)) for kk, _ in kv]
                    den = math.fsum(e)
                    want = sum(w * vv for w, (_, vv) in zip(e, kv)) / den
                    np.testing.assert_allclose(O[t, h], want, rtol=1e-12, atol=1e-13)
                    assert abs(L[h, t] - math.log(den)) < 1e-12


def test_paged_result_is_invariant_to_physical_page_order():
    from oracle import attention_paged_ref
    rng = np.random.default_rng(181)
    H, D, ps = 1, 4, 4
    num_pages = 6
    table = np.array([[4, 1, 5], [0, 2, 3]])
    lens_k = [10, 7]
    cu_q = np.array([0, 5, 9])
    k_cache = _rand((num_pages, ps, H, D), 182)
    v_cache = _rand((num_pages, ps, H, D), 183)
    q = _rand((9, H, D), 184)
    O, L = attention_paged_ref(q, k_cache, v_cache, cu_q, lens_k, table, 0.5, causal=True)
    perm = rng.permutation(num_pages)        # physical page p moves to slot perm[p]
    k2 = np.empty_like(k_cache)
    v2 = np.empty_like(v_cache)
    k2[perm] = k_cache
    v2[perm] = v_cache
    O2, L2 = attention_paged_ref(q, k2, v2, cu_q, lens_k, perm[table], 0.5, causal=True)
    np.testing.assert_array_equal(O, O2)
    np.testing.assert_array_equal(L, L2)
