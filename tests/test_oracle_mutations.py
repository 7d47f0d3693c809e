"""Plant plausible mistakes in a private copy of the oracle (CPU only) and check
that the pins catch each one: a dropped term, a wrong sign or index, an
off-by-one mask, a transposed operand.  The real oracle is never modified."""

import math
import os
import types

import numpy as np
import pytest

import oracle.attention as real

SRC = open(real.__file__).read()

MUTATIONS = {
    "mask_off_by_one": ("valid = cols[None, :] < lim[:, None]", "valid = cols[None, :] <= lim[:, None]"),
    "causal_diagonal_dropped": ("row_index.astype(np.int64) + 1", "row_index.astype(np.int64)"),
    "lse_drops_max": ("lse[has_key] = m + np.log(total)", "lse[has_key] = np.log(total)"),
    "no_max_subtraction": ("p = np.exp(sv - m[:, None])", "p = np.exp(sv)"),
    "min_instead_of_max": ("m = np.max(sv, axis=1)", "m = np.min(sv, axis=1)"),
    "scale_dropped": ("s = (q_rows @ k.T) * np.float64(scale)", "s = (q_rows @ k.T)"),
    "transposed_product": ("out[has_key] = (p @ v) / total[:, None]",
                           "out[has_key] = (p @ v[::-1]) / total[:, None]"),
    "kv_len_ignored": ("lim = np.full((n,), min(max(int(kv_len), 0), Sk), dtype=np.int64)",
                       "lim = np.full((n,), Sk, dtype=np.int64)"),
    "empty_row_lse_zero": ("lse = np.full((n,), -np.inf, dtype=np.float64)",
                           "lse = np.full((n,), 0.0, dtype=np.float64)"),
}


def _mutant(name):
    old, new = MUTATIONS[name]
    assert SRC.count(old) == 1, name
    mod = types.ModuleType("oracle_mutant_" + name)
    exec(compile(SRC.replace(old, new), "<mutant " + name + ">", "exec"), mod.__dict__)
    return mod


def _brute(q, k, v, scale, causal, kv):
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    O = np.zeros((B, H, Sq, v.shape[3]))
    L = np.full((B, H, Sq), -np.inf)
    for b in range(B):
        for h in range(H):
            for i in range(Sq):
                w = [(j, math.exp(scale * math.fsum(q[b, h, i] * k[b, h, j])))
                     for j in range(Sk) if j < min(max(kv[b], 0), Sk) and (not causal or j <= i)]
                if w:
                    den = math.fsum(e for _, e in w)
                    O[b, h, i] = sum(e * v[b, h, j] for j, e in w) / den
                    L[b, h, i] = math.log(den)
    return O, L


def _pins_pass(mod) -> bool:
    """A reduced set of the pins (brute force incl. padded / empty rows, large
    scores, out-of-range kv_lens); True iff the module passes all of them."""
    rng = np.random.default_rng(3)
    B, H, Sq, Sk, D = 3, 1, 5, 6, 4
    q, k, v = (rng.normal(size=(B, H, n, D)) for n in (Sq, Sk, Sk))
    try:
        for causal in (False, True):
            for kv in ([6, 2, 0], [9, -1, 3]):
                with np.errstate(all="ignore"):
                    O, L = mod.attention_ref(q, k, v, 0.5, causal=causal, kv_lens=kv)
                Ob, Lb = _brute(q, k, v, 0.5, causal, kv)
                if not np.allclose(O, Ob, rtol=1e-12, atol=1e-13, equal_nan=False):
                    return False
                if not np.array_equal(np.isfinite(L), np.isfinite(Lb)):
                    return False
                f = np.isfinite(Lb)
                if not np.allclose(L[f], Lb[f], rtol=1e-12, atol=1e-13):
                    return False
        # large scores: a softmax without the max subtraction overflows
        with np.errstate(all="ignore"):
            O, L = mod.attention_ref(q * 60, k * 60, v, 1.0)
        if not (np.all(np.isfinite(O)) and np.all(np.isfinite(L))):
            return False
    except Exception:
        return False
    return True


def test_real_oracle_passes_reduced_pins():
    assert _pins_pass(real)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name):
    assert not _pins_pass(_mutant(name)), f"planted mistake {name} went unnoticed"


PAGED_MUTATIONS = {
    "page_and_slot_swapped": ("slots = [j % page_size for j in range(n)]", "slots = [j // page_size for j in range(n)]"),
    "table_row_of_next_sequence": ("pages = [int(table[b, j // page_size]) for j in range(n)]",
                                   "pages = [int(table[(b + 1) % table.shape[0], j // page_size]) for j in range(n)]"),
    "seqlen_off_by_one": ("n = min(max(int(seqlens_k[b]), 0), table.shape[1] * page_size)",
                          "n = min(max(int(seqlens_k[b]) - 1, 0), table.shape[1] * page_size)"),
}


def _paged_pins_pass(mod) -> bool:
    """Shuffled page table against a per-key brute force (both masks)."""
    rng = np.random.default_rng(9)
    H, D, ps = 2, 3, 2
    lens_q, lens_k = [3, 2], [5, 3]
    table = rng.permutation(8)[:6].reshape(2, 3)
    kc, vc = rng.normal(size=(8, ps, H, D)), rng.normal(size=(8, ps, H, D))
    cu_q = np.array([0, 3, 5])
    q = rng.normal(size=(5, H, D))
    try:
        for causal in (False, True):
            O, L = mod.attention_paged_ref(q, kc, vc, cu_q, lens_k, table, 0.8, causal=causal)
            for b in range(2):
                for i in range(lens_q[b]):
                    t = cu_q[b] + i
                    for h in range(H):
                        keys = [j for j in range(lens_k[b]) if not causal or j <= i]
                        e = [math.exp(0.8 * math.fsum(q[t, h] * kc[table[b][j // ps], j % ps, h])) for j in keys]
                        want = sum(w * vc[table[b][j // ps], j % ps, h] for w, j in zip(e, keys)) / math.fsum(e)
                        if not np.allclose(O[t, h], want, rtol=1e-12, atol=1e-13):
                            return False
                        if abs(L[h, t] - math.log(math.fsum(e))) > 1e-12:
                            return False
    except Exception:
        return False
    return True


def test_real_paged_oracle_passes_pins():
    assert _paged_pins_pass(real)


@pytest.mark.parametrize("name", sorted(PAGED_MUTATIONS))
def test_paged_pins_catch_planted_mistake(name):
    old, new = PAGED_MUTATIONS[name]
    assert SRC.count(old) == 1, name
    mod = types.ModuleType("oracle_paged_mutant_" + name)
    exec(compile(SRC.replace(old, new), "<mutant " + name + ">", "exec"), mod.__dict__)
    assert not _paged_pins_pass(mod), f"planted mistake {name} went unnoticed"
