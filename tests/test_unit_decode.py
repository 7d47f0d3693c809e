"""CPU checks of the host-side arithmetic behind the kernel's work-unit decode.

The kernel divides by divisors fixed for a launch (heads, query tiles, key
ranges, head groups, grid size) with one multiply-high, an add and a shift
(Granlund and Montgomery, "Division by invariant integers using
multiplication", 1994): s = ceil(log2 d), m = floor(2^32 (2^s - d) / d) + 1,
floor(n / d) = (mulhi(n, m) + n) >> s.  These tests check that method against
exact integer division over the range the kernel uses (0 <= n < 2^31), and
that the unit order it decodes (heads-major; causal head groups with a
shorter last group) visits every (head, query tile) exactly once.  The GPU
parity tests check the kernel's own implementation end to end."""

import random

import pytest


def make(d):
    s = 0
    while (1 << s) < d:
        s += 1
    m = ((1 << 32) * ((1 << s) - d)) // d + 1
    return m, s


def fdiv(n, d):
    m, s = make(d)
    assert 0 <= m < (1 << 32)
    t = (n * m) >> 32
    assert t + n < (1 << 32)
    return (t + n) >> s


def test_division_exact_small_divisors_exhaustive():
    for d in range(1, 1025):
        for n in range(0, 4 * d + 3):
            assert fdiv(n, d) == n // d, (n, d)


def test_division_exact_at_the_edges_and_at_random():
    rng = random.Random(1)
    divisors = [rng.randrange(1, 1 << 31) for _ in range(2000)]
    divisors += [(1 << k) + e for k in range(1, 31) for e in (-1, 0, 1)]
    for d in divisors:
        ns = [0, 1, (1 << 31) - 1, (1 << 31) - 2] + [rng.randrange(0, 1 << 31) for _ in range(50)]
        for q in (1, 2, 7, ((1 << 31) - 1) // d):
            ns += [q * d + r for r in (-1, 0, 1) if 0 <= q * d + r < (1 << 31)]
        for n in ns:
            assert fdiv(n, d) == n // d, (n, d)


def _decode(t_in, B, H, n_qtiles, splits, causal, head_group):
    """The kernel's unit decode, with its divisions done by the method above."""
    bh_count = B * H
    t = fdiv(t_in, splits)
    split = t_in - t * splits
    if causal:
        groups = (bh_count + head_group - 1) // head_group
        grp = fdiv(t, head_group * n_qtiles)
        w = t - grp * head_group * n_qtiles
        heads = bh_count - (groups - 1) * head_group if grp == groups - 1 else head_group
        wq = fdiv(w, heads)
        qt = n_qtiles - 1 - wq
        bh = grp * head_group + (w - wq * heads)
    else:
        bh = fdiv(t, n_qtiles)
        qt = t - bh * n_qtiles
    b = fdiv(bh, H)
    return b, bh - b * H, qt, split


@pytest.mark.parametrize("B,H,n_qtiles,splits,causal,head_group", [
    (2, 16, 64, 1, False, 32), (2, 16, 64, 1, True, 12), (1, 8, 256, 1, True, 8), (4, 8, 8, 1, True, 32),
    (3, 5, 7, 3, True, 4), (3, 5, 7, 3, False, 4), (1, 8, 1, 16, False, 8), (8, 16, 16, 1, False, 128),
])
def test_unit_order_visits_every_tile_once(B, H, n_qtiles, splits, causal, head_group):
    seen = set()
    total = B * H * n_qtiles * splits
    for t in range(total):
        u = _decode(t, B, H, n_qtiles, splits, causal, head_group)
        assert 0 <= u[0] < B and 0 <= u[1] < H and 0 <= u[2] < n_qtiles and 0 <= u[3] < splits
        seen.add(u)
    assert len(seen) == total
