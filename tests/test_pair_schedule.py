"""The static deal of causal two-tile units (attn_fwd_pair_schedule), on the CPU.

The deal decides only which block runs which unit, never what a unit
computes; a wrong deal shows up as a missing unit in the GPU parity tests
(NaN-filled outputs) or as lost time.  Here: every unit goes to an existing
block, the first wave is one unit per block in order, the blocks' work is
balanced far better than a round-robin deal of the same order, and the
arguments the library must refuse are refused."""

import math

import numpy as np
import pytest

from exact_attention_86_gb300 import attn


@pytest.fixture(scope="module")
def lib():
    return attn.lib()


def _order(B, H, Sq, head_group):
    """(pair index) of each unit in the kernel's order: head groups, pairs
    from the last one down, the group's heads innermost."""
    bh = B * H
    n_pairs = math.ceil(Sq / 256)
    out = []
    for g0 in range(0, bh, head_group):
        heads = min(head_group, bh - g0)
        for wq in range(n_pairs):
            out += [n_pairs - 1 - wq] * heads
    return out


def _key_steps(pr, Sq):
    # causal, Sq == Sk: tile A of pair pr needs 2 pr + 1 key tiles, tile B one more
    rows_b = min(128, Sq - 256 * pr - 128)
    return 2 * pr + (2 if rows_b > 0 else 1)


@pytest.mark.parametrize("B,H,S,hg,grid", [(2, 16, 8192, 12, 152), (1, 8, 32768, 8, 152), (4, 8, 2048, 32, 152),
                                           (3, 5, 3000, 4, 100), (1, 1, 8192, 1, 152)])
def test_deal_is_complete_and_balanced(lib, B, H, S, hg, grid):
    owner = attn.attn_fwd_pair_schedule(B, H, S, S, hg, grid)
    order = _order(B, H, S, hg)
    assert owner is not None and len(owner) == len(order)
    owner = np.frombuffer(owner, dtype=np.uint8).astype(int)
    assert owner.min() >= 0 and owner.max() < grid
    n = len(order)
    first = min(n, grid)
    assert list(owner[:first]) == list(range(first))  # all blocks start idle: one unit each, in order
    steps = np.array([_key_steps(pr, S) for pr in order])
    load = np.bincount(owner, weights=steps + 2, minlength=grid)[:grid]
    if n >= 4 * grid:
        # greedy list scheduling: no block ends more than about one unit
        # after the mean (the library's model weighs a pair's key steps a
        # little differently from this count, hence the slack)
        assert load.max() - load.mean() <= 1.5 * (steps.max() + 2)
        # and it beats a round-robin deal of the same order
        rr = np.bincount(np.arange(n) % grid, weights=steps + 2, minlength=grid)
        assert load.max() < rr.max()


def test_refusals(lib):
    f = attn.attn_fwd_pair_schedule
    assert f(16, 16, 8192, 8192, 4, 152) is None          # 8192 units > 4096
    assert f(2, 16, 8192, 8192, 0, 152) is None           # head_group < 1
    assert f(2, 16, 8192, 8192, 4, 0) is None             # grid < 1
    assert f(2, 16, 8192, 8192, 4, 257) is None           # a block index must fit a byte
    assert f(-1, 16, 8192, 8192, 4, 152) is None
    assert f(0, 16, 8192, 8192, 4, 152) == b""            # nothing to deal
