"""The kernel's barrier protocol, checked on a CPU model under random
timings (see pipeline_model)."""

import random

import pytest

from pipeline_model import run


def _units(seed):
    rng = random.Random(seed)
    return [rng.choice([1, 2, 3, 5, 8, 16, 64]) for _ in range(rng.randint(1, 6))]


@pytest.mark.parametrize("slots", [5, 12])   # the ring depths of D = 128 and D = 64
def test_per_kind_full_barriers_never_alias_or_deadlock(slots):
    for seed in range(400):
        run(_units(seed), slots, per_kind=True, seed=seed)


def test_shared_full_barrier_with_odd_depth_aliases():
    """The model has teeth: one full barrier per slot with an odd ring depth
    lets the QK issuer pass a K wait on the phase of an older fill."""
    failures = 0
    for seed in range(200):
        try:
            run(_units(seed), 5, per_kind=False, seed=seed)
        except AssertionError as e:
            assert "aliasing" in str(e) or "read slot" in str(e) or "overwritten" in str(e), str(e)
            failures += 1
    assert failures > 0


def test_shared_full_barrier_with_even_depth_is_safe():
    for seed in range(200):
        run(_units(seed), 12, per_kind=False, seed=seed)
