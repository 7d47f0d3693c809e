"""The kernel's barrier protocol, checked on a CPU model under random
timings (see pipeline_model)."""

import random

import pytest

from pipeline_model import run, run_pair


def _units(seed):
    rng = random.Random(seed)
    return [rng.choice([1, 2, 3, 5, 8, 16, 64]) for _ in range(rng.randint(1, 6))]


# packed and paged batches: K and V in rings of their own, each with its own
# producer (bf16 D=128: 3 + 3 slots; bf16 D=64: 6 + 6; the 3 + 2 layout of
# an earlier five-slot ring stays covered)
@pytest.mark.parametrize("p_in_s,rings", [(False, (3, 3)), (False, (3, 2)), (False, (6, 6)), (True, (3, 3)),
                                          (True, (3, 2)), (True, (6, 6))])
def test_split_ring_protocol_never_aliases_or_deadlocks(p_in_s, rings):
    for seed in range(400):
        run(_units(seed), 0, per_kind=False, seed=seed, p_in_s=p_in_s, rings=rings)


@pytest.mark.parametrize("p_in_s,mistake", [
    (False, "qk_skips_buffer_wait"), (False, "p_store_skips_p_free"), (False, "rescale_skips_p_free"),
    (True, "qk_skips_buffer_wait"), (True, "rescale_skips_p_free"), (False, "producer_skips_kv_empty"),
])
def test_model_with_split_rings_catches_a_skipped_wait(p_in_s, mistake):
    failures = 0
    for seed in range(300):
        try:
            run(_units(seed), 0, per_kind=False, seed=seed, rescale_p=0.6, mistake=mistake, p_in_s=p_in_s,
                rings=(3, 2))
        except AssertionError:
            failures += 1
    assert failures > 0, mistake


# padded batches: one ring of alternating K and V positions, one producer
# (bf16 D=128: 6 slots; bf16 D=64 and E4M3: 12; the odd depth 5 of an
# earlier layout stays covered)
@pytest.mark.parametrize("p_in_s,slots", [(False, 6), (False, 5), (False, 12), (True, 12)])
def test_single_ring_protocol_never_aliases_or_deadlocks(p_in_s, slots):
    for seed in range(400):
        run(_units(seed), slots, per_kind=True, seed=seed, p_in_s=p_in_s)


@pytest.mark.parametrize("p_in_s,mistake", [
    (False, "qk_skips_buffer_wait"), (False, "p_store_skips_p_free"), (False, "rescale_skips_p_free"),
    (True, "qk_skips_buffer_wait"), (True, "rescale_skips_p_free"), (False, "producer_skips_kv_empty"),
])
def test_model_catches_a_skipped_wait(p_in_s, mistake):
    """The model has teeth: leaving out any one of the waits that guard the
    TMEM buffers shows up as a hazard in some random schedule.  (The E4M3
    protocol's o_free wait is implied by the softmax's own order, which the
    model confirms by never needing it; the kernel keeps it.)"""
    failures = 0
    for seed in range(300):
        try:
            run(_units(seed), 5, per_kind=True, seed=seed, rescale_p=0.6, mistake=mistake, p_in_s=p_in_s)
        except AssertionError:
            failures += 1
    assert failures > 0, mistake


def test_odd_depth_with_one_full_barrier_per_slot_aliases_in_the_bf16_protocol():
    """With S released by the softmax, the QK^T issuer can run ahead of the
    V fills; one full barrier per slot with an odd depth then aliases (the
    fault the per-kind barriers fixed)."""
    failures = 0
    for seed in range(200):
        try:
            run(_units(seed), 5, per_kind=False, seed=seed)
        except AssertionError as e:
            assert "aliasing" in str(e) or "read slot" in str(e) or "overwritten" in str(e), str(e)
            failures += 1
    assert failures > 0


@pytest.mark.parametrize("p_in_s,slots", [(False, 12), (True, 5), (True, 12)])
def test_one_full_barrier_per_slot_holds_with_even_depth_or_p_over_s(p_in_s, slots):
    """An even depth keeps each slot to one kind; and with the P V commit
    releasing the S buffers (E4M3 protocol) the QK^T issuer reaches K_j only
    after the V fills before it have landed.  The kernel keeps one full
    barrier per kind all the same."""
    for seed in range(200):
        run(_units(seed), slots, per_kind=False, seed=seed, p_in_s=p_in_s)


# ------------------------------------------------------------ dK/dV backward
from bwd_pipeline_model import run as run_bwd  # noqa: E402


def _bwd_units(seed):
    rng = random.Random(seed)
    return [rng.choice([0, 1, 2, 3, 5, 8, 40]) for _ in range(rng.randint(1, 6))]


@pytest.mark.parametrize("kernel", ["dkdv", "dq"])
@pytest.mark.parametrize("slots", [4, 8])  # D = 128, D = 64
def test_backward_protocols_never_alias_or_deadlock(kernel, slots):
    for seed in range(400):
        run_bwd(_bwd_units(seed), slots, seed=seed, kernel=kernel)


@pytest.mark.parametrize("kernel,mistake", [
    ("dkdv", "s_skips_s_free"), ("dkdv", "dp_skips_d_free"), ("dkdv", "products_skip_pd_full"),
    ("dkdv", "producer_skips_qd_empty"), ("dkdv", "epilogue_skips_out_full"), ("dkdv", "kv_load_skips_kv_empty"),
    ("dq", "s_skips_s_free"), ("dq", "products_skip_pd_full"), ("dq", "producer_skips_qd_empty"),
    ("dq", "epilogue_skips_out_full"), ("dq", "kv_load_skips_kv_empty"),
])
def test_backward_models_catch_a_skipped_wait(kernel, mistake):
    failures = 0
    for seed in range(300):
        try:
            run_bwd(_bwd_units(seed), 4, seed=seed, mistake=mistake, kernel=kernel)
        except AssertionError:
            failures += 1
    assert failures > 0, (kernel, mistake)


# the padded forward with two query tiles per unit (5 slots at D = 128, 12 at
# D = 64): unit lists of (K tiles of tile A, of tile B) as causal and
# non-causal batches give them (n_A = n_B, or n_A = n_B - 1, or tile B absent)
def _pair_units(seed):
    rng = random.Random(seed)
    out = []
    for _ in range(rng.randint(1, 6)):
        n = rng.choice([1, 2, 3, 5, 8, 16])
        out.append(rng.choice([(n, n), (n - 1, n), (n, 0), (0, 0)]))
    return out


@pytest.mark.parametrize("slots", [5, 12])
def test_pair_protocol_never_aliases_or_deadlocks(slots):
    for seed in range(400):
        run_pair(_pair_units(seed), slots, seed=seed)


@pytest.mark.parametrize("mistake", ["qk_skips_p_free", "producer_skips_kv_empty", "pv_skips_p_full"])
def test_pair_model_catches_a_skipped_wait(mistake):
    failures = 0
    for seed in range(300):
        try:
            run_pair(_pair_units(seed), 5, seed=seed, mistake=mistake)
        except AssertionError:
            failures += 1
    assert failures > 0, mistake
