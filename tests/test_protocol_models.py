"""The barrier protocols of the persistent tensor-core kernels, checked on
random interleavings (see protocol_models.py): the protocols as built finish
without a hazard on every run, and leaving out any one wait that guards a
buffer or a phase makes some run fail."""
import random

import pytest

import protocol_models as pm

N_RUNS = 1500


def _forward_cases():
    for seed in range(N_RUNS):
        rng = random.Random(10_000 + seed)
        yield pm.pairs_for(rng, rng.randint(1, 5)), seed, rng.choice([2, 4])


def _backward_cases():
    for seed in range(N_RUNS):
        rng = random.Random(7 + seed)
        yield [rng.randint(1, 5) for _ in range(rng.randint(1, 4))], seed


def test_forward_protocol_never_fails():
    for pairs, seed, stages in _forward_cases():
        assert pm.run_forward(pairs, seed, stages)


@pytest.mark.parametrize("pieces", [False, True], ids=["one_piece", "two_pieces"])
def test_backward_protocol_never_fails(pieces):
    for items, seed in _backward_cases():
        assert pm.run_backward(items, seed, pieces=pieces)


@pytest.mark.parametrize("wait", ["epi", "qfree", "vfree", "kfree"])
def test_forward_needs_every_wait(wait):
    for pairs, seed, stages in _forward_cases():
        try:
            pm.run_forward(pairs, seed, stages, skip=(wait,))
        except AssertionError:
            return
    pytest.fail(f"leaving out the {wait} wait went unnoticed")


@pytest.mark.parametrize("pieces", [False, True], ids=["one_piece", "two_pieces"])
@pytest.mark.parametrize("wait", ["itemdone", "dsfree", "stfree", "dqfree_first"])
def test_backward_needs_every_wait(wait, pieces):
    for items, seed in _backward_cases():
        try:
            pm.run_backward(items, seed, skip=(wait,), pieces=pieces)
        except AssertionError:
            return
    pytest.fail(f"leaving out the {wait} wait went unnoticed")


def test_backward_ring_needs_its_free_wait():
    """The wait for a record slot's readers keeps the producer from overwriting
    a record a role has not read: with a one-slot ring, leaving it out fails on
    some run.  (The kernel's ring has four slots; the reducer, which this model
    folds into the compute roles, can trail them by a step.)"""
    for items, seed in _backward_cases():
        try:
            pm.run_backward(items, seed, skip=("itemfree",), ring_slots=1)
        except AssertionError:
            return
    pytest.fail("leaving out the itemfree wait went unnoticed")


def test_backward_ring_of_four_never_fails():
    for items, seed in list(_backward_cases())[:500]:
        assert pm.run_backward(items, seed, ring_slots=4)


def test_backward_accumulator_release_is_implied():
    """The MMA thread's wait for the epilogue to have read the dK / dV
    accumulators is also implied by its wait for the next tile's P^T, which the
    compute warps publish only after their epilogue: dropping it never fails."""
    for items, seed in list(_backward_cases())[:300]:
        assert pm.run_backward(items, seed, skip=("accfree",))
