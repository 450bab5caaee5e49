"""The CPU oracle against its pins (hand-worked fixtures, closed forms,
float64 / int64 brute force, invariants and library special cases)."""
import pytest

import oracle
import synth
from tests import pins


@pytest.fixture(scope="module")
def ora():
    return oracle.get()


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(ora, check):
    check(ora)


def test_route_invariants_ds4_shape(ora):
    # router in the DS4 shape (Q8_0, hidden 4096, 256 experts, top-6)
    pins.check_route_invariants(ora, synth.DS4_ROUTER_ONLY, seed=3, T=8)


def test_expert_stages_ds4_rows(ora):
    pins.check_expert_stages(ora, synth.MICRO, seed=41, experts=(1, 7, None))


def test_layer_vs_textbook_micro(ora):
    pins.check_layer_vs_textbook(ora, synth.MICRO, seed=43, T=6, tol=3e-2)


def test_layer_vs_textbook_hash(ora):
    pins.check_layer_vs_textbook(ora, synth.MICRO_HASH, seed=45, T=6, tol=3e-2)
