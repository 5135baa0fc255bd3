"""The fp64 oracle against the facts the pages and the mathematics fix (no GPU)."""
import numpy as np
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_threads_do_not_change_results(orc):
    rng = np.random.default_rng(3)
    B, T, H, dk, dv = 2, 33, 3, 8, 8
    args = [rng.normal(size=(B, T, H, dk)), rng.normal(size=(B, T, H, dk)), rng.normal(size=(B, T, H, dv)),
            rng.uniform(0.5, 1, size=(B, T, H)), rng.uniform(0, 1, size=(B, T, H)), 1e-6,
            rng.normal(size=(B, H, dk, dv))]
    o1, s1 = orc.recurrent(*args, nthreads=1)
    o4, s4 = orc.recurrent(*args, nthreads=4)
    assert np.array_equal(o1, o4) and np.array_equal(s1, s4)


def test_empty_sequence_returns_initial_state(orc):
    rng = np.random.default_rng(4)
    S0 = rng.normal(size=(1, 2, 4, 4))
    z = np.zeros((1, 0, 2, 4))
    o, ST = orc.recurrent(z, z, z, np.zeros((1, 0, 2)), np.zeros((1, 0, 2)), 1e-6, S0)
    assert o.shape == (1, 0, 2, 4)
    assert np.array_equal(ST, S0)
