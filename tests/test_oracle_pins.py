"""The CPU oracle against closed forms, invariants, library routines and exact
rational arithmetic (no GPU)."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin, oracle_lib):
    err, tol = pin(oracle_lib)
    assert err <= tol, f"{pin.__name__}: max abs error {err:.3e} > {tol:.1e}"
