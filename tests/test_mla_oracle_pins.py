"""The MLA decode oracle against closed forms, invariants and library routines (no GPU)."""
import pytest

import mla_oracle_pins as P


@pytest.fixture(scope="session")
def mla_oracle_lib():
    import oracle.mla
    return oracle.mla.load()


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin, mla_oracle_lib):
    err, tol = pin(mla_oracle_lib)
    assert err <= tol, f"{pin.__name__}: max abs error {err:.3e} > {tol:.1e}"
