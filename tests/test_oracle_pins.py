"""The fp64 oracle against closed forms, invariants, library special cases and worked examples."""
import pytest

import oracle
import _pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("check", _pins.ALL_CHECKS, ids=lambda f: f.__name__[len("check_"):])
def test_pin(check, lib):
    check(lib)
