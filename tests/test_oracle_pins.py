"""The fp64 oracle against its pins (CPU only).

Each pin lives in ``tests/pins.py``; see its docstring for what each one fixes.
"""
import pytest

import oracle
import pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(oracle._load())
