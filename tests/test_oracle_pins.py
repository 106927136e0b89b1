"""The CPU oracle against what the formats and the mathematics fix.

Each check lives in oracle_checks.py; see its docstring for where every
expected value comes from (published format tables under tests/golden/,
PyTorch's float8_e4m3fn conversion, numpy's float16 rounding, closed forms,
invariants and an independent dense float64 expansion).
"""
import pytest

import oracle_checks as oc
from oracle import oracle


@pytest.fixture(scope="module")
def o():
    return oracle.get()


@pytest.mark.parametrize("check", oc.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(o, check):
    check(o)
