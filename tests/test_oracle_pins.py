"""The CPU oracle against facts that do not come from itself (see ``oracle_checks.py`` for the list)."""
import pytest

import oracle
import oracle_checks as C


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("check", C.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(orc, check):
    check(orc)
