"""The CPU oracle against what the pages and the number formats fix.

See ``tests/pins.py`` for what each check compares against.  These run on the
CPU only and take a few seconds.
"""

import pytest

import oracle
from tests import pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(oracle)
