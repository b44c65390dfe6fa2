"""SnapKV oracle against brute force, torch routines and invariants (CPU)."""
import pytest

import oracle.snapkv as snapkv
from tests import oracle_pins as pins


@pytest.mark.parametrize("check", pins.SNAPKV_CHECKS, ids=lambda f: f.__name__)
def test_snapkv_oracle_pin(check):
    check(snapkv)
