"""Quest oracle against brute force, closed forms, torch routines and invariants (CPU)."""
import pytest

import oracle.quest as quest
from tests import oracle_pins as pins


@pytest.mark.parametrize("check", pins.QUEST_CHECKS, ids=lambda f: f.__name__)
def test_quest_oracle_pin(check):
    check(quest)
