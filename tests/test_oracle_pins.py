"""The float64 oracle against its pins (closed forms, brute force, the
worked scan trace of the paper's Appendix A, the no-leak invariant)."""
import pytest

from oracle import rlca_ref
from tests import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(rlca_ref)


def test_app_a_fixture_parses():
    rows = pins.load_app_a_trace()
    labels = [r[0] for r in rows]
    assert labels[:4] == ["T1", "T2", "T3", "T4"]
    assert "T1..2" in labels and "T3..4" in labels and "T4-pass2" in labels
