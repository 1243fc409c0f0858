"""The CPU oracle against its pins (no GPU needed).

Every pin compares the oracle with something other than itself; see `tests/pins.py` for the
source of truth behind each one. The last test plants known mistakes in the oracle (on the CPU)
and checks that each one fails at least one pin.
"""
import numpy as np
import pytest

import oracle
from tests import pins


@pytest.fixture(autouse=True)
def _no_mutation(oracle_lib):
    oracle.set_mutation(0)
    yield
    oracle.set_mutation(0)


@pytest.mark.parametrize("pin", pins.ALL_PINS + [pins.pin_sampled_entry_points_agree],
                         ids=lambda f: f.__name__)
def test_pin(pin):
    fails = pin()
    assert not fails, "\n".join(fails)


@pytest.mark.parametrize("name", sorted(oracle.MUTATIONS))
def test_planted_mistake_is_caught(name):
    oracle.set_mutation(name)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            if pin():
                caught.append(pin.__name__)
        except Exception as e:  # a crash under a planted mistake also counts as caught
            caught.append(f"{pin.__name__} raised {type(e).__name__}")
    oracle.set_mutation(0)
    assert caught, f"planted mistake {name!r} passed every pin"


def test_oracle_rejects_bad_head_grouping():
    q = np.zeros((1, 3, 2, 4), np.float32)
    k = np.zeros((1, 2, 2, 4), np.float32)
    with pytest.raises(ValueError):
        oracle.fwd(q, k, k, scale=1.0, causal=False)
