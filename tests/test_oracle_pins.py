"""The CPU oracle against brute force, closed forms and invariants (no GPU)."""
import pytest

import oracle
from tests import _pins


@pytest.fixture(scope="module")
def o():
    return oracle.Oracle()


@pytest.mark.parametrize("pin", _pins.PINS, ids=lambda f: f.__name__)
def test_pin(o, pin):
    pin(o)


def test_exchange_helper_matches_run(o):
    import numpy as np
    S = np.array([[2, 0, 1], [1, 1, 0], [0, 3, 2]], dtype=np.int64)
    inp = _pins.tagged_inputs(S, 9)
    outs, so = o.exchange(inp, S, 9)
    ref_outs, ref_so = _pins.scatter_reference(inp, S, 9)
    for a, b in zip(outs, ref_outs):
        assert np.array_equal(a, b)
    assert np.array_equal(so, ref_so)
