"""The float64 oracle checked against what the pages and mathematics fix."""
import pytest

import oracle.attention as A
from pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(A)


def test_fp16_overflow_threshold():
    """Why the shift is needed: e^x overflows fp16 just above ln(65504) = 11.09
    ("The Online Softmax Recurrence", "The obstacle")."""
    import math

    import numpy as np

    assert abs(math.log(65504.0) - 11.09) < 5e-3
    with np.errstate(over="ignore"):
        assert np.isinf(np.exp(np.float16(11.1)))
        assert np.isfinite(np.exp(np.float16(11.08)))
