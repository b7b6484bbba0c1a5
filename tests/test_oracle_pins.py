"""The CPU oracle against brute force, library routines, closed forms and hand-worked trees (no GPU)."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(orc, pin):
    pin(orc.lib())


def test_oracle_rejects_bad_input(orc):
    import numpy as np
    x = np.zeros((1, 2, 16), np.float32)
    x[0, 1, 3] = np.nan
    with pytest.raises(orc.OracleError):
        orc.topm(x, 4)
    assert orc.tree_size(4, 3) == 4 + 16 + 64
    assert orc.tree_size(151936, 16, cap=1 << 40) == 1 << 40
