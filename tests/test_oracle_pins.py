"""The CPU oracle against facts other than itself (no GPU needed)."""
import pytest

import oracle
from tests import oracle_pins as pins


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_invalid_tree_rejected(orc):
    import numpy as np
    with pytest.raises(ValueError):
        orc.tree_anc(np.asarray([[-1, 1]], dtype=np.int32))   # parent must precede the node
    with pytest.raises(ValueError):
        orc.tree_anc(np.full((1, 65), -1, dtype=np.int32))    # more nodes than mask bits
