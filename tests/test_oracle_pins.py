"""The committed fp64 oracle against facts the recurrence's definition and mathematics fix."""
import pytest

import oracle
from oracle_pins import PINS


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(orc, pin):
    pin(orc)


def test_threads_do_not_change_results(orc):
    from oracle_pins import random_case
    import numpy as np

    c = random_case(21, 0, H=5, lengths=[9, 30, 2])
    a = orc.prefill(**c, threads=1)
    b = orc.prefill(**c, threads=4)
    for x, y in zip(a[:2], b[:2]):
        assert np.array_equal(x, y)


def test_rejects_bad_arguments(orc):
    from oracle_pins import random_case

    c = random_case(22, 16, H=1)
    with pytest.raises(ValueError):
        orc.prefill(**c, chunk=16, ckpt_stride=24)   # checkpoint inside a chunk
    with pytest.raises(ValueError):
        orc.prefill(**c, chunk=200)                  # exp(+-G) would overflow fp64
