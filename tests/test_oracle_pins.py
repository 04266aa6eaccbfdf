"""The CPU oracle against its pins (values printed on the pages, closed forms,
brute force, invariants, independent library routines)."""
import pytest

from tests import oracle_pins


@pytest.mark.parametrize("name", sorted(oracle_pins.PINS))
def test_pin(ora, name):
    oracle_pins.PINS[name](ora)


def test_pool_result_equals_serial_bitwise(ora):
    import oracle
    oracle_pins.pool_equals_serial(ora, oracle.get(openmp=True))
