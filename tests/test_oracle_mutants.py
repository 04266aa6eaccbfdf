"""Mutation testing of the oracle's pins.

Each build of the oracle with W4_ORACLE_MUTANT=n carries one planted mistake
(the list is in oracle/w4_oracle.c, after the pitfalls table of "Fused int4
and int8 dequantize-matmul in C", section 5).  A mutant is killed when at
least one pin fails on it; every mutant must be killed.
"""
import pytest

from tests import oracle_pins

MUTANTS = [1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15, 16, 17, 18, 19, 20, 21, 22, 23, 24, 25, 26, 27, 28, 29,
           30, 31, 32, 33, 34, 35, 36]
# pins too slow to repeat for every mutant, and not needed to kill any of them
_SKIP = {"f16_bruteforce", "bf16"}
# mutants whose mistake crashes the reading process (s11: the unchecked NULL
# weights are dereferenced): their pin runs in a child process, and a child
# that dies or fails the pin kills the mutant
_IN_CHILD = {11: "null_pointers"}


def _pin_in_child(mutant: int, pin: str) -> bool:
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import oracle; from tests import oracle_pins; "
            f"oracle_pins.PINS[{pin!r}](oracle.get(mutant={mutant}))")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, timeout=300)
    return r.returncode == 0


@pytest.mark.parametrize("mutant", MUTANTS)
def test_mutant_is_killed(mutant):
    import oracle
    o = oracle.get(mutant=mutant)
    assert o.mutant == mutant
    failed = []
    for name, fn in sorted(oracle_pins.PINS.items()):
        if name in _SKIP:
            continue
        if _IN_CHILD.get(mutant) == name:
            if not _pin_in_child(mutant, name):
                failed.append(name)
            continue
        try:
            fn(o)
        except AssertionError:
            failed.append(name)
    if mutant == 12:
        # a partition that drops a row also shows up against the serial build
        try:
            oracle_pins.pool_equals_serial(oracle.get(), oracle.get(mutant=12, openmp=True))
        except AssertionError:
            failed.append("pool_equals_serial")
    assert failed, f"mutant {mutant} survived every pin"
