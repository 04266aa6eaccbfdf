"""GB300 (sm_103a) fused int4 dequantize-matmul: W4A8 linear_q4 and group-wise W4A16.

The compute path is the C-ABI library ``libw4gb300.so`` built from ``csrc/``;
``ops`` is a thin ctypes binding over it (argument marshalling only).
``synth`` holds the seeded input generators shared with the tests.
"""
import importlib

__all__ = ["ops", "synth"]


def __getattr__(name):
    if name in ("ops", "synth", "build"):
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
