"""GB300 (sm_103a) fused int4 dequantize-matmul: W4A8 linear_q4 and group-wise W4A16.

The compute path is the C-ABI library ``libw4gb300.so`` built from ``csrc/``;
``ops`` is a thin ctypes binding over it (argument marshalling only).
``synth`` holds the seeded input generators shared with the tests.
"""
__all__ = ["ops", "synth"]


def __getattr__(name):
    if name == "ops":
        from . import ops
        return ops
    raise AttributeError(name)
