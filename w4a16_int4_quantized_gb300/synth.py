"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module holds input generation only: a counter-based splitmix64 stream,
Box-Muller normals, and the rounding of those draws to the storage types the
kernels take (f32, bf16, f16 bit patterns, raw bytes).  It contains none of
the quantize / dot / linear arithmetic; that lives in the oracle (C, under
``oracle/``) and in the CUDA kernels, which never import each other.

Recipes follow the workloads of the pages:
  * weights W ~ N(0, 0.02) in f32, activations x ~ N(0, 1)
    (ftts-kernels int4 / int8 module docs: per-output-channel symmetric Q4/Q8);
  * group-wise W4A16: raw uniform bytes as signed nibbles, f16 scales
    |N(0, 0.01)| + 1e-4, x in bf16 ("Fused int4 and int8 dequantize-matmul in C",
    section 2.2 layout);
  * seeds are 1000 + workload index.
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """Counter-based splitmix64: element i is mix(seed + (offset + i + 1) * golden)."""
    with np.errstate(over="ignore"):
        ctr = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + ctr * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """Uniform doubles in the open interval (0, 1) from the top 53 bits."""
    z = splitmix64(seed, n, offset)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def normal(seed: int, n: int, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    """Box-Muller normals in double precision (pairs of uniforms -> cos branch)."""
    u1 = uniform01(seed, n, 0)
    u2 = uniform01(seed ^ 0x5DEECE66D, n, 0)
    r = np.sqrt(-2.0 * np.log(u1))
    return mean + std * r * np.cos(2.0 * np.pi * u2)


def raw_bytes(seed: int, n: int) -> np.ndarray:
    """n uniformly random bytes."""
    words = splitmix64(seed, (n + 7) // 8)
    return words.view(np.uint8)[:n].copy()


# ---------------------------------------------------------------- storage types

def to_f32(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round f32 values to bf16 (round-to-nearest-even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(np.asarray(a, dtype=np.float32))
    rounded = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    out = rounded.astype(np.uint16)
    out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_f16_bits(a: np.ndarray) -> np.ndarray:
    """Round to IEEE half (numpy's round-to-nearest-even) and return the bit patterns."""
    return np.ascontiguousarray(a, dtype=np.float64).astype(np.float16).view(np.uint16)


# ---------------------------------------------------------------- recipes

def weights_f32(seed: int, n: int, k: int, std: float = 0.02) -> np.ndarray:
    """Dense f32 weight [n, k] ~ N(0, std)."""
    return to_f32(normal(seed, n * k, std).reshape(n, k))


def activations_f32(seed: int, m: int, k: int, std: float = 1.0) -> np.ndarray:
    """Dense f32 activations [m, k] ~ N(0, std)."""
    return to_f32(normal(seed, m * k, std).reshape(m, k))


def activations_bf16(seed: int, m: int, k: int) -> np.ndarray:
    """bf16 bit patterns [m, k] of N(0, 1) draws."""
    return f32_to_bf16_bits(normal(seed, m * k, 1.0).astype(np.float32)).reshape(m, k)


def packed_signed_nibbles(seed: int, n: int, k: int) -> np.ndarray:
    """Row-major packed int4 [n, ceil(k/2)] of uniform random nibbles.

    For odd k the unused high nibble of each row's last byte is set to 0x0,
    the signed code whose value is zero.
    """
    kb = (k + 1) // 2
    b = raw_bytes(seed, n * kb).reshape(n, kb)
    if k % 2:
        b[:, -1] &= 0x0F
    return b


def group_scales_f16(seed: int, n: int, ngroups: int) -> np.ndarray:
    """f16 bit patterns [n, ngroups] of |N(0, 0.01)| + 1e-4."""
    v = np.abs(normal(seed, n * ngroups, 0.01)) + 1e-4
    return to_f16_bits(v).reshape(n, ngroups)


def w4a16_inputs(seed: int, m: int, n: int, k: int, g: int):
    """(x_bf16 [m,k], packed [n,ceil(k/2)], scales_f16 [n, kp/g]) for group-wise W4A16."""
    kp = k + (k & 1)
    x = activations_bf16(seed, m, k)
    w = packed_signed_nibbles(seed + 1, n, k)
    s = group_scales_f16(seed + 2, n, kp // g)
    return x, w, s


def w4a8_inputs(seed: int, m: int, n: int, k: int):
    """(x_f32 [m,k] ~ N(0,1), W_f32 [n,k] ~ N(0,0.02)) before quantization."""
    return activations_f32(seed, m, k), weights_f32(seed + 1, n, k)


def q4_group_inputs(seed: int, m: int, n: int, k: int, g: int):
    """Grouped asymmetric W4A8 inputs: int8 codes xq [m, k] in [-127, 127],
    sx [m] in [0.5, 1.5), raw nibbles (every value 0..15) packed [n, kp/2],
    f16 scales and zero points 0..15, both [n, kp/g]."""
    kp = k + (k & 1)
    xq = raw_bytes(seed, m * k).view(np.int8).reshape(m, k).copy()
    xq[xq == -128] = -127
    sx = (uniform01(seed + 1, m) + 0.5).astype(np.float32)
    w = raw_bytes(seed + 2, n * (kp // 2)).reshape(n, kp // 2)
    s = group_scales_f16(seed + 3, n, kp // g)
    z = (raw_bytes(seed + 4, n * (kp // g)) & 0x0F).reshape(n, kp // g)
    return xq, sx, w, s, z


MICRODECODER_LAYERS = 5
MICRODECODER_PASSES = 15
# (name, N, K) of one microdecoder layer, in dataflow order.
MICRODECODER_LINEARS = (
    ("q", 1024, 1024), ("k", 1024, 1024), ("v", 1024, 1024), ("o", 1024, 1024),
    ("gate", 3072, 1024), ("up", 3072, 1024), ("down", 1024, 3072),
)


def microdecoder_weights(seed: int):
    """List over layers of {name: W_f32 [N, K]} with W ~ N(0, 0.02)."""
    layers = []
    s = seed
    for _ in range(MICRODECODER_LAYERS):
        d = {}
        for name, n, k in MICRODECODER_LINEARS:
            s += 1
            d[name] = weights_f32(s, n, k)
        layers.append(d)
    return layers
