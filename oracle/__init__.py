"""CPU oracle for the fused int4 dequantize-matmul -- TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  It wraps the plain C in ``w4_oracle.c`` (built with
gcc, ``-ffp-contract=off``, no fast-math) through ctypes and shares no code
with the CUDA library.  The row-parallel build of the same source
(``openmp=True``) is bitwise identical to the serial one and is what the
benchmark times.

See ``w4_oracle.h`` for the functions, the passages each one follows, and
the one parity-unpinned convention (the order of the two f32 scales).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4_oracle.c")
_HDR = os.path.join(_HERE, "w4_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()

REF_OK, REF_EINVAL, REF_ESHAPE = 0, 1, 2


def lib_path(mutant: int = 0, openmp: bool = False) -> str:
    name = "libw4oracle"
    if openmp:
        name += "_omp"
    if mutant:
        name += f"_mut{mutant}"
    return os.path.join(_BUILD, name + ".so")


def build(mutant: int = 0, openmp: bool = False, force: bool = False) -> str:
    """Compile the oracle (or one planted-mistake variant of it) with gcc."""
    out = lib_path(mutant, openmp)
    with _lock:
        newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
        if not force and os.path.exists(out) and os.path.getmtime(out) >= newest:
            return out
        os.makedirs(_BUILD, exist_ok=True)
        cmd = ["cc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               f"-DW4_ORACLE_MUTANT={int(mutant)}", "-o", out + ".tmp", _SRC, "-lm"]
        if openmp:
            cmd.insert(1, "-fopenmp")
        subprocess.run(cmd, check=True, capture_output=True)
        os.replace(out + ".tmp", out)
    return out


def _p(a):
    return a.ctypes.data_as(C.c_void_p) if a is not None else None


class Oracle:
    """numpy front end to one build of the C oracle."""

    def __init__(self, mutant: int = 0, openmp: bool = False):
        self.lib = C.CDLL(build(mutant, openmp))
        L = self.lib
        i64, vp, i32 = C.c_int64, C.c_void_p, C.c_int
        L.ref_f16_to_f32.restype = C.c_float
        L.ref_f16_to_f32.argtypes = [C.c_uint16]
        L.ref_bf16_to_f32.restype = C.c_float
        L.ref_bf16_to_f32.argtypes = [C.c_uint16]
        L.ref_f32_to_bf16_rne.restype = C.c_uint16
        L.ref_f32_to_bf16_rne.argtypes = [C.c_float]
        L.ref_nibble_signed.restype = i32
        L.ref_nibble_signed.argtypes = [C.c_uint]
        L.ref_nibble_biased.restype = i32
        L.ref_nibble_biased.argtypes = [C.c_uint]
        L.ref_quantize_row.restype = None
        L.ref_quantize_row.argtypes = [vp, i64, i32, vp, vp]
        for name, nargs in (("ref_quantize_row_q8", 6), ("ref_quantize_matrix_q4", 5),
                            ("ref_quantize_matrix_q8", 5)):
            getattr(L, name).restype = i32
        L.ref_quantize_row_q8.argtypes = [vp, i64, i64, vp, vp, vp]
        L.ref_quantize_matrix_q4.argtypes = [vp, i64, i64, vp, vp]
        L.ref_quantize_matrix_q8.argtypes = [vp, i64, i64, vp, vp]
        L.ref_dot_i32_q4.restype = C.c_int32
        L.ref_dot_i32_q4.argtypes = [vp, vp, i64]
        L.ref_dot_naive_q4.restype = C.c_int64
        L.ref_dot_naive_q4.argtypes = [vp, vp, i64]
        L.ref_dot_i32.restype = C.c_int32
        L.ref_dot_i32.argtypes = [vp, vp, i64]
        L.ref_linear_q4.restype = i32
        L.ref_linear_q4.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64]
        L.ref_linear_q8.restype = i32
        L.ref_linear_q8.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64]
        L.ref_linear_w8a32.restype = i32
        L.ref_linear_w8a32.argtypes = [vp, vp, vp, vp, i64, i64, i64]
        L.ref_linear_w4a16_exact.restype = i32
        L.ref_linear_w4a16_exact.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64]
        L.ref_linear_w8a16_exact.restype = i32
        L.ref_linear_w8a16_exact.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64]
        L.ref_blocks_b32.restype = i32
        L.ref_blocks_b32.argtypes = [vp, vp, vp, i64, i64]
        L.ref_linear_w4a16_b32_exact.restype = i32
        L.ref_linear_w4a16_b32_exact.argtypes = [vp, vp, vp, vp, i64, i64, i64]
        L.ref_linear_q4_group.restype = i32
        L.ref_linear_q4_group.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64]
        L.ref_linear_w4a16_lanes.restype = i32
        L.ref_linear_w4a16_lanes.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64]
        L.ref_linear_w4a16_bf16dequant.restype = i32
        L.ref_linear_w4a16_bf16dequant.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64]
        L.ref_pack_interleaved_n64.restype = i32
        L.ref_pack_interleaved_n64.argtypes = [vp, vp, i64, i64]
        L.ref_unpack_interleaved_n64.restype = i32
        L.ref_unpack_interleaved_n64.argtypes = [vp, vp, i64, i64, C.c_uint]
        L.ref_mutant_id.restype = i32
        self.mutant = L.ref_mutant_id()

    # -- element decoders
    def f16_to_f32(self, h: int) -> float:
        return float(self.lib.ref_f16_to_f32(int(h) & 0xFFFF))

    def bf16_to_f32(self, b: int) -> float:
        return float(self.lib.ref_bf16_to_f32(int(b) & 0xFFFF))

    def f32_to_bf16(self, f: float) -> int:
        return int(self.lib.ref_f32_to_bf16_rne(float(np.float32(f))))

    def nibble_signed(self, u: int) -> int:
        return int(self.lib.ref_nibble_signed(u))

    def nibble_biased(self, u: int) -> int:
        return int(self.lib.ref_nibble_biased(u))

    # -- quantizers
    def quantize_row(self, v, Q: int):
        v = np.ascontiguousarray(v, dtype=np.float32).ravel()
        q = np.zeros(v.size, np.int8)
        s = np.zeros(1, np.float32)
        self.lib.ref_quantize_row(_p(v), v.size, int(Q), _p(q), _p(s))
        return q, float(s[0])

    def quantize_row_q8(self, x):
        x = np.ascontiguousarray(x, dtype=np.float32)
        M, K = x.shape
        q = np.zeros((M, K), np.int8)
        sx = np.zeros(M, np.float32)
        rs = np.zeros(M, np.int32)
        rc = self.lib.ref_quantize_row_q8(_p(x), M, K, _p(q), _p(sx), _p(rs))
        assert rc == REF_OK, rc
        return q, sx, rs

    def quantize_matrix_q4(self, W):
        W = np.ascontiguousarray(W, dtype=np.float32)
        N, K = W.shape
        packed = np.zeros((N, (K + 1) // 2), np.uint8)
        sw = np.zeros(N, np.float32)
        rc = self.lib.ref_quantize_matrix_q4(_p(W), N, K, _p(packed), _p(sw))
        assert rc == REF_OK, rc
        return packed, sw

    def quantize_matrix_q8(self, W):
        W = np.ascontiguousarray(W, dtype=np.float32)
        N, K = W.shape
        q = np.zeros((N, K), np.int8)
        sw = np.zeros(N, np.float32)
        rc = self.lib.ref_quantize_matrix_q8(_p(W), N, K, _p(q), _p(sw))
        assert rc == REF_OK, rc
        return q, sw

    # -- dots
    def dot_i32_q4(self, xq, wrow, K: int) -> int:
        xq = np.ascontiguousarray(xq, dtype=np.int8)
        wrow = np.ascontiguousarray(wrow, dtype=np.uint8)
        return int(self.lib.ref_dot_i32_q4(_p(xq), _p(wrow), int(K)))

    def dot_naive_q4(self, xq, wrow, K: int) -> int:
        xq = np.ascontiguousarray(xq, dtype=np.int8)
        wrow = np.ascontiguousarray(wrow, dtype=np.uint8)
        return int(self.lib.ref_dot_naive_q4(_p(xq), _p(wrow), int(K)))

    def dot_i32(self, a, b) -> int:
        a = np.ascontiguousarray(a, dtype=np.int8)
        b = np.ascontiguousarray(b, dtype=np.int8)
        return int(self.lib.ref_dot_i32(_p(a), _p(b), a.size))

    # -- linears
    def linear_q4(self, xq, sx, w, sw, K: int):
        xq = np.ascontiguousarray(xq, dtype=np.int8)
        sx = np.ascontiguousarray(sx, dtype=np.float32)
        w = np.ascontiguousarray(w, dtype=np.uint8)
        sw = np.ascontiguousarray(sw, dtype=np.float32)
        M, N = xq.shape[0], w.shape[0]
        y = np.zeros((M, N), np.float32)
        rc = self.lib.ref_linear_q4(_p(xq), _p(sx), _p(w), _p(sw), _p(y), M, N, int(K))
        assert rc == REF_OK, rc
        return y

    def linear_q8(self, xq, sx, wq, sw):
        xq = np.ascontiguousarray(xq, dtype=np.int8)
        sx = np.ascontiguousarray(sx, dtype=np.float32)
        wq = np.ascontiguousarray(wq, dtype=np.int8)
        sw = np.ascontiguousarray(sw, dtype=np.float32)
        M, K = xq.shape
        N = wq.shape[0]
        y = np.zeros((M, N), np.float32)
        rc = self.lib.ref_linear_q8(_p(xq), _p(sx), _p(wq), _p(sw), _p(y), M, N, K)
        assert rc == REF_OK, rc
        return y

    def linear_w8a32(self, x, wq, s):
        x = np.ascontiguousarray(x, dtype=np.float32)
        wq = np.ascontiguousarray(wq, dtype=np.int8)
        s = np.ascontiguousarray(s, dtype=np.float32)
        M, K = x.shape
        N = wq.shape[0]
        y = np.zeros((M, N), np.float32)
        rc = self.lib.ref_linear_w8a32(_p(x), _p(wq), _p(s), _p(y), M, N, K)
        assert rc == REF_OK, rc
        return y

    def _w4a16_args(self, x, w, s):
        x = np.ascontiguousarray(x, dtype=np.uint16)
        w = np.ascontiguousarray(w, dtype=np.uint8)
        s = np.ascontiguousarray(s, dtype=np.uint16)
        return x, w, s

    def linear_w4a16_exact(self, x, w, s, K: int, G: int):
        x, w, s = self._w4a16_args(x, w, s)
        M, N = x.shape[0], w.shape[0]
        y = np.zeros((M, N), np.float64)
        a = np.zeros((M, N), np.float64)
        rc = self.lib.ref_linear_w4a16_exact(_p(x), _p(w), _p(s), _p(y), _p(a), M, N, int(K), int(G))
        assert rc == REF_OK, rc
        return y, a

    def linear_w8a16_exact(self, x, wq, sw):
        """linear_w8a16 in double: (y64, abs64)."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        wq = np.ascontiguousarray(wq, dtype=np.int8)
        sw = np.ascontiguousarray(sw, dtype=np.float32)
        M, K = x.shape
        N = wq.shape[0]
        y = np.zeros((M, N), np.float64)
        a = np.zeros((M, N), np.float64)
        rc = self.lib.ref_linear_w8a16_exact(_p(x), _p(wq), _p(sw), _p(y), _p(a), M, N, K)
        assert rc == REF_OK, rc
        return y, a

    def blocks_b32(self, w, s, K: int):
        w = np.ascontiguousarray(w, dtype=np.uint8)
        s = np.ascontiguousarray(s, dtype=np.uint16)
        N = w.shape[0]
        nb = (K + (K & 1)) // 32
        out = np.zeros((N, nb * 18), np.uint8)
        rc = self.lib.ref_blocks_b32(_p(w), _p(s), _p(out), N, int(K))
        assert rc == REF_OK, rc
        return out

    def linear_w4a16_b32_exact(self, x, blocks, K: int):
        x = np.ascontiguousarray(x, dtype=np.uint16)
        blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
        M, N = x.shape[0], blocks.shape[0]
        y = np.zeros((M, N), np.float64)
        a = np.zeros((M, N), np.float64)
        rc = self.lib.ref_linear_w4a16_b32_exact(_p(x), _p(blocks), _p(y), _p(a), M, N, int(K))
        assert rc == REF_OK, rc
        return y, a

    def linear_q4_group(self, xq, sx, w, s, z, K: int, G: int):
        """Grouped asymmetric W4A8 in double: (y64, abs64)."""
        xq = np.ascontiguousarray(xq, dtype=np.int8)
        sx = np.ascontiguousarray(sx, dtype=np.float32)
        w = np.ascontiguousarray(w, dtype=np.uint8)
        s = np.ascontiguousarray(s, dtype=np.uint16)
        z = np.ascontiguousarray(z, dtype=np.uint8)
        M, N = xq.shape[0], w.shape[0]
        y = np.zeros((M, N), np.float64)
        a = np.zeros((M, N), np.float64)
        rc = self.lib.ref_linear_q4_group(_p(xq), _p(sx), _p(w), _p(s), _p(z), _p(y), _p(a), M, N, int(K), int(G))
        assert rc == REF_OK, rc
        return y, a

    def linear_w4a16_lanes(self, x, w, s, K: int, G: int):
        x, w, s = self._w4a16_args(x, w, s)
        M, N = x.shape[0], w.shape[0]
        y = np.zeros((M, N), np.float32)
        rc = self.lib.ref_linear_w4a16_lanes(_p(x), _p(w), _p(s), _p(y), M, N, int(K), int(G))
        assert rc == REF_OK, rc
        return y

    def linear_w4a16_bf16dequant(self, x, w, s, K: int, G: int):
        x, w, s = self._w4a16_args(x, w, s)
        M, N = x.shape[0], w.shape[0]
        y = np.zeros((M, N), np.float64)
        rc = self.lib.ref_linear_w4a16_bf16dequant(_p(x), _p(w), _p(s), _p(y), M, N, int(K), int(G))
        assert rc == REF_OK, rc
        return y

    def w4a16_status(self, M, N, K, G) -> int:
        """Return code of the W4A16 shape check alone (no data read)."""
        x = np.zeros(max(M * K, 1), np.uint16)
        w = np.zeros(max(N * ((K + 1) // 2), 1), np.uint8)
        s = np.zeros(max(N * 8, 1), np.uint16)
        y = np.zeros(max(M * N, 1), np.float32)
        if M < 0 or N < 0 or K < 0 or G <= 0 or G % 2 or (K + (K & 1)) % G:
            return int(self.lib.ref_linear_w4a16_lanes(_p(x), _p(w), _p(s), _p(y), M, N, K, G))
        return REF_OK

    # -- interleaved layout
    def pack_interleaved_n64(self, w_rm, K: int):
        w_rm = np.ascontiguousarray(w_rm, dtype=np.uint8)
        N = w_rm.shape[0]
        out = np.zeros((N // 64, K, 32), np.uint8)
        rc = self.lib.ref_pack_interleaved_n64(_p(w_rm), _p(out), N, int(K))
        assert rc == REF_OK, rc
        return out

    def unpack_interleaved_n64(self, w_il, N: int, K: int, pad: int):
        w_il = np.ascontiguousarray(w_il, dtype=np.uint8)
        out = np.zeros((N, (K + 1) // 2), np.uint8)
        rc = self.lib.ref_unpack_interleaved_n64(_p(w_il), _p(out), int(N), int(K), int(pad))
        assert rc == REF_OK, rc
        return out


_cache: dict = {}


def get(mutant: int = 0, openmp: bool = False) -> Oracle:
    key = (mutant, openmp)
    if key not in _cache:
        _cache[key] = Oracle(mutant, openmp)
    return _cache[key]
