"""The C-ABI library on the host: it loads without a GPU, exports every symbol
include/w4.h declares, and validates arguments before touching the device
(error order of "Fused int4 and int8 dequantize-matmul in C", section 4:
EINVAL for negative dims / NULL pointers, ESHAPE for shapes the layout cannot
describe, M or N == 0 a no-op).  Only calls that fail validation or return
before any launch run here: no CUDA work is attempted."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4.h")


@pytest.fixture(scope="module")
def lib():
    from w4a16_int4_quantized_gb300 import build
    build.build()
    from w4a16_int4_quantized_gb300 import ops
    return ops


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w4_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("w4_quantize_row_q8", "w4_quantize_matrix_q4", "w4_dot_i32_q4", "w4_linear_q4",
                 "w4_linear_q8", "w4_linear_w4a16_group", "w4_pack_interleaved_n64"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    syms = declared_symbols()
    assert syms
    missing = [s for s in syms if not hasattr(lib.raw, s)]
    assert not missing, missing
    bound = {name for name, _, _ in lib.SIGNATURES}
    assert set(syms) == bound, set(syms) ^ bound


def test_version_and_strings(lib):
    assert lib.version() >= 100
    assert lib.raw.w4_status_string(2).decode().startswith("W4_ESHAPE")


FAKE = C.c_void_p(0x1000)   # never dereferenced: validation rejects the call first


def test_linear_q4_validation(lib):
    r = lib.raw
    f = lambda M, N, K, layout=0, y=FAKE, x=FAKE, w=FAKE: r.w4_linear_q4(x, FAKE, w, FAKE, y, M, N, K, layout,
                                                                          None, 0, 0, None)
    assert f(-1, 4, 4) == lib.W4_EINVAL
    assert f(1, -4, 4) == lib.W4_EINVAL
    assert f(1, 4, -4) == lib.W4_EINVAL
    assert f(1, 4, 4, layout=7) == lib.W4_EINVAL
    assert f(1, 65, 4, layout=1) == lib.W4_ESHAPE        # interleaved layout needs N % 64 == 0
    assert f(1, 4, 2_000_000) == lib.W4_ESHAPE           # i32 accumulator bound
    assert f(0, 4, 4) == lib.W4_OK                       # M == 0: nothing launched
    assert f(4, 0, 4) == lib.W4_OK
    assert f(1, 4, 4, y=None) == lib.W4_EINVAL
    assert f(1, 4, 4, w=None) == lib.W4_EINVAL
    assert f(1, 4, 4, x=None) == lib.W4_EINVAL


def test_linear_w4a16_validation(lib):
    r = lib.raw
    f = lambda M, N, K, G, layout=0, s=FAKE: r.w4_linear_w4a16_group(FAKE, FAKE, s, FAKE, M, N, K, G, layout,
                                                                      None, 0, 0, None)
    assert f(1, 2, 4, 3) == lib.W4_ESHAPE     # G odd
    assert f(1, 2, 4, 0) == lib.W4_ESHAPE     # G <= 0
    assert f(1, 2, 4, -2) == lib.W4_ESHAPE
    assert f(1, 2, 12, 8) == lib.W4_ESHAPE    # Kp % G != 0
    assert f(1, 2, 2047, 48) == lib.W4_ESHAPE  # odd K: Kp = 2048, not a multiple of 48
    assert f(-1, 2, 4, 2) == lib.W4_EINVAL
    assert f(0, 2, 4, 2) == lib.W4_OK
    assert f(1, 2, 4, 2, s=None) == lib.W4_EINVAL
    assert f(1, 65, 4, 2, layout=1) == lib.W4_ESHAPE


def test_other_validation(lib):
    r = lib.raw
    assert r.w4_quantize_row_q8(FAKE, -1, 4, FAKE, FAKE, None, None) == lib.W4_EINVAL
    assert r.w4_quantize_row_q8(FAKE, 0, 4, FAKE, FAKE, None, None) == lib.W4_OK
    assert r.w4_quantize_row_q8(FAKE, 2, 4, FAKE, None, None, None) == lib.W4_EINVAL
    assert r.w4_quantize_matrix_q4(FAKE, 3, -1, FAKE, FAKE, None) == lib.W4_EINVAL
    assert r.w4_quantize_matrix_q4(None, 0, 8, None, None, None) == lib.W4_OK
    assert r.w4_quantize_matrix_q8(FAKE, 3, 4, FAKE, None, None) == lib.W4_EINVAL
    assert r.w4_dot_i32_q4(FAKE, FAKE, -1, FAKE, None) == lib.W4_EINVAL
    assert r.w4_dot_i32_q4(FAKE, FAKE, 2_000_000, FAKE, None) == lib.W4_ESHAPE
    assert r.w4_dot_i32_q4(FAKE, FAKE, 8, None, None) == lib.W4_EINVAL
    assert r.w4_pack_interleaved_n64(FAKE, FAKE, 100, 8, None) == lib.W4_ESHAPE
    assert r.w4_pack_interleaved_n64(FAKE, FAKE, 0, 8, None) == lib.W4_OK
    assert r.w4_linear_q8(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 200_000, None, 0, 0, None) == lib.W4_ESHAPE
    assert r.w4_linear_q8(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 8, None, 0, 0, None) == lib.W4_EINVAL
    assert r.w4_device_status(None, 0) == lib.W4_EINVAL


def test_workspace_query_is_host_only(lib):
    for op in (lib.OP_LINEAR_Q4, lib.OP_LINEAR_Q8, lib.OP_LINEAR_W4A16):
        assert lib.workspace_bytes(op, 1, 2048, 2048, 128) == 0        # decode needs no scratch
        assert lib.workspace_bytes(op, 2048, 2048, 2048, 128) >= 0


def test_chain_validation(lib):
    """w4_chain_q4 rejects malformed chains on the host, in the header's order."""
    r = lib.raw
    mk = lambda *rows: (lib.ChainLinear * len(rows))(*[lib.ChainLinear(0x1000, 0x2000, 0x3000, N, K, inp, 0)
                                                         for N, K, inp in rows])
    ws = C.c_void_p(0x4000)
    f = lambda arr, n=None, K0=64, passes=2, po=None, x0=FAKE, wsb=1 << 20: r.w4_chain_q4(
        x0, K0, arr, len(arr) if n is None else n, passes, (len(arr) - 1) if po is None else po, ws, wsb, None)
    ok = mk((96, 64, -1), (64, 96, 0))                    # h(64) -> 96 -> 64 = next h
    assert f(ok, passes=0) == lib.W4_OK                   # nothing to run: no launch
    assert f(ok, n=0) == lib.W4_EINVAL
    assert f(ok, n=65) == lib.W4_EINVAL
    assert f(ok, passes=-1) == lib.W4_EINVAL
    assert f(ok, K0=0) == lib.W4_EINVAL
    assert f(ok, po=2) == lib.W4_EINVAL
    assert f(mk((96, 64, 0), (64, 96, 0))) == lib.W4_EINVAL            # input must be an earlier linear
    assert f(mk((96, 64, -1), (64, 96, -2))) == lib.W4_EINVAL
    bad = mk((96, 64, -1), (64, 96, 0))
    bad[1].reserved = 1
    assert f(bad) == lib.W4_EINVAL
    assert f(mk((96, 48, -1), (48, 96, 0)), K0=48) == lib.W4_ESHAPE    # K % 32
    assert f(mk((96, 64, -1), (64, 64, 0))) == lib.W4_ESHAPE            # K is not the input's length
    assert f(mk((96, 64, -1), (32, 96, 0))) == lib.W4_ESHAPE            # pass output N != K0 with passes > 1
    assert f(mk((64, 64, -1), (64, 64, 0)), po=0) == lib.W4_ESHAPE     # pass output of depth 0 races its readers
    # depth rule: the two depth-1 linears read different vectors
    assert f(mk((64, 64, -1), (64, 64, -1), (64, 64, 0), (64, 64, 1)), po=3) == lib.W4_ESHAPE
    assert f(ok, x0=None) == lib.W4_EINVAL
    assert f(ok, x0=C.c_void_p(0x1004)) == lib.W4_EINVAL                # x0 not 16-byte aligned
    need = r.w4_chain_workspace_bytes(ok, 2, 64)
    assert need == 256 + 8 * (2 * 64 + 96)                              # header + pass output x2 + linear 0
    assert f(ok, wsb=need - 1) == lib.W4_EINVAL                          # workspace too small
    assert r.w4_chain_workspace_bytes(None, 2, 64) == 0


def test_chain_timeout_entry_validation(lib):
    """The timeout test entry point checks its own two arguments first, then
    the chain exactly as w4_chain_q4 does (passes = 0: nothing launches)."""
    r = lib.raw
    rows = [(96, 64, -1), (64, 96, 0)]
    arr = (lib.ChainLinear * 2)(*[lib.ChainLinear(0x1000, 0x2000, 0x3000, N, K, inp, 0) for N, K, inp in rows])
    ws = C.c_void_p(0x4000)
    f = lambda wait_ns, hold, n=2, passes=0, K0=64: r.w4_chain_q4_test_timeout(
        FAKE, K0, arr, n, passes, 1, ws, 1 << 20, wait_ns, hold, None)
    assert f(1_000_000, -1) == lib.W4_OK
    assert f(1_000_000, 7) == lib.W4_OK                   # no stage has index 7: nothing is held
    assert f(1, -1) == lib.W4_OK and f(1_000_000_000, -1) == lib.W4_OK
    assert f(0, -1) == lib.W4_EINVAL
    assert f(1_000_000_001, -1) == lib.W4_EINVAL
    assert f(1_000_000, -2) == lib.W4_EINVAL
    assert f(1_000_000, -1, n=0) == lib.W4_EINVAL          # then the chain's own checks
    assert f(1_000_000, -1, K0=48) == lib.W4_ESHAPE


def test_linear_q4_group_validation(lib):
    r = lib.raw
    f = lambda M, N, K, G, layout=0, z=FAKE: r.w4_linear_q4_group(FAKE, FAKE, FAKE, FAKE, z, FAKE, M, N, K, G,
                                                                  layout, None, 0, 0, None)
    assert f(-1, 2, 4, 2) == lib.W4_EINVAL
    assert f(1, 2, 4, 2, layout=5) == lib.W4_EINVAL
    assert f(1, 2, 4, 3) == lib.W4_ESHAPE          # G odd
    assert f(1, 2, 12, 8) == lib.W4_ESHAPE         # Kp % G
    assert f(1, 65, 4, 2, layout=1) == lib.W4_ESHAPE
    assert f(0, 2, 4, 2) == lib.W4_OK
    assert f(1, 2, 4, 2, z=None) == lib.W4_EINVAL  # zero points required
    assert lib.workspace_bytes(lib.OP_LINEAR_Q4_GROUP, 1, 2048, 2048, 128) == 0
    assert lib.workspace_bytes(lib.OP_LINEAR_Q4_GROUP, 2048, 2048, 2048, 128) > 0


def test_linear_w8a16_validation(lib):
    r = lib.raw
    f = lambda M, N, K, y=FAKE, x=FAKE: r.w4_linear_w8a16(x, FAKE, FAKE, y, M, N, K, None, 0, 0, None)
    assert f(-1, 4, 4) == lib.W4_EINVAL
    assert f(0, 4, 4) == lib.W4_OK
    assert f(1, 4, 4, y=None) == lib.W4_EINVAL
    assert f(1, 4, 4, x=None) == lib.W4_EINVAL
    assert lib.workspace_bytes(lib.OP_LINEAR_W8A16, 1, 2048, 2048) == 0
    assert lib.workspace_bytes(lib.OP_LINEAR_W8A16, 2048, 2048, 2048) == 2048 * 2048 * 2


def test_block32_validation(lib):
    r = lib.raw
    f = lambda K, G, layout=2, s=None: r.w4_linear_w4a16_group(FAKE, FAKE, s, FAKE, 1, 8, K, G, layout, None, 0, 0, None)
    assert f(64, 64) == lib.W4_ESHAPE          # blocks are groups of 32
    assert f(64, 32, layout=3) == lib.W4_EINVAL
    assert f(64, 32, layout=0) == lib.W4_EINVAL  # the plane layouts need the scales
    assert r.w4_linear_q4(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 4, 2, None, 0, 0, None) == lib.W4_EINVAL
    assert r.w4_pack_block32(FAKE, FAKE, FAKE, 4, 48, None) == lib.W4_ESHAPE
    assert r.w4_pack_block32(FAKE, FAKE, FAKE, 0, 64, None) == lib.W4_OK


def test_linear_q4_f32_validation(lib):
    r = lib.raw
    f = lambda M=1, N=8, K=64, layout=0, sx=FAKE, xq=FAKE: r.w4_linear_q4_f32(
        FAKE, FAKE, FAKE, FAKE, xq, sx, M, N, K, layout, None, 0, 0, None)
    assert f(layout=3) == lib.W4_EINVAL
    assert f(K=1000001) == lib.W4_ESHAPE
    assert f(layout=1, N=100) == lib.W4_ESHAPE
    assert f(sx=None) == lib.W4_EINVAL
    assert f(xq=None) == lib.W4_EINVAL
    assert f(M=0) == lib.W4_OK
    assert f(M=-1) == lib.W4_EINVAL


def test_workspace_bytes_formula(lib):
    """Scratch of the tensor-core GEMM: the f16 image of the int8 / f32
    activations, M * round_up(K, 8) * 2 bytes for M > 16; none for W4A16 or
    the decode kernels."""
    r = lib.raw
    ops = lib
    for op in (ops.OP_LINEAR_Q4, ops.OP_LINEAR_Q8, ops.OP_LINEAR_Q4_GROUP, ops.OP_LINEAR_W8A16):
        assert r.w4_workspace_bytes(op, 16, 2048, 2048, 128) == 0
        assert r.w4_workspace_bytes(op, 17, 2048, 2048, 128) == 17 * 2048 * 2
        assert r.w4_workspace_bytes(op, 2048, 13312, 2047, 128) == 2048 * 2048 * 2
        assert r.w4_workspace_bytes(op, 32, 64, 100, 4) == 32 * 104 * 2
        assert r.w4_workspace_bytes(op, 32, 0, 100, 4) == 0
        assert r.w4_workspace_bytes(op, 32, 64, 0, 4) == 0
    assert r.w4_workspace_bytes(ops.OP_LINEAR_W4A16, 2048, 13312, 2048, 128) == 0
    assert r.w4_workspace_bytes(99, 2048, 13312, 2048, 128) == 0


def test_noalloc_validation(lib):
    r = lib.raw
    f = lambda M=1, N=8, K=64, layout=0: r.w4_linear_q4_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, M, N, K, layout, None)
    assert f(M=4096, K=2048) == lib.W4_ESHAPE      # 16 MiB of scratch > the fixed 8 MiB
    assert f(layout=3) == lib.W4_EINVAL
    assert f(K=2_000_000) == lib.W4_ESHAPE
    assert f(M=-1) == lib.W4_EINVAL
    assert f(M=0) == lib.W4_OK


def test_probe_and_version(lib):
    r = lib.raw
    v = C.c_double(0.0)
    assert r.w4_probe_mma_peak(2, FAKE, 1 << 20, C.byref(v), None) == lib.W4_EINVAL   # unknown kind
    assert r.w4_probe_mma_peak(0, None, 1 << 20, C.byref(v), None) == lib.W4_EINVAL   # no scratch
    assert r.w4_probe_mma_peak(1, FAKE, 1 << 20, None, None) == lib.W4_EINVAL        # no result pointer
    ver = r.w4_version()
    assert ver >= 100 and ver // 10000 < 100


def test_missing_library_fails_loudly(lib):
    """No fallback: without the built library the binding refuses to load."""
    with pytest.raises(RuntimeError, match="not built"):
        lib.load(os.path.join(ROOT, "no_such_dir", "libw4gb300.so"))


def test_product_never_touches_the_oracle():
    """The package (binding, build script, generators) neither imports nor
    names the oracle's module or library: the oracle is test infrastructure."""
    pkg = os.path.join(ROOT, "w4a16_int4_quantized_gb300")
    files = [os.path.join(pkg, f) for f in os.listdir(pkg) if f.endswith(".py")]
    csrc = os.path.join(pkg, "csrc")
    files += [os.path.join(csrc, f) for f in os.listdir(csrc)]
    for path in files:
        text = open(path, encoding="utf-8").read()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), path
        assert "w4oracle" not in text and "w4_oracle" not in text, path
