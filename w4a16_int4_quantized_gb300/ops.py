"""Thin Python binding over the C ABI of libw4gb300 (include/w4.h).

Argument marshalling only: every function passes torch tensors' device
pointers, sizes and the current CUDA stream to the ``w4_*`` entry point of
the same name, and raises ``W4Error`` on a non-OK status.  All arithmetic
runs in the library's CUDA kernels; if the library is missing this module
raises on import of the first call -- there is no CPU fallback.

``raw`` is the ctypes handle itself, for callers (and tests) that want to
drive the C functions with plain pointers.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libw4gb300.so")

W4_OK, W4_EINVAL, W4_ESHAPE, W4_ECUDA = 0, 1, 2, 3
LAYOUT_ROWMAJOR, LAYOUT_N64, LAYOUT_B32 = 0, 1, 2
FLAG_PDL = 1
OP_LINEAR_Q4, OP_LINEAR_Q8, OP_LINEAR_W4A16, OP_LINEAR_Q4_GROUP, OP_LINEAR_W8A16 = 0, 1, 2, 3, 4
CHAIN_MAX_LINEARS, CHAIN_MAX_K = 64, 8192


class ChainLinear(C.Structure):
    """w4_chain_linear of include/w4.h."""
    _fields_ = [("w", C.c_void_p), ("sw", C.c_void_p), ("y", C.c_void_p),
                ("N", C.c_int32), ("K", C.c_int32), ("input", C.c_int32), ("reserved", C.c_int32)]


# (name, restype, argtypes) of every exported symbol, in header order.
_vp, _i64, _i32, _u32, _sz = C.c_void_p, C.c_int64, C.c_int32, C.c_uint32, C.c_size_t
SIGNATURES = [
    ("w4_quantize_row_q8", _i32, [_vp, _i64, _i64, _vp, _vp, _vp, _vp]),
    ("w4_quantize_matrix_q4", _i32, [_vp, _i64, _i64, _vp, _vp, _vp]),
    ("w4_quantize_matrix_q8", _i32, [_vp, _i64, _i64, _vp, _vp, _vp]),
    ("w4_dot_i32_q4", _i32, [_vp, _vp, _i64, _vp, _vp]),
    ("w4_linear_q4", _i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _sz, _u32, _vp]),
    ("w4_linear_q4_f32", _i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _sz, _u32, _vp]),
    ("w4_linear_q8", _i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _sz, _u32, _vp]),
    ("w4_linear_w4a16_group", _i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i32, _vp, _sz, _u32, _vp]),
    ("w4_linear_q4_noalloc", _i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp]),
    ("w4_linear_w8a16", _i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _sz, _u32, _vp]),
    ("w4_linear_q4_group", _i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i32, _vp, _sz, _u32, _vp]),
    ("w4_chain_q4", _i32, [_vp, _i32, _vp, _i32, _i32, _i32, _vp, _sz, _vp]),
    ("w4_chain_q4_test_timeout", _i32, [_vp, _i32, _vp, _i32, _i32, _i32, _vp, _sz, C.c_uint64, _i32, _vp]),
    ("w4_chain_workspace_bytes", _sz, [_vp, _i32, _i32]),
    ("w4_pack_interleaved_n64", _i32, [_vp, _vp, _i64, _i64, _vp]),
    ("w4_pack_block32", _i32, [_vp, _vp, _vp, _i64, _i64, _vp]),
    ("w4_workspace_bytes", _sz, [_i32, _i64, _i64, _i64, _i64]),
    ("w4_device_status", _i32, [_vp, _i32]),
    ("w4_last_cuda_error", _i32, []),
    ("w4_status_string", C.c_char_p, [_i32]),
    ("w4_probe_mma_peak", _i32, [_i32, _vp, _i64, _vp, _vp]),
    ("w4_version", _i32, []),
]


class W4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = raw.w4_status_string(status).decode() if raw is not None else str(status)
        if status == W4_ECUDA and raw is not None:
            msg += f" (cudaError {raw.w4_last_cuda_error()})"
        super().__init__(f"{what}: {msg}")


def load(path: str = LIB_PATH) -> C.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(f"libw4gb300 not built ({path}); run __graft_entry__.build() or "
                           "python -m w4a16_int4_quantized_gb300.build")
    lib = C.CDLL(path)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


raw = load()


def _check(status: int, what: str) -> None:
    if status != W4_OK:
        raise W4Error(status, what)


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr() or None


def _stream(stream=None) -> int | None:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream or None


# ---------------------------------------------------------------- quantizers

def quantize_row_q8(x: torch.Tensor, stream=None):
    """x f32 [M, K] (cuda) -> (q int8 [M, K], sx f32 [M], rowsum int32 [M])."""
    assert x.dtype == torch.float32 and x.is_contiguous() and x.dim() == 2
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    sx = torch.empty(M, dtype=torch.float32, device=x.device)
    rs = torch.empty(M, dtype=torch.int32, device=x.device)
    _check(raw.w4_quantize_row_q8(_ptr(x), M, K, _ptr(q), _ptr(sx), _ptr(rs), _stream(stream)),
           "w4_quantize_row_q8")
    return q, sx, rs


def quantize_matrix_q4(W: torch.Tensor, stream=None):
    """W f32 [N, K] -> (packed uint8 [N, ceil(K/2)], sw f32 [N])."""
    assert W.dtype == torch.float32 and W.is_contiguous() and W.dim() == 2
    N, K = W.shape
    packed = torch.empty((N, (K + 1) // 2), dtype=torch.uint8, device=W.device)
    sw = torch.empty(N, dtype=torch.float32, device=W.device)
    _check(raw.w4_quantize_matrix_q4(_ptr(W), N, K, _ptr(packed), _ptr(sw), _stream(stream)),
           "w4_quantize_matrix_q4")
    return packed, sw


def quantize_matrix_q8(W: torch.Tensor, stream=None):
    """W f32 [N, K] -> (q int8 [N, K], sw f32 [N])."""
    assert W.dtype == torch.float32 and W.is_contiguous() and W.dim() == 2
    N, K = W.shape
    q = torch.empty((N, K), dtype=torch.int8, device=W.device)
    sw = torch.empty(N, dtype=torch.float32, device=W.device)
    _check(raw.w4_quantize_matrix_q8(_ptr(W), N, K, _ptr(q), _ptr(sw), _stream(stream)), "w4_quantize_matrix_q8")
    return q, sw


# ---------------------------------------------------------------- dot / linears

def dot_i32_q4(xq: torch.Tensor, wrow: torch.Tensor, K: int | None = None, stream=None) -> torch.Tensor:
    """Exact biased-Q4 dot of one row -> int32 device scalar."""
    K = xq.numel() if K is None else K
    out = torch.empty(1, dtype=torch.int32, device=xq.device)
    _check(raw.w4_dot_i32_q4(_ptr(xq), _ptr(wrow), K, _ptr(out), _stream(stream)), "w4_dot_i32_q4")
    return out


def _workspace(op, M, N, K, G, workspace, device):
    need = raw.w4_workspace_bytes(op, M, N, K, G)
    if need == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    return workspace, workspace.numel()


def linear_q4(xq, sx, w, sw, K: int | None = None, N: int | None = None, layout: int = LAYOUT_ROWMAJOR,
              flags: int = 0, out=None, workspace=None, stream=None) -> torch.Tensor:
    """W4A8: y[M, N] = (f32(sum xq * (u - 8)) * sx[m]) * sw[n]."""
    M = xq.shape[0]
    K = xq.shape[1] if K is None else K
    N = sw.numel() if N is None else N
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=xq.device)
    ws, wsb = _workspace(OP_LINEAR_Q4, M, N, K, 0, workspace, xq.device)
    _check(raw.w4_linear_q4(_ptr(xq), _ptr(sx), _ptr(w), _ptr(sw), _ptr(y), M, N, K, layout,
                            _ptr(ws), wsb, flags, _stream(stream)), "w4_linear_q4")
    return y


def linear_q4_f32(x, w, sw, K: int | None = None, N: int | None = None, layout: int = LAYOUT_ROWMAJOR,
                  flags: int = 0, out=None, xq=None, sx=None, workspace=None, stream=None):
    """quantize_row_q8(x) then linear_q4 in one call -> (y [M, N], xq [M, K], sx [M])."""
    assert x.dtype == torch.float32 and x.dim() == 2
    M = x.shape[0]
    K = x.shape[1] if K is None else K
    N = sw.numel() if N is None else N
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=x.device)
    xq = xq if xq is not None else torch.empty((M, K), dtype=torch.int8, device=x.device)
    sx = sx if sx is not None else torch.empty(M, dtype=torch.float32, device=x.device)
    ws, wsb = _workspace(OP_LINEAR_Q4, M, N, K, 0, workspace, x.device)
    _check(raw.w4_linear_q4_f32(_ptr(x), _ptr(w), _ptr(sw), _ptr(y), _ptr(xq), _ptr(sx), M, N, K, layout,
                                _ptr(ws), wsb, flags, _stream(stream)), "w4_linear_q4_f32")
    return y, xq, sx


NOALLOC_SCRATCH_BYTES = 8 << 20


def linear_q4_noalloc(xq, sx, w, sw, K: int | None = None, N: int | None = None, layout: int = LAYOUT_ROWMAJOR,
                      out=None, stream=None) -> torch.Tensor:
    """linear_q4 for callers that may not allocate device scratch: large
    batches use the library's fixed NOALLOC_SCRATCH_BYTES array instead (calls
    on one device share it, so keep them on one stream).  `out` must be given
    by callers that may not allocate at all."""
    M = xq.shape[0]
    K = xq.shape[1] if K is None else K
    N = sw.numel() if N is None else N
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=xq.device)
    st = raw.w4_linear_q4_noalloc(_ptr(xq), _ptr(sx), _ptr(w), _ptr(sw), _ptr(y), M, N, K, layout, _stream(stream))
    if st == W4_ESHAPE and raw.w4_workspace_bytes(OP_LINEAR_Q4, M, N, K, 0) > NOALLOC_SCRATCH_BYTES:
        raise W4Error(st, f"w4_linear_q4_noalloc: batch needs {raw.w4_workspace_bytes(OP_LINEAR_Q4, M, N, K, 0)} "
                          f"bytes of scratch, above the fixed {NOALLOC_SCRATCH_BYTES}")
    _check(st, "w4_linear_q4_noalloc")
    return y


def linear_q8(xq, sx, w, sw, flags: int = 0, out=None, workspace=None, stream=None) -> torch.Tensor:
    """W8A8: y[M, N] = (f32(sum xq * w) * sx[m]) * sw[n]."""
    M, K = xq.shape
    N = w.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=xq.device)
    ws, wsb = _workspace(OP_LINEAR_Q8, M, N, K, 0, workspace, xq.device)
    _check(raw.w4_linear_q8(_ptr(xq), _ptr(sx), _ptr(w), _ptr(sw), _ptr(y), M, N, K,
                            _ptr(ws), wsb, flags, _stream(stream)), "w4_linear_q8")
    return y


def linear_w4a16_group(x, w, scales, G: int, K: int | None = None, N: int | None = None,
                       layout: int = LAYOUT_ROWMAJOR, flags: int = 0, out=None, workspace=None,
                       stream=None) -> torch.Tensor:
    """Group-wise W4A16: y = sum_g s[n, g] * sum_{k in g} x[m, k] * q[n, k].

    x: bf16 [M, K] (torch.bfloat16, or int16/uint16 bit patterns);
    w: packed signed nibbles; scales: f16 [N, Kp/G] (torch.float16 or 16-bit patterns).
    """
    assert x.element_size() == 2 and scales.element_size() == 2
    M = x.shape[0]
    K = x.shape[1] if K is None else K
    N = scales.shape[0] if N is None else N
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=x.device)
    ws, wsb = _workspace(OP_LINEAR_W4A16, M, N, K, G, workspace, x.device)
    _check(raw.w4_linear_w4a16_group(_ptr(x), _ptr(w), _ptr(scales), _ptr(y), M, N, K, G, layout,
                                     _ptr(ws), wsb, flags, _stream(stream)), "w4_linear_w4a16_group")
    return y


def linear_w8a16(x, w, sw, flags: int = 0, out=None, workspace=None, stream=None) -> torch.Tensor:
    """W8A16: y[M, N] = sw[n] * sum_k x[m, k] * q[n, k], x f32, q int8."""
    M, K = x.shape
    N = sw.numel()
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=x.device)
    ws, wsb = _workspace(OP_LINEAR_W8A16, M, N, K, 0, workspace, x.device)
    _check(raw.w4_linear_w8a16(_ptr(x), _ptr(w), _ptr(sw), _ptr(y), M, N, K, _ptr(ws), wsb, flags, _stream(stream)),
           "w4_linear_w8a16")
    return y


def linear_q4_group(xq, sx, w, scales, zeros, G: int, K: int | None = None, N: int | None = None,
                    layout: int = LAYOUT_ROWMAJOR, flags: int = 0, out=None, workspace=None,
                    stream=None) -> torch.Tensor:
    """Grouped asymmetric W4A8: y = sx[m] * sum_g (sum_{k in g} xq * (u - z[n, g])) * s[n, g]."""
    M = xq.shape[0]
    K = xq.shape[1] if K is None else K
    N = scales.shape[0] if N is None else N
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=xq.device)
    ws, wsb = _workspace(OP_LINEAR_Q4_GROUP, M, N, K, G, workspace, xq.device)
    _check(raw.w4_linear_q4_group(_ptr(xq), _ptr(sx), _ptr(w), _ptr(scales), _ptr(zeros), _ptr(y), M, N, K, G,
                                  layout, _ptr(ws), wsb, flags, _stream(stream)), "w4_linear_q4_group")
    return y


def chain_descriptors(linears):
    """ctypes array of w4_chain_linear for (w, sw, y, input) tuples."""
    arr = (ChainLinear * len(linears))()
    for i, (w, sw, y, inp) in enumerate(linears):
        arr[i] = ChainLinear(_ptr(w), _ptr(sw), _ptr(y), sw.numel(), 2 * w.shape[-1], inp, 0)
    return arr


def chain_workspace_bytes(linears, K0: int) -> int:
    return raw.w4_chain_workspace_bytes(chain_descriptors(linears), len(linears), K0)


def chain_q4(x0, linears, passes: int, pass_output: int, workspace=None, stream=None):
    """Runs a chain of M = 1 W4A8 linears as one kernel.  linears: sequence of
    (w, sw, y, input) with w packed [N][K/2] uint8, sw [N] f32, y [N] f32
    (written), input = -1 for the pass input or the index of an earlier
    linear.  Returns the y tensors."""
    arr = chain_descriptors(linears)
    need = raw.w4_chain_workspace_bytes(arr, len(linears), x0.numel())
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x0.device)
    _check(raw.w4_chain_q4(_ptr(x0), x0.numel(), arr, len(linears), passes, pass_output, _ptr(workspace),
                           workspace.numel(), _stream(stream)), "w4_chain_q4")
    return [y for _, _, y, _ in linears]


def chain_q4_test_timeout(x0, linears, passes: int, pass_output: int, wait_limit_ns: int, hold_stage: int,
                          workspace=None, stream=None) -> int:
    """w4_chain_q4_test_timeout: the chain with a short wait limit and,
    hold_stage >= 0, one stage whose outputs are never published.  Returns
    the call's status (the device status word reports the timeout)."""
    arr = chain_descriptors(linears)
    need = raw.w4_chain_workspace_bytes(arr, len(linears), x0.numel())
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x0.device)
    return raw.w4_chain_q4_test_timeout(_ptr(x0), x0.numel(), arr, len(linears), passes, pass_output,
                                        _ptr(workspace), workspace.numel(), int(wait_limit_ns), int(hold_stage),
                                        _stream(stream))


def pack_interleaved_n64(w: torch.Tensor, K: int, stream=None) -> torch.Tensor:
    """Row-major packed int4 [N, ceil(K/2)] -> interleaved [N/64, K, 32]."""
    N = w.shape[0]
    il = torch.empty((N // 64, K, 32), dtype=torch.uint8, device=w.device)
    _check(raw.w4_pack_interleaved_n64(_ptr(w), _ptr(il), N, K, _stream(stream)), "w4_pack_interleaved_n64")
    return il


def linear_w4a16_b32(x, blocks, K: int | None = None, N: int | None = None, flags: int = 0, out=None,
                     stream=None) -> torch.Tensor:
    """Group-wise W4A16 (G = 32) reading inline-scale blocks [N][Kp/32 * 18]."""
    assert x.element_size() == 2
    M = x.shape[0]
    K = x.shape[1] if K is None else K
    N = blocks.shape[0] if N is None else N
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=x.device)
    _check(raw.w4_linear_w4a16_group(_ptr(x), _ptr(blocks), None, _ptr(y), M, N, K, 32, LAYOUT_B32, None, 0, flags,
                                     _stream(stream)), "w4_linear_w4a16_group")
    return y


def pack_block32(w: torch.Tensor, scales: torch.Tensor, K: int, stream=None) -> torch.Tensor:
    """W4A16 planes (packed [N][Kp/2], f16 scales [N][Kp/32]) -> inline-scale blocks [N][Kp/32 * 18]."""
    N = w.shape[0]
    nb = (K + (K & 1)) // 32
    out = torch.empty((N, nb * 18), dtype=torch.uint8, device=w.device)
    _check(raw.w4_pack_block32(_ptr(w), _ptr(scales), _ptr(out), N, K, _stream(stream)), "w4_pack_block32")
    return out


def workspace_bytes(op: int, M: int, N: int, K: int, G: int = 0) -> int:
    return int(raw.w4_workspace_bytes(op, M, N, K, G))


def device_status(clear: bool = False) -> int:
    v = C.c_uint32(0)
    _check(raw.w4_device_status(C.byref(v), 1 if clear else 0), "w4_device_status")
    return int(v.value)


def probe_mma_peak(kind: int) -> float:
    """Measured legacy mma.sync throughput in tera-ops/s (0: s8 m16n8k32, 1: bf16 m16n8k16)."""
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    scratch = torch.empty(4 * sms * 256, dtype=torch.int32, device="cuda")
    v = C.c_double(0.0)
    _check(raw.w4_probe_mma_peak(kind, _ptr(scratch), scratch.numel(), C.byref(v), _stream()), "w4_probe_mma_peak")
    return float(v.value)


def version() -> int:
    return int(raw.w4_version())
