"""w4_linear_q4_noalloc: the W4A8 linear for callers that cannot allocate
device memory while they run (a serving process with a memory budget fixed
at start-up, a host framework whose allocator owns the device, a loop where
an allocation could block).  Large batches use a fixed scratch array inside
the library instead of caller workspace; the result must be the same as
w4_linear_q4's and the CPU oracle's, bit for bit (the W4A8 bar), on
consecutive calls that reuse that array with different shapes.

This file is collected last on purpose, and passes alone in a fresh process
as well as after the rest of the suite.
"""
import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from w4a16_int4_quantized_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a16_int4_quantized_gb300 import build
    build.build()
    from w4a16_int4_quantized_gb300 import ops as o
    return o


def _case(ops, seed, M, N, K):
    x, W = synth.w4a8_inputs(seed, M, N, K)
    xq, sx, _ = ops.quantize_row_q8(torch.from_numpy(x).cuda())
    w, sw = ops.quantize_matrix_q4(torch.from_numpy(W).cuda())
    return xq, sx, w, sw


def _reference(ops, xq, sx, w, sw, M, N, K):
    """The existing entry point, with caller-allocated workspace."""
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    need = ops.raw.w4_workspace_bytes(ops.OP_LINEAR_Q4, M, N, K, 0)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    st = ops.raw.w4_linear_q4(xq.data_ptr(), sx.data_ptr(), w.data_ptr(), sw.data_ptr(), y.data_ptr(), M, N, K,
                              ops.LAYOUT_ROWMAJOR, ws.data_ptr(), need, 0, None)
    assert st == ops.W4_OK
    return y


def _noalloc(ops, xq, sx, w, sw, M, N, K):
    y = torch.full((M, N), -1.0, dtype=torch.float32, device="cuda")
    st = ops.raw.w4_linear_q4_noalloc(xq.data_ptr(), sx.data_ptr(), w.data_ptr(), sw.data_ptr(), y.data_ptr(),
                                      M, N, K, ops.LAYOUT_ROWMAJOR, None)
    assert st == ops.W4_OK
    return y


def test_noalloc_matches_linear_q4_on_consecutive_calls(ops):
    # two different batches back to back: the second reuses (and must fully
    # rewrite) the scratch the first one filled; both take the tensor-core
    # path that needs scratch (M > 16)
    for seed, (M, N, K) in ((301, (300, 256, 1024)), (302, (64, 384, 2048))):
        assert ops.raw.w4_workspace_bytes(ops.OP_LINEAR_Q4, M, N, K, 0) > 0
        xq, sx, w, sw = _case(ops, seed, M, N, K)
        got = _noalloc(ops, xq, sx, w, sw, M, N, K)
        want = _reference(ops, xq, sx, w, sw, M, N, K)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int32), want.view(torch.int32)), (M, N, K)
        # and directly against the CPU oracle's linear_q4 on the same codes
        import oracle
        ref = oracle.get().linear_q4(xq.cpu().numpy(), sx.cpu().numpy(), w.cpu().numpy(), sw.cpu().numpy(), K)
        assert np.array_equal(got.cpu().numpy().view(np.int32), ref.view(np.int32)), (M, N, K)
    assert ops.device_status() == 0


def test_noalloc_rejects_batches_beyond_the_fixed_scratch(ops):
    M, N, K = 4096, 128, 2048   # needs 16 MiB of scratch, the array holds 8 MiB
    assert ops.raw.w4_workspace_bytes(ops.OP_LINEAR_Q4, M, N, K, 0) > ops.NOALLOC_SCRATCH_BYTES
    fake = C.c_void_p(0x1000)   # rejected on the host before anything is read or launched
    st = ops.raw.w4_linear_q4_noalloc(fake, fake, fake, fake, fake, M, N, K, ops.LAYOUT_ROWMAJOR, None)
    assert st == ops.W4_ESHAPE
