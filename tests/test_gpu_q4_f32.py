"""w4_linear_q4_f32: quantize_row_q8 followed by linear_q4 in one call
(docs.rs ftts_kernels::int4 / ::int8).  For M <= 8 on large row-major N the
rows are quantised inside the linear's thread blocks; every route must give
the oracle's codes, scales and outputs bit for bit."""
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
    o.device_status(clear=True)
    return o


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


def check(ops, ora, x, W, flags=0, layout=0):
    M, K = x.shape
    N = W.shape[0]
    wq, sw = ora.quantize_matrix_q4(W)
    wd = dev(wq)
    if layout == ops.LAYOUT_N64:
        wd = ops.pack_interleaved_n64(wd, K)
    y, xq, sx = ops.linear_q4_f32(dev(x), wd, dev(sw), K=K, N=N, layout=layout, flags=flags)
    xq0, sx0, _ = ora.quantize_row_q8(x)
    assert np.array_equal(host(xq), xq0)
    assert np.array_equal(bits(host(sx)), bits(sx0))
    assert np.array_equal(bits(host(y)), bits(ora.linear_q4(xq0, sx0, wq, sw, K)))
    assert ops.device_status() == 0


@pytest.mark.parametrize("flags", [0, 1])
@pytest.mark.parametrize("M", [1, 3, 8])
@pytest.mark.parametrize("N,K", [(2048, 2048), (13312, 2048), (1024, 1024), (2048, 2047), (3072, 4096),
                                 (512, 2048), (37, 200), (1024, 1000), (1100, 1056), (1536, 2040), (4099, 2045)])
def test_linear_q4_f32_bitexact(ops, ora, flags, M, N, K):
    x = synth.activations_f32(151 + M + K, M, K)
    W = synth.weights_f32(152 + N + K, N, K)
    check(ops, ora, x, W, flags=flags)


@pytest.mark.parametrize("M", [9, 16, 40, 300, 2048])
def test_linear_q4_f32_batches(ops, ora, M):
    x = synth.activations_f32(161 + M, M, 2048)
    W = synth.weights_f32(162, 2048 if M <= 300 else 384, 2048)
    check(ops, ora, x, W, flags=1)


@pytest.mark.parametrize("K", [8, 1024, 2056, 4096])
def test_linear_q4_f32_prefill_rows(ops, ora, K):
    """M > 16: one pass quantises the rows and writes the f16 image the
    tensor-core GEMM reads; rows of at most 2048 columns stay in registers,
    longer rows are read twice.  Row 0 holds exact ties, row 1 is zero,
    row 2 has a tiny amax (the reciprocal of the scale overflows)."""
    M = 40
    x = synth.activations_f32(165 + K, M, K)
    x[0, :] = (np.arange(K) % 254 - 127).astype(np.float32) + 0.5
    x[0, 0] = 127.0
    x[1, :] = 0.0
    x[2, :] = np.float32(1e-40) * ((np.arange(K) % 5) - 2)
    W = synth.weights_f32(166 + K, 256, K)
    check(ops, ora, x, W, flags=1)
    check(ops, ora, x, synth.weights_f32(167 + K, 256, K), flags=1, layout=ops.LAYOUT_N64)


def test_linear_q4_f32_interleaved(ops, ora):
    x = synth.activations_f32(171, 2, 2048)
    W = synth.weights_f32(172, 2048, 2048)
    check(ops, ora, x, W, layout=ops.LAYOUT_N64)


def test_linear_q4_f32_ties_and_zero_rows(ops, ora):
    """Row 0: scale exactly 1 (amax 127) and values on half-integers, so every
    code is a round-half-to-even decision; row 1 all zeros (scale 0, codes 0);
    row 2 a tiny amax (the reciprocal of the scale overflows)."""
    K = 2048
    x = np.zeros((3, K), np.float32)
    x[0, :] = (np.arange(K) % 254 - 127).astype(np.float32) + 0.5
    x[0, 0] = 127.0
    x[0, 1::7] = -x[0, 1::7]
    x[2, :] = np.float32(1e-40) * ((np.arange(K) % 5) - 2)
    W = synth.weights_f32(181, 2048, K)
    check(ops, ora, x, W, flags=1)
    for m in range(3):  # alone: the one-row integer-dot kernel
        check(ops, ora, np.ascontiguousarray(x[m:m + 1]), W, flags=1)


@pytest.mark.parametrize("K", [32, 1024, 2048, 2047, 4096, 4128])
def test_linear_q4_one_row(ops, ora, K):
    """M = 1 through both entry points with PDL (the integer-dot kernel where
    K allows), against the oracle's bits."""
    x = synth.activations_f32(191 + K, 1, K)
    W = synth.weights_f32(192 + K, 2048, K)
    check(ops, ora, x, W, flags=1)
    xq, sx, _ = ora.quantize_row_q8(x)
    wq, sw = ora.quantize_matrix_q4(W)
    y = host(ops.linear_q4(dev(xq), dev(sx), dev(wq), dev(sw), K=K, flags=ops.FLAG_PDL))
    assert np.array_equal(bits(y), bits(ora.linear_q4(xq, sx, wq, sw, K)))
