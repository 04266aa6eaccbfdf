"""Prefill (M > 16) linears on the tcgen05 tensor-core path vs the CPU oracle.

W4A8 and W8A8 are bit-exact: the weights and activation codes are exact f16
integers and every partial sum is an integer below 2^24, so the f32 tensor
accumulator holds the exact i32 dot product.  The adversarial cases (all
extremes, alternating extremes, heavy cancellation, every nibble code) check
that the tensor core's accumulation really is exact at the sizes used, in the
spirit of the all-extreme selftest of docs.rs ftts_kernels::int8 ("Tier law").

W4A16 dequantises each weight once to bf16(q * s) in shared memory; the bound
is |y - y_exact| <= 4e-3 * sum_k |x_k W_nk| + 1e-6, and against the oracle that
dequantises the same way it must agree to fp32 accumulation error.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from tests.oracle_pins import np_pack
from tests.test_gpu_parity import bits, dev, host
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


SHAPES = [(17, 128, 256), (256, 128, 2048), (300, 200, 512), (512, 384, 1024), (33, 2048, 2048)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_w4a8_bitexact(ops, ora, M, N, K):
    x, W = synth.w4a8_inputs(201 + M + N, M, N, K)
    xq, sx, _ = ora.quantize_row_q8(x)
    w, sw = ora.quantize_matrix_q4(W)
    want = ora.linear_q4(xq, sx, w, sw, K)
    y = host(ops.linear_q4(dev(xq), dev(sx), dev(w), dev(sw), K=K))
    assert np.array_equal(bits(y), bits(want))


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_w8a8_bitexact(ops, ora, M, N, K):
    x, W = synth.w4a8_inputs(211 + M + N, M, N, K)
    xq, sx, _ = ora.quantize_row_q8(x)
    wq, sw = ora.quantize_matrix_q8(W)
    want = ora.linear_q8(xq, sx, wq, sw)
    y = host(ops.linear_q8(dev(xq), dev(sx), dev(wq), dev(sw)))
    assert np.array_equal(bits(y), bits(want))


@pytest.mark.parametrize("K", [2048, 3072, 16384])
def test_gemm_int_exactness_adversarial(ops, ora, K):
    """Extreme and cancelling integer sums through the f32 tensor accumulator."""
    M, N = 64, 128
    rng = np.random.default_rng(K)
    rows = [np.full(K, 127), np.where(np.arange(K) % 2 == 0, 127, -127),
            np.concatenate([np.full(K // 2, 127), np.full(K - K // 2, -127)]),
            rng.integers(-127, 128, K)]
    xq = np.stack([rows[i % len(rows)] for i in range(M)]).astype(np.int8)
    codes = []
    for n in range(N):
        kind = n % 4
        if kind == 0:
            codes.append(np.full(K, 15))                              # q = 7 everywhere
        elif kind == 1:
            codes.append(np.zeros(K, np.int64))                       # q = -8 everywhere (never emitted, must decode)
        elif kind == 2:
            codes.append(np.where(np.arange(K) % 2 == 0, 15, 1))      # +7 / -7 alternating
        else:
            codes.append(rng.integers(0, 16, K))
    u = np.stack(codes)
    w = np_pack(u, 8)
    ones_m, ones_n = np.ones(M, np.float32), np.ones(N, np.float32)
    want = ora.linear_q4(xq, ones_m, w, ones_n, K)
    exact = xq.astype(np.int64) @ (u - 8).T
    assert np.array_equal(want.astype(np.int64), exact)
    y = host(ops.linear_q4(dev(xq), dev(ones_m), dev(w), dev(ones_n), K=K))
    assert np.array_equal(y.astype(np.int64), exact)
    wq = np.clip((u - 8) * 16, -127, 127).astype(np.int8)      # large int8 weights
    y8 = host(ops.linear_q8(dev(xq), dev(ones_m), dev(wq), dev(ones_n)))
    # |acc| may exceed 2^24 here: the f32 output is the rounded exact integer, as in the oracle
    assert np.array_equal(bits(y8), bits(ora.linear_q8(xq, ones_m, wq, ones_n)))


W4A16_SHAPES = [(17, 128, 256, 32), (256, 128, 2048, 128), (300, 200, 512, 64), (64, 2048, 2048, 32),
                (512, 384, 1024, 128)]


@pytest.mark.parametrize("M,N,K,G", W4A16_SHAPES)
def test_gemm_w4a16(ops, ora, M, N, K, G):
    x, w, s = synth.w4a16_inputs(221 + M + N + G, M, N, K, G)
    y = host(ops.linear_w4a16_group(dev(x), dev(w), dev(s), G, K=K)).astype(np.float64)
    ye, a = ora.linear_w4a16_exact(x, w, s, K, G)
    assert np.all(np.abs(y - ye) <= 4e-3 * a + 1e-6), float((np.abs(y - ye) / (a + 1e-30)).max())
    # against the same dequantisation to bf16: only fp32 accumulation error remains
    yb = ora.linear_w4a16_bf16dequant(x, w, s, K, G)
    assert np.all(np.abs(y - yb) <= 1e-5 * a + 1e-6), float((np.abs(y - yb) / (a + 1e-30)).max())


@pytest.mark.parametrize("N", [2048, 3072, 13312])
def test_prefill_full_size_sampled(ops, ora, N):
    """Prefill workload at full size (M = 2048, K = 2048), sampled output channels."""
    M, K, G = 2048, 2048, 128
    rows = np.sort(np.random.default_rng(N).choice(N, 48, replace=False))
    x, W = synth.w4a8_inputs(231 + N, M, N, K)
    xq_t, sx_t, _ = ops.quantize_row_q8(dev(x))
    w_t, sw_t = ops.quantize_matrix_q4(dev(W))
    y = host(ops.linear_q4(xq_t, sx_t, w_t, sw_t, K=K))
    xq, sx, w, sw = host(xq_t), host(sx_t), host(w_t), host(sw_t)
    want = ora.linear_q4(xq, sx, w[rows], sw[rows], K)
    assert np.array_equal(bits(np.ascontiguousarray(y[:, rows])), bits(want))
    xb, wb, sb = synth.w4a16_inputs(241 + N, M, N, K, G)
    yb = host(ops.linear_w4a16_group(dev(xb), dev(wb), dev(sb), G, K=K)).astype(np.float64)
    ye, a = ora.linear_w4a16_exact(xb, wb[rows], sb[rows], K, G)
    assert np.all(np.abs(yb[:, rows] - ye) <= 4e-3 * a + 1e-6)


@pytest.mark.parametrize("M,N,K,G", [(40, 128, 512, 128), (300, 192, 1024, 32), (33, 2048, 2048, 128)])
def test_gemm_interleaved_w4a16_matches_rowmajor(ops, ora, M, N, K, G):
    """Prefill straight from the [N/64][K][32 B] layout: the same dequantised
    bf16 tile as the row-major GEMM (the interleave is undone in shared
    memory), so the same bits; N = 192 has an odd number of 64-channel blocks."""
    x, w, s = synth.w4a16_inputs(251 + M + G, M, N, K, G)
    y = host(ops.linear_w4a16_group(dev(x), dev(w), dev(s), G, K=K))
    il = ops.pack_interleaved_n64(dev(w), K)
    y2 = host(ops.linear_w4a16_group(dev(x), il, dev(s), G, K=K, N=N, layout=ops.LAYOUT_N64))
    assert np.array_equal(bits(y2), bits(y))
    ye, a = ora.linear_w4a16_exact(x, w, s, K, G)
    assert np.all(np.abs(y2.astype(np.float64) - ye) <= 4e-3 * a + 1e-6)


@pytest.mark.parametrize("M,N,K", [(33, 128, 256), (300, 192, 1000), (64, 2048, 2047), (520, 384, 2048)])
def test_gemm_interleaved_w4a8_bitexact(ops, ora, M, N, K):
    """W4A8 prefill from the interleaved layout: bit-exact with the oracle
    (ragged M, odd block count, K not a multiple of 64, odd K)."""
    x, W = synth.w4a8_inputs(261 + M + N, M, N, K)
    xq, sx, _ = ora.quantize_row_q8(x)
    w, sw = ora.quantize_matrix_q4(W)
    want = ora.linear_q4(xq, sx, w, sw, K)
    il = ops.pack_interleaved_n64(dev(w), K)
    y = host(ops.linear_q4(dev(xq), dev(sx), il, dev(sw), K=K, N=N, layout=ops.LAYOUT_N64))
    assert np.array_equal(bits(y), bits(want))


def test_gemm_device_status_clean(ops):
    torch.cuda.synchronize()
    assert ops.device_status() == 0
