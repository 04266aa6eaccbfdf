"""GPU parity of the grouped asymmetric W4A8 linear (vllm-omni "The 4-bit CPU
path", W4A8 with the checkpoint's zero points) against the oracle:
|y - y_ref| <= 1e-5 * sum|terms| + 1e-6 for M <= 16 (the exact integer
group sums, scaled and summed in f32), 4e-3 for the M > 16 tensor-core path
(f16 rounding of (u - z) * s)."""
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


def run(ops, args, G, K, layout=0):
    xq, sx, w, s, z = args
    wd = dev(w)
    if layout == 1:
        wd = ops.pack_interleaved_n64(wd, K)
    return host(ops.linear_q4_group(dev(xq), dev(sx), wd, dev(s), dev(z), G, K=K, N=w.shape[0], layout=layout))


@pytest.mark.parametrize("M", [1, 3, 8, 16])
@pytest.mark.parametrize("N,K,G", [(256, 2048, 128), (2048, 2048, 32), (192, 1000, 8), (128, 2047, 128)])
@pytest.mark.parametrize("layout", [0, 1])
def test_decode_parity(ops, ora, M, N, K, G, layout):
    args = synth.q4_group_inputs(800 + M + N + G, M, N, K, G)
    y = run(ops, args, G, K, layout).astype(np.float64)
    ye, a = ora.linear_q4_group(*args, K, G)
    assert np.all(np.abs(y - ye) <= 1e-5 * a + 1e-6), float((np.abs(y - ye) / (a + 1e-30)).max())


def test_decode_batch_and_layout_invariance(ops):
    """The K split depends on (N, K, G) only: M = 1 and every row of M = 16,
    row-major and interleaved, give the same bits."""
    N, K, G = 2048, 2048, 128
    xq, sx, w, s, z = synth.q4_group_inputs(830, 16, N, K, G)
    y16 = run(ops, (xq, sx, w, s, z), G, K)
    y16il = run(ops, (xq, sx, w, s, z), G, K, layout=1)
    for m in (0, 5, 15):
        y1 = run(ops, (xq[m:m + 1], sx[m:m + 1], w, s, z), G, K)
        assert np.array_equal(y1[0].view(np.uint32), y16[m].view(np.uint32))
    assert np.array_equal(y16.view(np.uint32), y16il.view(np.uint32))


def test_symmetric_case_is_linear_q4(ops):
    """Zero points 8 and one scale per row: the per-channel linear_q4, to rounding."""
    M, N, K, G = 4, 512, 1024, 128
    x, W = synth.w4a8_inputs(840, M, N, K)
    xq, sx, _ = ops.quantize_row_q8(dev(x))
    w, sw = ops.quantize_matrix_q4(dev(W))
    s16 = sw.to(torch.float16)
    s = s16.view(torch.int16)[:, None].repeat(1, K // G).contiguous()
    z = torch.full((N, K // G), 8, dtype=torch.uint8, device="cuda")
    y = host(ops.linear_q4_group(xq, sx, w, s, z, G, K=K)).astype(np.float64)
    y1 = host(ops.linear_q4(xq, sx, w, s16.float(), K=K)).astype(np.float64)
    assert np.all(np.abs(y - y1) <= 1e-5 * np.abs(y1) + 1e-6)


@pytest.mark.parametrize("M,N,K,G", [(33, 256, 2048, 128), (300, 200, 1024, 32), (64, 384, 2047, 128)])
def test_prefill_parity(ops, ora, M, N, K, G):
    args = synth.q4_group_inputs(850 + M + N, M, N, K, G)
    y = run(ops, args, G, K).astype(np.float64)
    ye, a = ora.linear_q4_group(*args, K, G)
    assert np.all(np.abs(y - ye) <= 4e-3 * a + 1e-6), float((np.abs(y - ye) / (a + 1e-30)).max())


def test_prefill_full_size_sampled(ops, ora):
    """M = 2048, K = 2048, N = 13312, G = 128: 48 sampled output channels."""
    M, N, K, G = 2048, 13312, 2048, 128
    xq, sx, w, s, z = synth.q4_group_inputs(860, M, N, K, G)
    y = run(ops, (xq, sx, w, s, z), G, K).astype(np.float64)
    rows = np.sort(np.random.default_rng(861).choice(N, 48, replace=False))
    ye, a = ora.linear_q4_group(xq, sx, w[rows], s[rows], z[rows], K, G)
    assert np.all(np.abs(y[:, rows] - ye) <= 4e-3 * a + 1e-6)


def test_edges(ops):
    xq, sx, w, s, z = synth.q4_group_inputs(870, 2, 64, 64, 32)
    y = ops.linear_q4_group(dev(xq), dev(sx), dev(w), dev(s), dev(z), 32, K=0)
    assert np.array_equal(host(y), np.zeros((2, 64), np.float32))                   # K = 0: zeros
    assert ops.raw.w4_linear_q4_group(None, None, None, None, None, None, 0, 64, 64, 32, 0, None, 0, 0, None) == 0
    assert ops.device_status() == 0
