"""GPU parity of linear_w8a16 (docs.rs ftts_kernels::int8, linear_w8a16: f32
activations times the per-channel Q8 matrix) against the oracle's exact-product
reference: within 1e-5 * sum|x * q * sw| + 1e-6 for M <= 16, 4e-3 for the
M > 16 tensor-core path (x rounded once to bf16)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from tests.golden import load_kv
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


def inputs(seed, M, N, K):
    x = synth.activations_f32(seed, M, K)
    wq = synth.raw_bytes(seed + 1, N * K).view(np.int8).reshape(N, K).copy()
    sw = (synth.uniform01(seed + 2, N) * 0.01 + 1e-3).astype(np.float32)
    return x, wq, sw


def test_hand_example(ops):
    """The printed W8A32 example ("Fused int4 ..." section 3): exact."""
    g = load_kv("hand_example_q8.txt")
    x = np.array(g["x"], np.float32).reshape(1, 4)
    wq = np.array(g["codes"], np.int8).reshape(2, 4)
    s = np.array(g["scales"], np.float32)
    y = host(ops.linear_w8a16(dev(x), dev(wq), dev(s)))
    assert np.array_equal(y, np.array([g["y"]], np.float32)), y


@pytest.mark.parametrize("M", [1, 3, 8, 16])
@pytest.mark.parametrize("N,K", [(256, 2048), (2048, 1024), (200, 1000), (13312, 2048)])
def test_decode_parity(ops, ora, M, N, K):
    x, wq, sw = inputs(900 + M + N + K, M, N, K)
    y = host(ops.linear_w8a16(dev(x), dev(wq), dev(sw))).astype(np.float64)
    ye, a = ora.linear_w8a16_exact(x, wq, sw)
    assert np.all(np.abs(y - ye) <= 1e-5 * a + 1e-6), float((np.abs(y - ye) / (a + 1e-30)).max())


def test_decode_batch_invariance(ops):
    N, K = 2048, 2048
    x, wq, sw = inputs(930, 16, N, K)
    y16 = host(ops.linear_w8a16(dev(x), dev(wq), dev(sw)))
    for m in (0, 7, 15):
        y1 = host(ops.linear_w8a16(dev(x[m:m + 1]), dev(wq), dev(sw)))
        assert np.array_equal(y1[0].view(np.uint32), y16[m].view(np.uint32))


@pytest.mark.parametrize("M,N,K", [(33, 256, 2048), (300, 200, 1024), (64, 384, 1000)])
def test_prefill_parity(ops, ora, M, N, K):
    x, wq, sw = inputs(940 + M + N, M, N, K)
    y = host(ops.linear_w8a16(dev(x), dev(wq), dev(sw))).astype(np.float64)
    ye, a = ora.linear_w8a16_exact(x, wq, sw)
    assert np.all(np.abs(y - ye) <= 4e-3 * a + 1e-6), float((np.abs(y - ye) / (a + 1e-30)).max())


def test_prefill_full_size_sampled(ops, ora):
    M, N, K = 2048, 13312, 2048
    x, wq, sw = inputs(950, M, N, K)
    y = host(ops.linear_w8a16(dev(x), dev(wq), dev(sw))).astype(np.float64)
    rows = np.sort(np.random.default_rng(951).choice(N, 32, replace=False))
    ye, a = ora.linear_w8a16_exact(x, wq[rows], sw[rows])
    assert np.all(np.abs(y[:, rows] - ye) <= 4e-3 * a + 1e-6)


def test_edges(ops):
    x, wq, sw = inputs(960, 2, 64, 64)
    y = ops.linear_w8a16(dev(x[:, :0]), dev(wq[:, :0]), dev(sw))
    assert np.array_equal(host(y), np.zeros((2, 64), np.float32))
    assert ops.device_status() == 0
