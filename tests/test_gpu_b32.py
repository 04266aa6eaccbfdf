"""Inline-scale blocks of 32 (W4_LAYOUT_B32; written from "Fused int4 and int8
dequantize-matmul in C", Going further: blocks of 32 with the scale stored
inline next to the codes): the device packer equals the oracle's bytes, and
the linear reading the blocks is group-wise W4A16 with G = 32 -- within
1e-5 * sum|terms| of the oracle, and the same bits as the plane form when
both take the same K split."""
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


@pytest.mark.parametrize("N,K", [(7, 64), (64, 2047), (300, 4096)])
def test_pack_block32_bytes(ops, ora, N, K):
    _, w, s = synth.w4a16_inputs(970 + K, 1, N, K, 32)
    got = host(ops.pack_block32(dev(w), dev(s), K))
    assert np.array_equal(got, ora.blocks_b32(w, s, K))


@pytest.mark.parametrize("M", [1, 5, 16, 40])
@pytest.mark.parametrize("N,K", [(2048, 2048), (13312, 2048), (200, 4096), (96, 1056), (40, 1055)])
def test_linear_b32_parity(ops, ora, M, N, K):
    x, w, s = synth.w4a16_inputs(980 + M + N + K, M, N, K, 32)
    blocks = ora.blocks_b32(w, s, K)
    y = host(ops.linear_w4a16_b32(dev(x), dev(blocks), K=K)).astype(np.float64)
    ye, a = ora.linear_w4a16_b32_exact(x, blocks, K)
    assert np.all(np.abs(y - ye) <= 1e-5 * a + 1e-6), float((np.abs(y - ye) / (a + 1e-30)).max())


@pytest.mark.parametrize("M", [1, 16])
def test_b32_same_bits_as_planes(ops, M):
    """N >= 1024: both layouts split K the same way, so the same arithmetic."""
    N, K = 2048, 2048
    x, w, s = synth.w4a16_inputs(990 + M, M, N, K, 32)
    yp = host(ops.linear_w4a16_group(dev(x), dev(w), dev(s), 32, K=K))
    yb = host(ops.linear_w4a16_b32(dev(x), ops.pack_block32(dev(w), dev(s), K), K=K))
    assert np.array_equal(yb.view(np.uint32), yp.view(np.uint32))
    assert ops.device_status() == 0
