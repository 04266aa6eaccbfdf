"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Bar: bit-exact for codes, scales, i32 dots and the W4A8 / W8A8 f32 outputs;
W4A16 within |y - y_exact| <= 1e-5 * sum_k |x_k W_nk| + 1e-6 (the bound the
workload states for fp32 accumulation; y_exact is the oracle's exact-product
sum).  Shapes span several tiles, ragged tails and the degenerate cases, and
the full workload sizes are checked on sampled output channels.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from tests.oracle_pins import np_pack
from w4a16_int4_quantized_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_REL, TOL_ABS = 1e-5, 1e-6


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


# ------------------------------------------------------------------ quantizers

SPECIAL_ROWS = [
    np.zeros(40, np.float32),                                         # amax == 0
    np.array([127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5] * 5, np.float32),  # exact ties
    np.full(40, 1e-44, np.float32),                                   # subnormal amax, scale underflows
    (np.arange(40, dtype=np.float32) - 20) * np.float32(3e-39),       # subnormal range
    np.array([3e38, -3e38] + [1.0] * 38, np.float32),                 # huge values
]


@pytest.mark.parametrize("M,K", [(1, 2048), (3, 33), (16, 2047), (7, 1), (2048, 2048)])
def test_quantize_row_q8_bitexact(ops, ora, M, K):
    x = synth.activations_f32(11 + K, M, K)
    q, sx, rs = ops.quantize_row_q8(dev(x))
    rq, rsx, rrs = ora.quantize_row_q8(x)
    assert np.array_equal(host(q), rq)
    assert np.array_equal(bits(host(sx)), bits(rsx))
    assert np.array_equal(host(rs), rrs)


def test_quantize_special_rows(ops, ora):
    x = np.stack(SPECIAL_ROWS)
    q, sx, rs = ops.quantize_row_q8(dev(x))
    rq, rsx, rrs = ora.quantize_row_q8(x)
    assert np.array_equal(host(q), rq) and np.array_equal(bits(host(sx)), bits(rsx))
    assert np.array_equal(host(rs), rrs)
    p, sw = ops.quantize_matrix_q4(dev(x))
    rp, rsw = ora.quantize_matrix_q4(x)
    assert np.array_equal(host(p), rp) and np.array_equal(bits(host(sw)), bits(rsw))


@pytest.mark.parametrize("N,K", [(2048, 2048), (37, 2047), (5, 1), (64, 3), (13312, 2048)])
def test_quantize_matrix_q4_bitexact(ops, ora, N, K):
    W = synth.weights_f32(21 + K, N, K)
    p, sw = ops.quantize_matrix_q4(dev(W))
    rp, rsw = ora.quantize_matrix_q4(W)
    assert np.array_equal(host(p), rp)
    assert np.array_equal(bits(host(sw)), bits(rsw))


@pytest.mark.parametrize("N,K", [(1024, 1024), (37, 200), (3, 1)])
def test_quantize_matrix_q8_bitexact(ops, ora, N, K):
    W = synth.weights_f32(31 + K, N, K)
    q, sw = ops.quantize_matrix_q8(dev(W))
    rq, rsw = ora.quantize_matrix_q8(W)
    assert np.array_equal(host(q), rq) and np.array_equal(bits(host(sw)), bits(rsw))


# ------------------------------------------------------------------ dot

@pytest.mark.parametrize("K", [1, 7, 2047, 2048, 3072])
def test_dot_i32_q4(ops, ora, K):
    xq = synth.raw_bytes(41 + K, K).view(np.int8).copy()
    xq[xq == -128] = -127
    w = synth.raw_bytes(42 + K, (K + 1) // 2)
    got = int(host(ops.dot_i32_q4(dev(xq), dev(w), K))[0])
    assert got == ora.dot_i32_q4(xq, w, K) == ora.dot_naive_q4(xq, w, K)
    # all-extreme row (selftest-style): 127 * 7 * K
    xe = np.full(K, 127, np.int8)
    we = np_pack(np.full((1, K), 15), 8)[0]
    assert int(host(ops.dot_i32_q4(dev(xe), dev(we), K))[0]) == 127 * 7 * K


# ------------------------------------------------------------------ W4A8 / W8A8 linears

def w4a8_case(ora, seed, M, N, K):
    x, W = synth.w4a8_inputs(seed, M, N, K)
    xq, sx, _ = ora.quantize_row_q8(x)
    w, sw = ora.quantize_matrix_q4(W)
    return xq, sx, w, sw


LIN_SHAPES = [(2048, 2048), (37, 200), (64, 2047), (3072, 2048), (1024, 3072), (100, 64), (1, 32), (1024, 32)]


@pytest.mark.parametrize("M", [1, 2, 4, 8, 9, 16])
@pytest.mark.parametrize("N,K", LIN_SHAPES)
def test_linear_q4_bitexact(ops, ora, M, N, K):
    xq, sx, w, sw = w4a8_case(ora, 51 + N + K, M, N, K)
    want = ora.linear_q4(xq, sx, w, sw, K)
    y = ops.linear_q4(dev(xq), dev(sx), dev(w), dev(sw), K=K)
    assert np.array_equal(bits(host(y)), bits(want))
    if N % 64 == 0:
        il = ops.pack_interleaved_n64(dev(w), K)
        assert np.array_equal(host(il), ora.pack_interleaved_n64(w, K))
        y2 = ops.linear_q4(dev(xq), dev(sx), il, dev(sw), K=K, N=N, layout=ops.LAYOUT_N64)
        assert np.array_equal(bits(host(y2)), bits(want))


@pytest.mark.parametrize("M", [1, 4, 16])
def test_linear_q4_random_bytes_every_nibble(ops, ora, M):
    """Random packed bytes include nibble 0 (= -8), which the quantizer never emits."""
    N, K = 256, 1024
    xq = synth.raw_bytes(61, M * K).view(np.int8).reshape(M, K).copy()
    xq[xq == -128] = -127
    w = synth.raw_bytes(62, N * K // 2).reshape(N, K // 2)
    sx = np.abs(synth.normal(63, M, 0.01)).astype(np.float32) + 1e-3
    sw = np.abs(synth.normal(64, N, 0.01)).astype(np.float32) + 1e-3
    want = ora.linear_q4(xq, sx, w, sw, K)
    y = ops.linear_q4(dev(xq), dev(sx), dev(w), dev(sw), K=K)
    assert np.array_equal(bits(host(y)), bits(want))


@pytest.mark.parametrize("K", [2047, 2048, 3072])
@pytest.mark.parametrize("M", [1, 16])
def test_linear_q4_all_extreme(ops, M, K):
    N = 64
    xq = np.full((M, K), 127, np.int8)
    w = np_pack(np.full((N, K), 15), 8)
    ones_m, ones_n = np.ones(M, np.float32), np.ones(N, np.float32)
    y = host(ops.linear_q4(dev(xq), dev(ones_m), dev(w), dev(ones_n), K=K))
    assert np.all(y == np.float32(127 * 7 * K))
    xa = np.tile(np.where(np.arange(K) % 2 == 0, 127, -127).astype(np.int8), (M, 1))
    wa = np_pack(np.tile(np.where(np.arange(K) % 2 == 0, 15, 1), (N, 1)), 8)
    y = host(ops.linear_q4(dev(xa), dev(ones_m), dev(wa), dev(ones_n), K=K))
    assert np.all(y == np.float32(127 * 7 * K))


@pytest.mark.parametrize("K", [16384, 65536, 131072])
def test_linear_q4_extreme_long_rows(ops, ora, K):
    """Extreme codes (x = +-127, nibbles 0 = -8 and 15 = +7) on rows long
    enough that a warp's partial sums approach and pass 2^24: the integer
    result must stay exact whichever accumulation the kernels pick."""
    N, M = 1024, 2
    xq = np.full((M, K), 127, np.int8)
    xq[1, 1::2] = -127
    w = np.zeros((N, K // 2), np.uint8)
    w[1::2, ::3] = 0xFF
    w[2::4, :] = 0xF0
    sx = np.ones(M, np.float32)
    sw = np.ones(N, np.float32)
    want = ora.linear_q4(xq, sx, w, sw, K)
    wd, swd = dev(w), dev(sw)
    for flags in (0, ops.FLAG_PDL):
        y = host(ops.linear_q4(dev(xq), dev(sx), wd, swd, K=K, flags=flags))
        assert np.array_equal(bits(y), bits(want))
    y, xq_d, sx_d = ops.linear_q4_f32(dev(xq.astype(np.float32)), wd, swd, K=K, flags=ops.FLAG_PDL)
    assert np.array_equal(host(xq_d), xq) and np.all(host(sx_d) == 1.0)
    assert np.array_equal(bits(host(y)), bits(want))
    assert ops.device_status() == 0


@pytest.mark.parametrize("M", [1, 3, 16])
@pytest.mark.parametrize("N,K", [(1024, 1024), (37, 200), (3072, 1024), (64, 64)])
def test_linear_q8_bitexact(ops, ora, M, N, K):
    x, W = synth.w4a8_inputs(71 + N, M, N, K)
    xq, sx, _ = ora.quantize_row_q8(x)
    wq, sw = ora.quantize_matrix_q8(W)
    want = ora.linear_q8(xq, sx, wq, sw)
    y = ops.linear_q8(dev(xq), dev(sx), dev(wq), dev(sw))
    assert np.array_equal(bits(host(y)), bits(want))


@pytest.mark.parametrize("M", [1, 4, 16])
@pytest.mark.parametrize("N", [13312, 3072])
def test_linear_q4_full_size_sampled(ops, ora, M, N):
    """Decode-batch workload at full size (K = 2048), both layouts; sampled channels."""
    K = 2048
    x, W = synth.w4a8_inputs(81 + M, M, N, K)
    xq_t, sx_t, _ = ops.quantize_row_q8(dev(x))
    w_t, sw_t = ops.quantize_matrix_q4(dev(W))
    y = host(ops.linear_q4(xq_t, sx_t, w_t, sw_t, K=K))
    il = ops.pack_interleaved_n64(w_t, K)
    y2 = host(ops.linear_q4(xq_t, sx_t, il, sw_t, K=K, N=N, layout=ops.LAYOUT_N64))
    assert np.array_equal(bits(y), bits(y2))
    rows = np.sort(np.random.default_rng(M).choice(N, 384, replace=False))
    xq, sx, w, sw = host(xq_t), host(sx_t), host(w_t), host(sw_t)
    want = ora.linear_q4(xq, sx, w[rows], sw[rows], K)
    assert np.array_equal(bits(np.ascontiguousarray(y[:, rows])), bits(want))


# ------------------------------------------------------------------ W4A16

def w4a16_check(y, ora, x, w, s, K, G):
    ye, a = ora.linear_w4a16_exact(x, w, s, K, G)
    err = np.abs(y.astype(np.float64) - ye)
    bound = TOL_REL * a + TOL_ABS
    assert np.all(err <= bound), (float((err / bound).max()), np.unravel_index(np.argmax(err / bound), err.shape))


@pytest.mark.parametrize("M", [1, 2, 4, 8, 9, 16])
@pytest.mark.parametrize("N,K,G", [(2048, 2048, 32), (2048, 2047, 32), (3072, 2048, 128), (64, 384, 64),
                                   (37, 384, 32), (100, 1024, 256), (64, 2048, 2048),
                                   (1024, 1024, 128), (1024, 32, 32), (1088, 1024, 128)])
def test_linear_w4a16(ops, ora, M, N, K, G):
    x, w, s = synth.w4a16_inputs(91 + N + K + G, M, N, K, G)
    y = host(ops.linear_w4a16_group(dev(x), dev(w), dev(s), G, K=K))
    w4a16_check(y, ora, x, w, s, K, G)
    if N % 64 == 0:
        il = ops.pack_interleaved_n64(dev(w), K)
        y2 = host(ops.linear_w4a16_group(dev(x), il, dev(s), G, K=K, N=N, layout=ops.LAYOUT_N64))
        assert np.array_equal(bits(y2), bits(y)), "interleaved layout must match row-major bit for bit"


@pytest.mark.parametrize("N,K,G", [(37, 384, 2), (19, 200, 40), (21, 2047, 2), (64, 100, 10)])
@pytest.mark.parametrize("M", [1, 5])
def test_linear_w4a16_generic_shapes(ops, ora, M, N, K, G):
    x, w, s = synth.w4a16_inputs(101 + K + G, M, N, K, G)
    y = host(ops.linear_w4a16_group(dev(x), dev(w), dev(s), G, K=K))
    w4a16_check(y, ora, x, w, s, K, G)


def test_w4a16_hand_example(ops):
    from tests.golden import load_kv
    g = load_kv("hand_example_w4a16.txt")
    x = synth.f32_to_bf16_bits(np.array([g["x"]], np.float32))
    w = np.array(g["bytes"], np.uint8).reshape(2, 2)
    s = np.array(g["scales_f16"], np.uint16).reshape(2, 2)
    y = host(ops.linear_w4a16_group(dev(x), dev(w), dev(s), g["G"], K=g["K"]))
    assert np.array_equal(y, np.array([g["y"]], np.float32))


@pytest.mark.parametrize("N,K,G", [(2048, 2048, 32), (3072, 2048, 128), (13312, 2048, 128)])
def test_w4a16_batch_invariance(ops, N, K, G):
    """Rows computed alone equal the same rows inside a batch, bit for bit
    ("Fused int4 ..." batch_invariant_rows): the K split does not depend on M."""
    M = 12
    x, w, s = synth.w4a16_inputs(111, M, N, K, G)
    wd, sd = dev(w), dev(s)
    yb = host(ops.linear_w4a16_group(dev(x), wd, sd, G, K=K))
    for m in range(M):
        y1 = host(ops.linear_w4a16_group(dev(x[m:m + 1]), wd, sd, G, K=K))
        assert np.array_equal(bits(y1[0]), bits(yb[m])), m


@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
@pytest.mark.parametrize("N,K,G", [(2048, 2048, 32), (2048, 2047, 32), (13312, 2048, 128), (1024, 1024, 128),
                                   (3072, 2048, 128), (4096, 8192, 128), (1000, 4096, 32), (1100, 1024, 64),
                                   (5000, 2048, 32), (2056, 512, 128), (3000, 1022, 2)])
def test_w4a16_pdl_same_bits(ops, ora, M, N, K, G):
    """With W4_FLAG_PDL, large-N decode calls stream whole-SM row ranges with
    bulk copies (a different kernel); the arithmetic, and so every bit, is the
    one of the call without the flag.  Sampled rows against the oracle."""
    x, w, s = synth.w4a16_inputs(131 + M + N + K, M, N, K, G)
    xd, wd, sd = dev(x), dev(w), dev(s)
    y0 = host(ops.linear_w4a16_group(xd, wd, sd, G, K=K))
    y1 = host(ops.linear_w4a16_group(xd, wd, sd, G, K=K, flags=ops.FLAG_PDL))
    assert np.array_equal(bits(y1), bits(y0))
    rows = np.sort(np.random.default_rng(N + M).choice(N, min(N, 192), replace=False))
    w4a16_check(np.ascontiguousarray(y1[:, rows]), ora, x, w[rows], s[rows], K, G)
    assert ops.device_status() == 0


@pytest.mark.parametrize("M", [1, 8, 16])
@pytest.mark.parametrize("N,K", [(2048, 2048), (13312, 2048)])
def test_linear_q4_pdl_bitexact(ops, ora, M, N, K):
    """The PDL-launched row quantizer followed by a PDL linear: the oracle's bits."""
    x = synth.activations_f32(141 + M, M, K)
    W = synth.weights_f32(142 + N, N, K)
    wq, sw = ora.quantize_matrix_q4(W)
    xq_d, sx_d, _ = ops.quantize_row_q8(dev(x))
    y = host(ops.linear_q4(xq_d, sx_d, dev(wq), dev(sw), K=K, flags=ops.FLAG_PDL))
    xq, sx, _ = ora.quantize_row_q8(x)
    assert np.array_equal(host(xq_d), xq) and np.array_equal(bits(host(sx_d)), bits(sx))
    assert np.array_equal(bits(y), bits(ora.linear_q4(xq, sx, wq, sw, K)))


@pytest.mark.parametrize("M", [1, 4, 16])
@pytest.mark.parametrize("N", [13312, 3072])
def test_linear_w4a16_full_size_sampled(ops, ora, M, N):
    K, G = 2048, 128
    x, w, s = synth.w4a16_inputs(121 + M, M, N, K, G)
    y = host(ops.linear_w4a16_group(dev(x), dev(w), dev(s), G, K=K))
    il = ops.pack_interleaved_n64(dev(w), K)
    y2 = host(ops.linear_w4a16_group(dev(x), il, dev(s), G, K=K, N=N, layout=ops.LAYOUT_N64))
    assert np.array_equal(bits(y), bits(y2))
    rows = np.sort(np.random.default_rng(M + 7).choice(N, 256, replace=False))
    w4a16_check(np.ascontiguousarray(y[:, rows]), ora, x, w[rows], s[rows], K, G)


# ------------------------------------------------------------------ edge cases

def test_empty_and_zero_k(ops):
    canary = np.float32(-12345.0)
    y = dev(np.full((3, 5), canary, np.float32))
    e = torch.empty(0, device="cuda")
    # M == 0 / N == 0: no-op, y untouched
    ops.raw.w4_linear_q4(None, None, None, None, y.data_ptr(), 0, 5, 8, 0, None, 0, 0, None)
    ops.raw.w4_linear_q4(None, None, None, None, y.data_ptr(), 3, 0, 8, 0, None, 0, 0, None)
    assert np.all(host(y) == canary)
    # K == 0: y = 0
    sx = dev(np.ones(3, np.float32))
    sw = dev(np.ones(5, np.float32))
    st = ops.raw.w4_linear_q4(None, sx.data_ptr(), None, sw.data_ptr(), y.data_ptr(), 3, 5, 0, 0, None, 0, 0, None)
    assert st == ops.W4_OK and np.all(host(y) == 0)
    y.fill_(float(canary))
    st = ops.raw.w4_linear_w4a16_group(None, None, None, y.data_ptr(), 3, 5, 0, 2, 0, None, 0, 0, None)
    assert st == ops.W4_OK and np.all(host(y) == 0)
    del e


def test_errors_leave_y_untouched(ops):
    canary = np.float32(7.5)
    y = dev(np.full((2, 64), canary, np.float32))
    x = dev(np.zeros((2, 12), np.uint16))
    w = dev(np.zeros((64, 6), np.uint8))
    s = dev(np.zeros((64, 6), np.uint16))
    for G in (3, 0, 8):        # odd, non-positive, not dividing K
        st = ops.raw.w4_linear_w4a16_group(x.data_ptr(), w.data_ptr(), s.data_ptr(), y.data_ptr(), 2, 64, 12, G, 0,
                                           None, 0, 0, None)
        assert st == ops.W4_ESHAPE
    st = ops.raw.w4_linear_w4a16_group(x.data_ptr(), w.data_ptr(), s.data_ptr(), y.data_ptr(), 2, 63, 12, 2, 1,
                                       None, 0, 0, None)
    assert st == ops.W4_ESHAPE
    assert np.all(host(y) == canary)


def test_pdl_flag_same_bits(ops, ora):
    M, N, K, G = 4, 3072, 2048, 128
    x, w, s = synth.w4a16_inputs(131, M, N, K, G)
    a = host(ops.linear_w4a16_group(dev(x), dev(w), dev(s), G, K=K))
    b = host(ops.linear_w4a16_group(dev(x), dev(w), dev(s), G, K=K, flags=ops.FLAG_PDL))
    assert np.array_equal(bits(a), bits(b))
    xq, sx, wq, sw = w4a8_case(ora, 132, M, N, K)
    a = host(ops.linear_q4(dev(xq), dev(sx), dev(wq), dev(sw), K=K))
    b = host(ops.linear_q4(dev(xq), dev(sx), dev(wq), dev(sw), K=K, flags=ops.FLAG_PDL))
    assert np.array_equal(bits(a), bits(b))


def test_device_status_clean(ops):
    torch.cuda.synchronize()
    assert ops.device_status() == 0


@pytest.mark.parametrize("N,G", [(13312, 128), (7680, 32), (8192, 64)])
def test_w4a16_interleaved_m1_pdl_same_bits(ops, ora, N, G):
    """M = 1 under PDL from the interleaved [N/64][K][32 B] layout: the
    all-warp kernel turns each 64-channel block into row-major rows in shared
    memory, so the result equals the row-major call bit for bit (and G = 64
    takes the staged kernel, also bit-identical).  Sampled rows against the oracle."""
    K = 2048
    x, w, s = synth.w4a16_inputs(171 + N + G, 1, N, K, G)
    xd, wd, sd = dev(x), dev(w), dev(s)
    y0 = host(ops.linear_w4a16_group(xd, wd, sd, G, K=K))
    wil = ops.pack_interleaved_n64(wd, K)
    y1 = host(ops.linear_w4a16_group(xd, wil, sd, G, K=K, N=N, layout=ops.LAYOUT_N64, flags=ops.FLAG_PDL))
    y2 = host(ops.linear_w4a16_group(xd, wil, sd, G, K=K, N=N, layout=ops.LAYOUT_N64))
    assert np.array_equal(bits(y1), bits(y0))
    assert np.array_equal(bits(y2), bits(y0))
    rows = np.sort(np.random.default_rng(N).choice(N, 128, replace=False))
    w4a16_check(np.ascontiguousarray(y1[:, rows]), ora, x, w[rows], s[rows], K, G)
    assert ops.device_status() == 0


@pytest.mark.parametrize("N", [13312, 7680])
def test_linear_q4_interleaved_m1_pdl_bitexact(ops, ora, N):
    """W4A8 at M = 1 under PDL from the interleaved layout (the all-warp
    kernel transposes each 64-channel block in shared memory): the oracle's
    bits, the same as the row-major call."""
    K = 2048
    x = synth.activations_f32(181 + N, 1, K)
    W = synth.weights_f32(182 + N, N, K)
    wq, sw = ora.quantize_matrix_q4(W)
    xq, sx, _ = ora.quantize_row_q8(x)
    wil = ops.pack_interleaved_n64(dev(wq), K)
    y = host(ops.linear_q4(dev(xq), dev(sx), wil, dev(sw), K=K, N=N, layout=ops.LAYOUT_N64, flags=ops.FLAG_PDL))
    assert np.array_equal(bits(y), bits(ora.linear_q4(xq, sx, wq, sw, K)))
    assert ops.device_status() == 0
