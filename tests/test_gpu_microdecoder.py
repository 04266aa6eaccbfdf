"""The weight-resident microdecoder frame (docs.rs ftts_kernels::int4, "Why the
microdecoder": a 5-layer body re-read fifteen times per frame), W4A8 end to
end: every linear's f32 output is re-quantised per row (quantize_row_q8)
before it feeds the next linear.  The dataflow per layer (the pages give
only "5-layer body"): q, k, v read h; o reads Q8(v); gate and up read Q8(o);
down reads Q8(up); the next h is Q8(down).  Every step is exact or
bit-reproducible, so the GPU frame must equal the oracle's frame bit for bit.
"""
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


def oracle_chain(ora, x0, lins, passes, pass_output):
    """The chain semantics of w4_chain_q4 written out with the oracle's
    quantize_row_q8 and linear_q4 (lins: (packed, sw, input) per linear)."""
    h = np.ascontiguousarray(x0, np.float32).reshape(1, -1)
    ys = [None] * len(lins)
    for _ in range(passes):
        for i, (pk, sw, inp) in enumerate(lins):
            src = h if inp < 0 else ys[inp]
            q, s, _ = ora.quantize_row_q8(src)
            ys[i] = ora.linear_q4(q, s, pk, sw, src.shape[1])
        h = ys[pass_output]
    return ys


NAMES = [n for n, _, _ in synth.MICRODECODER_LINEARS]


def microdecoder_descriptors(n_layers):
    """(layer, name, input index) of the frame's dataflow, in order."""
    out = []
    for L in range(n_layers):
        base = 7 * L
        h_in = -1 if L == 0 else base - 1            # the previous layer's down
        ins = {"q": h_in, "k": h_in, "v": h_in, "o": base + 2, "gate": base + 3, "up": base + 3, "down": base + 5}
        out += [(L, name, ins[name]) for name in NAMES]
    return out


def oracle_frame(ora, layers, x0, passes):
    hq, hs, _ = ora.quantize_row_q8(x0)
    taps = []
    for _ in range(passes):
        for L in layers:
            lin = lambda name, q, s: ora.linear_q4(q, s, L[name][0], L[name][1], L[name][2])
            q_out, k_out, v_out = lin("q", hq, hs), lin("k", hq, hs), lin("v", hq, hs)
            vq, vs, _ = ora.quantize_row_q8(v_out)
            o_out = lin("o", vq, vs)
            oq, os_, _ = ora.quantize_row_q8(o_out)
            gate_out, up_out = lin("gate", oq, os_), lin("up", oq, os_)
            uq, us, _ = ora.quantize_row_q8(up_out)
            down_out = lin("down", uq, us)
            hq, hs, _ = ora.quantize_row_q8(down_out)
            taps.append((q_out, k_out, gate_out, down_out))
    return hq, hs, taps


def gpu_frame(ops, layers, x0, passes):
    hq, hs, _ = ops.quantize_row_q8(x0)
    taps = []
    for _ in range(passes):
        for L in layers:
            lin = lambda name, q, s: ops.linear_q4(q, s, L[name][0], L[name][1], K=L[name][2], flags=ops.FLAG_PDL)
            q_out, k_out, v_out = lin("q", hq, hs), lin("k", hq, hs), lin("v", hq, hs)
            vq, vs, _ = ops.quantize_row_q8(v_out)
            o_out = lin("o", vq, vs)
            oq, os_, _ = ops.quantize_row_q8(o_out)
            gate_out, up_out = lin("gate", oq, os_), lin("up", oq, os_)
            uq, us, _ = ops.quantize_row_q8(up_out)
            down_out = lin("down", uq, us)
            hq, hs, _ = ops.quantize_row_q8(down_out)
            taps.append((q_out, k_out, gate_out, down_out))
    return hq, hs, taps


def test_microdecoder_frame_bitexact(ops, ora):
    Wf = synth.microdecoder_weights(3003)
    x0 = synth.activations_f32(3004, 1, 1024)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    glayers, olayers = [], []
    for L in Wf:
        gl, ol = {}, {}
        for name, W in L.items():
            p, s = ops.quantize_matrix_q4(dev(W))
            rp, rs = ora.quantize_matrix_q4(W)
            torch.cuda.synchronize()
            assert np.array_equal(p.cpu().numpy(), rp) and np.array_equal(s.cpu().numpy(), rs)
            gl[name] = (p, s, W.shape[1])
            ol[name] = (rp, rs, W.shape[1])
        glayers.append(gl)
        olayers.append(ol)
    passes = 15
    gq, gs, gtaps = gpu_frame(ops, glayers, dev(x0), passes)
    oq, os_, otaps = oracle_frame(ora, olayers, x0, passes)
    torch.cuda.synchronize()
    assert np.array_equal(gq.cpu().numpy(), oq)
    assert np.array_equal(gs.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    for i, (gt, ot) in enumerate(zip(gtaps, otaps)):
        for a, b in zip(gt, ot):
            assert np.array_equal(a.cpu().numpy().view(np.uint32), b.view(np.uint32)), i
    assert ops.device_status() == 0


@pytest.fixture(scope="module")
def microdecoder(ops, ora):
    Wf = synth.microdecoder_weights(3003)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    g, o = [], []
    for L in Wf:
        gl, ol = {}, {}
        for name, W in L.items():
            gl[name] = ops.quantize_matrix_q4(dev(W))
            ol[name] = ora.quantize_matrix_q4(W)
        g.append(gl)
        o.append(ol)
    torch.cuda.synchronize()
    return g, o, synth.activations_f32(3004, 1, 1024)


@pytest.mark.parametrize("passes", [1, 2, 15])
def test_chain_microdecoder_bitexact(ops, ora, microdecoder, passes):
    """The frame as ONE persistent kernel: every linear's last-pass output
    equals the oracle's chain bit for bit."""
    g, o, x0 = microdecoder
    desc = microdecoder_descriptors(len(g))
    ys = [torch.full((1, g[L][name][1].numel()), float("nan"), device="cuda") for L, name, _ in desc]
    lins = [(g[L][name][0], g[L][name][1], ys[i], inp) for i, (L, name, inp) in enumerate(desc)]
    x0d = torch.from_numpy(x0).cuda()
    ops.chain_q4(x0d, lins, passes, len(desc) - 1)
    ref = oracle_chain(ora, x0, [(o[L][name][0], o[L][name][1], inp) for L, name, inp in desc], passes,
                       len(desc) - 1)
    torch.cuda.synchronize()
    for i, (L, name, _) in enumerate(desc):
        got = ys[i].cpu().numpy().view(np.uint32)
        assert np.array_equal(got, ref[i].view(np.uint32)), (passes, L, name)
    assert ops.device_status() == 0


def test_chain_matches_per_call_path(ops, microdecoder):
    """w4_chain_q4 == the same chain issued as quantize_row_q8 + linear_q4 calls."""
    g, _, x0 = microdecoder
    desc = microdecoder_descriptors(len(g))
    x0d = torch.from_numpy(x0).cuda()
    ys = [torch.empty((1, g[L][name][1].numel()), device="cuda") for L, name, _ in desc]
    ops.chain_q4(x0d, [(g[L][name][0], g[L][name][1], ys[i], inp) for i, (L, name, inp) in enumerate(desc)],
                 3, len(desc) - 1)
    h = x0d.reshape(1, -1)
    ref = [None] * len(desc)
    for _ in range(3):
        for i, (L, name, inp) in enumerate(desc):
            src = h if inp < 0 else ref[inp]
            q, s, _ = ops.quantize_row_q8(src)
            ref[i] = ops.linear_q4(q, s, g[L][name][0], g[L][name][1], K=src.shape[1])
        h = ref[-1]
    torch.cuda.synchronize()
    for a, b in zip(ys, ref):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def _random_chain(ops, ora, seed, shapes, K0):
    """shapes: (N, input) per linear; weights ~ N(0, 0.02) quantized on both sides."""
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    glins, olins = [], []
    for i, (N, inp) in enumerate(shapes):
        K = K0 if inp < 0 else shapes[inp][0]
        W = synth.weights_f32(seed + i, N, K)
        pk, sw = ops.quantize_matrix_q4(dev(W))
        glins.append((pk, sw, torch.full((1, N), float("nan"), device="cuda"), inp))
        olins.append(ora.quantize_matrix_q4(W) + (inp,))
    return glins, olins


def test_chain_ragged_and_wide(ops, ora):
    """Stages of several linears with ragged N; K at the maximum (8192: eight
    16-byte chunks per lane per row, so two rows already overflow the
    register prefetch into the direct-load path); K = 4960 (155 chunks: a
    partial last round of lanes); K = 352 (11 chunks: most lanes idle); a
    stage of ~9 rows per warp."""
    K0 = 8192
    shapes = [(4960, -1), (64, -1), (32, -1),   # depth 0: 5056 rows, K = 8192
              (8192, 0),                         # depth 1: K = 4960
              (21952, 3), (352, 3),              # depth 2: 22304 rows, K = 8192
              (8192, 5)]                         # depth 3: K = 352; the pass output (N = K0)
    glins, olins = _random_chain(ops, ora, 4100, shapes, K0)
    x0 = synth.activations_f32(4099, 1, K0)
    ops.chain_q4(torch.from_numpy(x0).cuda(), glins, 2, 6)
    ref = oracle_chain(ora, x0, olins, 2, 6)
    torch.cuda.synchronize()
    for i, (_, _, y, _) in enumerate(glins):
        assert np.array_equal(y.cpu().numpy().view(np.uint32), ref[i].view(np.uint32)), i
    assert ops.device_status() == 0


def test_chain_zero_input_and_noop(ops, ora):
    """x0 = 0: every scale is 0, every code 0, every output exactly +0.0.
    passes == 0 launches nothing and leaves y untouched."""
    glins, _ = _random_chain(ops, ora, 4200, [(64, -1), (96, 0), (64, 1)], 64)
    x0 = torch.zeros(64, device="cuda")
    ops.chain_q4(x0, glins, 0, 2)
    torch.cuda.synchronize()
    assert all(torch.isnan(y).all() for _, _, y, _ in glins)
    ops.chain_q4(x0, glins, 3, 2)
    torch.cuda.synchronize()
    for _, _, y, _ in glins:
        assert torch.equal(y.view(torch.int32), torch.zeros_like(y).view(torch.int32))
    assert ops.device_status() == 0


def _tie_inputs(amax: float, K: int, seed: int) -> np.ndarray:
    """x0 with max |x0| = amax, the rest exact and near half-integer multiples
    of the Q8 scale fl(amax / 127): the values whose code depends on the last
    bit of the quotient and on ties-to-even."""
    sx = np.float32(np.float32(amax) / np.float32(127))
    vals = [np.float32(amax)]
    for k in range(-127, 127):
        h = np.float32((k + 0.5) * float(sx))
        vals += [h, np.nextafter(h, np.float32(np.inf)), np.nextafter(h, np.float32(-np.inf))]
    vals = np.array(vals, np.float32)
    rng = np.random.default_rng(seed)
    vals = np.concatenate([vals, rng.uniform(-amax, amax, K).astype(np.float32)])[:K]
    vals[0] = np.float32(amax)
    return vals


@pytest.mark.parametrize("amax", [127.0, 100.0, 3.0e-3])
def test_chain_quantizer_ties(ops, ora, amax):
    """Unit-vector weights make y reveal every Q8 code of the chain's input
    (y_n = 7 q_n sx / 7 exactly per channel); a second linear re-quantises
    that output.  Bit-exact against the oracle's quantize_row_q8 + linear_q4."""
    K = 1024
    W = np.zeros((K, K), np.float32)
    W[np.arange(K), np.arange(K)] = 1.0
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    pk, sw = ops.quantize_matrix_q4(dev(W))
    W2 = synth.weights_f32(4300, 64, K)
    pk2, sw2 = ops.quantize_matrix_q4(dev(W2))
    x0 = _tie_inputs(amax, K, 4301)
    ys = [torch.empty((1, K), device="cuda"), torch.empty((1, 64), device="cuda")]
    ops.chain_q4(dev(x0), [(pk, sw, ys[0], -1), (pk2, sw2, ys[1], 0)], 1, 1)
    ref = oracle_chain(ora, x0, [ora.quantize_matrix_q4(W) + (-1,), ora.quantize_matrix_q4(W2) + (0,)], 1, 1)
    torch.cuda.synchronize()
    assert np.array_equal(ys[0].cpu().numpy().view(np.uint32), ref[0].view(np.uint32))
    assert np.array_equal(ys[1].cpu().numpy().view(np.uint32), ref[1].view(np.uint32))
    assert ops.device_status() == 0
