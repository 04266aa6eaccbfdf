"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

Each pin takes an ``oracle.Oracle`` and raises AssertionError on a mismatch.
None of them re-types the oracle's own arithmetic: they compare with values
printed on the pages (tests/golden/, each file citing its passage), closed
forms, brute force over tiny inputs, invariants, or independent library
routines (numpy's IEEE half decoder, torch's bfloat16 rounding, numpy float64
matmul of an independently decoded weight).  The same battery runs against
every planted mutant of the oracle (test_oracle_mutants.py), so each pin is
shown to catch the mistakes it is meant to catch.
"""
from __future__ import annotations

import numpy as np

from tests.golden import load_kv, load_table
from w4a16_int4_quantized_gb300 import synth

REF_OK, REF_EINVAL, REF_ESHAPE = 0, 1, 2

# ---------------------------------------------------------------- independent decoders

# Signed nibble table as printed ("Fused int4 ..." 2.2): from the golden file.
_NIB = np.array([r[1] for r in load_table("nibble_codes.txt")], dtype=np.int64)


def np_unpack_codes(packed: np.ndarray, K: int, biased: bool) -> np.ndarray:
    """Packed rows -> int64 codes [N, K] (low nibble = even column)."""
    packed = np.asarray(packed, dtype=np.uint8)
    lo = (packed & 0x0F).astype(np.int64)
    hi = (packed >> 4).astype(np.int64)
    u = np.empty((packed.shape[0], packed.shape[1] * 2), dtype=np.int64)
    u[:, 0::2] = lo
    u[:, 1::2] = hi
    u = u[:, :K]
    return u - 8 if biased else _NIB[u]


def np_pack(u: np.ndarray, pad: int) -> np.ndarray:
    """Raw nibble values u [N, K] in 0..15 -> packed bytes [N, ceil(K/2)]."""
    N, K = u.shape
    if K % 2:
        u = np.concatenate([u, np.full((N, 1), pad, dtype=u.dtype)], axis=1)
    return (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def np_f16(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def torch_bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.asarray(bits, dtype=np.uint16).astype(np.int16).copy()).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def np_dequant_w4a16(w: np.ndarray, s: np.ndarray, K: int, G: int) -> np.ndarray:
    """W64[n, k] = q[n, k] * s[n, k // G] in float64."""
    q = np_unpack_codes(w, K, biased=False).astype(np.float64)
    sc = np_f16(s)
    return q * np.repeat(sc, G, axis=1)[:, :K]


# ---------------------------------------------------------------- pins

def pin_hand_example_w4a16(o):
    g = load_kv("hand_example_w4a16.txt")
    x = synth.f32_to_bf16_bits(np.array(g["x"], np.float32)).reshape(1, -1)
    w = np.array(g["bytes"], np.uint8).reshape(2, 2)
    s = np.array(g["scales_f16"], np.uint16).reshape(2, 2)
    want = np.array(g["y"], np.float64).reshape(1, 2)
    y, _ = o.linear_w4a16_exact(x, w, s, g["K"], g["G"])
    assert np.array_equal(y, want), (y, want)
    yl = o.linear_w4a16_lanes(x, w, s, g["K"], g["G"])
    assert np.array_equal(yl.astype(np.float64), want), (yl, want)
    yb = o.linear_w4a16_bf16dequant(x, w, s, g["K"], g["G"])
    assert np.array_equal(yb, want), (yb, want)


def pin_hand_example_bytes(o):
    """The printed bytes decode, nibble by nibble, to the printed codes."""
    g = load_kv("hand_example_w4a16.txt")
    codes = np.array(g["codes"]).reshape(2, 4)
    by = np.array(g["bytes"], np.uint8).reshape(2, 2)
    got = np.array([[o.nibble_signed(int(b >> (4 * h)) & 0xF) for b in row for h in (0, 1)] for row in by])
    assert np.array_equal(got, codes), got
    assert np.array_equal(np_unpack_codes(by, 4, False), codes)


def pin_hand_example_q8(o):
    g = load_kv("hand_example_q8.txt")
    x = np.array(g["x"], np.float32).reshape(1, 4)
    wq = np.array(g["codes"], np.int8).reshape(2, 4)
    s = np.array(g["scales"], np.float32)
    want = np.array(g["y"], np.float32).reshape(1, 2)
    assert np.array_equal(o.linear_w8a32(x, wq, s), want)
    # W8A8 with xq = x (exact small integers) and sx = 1 reproduces it.
    y = o.linear_q8(x.astype(np.int8), np.ones(1, np.float32), wq, s)
    assert np.array_equal(y, want), y


def pin_every_nibble_code(o):
    table = load_table("nibble_codes.txt")
    for u, v in table:
        assert o.nibble_signed(u) == v, (u, o.nibble_signed(u), v)
        assert o.nibble_biased(u) == u - 8
    # both nibble positions through the full W4A16 linear: one weight row of
    # two columns, unit activations, scale 1.0 (f16 0x3C00).
    w = np.array([[lo | (hi << 4)] for lo in range(16) for hi in range(16)], np.uint8)
    s = np.full((256, 1), 0x3C00, np.uint16)
    e0 = synth.f32_to_bf16_bits(np.array([[1.0, 0.0]], np.float32))
    e1 = synth.f32_to_bf16_bits(np.array([[0.0, 1.0]], np.float32))
    y0, _ = o.linear_w4a16_exact(e0, w, s, 2, 2)
    y1, _ = o.linear_w4a16_exact(e1, w, s, 2, 2)
    lo = np.repeat(np.arange(16), 16)
    hi = np.tile(np.arange(16), 16)
    assert np.array_equal(y0[0], _NIB[lo].astype(np.float64)), "low nibble is column 2b"
    assert np.array_equal(y1[0], _NIB[hi].astype(np.float64)), "high nibble is column 2b+1"


def pin_f16_golden(o):
    for bits, val in load_table("f16_scales.txt"):
        assert o.f16_to_f32(bits) == val, (hex(bits), o.f16_to_f32(bits), val)


def pin_f16_bruteforce(o):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = np_f16(allbits)
    got = np.array([o.f16_to_f32(int(b)) for b in allbits], np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_bf16(o):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch_bf16_to_f64(allbits)
    got = np.array([o.bf16_to_f32(int(b)) for b in allbits], np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(got[~nan], ref[~nan])
    import torch
    f = synth.normal(7, 4096, 3.0).astype(np.float32)
    f[:4] = [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 0.0]   # exact ties
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([o.f32_to_bf16(v) for v in f], np.uint16)
    assert np.array_equal(got, want)


def pin_ties_to_even(o):
    q, s = o.quantize_row([7.0, 0.5, 1.5, 2.5, -2.5, -7.0, -0.5, 6.5], 7)
    assert s == 1.0 and list(q) == [7, 0, 2, 2, -2, -7, 0, 6], (q, s)
    q, s = o.quantize_row([127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5], 127)
    assert s == 1.0 and list(q) == [127, 0, 2, 2, 0, -2, -2, 126], (q, s)


def pin_negation_symmetry(o):
    for Q in (7, 127):
        for r in range(8):
            v = synth.normal(100 + r, 257, 0.02).astype(np.float32)
            v[r] = -np.abs(v).max() * 1.5       # the extreme may be the negative one
            q1, s1 = o.quantize_row(v, Q)
            q2, s2 = o.quantize_row(-v, Q)
            assert s1 == s2 and np.array_equal(q1.astype(int), -q2.astype(int)), (Q, r)


def pin_quantizer_bounds(o):
    for Q in (7, 127):
        for r in range(6):
            v = synth.normal(200 + r, 300, 1.0).astype(np.float32)
            q, s = o.quantize_row(v, Q)
            qi = q.astype(np.int64)
            assert qi.min() >= -Q and qi.max() <= Q
            assert np.abs(qi).max() == Q
            # nearest code: |v - q*s| <= s/2 (+ the f32 rounding of v/s)
            err = np.abs(v.astype(np.float64) - qi * float(s))
            assert np.all(err <= 0.5 * float(s) * (1 + 1e-6)), err.max() / s
            # s is max|v| / Q to within one f32 rounding
            assert abs(float(s) * Q - float(np.abs(v).max())) <= 2 ** -23 * float(np.abs(v).max()) * Q
        q, s = o.quantize_row(np.zeros(16, np.float32), Q)
        assert s == 0.0 and not q.any()


def pin_quantize_matrix_q4_layout(o):
    for K in (9, 16):
        W = synth.weights_f32(300 + K, 5, K)
        packed, sw = o.quantize_matrix_q4(W)
        assert packed.shape == (5, (K + 1) // 2)
        codes = np_unpack_codes(packed, K, biased=True)
        for n in range(5):
            q, s = o.quantize_row(W[n], 7)
            assert s == sw[n] and np.array_equal(codes[n], q.astype(np.int64))
        if K % 2:
            assert np.all((packed[:, -1] >> 4) == 8), "odd K pads with the biased zero"


def pin_w4a8_hand(o):
    g = load_kv("w4a8_hand_example.txt")
    p, s = o.quantize_matrix_q4(np.array([g["codes"]], np.float32))
    assert s[0] == 1.0 and list(p[0]) == g["bytes"], (p, s)
    assert o.dot_i32_q4(np.array(g["xq"], np.int8), p[0], 4) == g["acc"]
    p, s = o.quantize_matrix_q4(np.array([g["odd_codes"]], np.float32))
    assert list(p[0]) == g["odd_bytes"], p
    assert o.dot_i32_q4(np.array(g["odd_xq"], np.int8), p[0], 3) == g["odd_acc"]


def pin_pad_nibble_wholebyte(o):
    """Odd K: a whole-byte dot (x padded with any value) equals the masked dot."""
    for K in (1, 3, 2047):
        W = synth.weights_f32(400 + K, 3, K)
        packed, _ = o.quantize_matrix_q4(W)
        x = synth.activations_f32(401 + K, 1, K)
        xq, _, _ = o.quantize_row_q8(x)
        xpad = np.concatenate([xq[0].astype(np.int64), [127]])
        for n in range(3):
            u = np.concatenate([(packed[n] & 0xF)[:, None], (packed[n] >> 4)[:, None]], 1).ravel().astype(np.int64)
            whole = int(np.dot(xpad, u - 8))
            assert o.dot_i32_q4(xq[0], packed[n], K) == whole


def pin_bias_cancellation(o):
    for K in (1, 7, 64, 1001):
        xq = (synth.raw_bytes(500 + K, K).view(np.int8)).copy()
        xq[xq == -128] = -127
        wrow = synth.raw_bytes(501 + K, (K + 1) // 2)       # every nibble, incl. 0 (= -8)
        want = int(np.dot(xq.astype(np.int64), np_unpack_codes(wrow[None], K, True)[0]))
        assert o.dot_naive_q4(xq, wrow, K) == want
        assert o.dot_i32_q4(xq, wrow, K) == want


def pin_brute_force_tiny(o):
    """K <= 3: every weight-code combination against a set of activation rows."""
    for K in (1, 2, 3):
        combos = np.array(np.meshgrid(*[np.arange(16)] * K, indexing="ij")).reshape(K, -1).T
        w = np_pack(combos, 8)
        vals = np.array([-127, -3, 0, 2, 127])
        xq = np.array(np.meshgrid(*[vals] * K, indexing="ij")).reshape(K, -1).T.astype(np.int8)
        ones_m = np.ones(xq.shape[0], np.float32)
        ones_n = np.ones(w.shape[0], np.float32)
        y = o.linear_q4(xq, ones_m, w, ones_n, K)
        want = xq.astype(np.int64) @ (combos - 8).T
        assert np.array_equal(y.astype(np.int64), want), K


def pin_linear_q4_random(o):
    M, N, K = 3, 37, 200
    x, W = synth.w4a8_inputs(600, M, N, K)
    xq, sx, rs = o.quantize_row_q8(x)
    assert np.array_equal(rs, xq.astype(np.int64).sum(1))
    packed, sw = o.quantize_matrix_q4(W)
    codes = np_unpack_codes(packed, K, True)
    acc = xq.astype(np.int64) @ codes.T
    y1 = o.linear_q4(xq, np.ones(M, np.float32), packed, np.ones(N, np.float32), K)
    assert np.array_equal(y1.astype(np.int64), acc)
    y = o.linear_q4(xq, sx, packed, sw, K).astype(np.float64)
    exact = acc * sx[:, None].astype(np.float64) * sw[None, :].astype(np.float64)
    assert np.all(np.abs(y - exact) <= 2 * 2.0 ** -24 * np.abs(exact) + 1e-30)


def pin_linear_q8_random(o):
    M, N, K = 3, 37, 200
    x, W = synth.w4a8_inputs(610, M, N, K)
    xq, sx, _ = o.quantize_row_q8(x)
    wq, sw = o.quantize_matrix_q8(W)
    acc = xq.astype(np.int64) @ wq.astype(np.int64).T
    y = o.linear_q8(xq, sx, wq, sw).astype(np.float64)
    exact = acc * sx[:, None].astype(np.float64) * sw[None, :].astype(np.float64)
    assert np.all(np.abs(y - exact) <= 2 * 2.0 ** -24 * np.abs(exact) + 1e-30)
    # q8_matches_dequantize_then_matmul: W8A32, K = 200
    y8 = o.linear_w8a32(x, wq, sw).astype(np.float64)
    ref = x.astype(np.float64) @ (wq.astype(np.float64) * sw[:, None]).T
    scale = np.abs(x).astype(np.float64) @ np.abs(wq.astype(np.float64) * sw[:, None]).T
    assert np.all(np.abs(y8 - ref) <= 1e-5 * scale + 1e-6)


def pin_all_extreme(o):
    for K in (1024, 2047, 2048, 3072):
        xq = np.full(K, 127, np.int8)
        w = np_pack(np.full((1, K), 15), 8)[0]
        assert o.dot_i32_q4(xq, w, K) == 127 * 7 * K
        assert 127 * 15 * K < 2 ** 31
        xa = np.where(np.arange(K) % 2 == 0, 127, -127).astype(np.int8)
        wa = np_pack(np.where(np.arange(K) % 2 == 0, 15, 1)[None], 8)[0]
        assert o.dot_i32_q4(xa, wa, K) == 127 * 7 * K
        y = o.linear_q4(xq[None], np.ones(1, np.float32), w[None], np.ones(1, np.float32), K)
        assert y[0, 0] == 127 * 7 * K
        wq = np.full((1, K), 127, np.int8)
        assert o.dot_i32(xq, wq[0]) == 127 * 127 * K


def pin_dequant_then_matmul_w4a16(o):
    for (M, N, K, G) in ((2, 37, 384, 2), (2, 37, 384, 32), (2, 37, 384, 64), (1, 37, 384, 384),
                         (3, 19, 200, 40), (1, 21, 2047, 32), (2, 9, 256, 128)):
        x, w, s = synth.w4a16_inputs(700 + K + G, M, N, K, G)
        y, a = o.linear_w4a16_exact(x, w, s, K, G)
        ref = torch_bf16_to_f64(x) @ np_dequant_w4a16(w, s, K, G).T
        scale = np.abs(torch_bf16_to_f64(x)) @ np.abs(np_dequant_w4a16(w, s, K, G)).T
        assert np.allclose(a, scale, rtol=1e-12, atol=0)
        assert np.all(np.abs(y - ref) <= 1e-12 * scale + 1e-300), (M, N, K, G)
        yl = o.linear_w4a16_lanes(x, w, s, K, G).astype(np.float64)
        assert np.all(np.abs(yl - ref) <= 1e-5 * scale + 1e-6), (M, N, K, G)
        yb = o.linear_w4a16_bf16dequant(x, w, s, K, G)
        assert np.all(np.abs(yb - ref) <= 2.0 ** -8 * scale + 1e-6), (M, N, K, G)


def pin_quantize_matrix_q8(o):
    # [int8] summary: the weight matrix is quantised row by row with the
    # activation recipe (scale = max|row| / 127, ties to even, [-127, 127]).
    # Hand row: max 127 gives s = 1 exactly, so the codes are rint(v).
    W = np.array([[127.0, 0.5, 1.5, 2.5, -2.5, 126.5],
                  [-254.0, 1.0, 3.0, -5.0, 127.0, 0.0]], np.float32)
    q, sw = o.quantize_matrix_q8(W)
    assert list(sw) == [1.0, 2.0], sw
    assert q[0].tolist() == [127, 0, 2, 2, -2, 126], q[0]
    assert q[1].tolist() == [-127, 0, 2, -2, 64, 0], q[1]   # 1.5 -> 2, 2.5 -> 2, 63.5 -> 64
    for K in (1, 37, 300):
        W = synth.weights_f32(900 + K, 7, K)
        W[3] *= 50.0                                   # rows on different scales
        W[5, K // 2] = -4.0 * float(np.abs(W[5]).max())  # a negative extreme
        q, sw = o.quantize_matrix_q8(W)
        qi = q.astype(np.int64)
        assert qi.min() >= -127 and np.all(np.abs(qi).max(axis=1) == 127), "codes in [-127, 127], the extreme at 127"
        amax = np.abs(W.astype(np.float64)).max(axis=1)
        assert np.all(np.abs(sw.astype(np.float64) * 127 - amax) <= 2.0 ** -23 * amax * 127)
        err = np.abs(W.astype(np.float64) - qi * sw[:, None].astype(np.float64))
        assert np.all(err <= 0.5 * sw[:, None] * (1 + 1e-6)), "nearest code per row"
        qn, swn = o.quantize_matrix_q8(-W)
        assert np.array_equal(sw, swn) and np.array_equal(qi, -qn.astype(np.int64)), "negation symmetry"
    assert not o.quantize_matrix_q8(np.zeros((2, 8), np.float32))[0].any()


def pin_bf16_dequant_one_hot(o):
    # One-hot activations make y[m, n] the dequantised weight w[n, m] itself:
    # bf16_rne(q * s), q * s exact in f32; compared with torch's bf16 rounding.
    import torch
    K, N, G = 64, 24, 32
    _, w, s = synth.w4a16_inputs(950, 1, N, K, G)
    s = s.copy()
    s[0, 0] = 0x3C0C          # 1 + 3 * 2^-8: q = 2 gives an exact bf16 tie
    s[1, 0] = 0x3C03          # 1 + 3 * 2^-10
    q = np_unpack_codes(w, K, biased=False)
    q[0, :] = 2
    q[1, :] = np.arange(K) % 16 - 8
    w = np_pack(q & 0xF, 0)
    eye = np.zeros((K, K), np.uint16)
    eye[np.arange(K), np.arange(K)] = 0x3F80   # bf16 1.0
    y = o.linear_w4a16_bf16dequant(eye, w, s, K, G)
    prod = (q.astype(np.float64) * np_f16(s)[:, np.arange(K) // G]).astype(np.float32)
    want = torch.from_numpy(prod).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(y.T, want), np.argwhere(y.T != want)[:4]
    assert want[0, 0] == 2.0 * (1 + 2.0 ** -6), "the tie rounds to even (up here)"


def pin_interleave_index_pattern(o):
    """Pack index patterns and read back where each nibble landed
    ("The weight layout, measured").  Two patterns together identify the
    channel (n % 16 and n // 16) and the column k of every nibble."""
    N, K = 128, 5
    n = np.arange(N)[:, None]
    k = np.arange(K)[None, :]
    for pattern in (lambda n, k: (n % 16) + 0 * k, lambda n, k: (n // 16 + 3 * k) % 16):
        u = pattern(n, k)
        w = np_pack(u, 8)
        il = o.pack_interleaved_n64(w, K)
        assert il.shape == (N // 64, K, 32)
        for b in range(N // 64):
            for kk in range(K):
                for d in range(32):
                    lo = pattern(64 * b + d, kk)
                    hi = pattern(64 * b + d + 32, kk)
                    assert il[b, kk, d] == lo | (hi << 4), (b, kk, d)
        assert np.array_equal(o.unpack_interleaved_n64(il, N, K, 8), w)
        assert np.array_equal(o.unpack_interleaved_n64(il, N, K, 0), np_pack(u, 0))


def pin_batch_invariance(o):
    M, N, K, G = 12, 24, 256, 32
    x, w, s = synth.w4a16_inputs(800, M, N, K, G)
    yb = o.linear_w4a16_lanes(x, w, s, K, G)
    for m in range(M):
        y1 = o.linear_w4a16_lanes(x[m:m + 1], w, s, K, G)
        assert np.array_equal(y1[0].view(np.uint32), yb[m].view(np.uint32)), m


def pin_shape_errors(o):
    st = o.w4a16_status
    assert st(1, 2, 4, 3) == REF_ESHAPE      # G odd
    assert st(1, 2, 4, 0) == REF_ESHAPE      # G <= 0
    assert st(1, 2, 4, -2) == REF_ESHAPE
    assert st(1, 2, 12, 8) == REF_ESHAPE     # K % G != 0
    assert st(1, 2, 10, 4) == REF_ESHAPE
    assert st(-1, 2, 4, 2) == REF_EINVAL
    assert st(1, 2, 4, 2) == REF_OK
    assert st(0, 2, 4, 2) == REF_OK


def pin_null_pointers(o):
    """shape_and_argument_errors, NULL half ("Fused int4 ..." section 4: EINVAL
    for NULL pointers, before any read, y untouched): each required pointer
    missing in turn, with the others valid."""
    import ctypes as C
    M, N, K, G = 1, 2, 4, 2
    x = np.zeros(M * K, np.uint16)
    w = np.zeros(N * K // 2, np.uint8)
    s = np.zeros(N * K // G, np.uint16)
    y = np.full(M * N, 7.0, np.float32)
    p = lambda a: a.ctypes.data_as(C.c_void_p)
    args = [p(x), p(w), p(s), p(y)]
    for i in range(4):
        a = list(args)
        a[i] = None
        assert o.lib.ref_linear_w4a16_lanes(*a, M, N, K, G) == REF_EINVAL, i
        assert np.all(y == 7.0)
    assert o.lib.ref_linear_w4a16_lanes(*args, M, N, K, G) == REF_OK
    xq, sx, sw = np.zeros(K, np.int8), np.ones(M, np.float32), np.ones(N, np.float32)
    y[:] = 7.0
    q4 = [p(xq), p(sx), p(w), p(sw), p(y)]
    for i in range(5):
        a = list(q4)
        a[i] = None
        assert o.lib.ref_linear_q4(*a, M, N, K) == REF_EINVAL, i
        assert np.all(y == 7.0)


# ---------------------------------------------------------------- inline-scale blocks of 32

def pin_b32_closed_form(o):
    """One block by hand: codes q_k = (k mod 16) - 8 (two runs of -8..7, sum -16),
    scale 0.5 (f16 0x3800), x = 1: y = 0.5 * -16 = -8; the block's bytes are
    [0x00, 0x38] then byte j = nib(2j) | nib(2j+1) << 4 of the signed codes."""
    q = (np.arange(32) % 16) - 8
    nibs = q & 0xF
    codes = (nibs[0::2] | (nibs[1::2] << 4)).astype(np.uint8)
    blk = np.concatenate([[0x00, 0x38], codes]).astype(np.uint8)[None]
    x = np.full((1, 32), 0x3F80, np.uint16)                # bf16 1.0
    y, a = o.linear_w4a16_b32_exact(x, blk, 32)
    assert y[0, 0] == -8.0 and a[0, 0] == 0.5 * 2 * (8 * 9 // 2 + 7 * 8 // 2), (y, a)
    b = o.blocks_b32(codes[None], np.array([[0x3800]], np.uint16), 32)
    assert np.array_equal(b, blk), b


def pin_b32_same_numbers_as_planes(o):
    """Blocks built from the planes give exactly the plane form's W4A16 (G = 32)
    result; odd K (pad nibble) included."""
    for (M, N, K) in ((2, 5, 64), (1, 9, 255), (3, 4, 1024)):
        x, w, s = synth.w4a16_inputs(730 + K, M, N, K, 32)
        blocks = o.blocks_b32(w, s, K)
        assert blocks.shape == (N, (K + (K & 1)) // 32 * 18)
        y, a = o.linear_w4a16_b32_exact(x, blocks, K)
        yp, ap = o.linear_w4a16_exact(x, w, s, K, 32)
        assert np.array_equal(y, yp) and np.array_equal(a, ap), K


# ---------------------------------------------------------------- linear_w8a16

def pin_w8a16_hand_example(o):
    """The printed W8A32 hand example ("Fused int4 ..." section 3): f32 x times
    int8 codes with one scale per row gives [-13, 5]; exact in double."""
    g = load_kv("hand_example_q8.txt")
    x = np.array(g["x"], np.float32).reshape(1, 4)
    wq = np.array(g["codes"], np.int8).reshape(2, 4)
    s = np.array(g["scales"], np.float32)
    y, a = o.linear_w8a16_exact(x, wq, s)
    assert np.array_equal(y, np.array([g["y"]], np.float64)), y
    assert np.array_equal(a, np.array([[0.5 * (1 + 4 + 9 + 32), 0.25 * (7 + 0 + 3 + 16)]])), a


def pin_w8a16_random(o):
    """Random f32 x and int8 codes (every value) against a float64 matmul, and
    against the pages' f32 order (ref_linear_w8a32) within f32 accumulation error."""
    M, N, K = 3, 29, 300
    x = synth.activations_f32(720, M, K)
    wq = synth.raw_bytes(721, N * K).view(np.int8).reshape(N, K)
    sw = (synth.uniform01(722, N) * 0.01 + 1e-3).astype(np.float32)
    y, a = o.linear_w8a16_exact(x, wq, sw)
    want = (x.astype(np.float64) @ wq.astype(np.float64).T) * sw[None, :].astype(np.float64)
    assert np.allclose(y, want, rtol=1e-12, atol=1e-12)
    assert np.allclose(a, np.abs(x.astype(np.float64)) @ np.abs(wq.astype(np.float64)).T * sw[None, :])
    y32 = o.linear_w8a32(x, wq, sw).astype(np.float64)
    assert np.all(np.abs(y32 - y) <= K * 2.0 ** -23 * a + 1e-30)


# ---------------------------------------------------------------- grouped asymmetric W4A8

def np_dequant_q4_group(w, s, z, K: int, G: int) -> np.ndarray:
    """W64[n, k] = (u[n, k] - z[n, k // G]) * f16(s[n, k // G]), raw nibbles decoded independently."""
    u = np_unpack_codes(w, K, biased=True) + 8
    g = np.arange(K) // G
    return (u - np.asarray(z, np.int64)[:, g]).astype(np.float64) * np_f16(s)[:, g]


def pin_q4_group_hand(o):
    """Worked by hand (not printed on the pages): K = 4, G = 2, xq = [1, 2, 3, 4], sx = 1.
    Row 0: u = [15, 8, 7, 12] (bytes 0x8F 0xC7), z = [8, 10], s = [0.5, 0.25]:
      g0 = 1*7 + 2*0 = 7, g1 = 3*(-3) + 4*2 = -1, y = 7*0.5 - 0.25 = 3.25, sum|terms| = 3.5 + 17*0.25.
    Row 1: u = [0, 15, 3, 3] (bytes 0xF0 0x33), z = [3, 3], s = [1, 2]:
      g0 = 1*(-3) + 2*12 = 21, g1 = 0, y = 21."""
    w = np.array([[0x8F, 0xC7], [0xF0, 0x33]], np.uint8)
    s = np.array([[0x3800, 0x3400], [0x3C00, 0x4000]], np.uint16)
    z = np.array([[8, 10], [3, 3]], np.uint8)
    xq = np.array([[1, 2, 3, 4]], np.int8)
    y, a = o.linear_q4_group(xq, np.ones(1, np.float32), w, s, z, 4, 2)
    assert y[0, 0] == 3.25 and y[0, 1] == 21.0, y
    assert a[0, 0] == 3.5 + 17 * 0.25 and a[0, 1] == 27.0, a


def pin_q4_group_symmetric_is_linear_q4(o):
    """Zero points all 8 and one scale per row: the grouped contract reduces to
    the (pinned) per-channel linear_q4 -- up to linear_q4's two f32 roundings."""
    M, N, K, G = 3, 29, 256, 64
    x, W = synth.w4a8_inputs(700, M, N, K)
    xq, sx, _ = o.quantize_row_q8(x)
    w, sw = o.quantize_matrix_q4(W)
    s16 = np.asarray(sw, np.float32).astype(np.float16)           # f16 scale, the same in every group
    s = np.repeat(s16.view(np.uint16)[:, None], K // G, axis=1)
    z = np.full((N, K // G), 8, np.uint8)
    y, _ = o.linear_q4_group(xq, sx, w, s, z, K, G)
    y1 = o.linear_q4(xq, sx, w, s16.astype(np.float32), K).astype(np.float64)
    assert np.all(np.abs(y - y1) <= 2 * 2.0 ** -24 * np.abs(y1) + 1e-30)


def pin_q4_group_random(o):
    """Random codes, zero points and scales against a float64 matmul of the
    independently dequantised weights; odd K; several groups per row."""
    for (M, N, K, G) in ((2, 13, 96, 32), (3, 7, 255, 128), (1, 40, 1000, 8)):
        Kp = K + (K & 1)
        xq = synth.raw_bytes(710 + K, M * K).view(np.int8).reshape(M, K).copy()
        xq[xq == -128] = -127
        sx = (synth.uniform01(711 + K, M) + 0.5).astype(np.float32)
        w = synth.raw_bytes(712 + K, N * (Kp // 2)).reshape(N, Kp // 2)
        s = synth.group_scales_f16(713 + K, N, Kp // G)
        z = (synth.raw_bytes(714 + K, N * (Kp // G)) & 0x0F).reshape(N, Kp // G)
        y, a = o.linear_q4_group(xq, sx, w, s, z, K, G)
        W64 = np_dequant_q4_group(w, s, z, K, G)
        want = sx[:, None].astype(np.float64) * (xq.astype(np.float64) @ W64.T)
        awant = np.abs(sx[:, None].astype(np.float64)) * (np.abs(xq.astype(np.float64)) @ np.abs(W64).T)
        assert np.allclose(y, want, rtol=1e-12, atol=1e-9), (M, N, K, G)
        assert np.allclose(a, awant, rtol=1e-12, atol=1e-9)


PINS = {name[4:]: fn for name, fn in globals().items() if name.startswith("pin_")}


def pool_equals_serial(serial, omp):
    """pool_result_equals_serial_bitwise: the row-parallel build, N = 37."""
    M, N, K, G = 3, 37, 256, 32
    x, w, s = synth.w4a16_inputs(900, M, N, K, G)
    a = serial.linear_w4a16_lanes(x, w, s, K, G)
    b = omp.linear_w4a16_lanes(x, w, s, K, G)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    xf, W = synth.w4a8_inputs(901, M, N, K)
    xq, sx, _ = serial.quantize_row_q8(xf)
    p, sw = serial.quantize_matrix_q4(W)
    assert np.array_equal(serial.linear_q4(xq, sx, p, sw, K).view(np.uint32),
                          omp.linear_q4(xq, sx, p, sw, K).view(np.uint32))
