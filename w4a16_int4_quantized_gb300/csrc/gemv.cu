// gemv.cu -- decode-regime linears (M <= 16) for W4A8, W8A8 and group-wise W4A16.
//
// What is computed (per output element):
//   W4A8  ("linear_q4", docs.rs ftts_kernels::int4):
//         acc = sum_k x[m][k] * u[n][k] - 8 * sum_k x[m][k]   (exact i32)
//         y   = (f32(acc) * sx[m]) * sw[n]
//   W8A8  ("linear_q8", docs.rs ftts_kernels::int8): acc = sum_k x*w, same epilogue.
//   W4A16 ("Fused int4 and int8 dequantize-matmul in C", 2.3):
//         y = sum_g s[n][g] * partial_g,  partial_g = sum_{k in g} x*q  (fp32)
//
// Design (GB300): the GEMV is HBM-bound -- a weight byte is used M times.
//  * Each CTA owns a tile of R output channels and a contiguous K range.
//    Its weight tile is fetched by one thread with bulk async copies
//    (cp.async.bulk, one per row, completing on an mbarrier), so the whole
//    tile is in flight at once without occupying registers.  With PDL the
//    copies are issued before griddepcontrol.wait: weights do not depend on
//    the previous kernel, so the fetch overlaps its tail.
//  * The packed tile lands in shared memory with a padded row stride; warps
//    read it in the register layout of mma.sync and unpack nibbles with
//    LOP3/PRMT-class integer ops.  The tensor core does the k-reduction:
//    m16n8k32 s8 for the integer kinds (a dp4a-style int8 dot product, 8
//    products per thread per instruction), m16n8k16 bf16 for W4A16 (the
//    signed codes are exact bf16 integers; the group scale is applied to the
//    f32 partial after the group's MMAs).  Activations are the MMA's N
//    dimension (8 per tile; 16 with two tiles), weights its M dimension.
//  * The k-slot <-> column assignment inside an MMA is free as long as both
//    operands agree, so x is staged in shared memory pre-permuted to match
//    the order the nibbles come out of a 32-bit word.
//  * K is split across the warps of a CTA and, for small N, across the CTAs
//    of a thread-block cluster; partial sums are combined in a fixed order
//    (warps in index order, then cluster ranks in order through distributed
//    shared memory), so the f32 result does not depend on scheduling.
//  * The interleaved [N/64][K][32 B] layout is fetched as one contiguous
//    bulk copy per 64-channel block and transposed in shared memory (4x4
//    byte transposes with PRMT) into the row-major tile; from there the
//    arithmetic is the row-major path's, so the two layouts agree bit for bit.
//  * Under PDL, large-N calls stream instead (gemv_stream_kernel): one CTA
//    per ~N/152 rows, its whole weight range requested by bulk copies at
//    entry, at most two CTAs per SM so the next launch prefetches while this
//    one computes -- the same arithmetic, so the same bits.  W4A8 at M = 1
//    uses integer dot products there (gemv_q4dp_kernel), and the fused
//    quantize + linear call quantises the activation row inside these
//    kernels (stage_x_q8).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>
#include <numeric>
#include <type_traits>

#include "w4.h"
#include "common.cuh"
#include "internal.h"

namespace w4 {
namespace {

template <int KIND> constexpr bool kGrouped = KIND == KIND_W4A16 || KIND == KIND_W4A8G;  // f16 group scales
template <int KIND> constexpr bool kIntAcc = KIND == KIND_W4A8 || KIND == KIND_W8A8;     // i32 accumulators
template <int KIND> constexpr bool kBiased = KIND == KIND_W4A8 || KIND == KIND_W4A8G;    // u - 8 MMA operands
template <int KIND> constexpr bool kW8 = KIND == KIND_W8A8 || KIND == KIND_W8A16;        // int8 weights, 32-B chunks
template <int KIND> constexpr int kXPlanes = KIND == KIND_W8A16 ? 2 : 1;  // f32 x as bf16 hi + lo

// Integer kinds: whether a warp may add its unit partials (exact integers in
// f32) in f32 and convert once -- every partial sum of the warp is an integer
// below 2^24 in magnitude, so each f32 addition is exact and the result is the
// i32 sum.  Columns per warp times the largest |x code * weight code|.
template <int KIND>
W4_DEV bool f32_sum_exact(int units_per_warp, int unit_k) {
    return (long long)units_per_warp * unit_k * 127 * (kW8<KIND> ? 128 : 8) < (1LL << 24);
}

// acc += part, exactly: in f32 (bits kept in the int) or per unit in i32.
W4_DEV void add_exact(int &acc, float part, bool f32sum) {
    if (f32sum) acc = __float_as_int(__int_as_float(acc) + part);
    else acc += __float2int_rn(part);
}
W4_DEV void finish_exact(int &acc, bool f32sum) {
    if (f32sum) acc = __float2int_rn(__int_as_float(acc));
}

struct GemvParams {
    const void *x;
    const uint8_t *w;
    const void *scale;
    const float *sx;
    const uint8_t *zeros;  // W4A8G: [N][ng]
    float *y;
    uint32_t *status;
    int M, N, K;
    int Kb;          // bytes per packed row (row-major)
    int ng;          // W4A16: scale groups per row
    int cpg;         // 32-column chunks per unit (a unit is one group for W4A16, one chunk otherwise)
    int units;       // units per row
    int upc;         // units per CTA (split-K granularity)
    int upp;         // units per transpose phase (interleaved layout)
    int R, WR, WK;   // rows per CTA, warps along rows, warps along K
    int unit_k;      // columns per unit
    int unit_bytes;  // packed bytes per unit per row
    int wstride;     // shared row stride of the (row-major) weight tile (bytes)
    int rawstride;   // inline-scale blocks: shared row stride of the raw block rows (bytes)
    int xstride;     // shared row stride of the activation tile (bytes)
    int sstride;     // shared row stride of the f32 scale tile (floats)
    int raw_off, w_off, x_off, sc_off, red_off, bar_off;
    int zc_off, xs_off;  // W4A8G: (8 - z) per [row][unit] (int), activation sums per [m][unit] (int)
    const float *xf;  // fused W4A8: f32 activations [M][K], quantised per row in every CTA
    int8_t *xq_out;   // fused W4A8: the Q8 codes [M][K] (written by CTA 0)
    float *sx_out;    // fused W4A8: the row scales [M] (written by CTA 0)
    int xq_off;       // fused W4A8: shared row scales [16] + per-warp row maxima [16 warps][8]
    int rb;           // streaming kernels: rows per mbarrier block
    int x_vec;       // activation rows can be read with aligned vector loads
    int s_vec;       // scale rows can be read as 16-byte vectors
    int x_al;        // the activation base is 16-byte aligned
    int x_pref;      // bytes of the activation row prefetched into L2 before the PDL wait (0: none)
};

// ---------------------------------------------------------------- MMA wrappers

W4_DEV void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Signed nibbles k0..k7 of a word -> four bf16x2 pairs of exact integers:
// P0 = (k0, k4), P1 = (k1, k5), P2 = (k2, k6), P3 = (k3, k7).
// 0x4300 | v is the bf16 128 + v (v < 128); with v = u ^ 8 = q + 8 the value
// is 136 + q, and subtracting 136 is exact.
W4_DEV void unpack_signed_bf16(uint32_t w, uint32_t (&p)[4]) {
    // one shift, one LOP3 ((v & 0x000F000F) ^ 0x43084308) and one bf16x2
    // subtraction per pair, written out so nothing else is generated around them
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t v = w, r;
        if (i > 0) asm("shr.b32 %0, %1, %2;" : "=r"(v) : "r"(w), "r"(4 * i));
        asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(v), "r"(0x000F000Fu), "r"(0x43084308u));
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(p[i]) : "r"(r), "r"(0x43084308u));
    }
}

// Biased nibbles (u = q + 8) of a word -> four f16x2 pairs of the exact
// integers q: P0 = (k0, k4), P1 = (k1, k5), P2 = (k2, k6), P3 = (k3, k7).
// 0x6400 | u is the f16 1024 + u; subtracting 1032 is exact.
W4_DEV void unpack_biased_f16(uint32_t w, uint32_t (&p)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t v = w, r;
        if (i > 0) asm("shr.b32 %0, %1, %2;" : "=r"(v) : "r"(w), "r"(4 * i));
        // (v & 0x000F000F) | 0x64006400
        asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(0x000F000Fu), "r"(0x64006400u));
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(p[i]) : "r"(r), "r"(0x64086408u));
    }
}

// Eight int8 values (lo = bytes 0-3, hi = bytes 4-7) -> four f16x2 pairs of
// the same integers, pair i made of the two bytes PRMT selector sel[i] puts
// in result bytes 0 and 2.  b ^ 0x80 = b + 128; 0x6400 | (b + 128) is the
// f16 1024 + 128 + b, and subtracting 1152 is exact.
W4_DEV void s8_to_f16_pairs(uint32_t lo, uint32_t hi, const uint32_t (&sel)[4], uint32_t (&p)[4]) {
    const __half2 off = __halves2half2(__ushort_as_half((unsigned short)0x6480), __ushort_as_half((unsigned short)0x6480));
    lo ^= 0x80808080u;
    hi ^= 0x80808080u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t v = (prmt(lo, hi, sel[i]) & 0x00FF00FFu) | 0x64006400u;
        __half2 h = *reinterpret_cast<const __half2 *>(&v);
        h = __hsub2(h, off);
        p[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
}

// Eight int8 values -> four bf16x2 pairs of the same integers (exact: |b| <= 128
// fits bf16's 8-bit significand), pair i from the bytes PRMT selector sel[i]
// puts in result bytes 0 and 2.
W4_DEV void s8_to_bf16_pairs(uint32_t lo, uint32_t hi, const uint32_t (&sel)[4], uint32_t (&p)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t v = prmt(lo, hi, sel[i]);  // bytes 0 and 2 hold the two values
        const int a = (int)(int8_t)(v & 0xFFu), b = (int)(int8_t)((v >> 16) & 0xFFu);
        __nv_bfloat162 h = __floats2bfloat162_rn((float)a, (float)b);
        p[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
}

W4_DEV void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Division by a CTA-invariant divisor d (< 2^16) of j < 2^16: floor(j / d)
// = umulhi(j, ceil(2^32 / d)).
// j / d for 0 <= j < 2^32 / d by one high multiply with ceil(2^32 / d); for
// d = 1 the multiplier (2^32) does not fit and is stored as 0, meaning j / 1.
W4_DEV uint32_t div_magic(uint32_t d) { return 0xFFFFFFFFu / d + 1u; }
W4_DEV int fast_div(int j, uint32_t magic) { return magic ? (int)__umulhi((uint32_t)j, magic) : j; }

// One unit (CPG chunks of 32 columns) of one warp: MMA partial sums for the
// warp's 16-row block (rows g, g + 8 of each thread) against MT 8-row
// activation tiles.  wr0 / wr8: the thread's word in the unit's first chunk
// of rows g and g + 8; xr[mt]: the thread's 8 activations of that chunk.
// Byte offset, inside a weight tile, of the thread's word of 16-byte chunk c
// of its row.  Row-major tiles arrive by TMA with the 128-byte swizzle:
// [segment][R rows][128 B], chunk (c mod 8) of a row stored at (c mod 8) xor
// (row mod 8); a warp's 8 rows then read 8 distinct bank groups.  The
// interleaved layout is transposed into padded rows of `wstride` bytes.
template <bool SWZ, int KIND>
W4_DEV int wword_off(int c, int g, int t, int R128) {
    if constexpr (SWZ) {
        if constexpr (kW8<KIND>) {
            const int c16 = 2 * c + (t >> 1);
            return (c16 >> 3) * R128 + (((c16 & 7) ^ g) << 4) + 8 * (t & 1);
        }
        return (c >> 3) * R128 + (((c & 7) ^ g) << 4) + 4 * t;
    } else {
        return kW8<KIND> ? 32 * c + 8 * t : 16 * c + 4 * t;
    }
}

// One unit (CPG chunks of 32 columns, starting at chunk c0 of the tile) of
// one warp: MMA partial sums for the warp's 16-row block (rows g, g + 8 of
// each thread) against MT 8-row activation tiles.  w0 / w8: rows g and g + 8
// of the tile; xr[mt]: the thread's activations of the unit's first chunk.
template <int KIND, bool SWZ, int RB, int MT, int CPG>
W4_DEV void unit_mma(const uint8_t *w0, const uint8_t *w8, int c0, int g, int t, int R128,
                     const uint8_t *const (&xr)[MT], const bool (&xvalid)[MT], int cpg_rt, float (&part)[MT][4],
                     int xlo = 0) {
    const uint32_t xsel8[4] = {0x0100u, 0x0302u, 0x0504u, 0x0706u};
    const int nc = CPG > 0 ? CPG : cpg_rt;
#pragma unroll
    for (int c = 0; c < (CPG > 0 ? CPG : 1); ++c) {
        for (int cc = (CPG > 0 ? c : 0); cc < (CPG > 0 ? c + 1 : nc); ++cc) {
            const int wo = wword_off<SWZ, KIND>(c0 + cc, g, t, R128);
            uint32_t pa[4], pb[4] = {0u, 0u, 0u, 0u};
            if constexpr (KIND == KIND_W4A16) {
                unpack_signed_bf16(*reinterpret_cast<const uint32_t *>(w0 + wo), pa);
                if (RB == 16) unpack_signed_bf16(*reinterpret_cast<const uint32_t *>(w8 + wo), pb);
            } else if constexpr (kBiased<KIND>) {
                unpack_biased_f16(*reinterpret_cast<const uint32_t *>(w0 + wo), pa);
                if (RB == 16) unpack_biased_f16(*reinterpret_cast<const uint32_t *>(w8 + wo), pb);
            } else if constexpr (KIND == KIND_W8A16) {
                const uint2 wa = *reinterpret_cast<const uint2 *>(w0 + wo);
                s8_to_bf16_pairs(wa.x, wa.y, xsel8, pa);
                if (RB == 16) {
                    const uint2 wb = *reinterpret_cast<const uint2 *>(w8 + wo);
                    s8_to_bf16_pairs(wb.x, wb.y, xsel8, pb);
                }
            } else {
                const uint2 wa = *reinterpret_cast<const uint2 *>(w0 + wo);
                s8_to_f16_pairs(wa.x, wa.y, xsel8, pa);
                if (RB == 16) {
                    const uint2 wb = *reinterpret_cast<const uint2 *>(w8 + wo);
                    s8_to_f16_pairs(wb.x, wb.y, xsel8, pb);
                }
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                // activations staged as f16/bf16 pairs in the order of the weight pairs
                uint4 xv = make_uint4(0u, 0u, 0u, 0u);
                if (xvalid[mt]) xv = *reinterpret_cast<const uint4 *>(xr[mt] + 64 * cc);
                if constexpr (KIND == KIND_W4A16) {
                    mma_bf16(part[mt], pa[0], pb[0], pa[1], pb[1], xv.x, xv.y);
                    mma_bf16(part[mt], pa[2], pb[2], pa[3], pb[3], xv.z, xv.w);
                } else if constexpr (KIND == KIND_W8A16) {
                    // x = hi + lo (two bf16 planes): two MMA pairs into the same f32 partial
                    uint4 xl = make_uint4(0u, 0u, 0u, 0u);
                    if (xvalid[mt]) xl = *reinterpret_cast<const uint4 *>(xr[mt] + xlo + 64 * cc);
                    mma_bf16(part[mt], pa[0], pb[0], pa[1], pb[1], xv.x, xv.y);
                    mma_bf16(part[mt], pa[2], pb[2], pa[3], pb[3], xv.z, xv.w);
                    mma_bf16(part[mt], pa[0], pb[0], pa[1], pb[1], xl.x, xl.y);
                    mma_bf16(part[mt], pa[2], pb[2], pa[3], pb[3], xl.z, xl.w);
                } else {
                    mma_f16(part[mt], pa[0], pb[0], pa[1], pb[1], xv.x, xv.y);
                    mma_f16(part[mt], pa[2], pb[2], pa[3], pb[3], xv.z, xv.w);
                }
            }
        }
    }
}

// W4A16 scales of rows [row0, row0 + rows) x units [u0, u0 + nun): 16-byte
// vectors into registers when the rows allow it (stored to shared memory as
// f32 after the PDL wait by store_scales), otherwise converted straight into
// shared memory.  Returns whether the vector path was taken.
template <int KIND>
W4_DEV bool prefetch_scales(const GemvParams &p, int row0, int rows, int u0, int nun, int nthr, uint4 (&sv)[2],
                            uint8_t *smem) {
    constexpr int kMaxSc = 2;
    const int tid = threadIdx.x;
    bool svec = false;
    const int spr = nun >> 3;  // 16-byte scale vectors per row
    svec = kGrouped<KIND> && p.s_vec && rows * spr <= kMaxSc * nthr;
    const uint32_t spr_magic = div_magic((uint32_t)max(spr, 1));
    if constexpr (kGrouped<KIND>) {
        const uint16_t *s16 = static_cast<const uint16_t *>(p.scale);
        if (svec) {
#pragma unroll
            for (int i = 0; i < kMaxSc; ++i) {
                const int j = tid + i * nthr;
                if (j < rows * spr) {
                    const int r = fast_div(j, spr_magic);
                    sv[i] = __ldg(reinterpret_cast<const uint4 *>(s16 + (size_t)(row0 + r) * p.ng + u0) + (j - r * spr));
                }
            }
        } else {
            const uint32_t nun_magic = div_magic((uint32_t)nun);
            float *scf = reinterpret_cast<float *>(smem + p.sc_off);
            for (int i = tid; i < rows * nun; i += nthr) {
                const int r = fast_div(i, nun_magic), gi = i - r * nun;
                scf[r * p.sstride + gi] = __half2float(__ushort_as_half(__ldg(s16 + (size_t)(row0 + r) * p.ng + u0 + gi)));
            }
        }
    }

    return svec;
}

// Activations of columns [k0, k0 + span_k) into shared memory: each group
// of 8 columns becomes four 16-bit pairs in the order of the weight pairs
// (zero beyond K): W4A16 bf16 (x0 x4)(x1 x5)(x2 x6)(x3 x7); W4A8 the same as
// exact f16; W8A8 f16 (x0 x1)(x2 x3)(x4 x5)(x6 x7).
template <int KIND>
W4_DEV void stage_x(const GemvParams &p, int k0, int span_k, int nthr, uint8_t *smem) {
    constexpr bool kInt = KIND != KIND_W4A16;
    const int tid = threadIdx.x;
    {
        const int per_row = span_k >> 3;  // 8-element groups
        const uint32_t pr_magic = div_magic((uint32_t)per_row);
        for (int j = tid; j < p.M * per_row; j += nthr) {
            const int m = fast_div(j, pr_magic), b8 = j - m * per_row;
            const int kk = k0 + 8 * b8;
            uint4 o;
            if constexpr (KIND == KIND_W8A16) {
                // f32 x -> bf16 hi = rn(x), lo = rn(x - hi), pairs (x0 x1)(x2 x3)(x4 x5)(x6 x7)
                const float *xr = static_cast<const float *>(p.x) + (size_t)m * p.K;
                float e[8];
                if (p.x_vec && kk + 8 <= p.K) {
                    const float4 a0 = __ldg(reinterpret_cast<const float4 *>(xr + kk));
                    const float4 a1 = __ldg(reinterpret_cast<const float4 *>(xr + kk + 4));
                    e[0] = a0.x; e[1] = a0.y; e[2] = a0.z; e[3] = a0.w;
                    e[4] = a1.x; e[5] = a1.y; e[6] = a1.z; e[7] = a1.w;
                } else {
#pragma unroll
                    for (int i2 = 0; i2 < 8; ++i2) e[i2] = (kk + i2 < p.K) ? xr[kk + i2] : 0.0f;
                }
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const __nv_bfloat162 h = __floats2bfloat162_rn(e[2 * q], e[2 * q + 1]);
                    const float2 hf = __bfloat1622float2(h);
                    const __nv_bfloat162 l = __floats2bfloat162_rn(e[2 * q] - hf.x, e[2 * q + 1] - hf.y);
                    hi[q] = *reinterpret_cast<const uint32_t *>(&h);
                    lo[q] = *reinterpret_cast<const uint32_t *>(&l);
                }
                *reinterpret_cast<uint4 *>(smem + p.x_off + (p.M + m) * p.xstride + 16 * b8) =
                    make_uint4(lo[0], lo[1], lo[2], lo[3]);
                o = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            } else if constexpr (kInt) {
                const int8_t *xr = static_cast<const int8_t *>(p.x) + (size_t)m * p.K;
                uint2 v;
                if (p.x_vec && kk + 8 <= p.K) {
                    v = __ldg(reinterpret_cast<const uint2 *>(xr + kk));
                } else {
                    uint32_t lo = 0, hi = 0;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t b = (kk + i < p.K) ? (uint32_t)(uint8_t)xr[kk + i] : 0u;
                        if (i < 4) lo |= b << (8 * i);
                        else hi |= b << (8 * (i - 4));
                    }
                    v = make_uint2(lo, hi);
                }
                const uint32_t xsel4[4] = {0x0400u, 0x0501u, 0x0602u, 0x0703u};
                const uint32_t xsel8[4] = {0x0100u, 0x0302u, 0x0504u, 0x0706u};
                uint32_t b[4];
                s8_to_f16_pairs(v.x, v.y, kBiased<KIND> ? xsel4 : xsel8, b);
                o = make_uint4(b[0], b[1], b[2], b[3]);
            } else {
                const uint16_t *xr = static_cast<const uint16_t *>(p.x) + (size_t)m * p.K;
                uint4 v;
                if (p.x_vec && kk + 8 <= p.K) {
                    v = __ldg(reinterpret_cast<const uint4 *>(xr + kk));
                } else {
                    uint32_t e[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) e[i] = (kk + i < p.K) ? (uint32_t)xr[kk + i] : 0u;
                    v = make_uint4(e[0] | (e[1] << 16), e[2] | (e[3] << 16), e[4] | (e[5] << 16), e[6] | (e[7] << 16));
                }
                o = make_uint4(prmt(v.x, v.z, 0x5410), prmt(v.x, v.z, 0x7632), prmt(v.y, v.w, 0x5410),
                               prmt(v.y, v.w, 0x7632));
            }
            *reinterpret_cast<uint4 *>(smem + p.x_off + m * p.xstride + 16 * b8) = o;
        }
    }

}

// Second half of prefetch_scales: the vector path's registers -> f32 in shared memory.
template <int KIND>
W4_DEV void store_scales(const GemvParams &p, int rows, int nun, int nthr, bool svec, const uint4 (&sv)[2],
                         uint8_t *smem) {
    constexpr int kMaxSc = 2;
    const int tid = threadIdx.x;
    const int spr = nun >> 3;
    const uint32_t spr_magic = div_magic((uint32_t)max(spr, 1));
    if constexpr (kGrouped<KIND>) {
        if (svec) {
            float *scf = reinterpret_cast<float *>(smem + p.sc_off);
#pragma unroll
            for (int i = 0; i < kMaxSc; ++i) {
                const int j = tid + i * nthr;
                if (j < rows * spr) {
                    const int r = fast_div(j, spr_magic), c8 = j - r * spr;
                    const uint32_t w4[4] = {sv[i].x, sv[i].y, sv[i].z, sv[i].w};
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        scf[r * p.sstride + 8 * c8 + e] =
                            __half2float(__ushort_as_half((unsigned short)(w4[e >> 1] >> (16 * (e & 1)))));
                }
            }
        }
    }
}

// Combines the K-split warps in index order, then the cluster's K splits in
// rank order (distributed shared memory), and writes y (rank 0, K-warp 0).
template <int KIND, int RB, int MT, typename Acc>
W4_DEV void combine_and_store(const GemvParams &p, Acc (&acc)[MT][4], int wr, int wk, int lane, int g, int t,
                              int rowbase, uint8_t *smem) {
    constexpr bool kInt = kIntAcc<KIND>;
    // ---- 5. combine the K-split warps in index order.
    uint32_t *red = reinterpret_cast<uint32_t *>(smem + p.red_off);
    constexpr int kVals = MT * 4;
    const int WK = p.WK;
    if (WK > 1) {
        if (wk > 0) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    red[((wk * p.WR + wr) * 32 + lane) * kVals + mt * 4 + i] = kInt ? (uint32_t)acc[mt][i]
                                                                                  : __float_as_uint((float)acc[mt][i]);
        }
        __syncthreads();
        if (wk == 0) {
            for (int w2 = 1; w2 < WK; ++w2)
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t v = red[((w2 * p.WR + wr) * 32 + lane) * kVals + mt * 4 + i];
                        if constexpr (kInt) acc[mt][i] += (int)v;
                        else acc[mt][i] += __uint_as_float(v);
                    }
        }
    }

    // ---- combine the cluster's K splits in rank order (distributed shared memory).
    const int S = gridDim.y;
    if (S > 1) {
        __syncthreads();  // red is reused below
        if (wk == 0) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    red[(wr * 32 + lane) * kVals + mt * 4 + i] = kInt ? (uint32_t)acc[mt][i]
                                                                     : __float_as_uint((float)acc[mt][i]);
        }
        cluster_sync();
        if (blockIdx.y == 0 && wk == 0) {
            for (int r = 1; r < S; ++r) {
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t v =
                            dsmem_ld_u32(dsmem_map(&red[(wr * 32 + lane) * kVals + mt * 4 + i], (uint32_t)r));
                        if constexpr (kInt) acc[mt][i] += (int)v;
                        else acc[mt][i] += __uint_as_float(v);
                    }
            }
        }
        cluster_sync();  // peers keep their shared memory alive until rank 0 has read it
    }

    // ---- epilogue.
    if (blockIdx.y != 0 || wk != 0) return;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (RB == 8 && i >= 2) continue;
            const int m = 8 * mt + 2 * t + (i & 1);
            const int n = rowbase + g + 8 * (i >> 1);
            if (m >= p.M || n >= p.N) continue;
            float out;
            if constexpr (kInt) {
                const float sw = static_cast<const float *>(p.scale)[n];
                out = __fmul_rn(__fmul_rn(__int2float_rn((int)acc[mt][i]), p.sx[m]), sw);
            } else if constexpr (KIND == KIND_W4A8G) {
                out = __fmul_rn((float)acc[mt][i], p.sx[m]);  // sx * sum_g acc_g * s_g
            } else if constexpr (KIND == KIND_W8A16) {
                out = __fmul_rn((float)acc[mt][i], static_cast<const float *>(p.scale)[n]);  // sw * sum x q
            } else {
                out = (float)acc[mt][i];
            }
            p.y[(size_t)m * p.N + n] = out;
        }
}

// W4A8G zero points of rows [row0, row0 + rows) x units [u0, u0 + nun) as
// (8 - z) ints in shared memory (weights-side: loaded before the PDL wait).
W4_DEV void load_zero_points(const GemvParams &p, int row0, int rows, int u0, int nun, int nthr, uint8_t *smem) {
    int *zc = reinterpret_cast<int *>(smem + p.zc_off);
    const uint32_t nun_magic = div_magic((uint32_t)nun);
    for (int i = threadIdx.x; i < rows * nun; i += nthr) {
        const int r = fast_div(i, nun_magic), gi = i - r * nun;
        zc[r * p.sstride + gi] = 8 - (int)__ldg(p.zeros + (size_t)(row0 + r) * p.ng + u0 + gi);
    }
}

// W4A8G: sum of the int8 activation codes of every (row m, unit) of the
// CTA's span, for the zero-point correction (x-side: after the PDL wait).
W4_DEV void stage_unit_sums(const GemvParams &p, int k0, int nun, int nthr, uint8_t *smem) {
    int *xs = reinterpret_cast<int *>(smem + p.xs_off);
    const uint32_t nun_magic = div_magic((uint32_t)nun);
    const int8_t *x = static_cast<const int8_t *>(p.x);
    for (int j = threadIdx.x; j < p.M * nun; j += nthr) {
        const int m = fast_div(j, nun_magic), u = j - m * nun;
        const int kb = k0 + u * p.unit_k, ke = min(p.K, kb + p.unit_k);
        int sum = 0;
        const int8_t *xr = x + (size_t)m * p.K;
        int k = kb;
        if (p.x_vec)
            for (; k + 16 <= ke; k += 16) {
                const int4 v = __ldg(reinterpret_cast<const int4 *>(xr + k));
                const int one = 0x01010101;
                sum = __dp4a(v.x, one, sum);
                sum = __dp4a(v.y, one, sum);
                sum = __dp4a(v.z, one, sum);
                sum = __dp4a(v.w, one, sum);
            }
        for (; k < ke; ++k) sum += xr[k];
        xs[m * p.upc + u] = sum;
    }
}

// ---------------------------------------------------------------- kernel
//
// One CTA: rows [row0, row0 + R) x the K range of split blockIdx.y.
//  1. every thread issues 128-bit loads of its share of the weight tile and
//     the W4A16 scales -- before the PDL wait, since no earlier kernel on the
//     stream writes weights;
//  2. griddepcontrol.wait, then 128-bit loads of the activation rows;
//  3. the tiles go to shared memory (padded rows, conflict-free for the MMA
//     fragment reads) and the CTA synchronises once;
//  4. warps run the tensor-core k-reduction over their units, four units at
//     a time with independent accumulators;
//  5. K-split warps, then cluster ranks, are combined in index order.
// A 32-column chunk is two m16n8k16 MMAs.  W4A16: bf16 operands (the signed
// codes are exact bf16 integers), the group scale multiplies the f32
// partial.  W4A8 / W8A8: f16 operands holding exact integers; each 32-column
// unit's partial (|sum| <= 32 * 127 * 128 < 2^24) is exact in the f32
// accumulator and is converted to i32 before it is added, so the integer
// result is exact for any K.
template <int KIND, int LAY, int RB, int MT, int CPG>
__global__ void __launch_bounds__(512) gemv_kernel(const __grid_constant__ GemvParams p) {
    constexpr bool N64 = LAY == 1;  // interleaved [N/64][K][32] layout
    constexpr bool B32 = LAY == 2;  // inline-scale blocks of 32
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wr = warp % p.WR, wk = warp / p.WR;
    const int g = lane >> 2, t = lane & 3;
    const int row0 = blockIdx.x * p.R;
    const int u0 = blockIdx.y * p.upc;
    const int nun = min(p.units, u0 + p.upc) - u0;  // >= 1 (host guarantees)
    const int k0 = u0 * p.unit_k;
    const int span_k = nun * p.unit_k;
    const int span_bytes = nun * p.unit_bytes;
    const int rows = min(p.R, p.N - row0);
    const int nthr = blockDim.x;

    // ---- 1. weight-side loads into registers (16-byte vectors), issued
    // before the PDL wait: no earlier kernel on the stream writes weights.
    constexpr int kMaxLd = 8;  // 16-byte loads per thread per round
    const int cpr = span_bytes >> 4;  // 16-byte chunks per row (row-major)
    const uint32_t cpr_magic = div_magic((uint32_t)max(cpr, 1));
    const int wchunks = N64 ? ((min(p.K, k0 + span_k) - k0) * 32) >> 4 : rows * cpr;
    const uint8_t *wsrc = N64 ? p.w + ((size_t)blockIdx.x * p.K + k0) * 32
                              : p.w + (size_t)row0 * p.Kb + (size_t)u0 * p.unit_bytes;
    uint4 wv[kMaxLd];
    {
        const int lim = min(wchunks, kMaxLd * nthr);
#pragma unroll
        for (int i = 0; i < kMaxLd; ++i) {
            const int j = tid + i * nthr;
            if (j < lim) {
                const uint8_t *src;
                if constexpr (N64) src = wsrc + 16 * (size_t)j;
                else {
                    const int r = fast_div(j, cpr_magic);
                    src = wsrc + (size_t)r * p.Kb + 16 * (j - r * cpr);
                }
                wv[i] = __ldg(reinterpret_cast<const uint4 *>(src));
            }
        }
    }
    constexpr int kMaxSc = 2;
    uint4 sv[kMaxSc];
    bool svec = false;
    if constexpr (!B32) svec = prefetch_scales<KIND>(p, row0, rows, u0, nun, nthr, sv, smem);  // B32: scales in the blocks
    if constexpr (KIND == KIND_W4A8G) load_zero_points(p, row0, rows, u0, nun, nthr, smem);

    griddep_wait();  // x may be written, and y read, by the previous kernel

    stage_x<KIND>(p, k0, span_k, nthr, smem);
    if constexpr (KIND == KIND_W4A8G) stage_unit_sums(p, k0, nun, nthr, smem);

    // ---- 3. weight tile into shared memory (further rounds for big tiles).
    for (int base = 0; base < wchunks; base += kMaxLd * nthr) {
        const int lim = min(wchunks - base, kMaxLd * nthr);
        if (base > 0) {
#pragma unroll
            for (int i = 0; i < kMaxLd; ++i) {
                const int j = base + tid + i * nthr;
                if (tid + i * nthr < lim) {
                    const uint8_t *src;
                    if constexpr (N64) src = wsrc + 16 * (size_t)j;
                    else {
                        const int r = fast_div(j, cpr_magic);
                        src = wsrc + (size_t)r * p.Kb + 16 * (j - r * cpr);
                    }
                    wv[i] = __ldg(reinterpret_cast<const uint4 *>(src));
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kMaxLd; ++i) {
            const int j = base + tid + i * nthr;
            if (tid + i * nthr < lim) {
                uint8_t *dst;
                if constexpr (N64) dst = smem + p.raw_off + 16 * j;
                else if constexpr (B32) {  // raw block rows, repacked below
                    const int r = fast_div(j, cpr_magic);
                    dst = smem + p.raw_off + r * p.rawstride + 16 * (j - r * cpr);
                } else {
                    const int r = fast_div(j, cpr_magic);
                    dst = smem + p.w_off + r * p.wstride + 16 * (j - r * cpr);
                }
                *reinterpret_cast<uint4 *>(dst) = wv[i];
            }
        }
    }
    store_scales<KIND>(p, rows, nun, nthr, svec, sv, smem);
    __syncthreads();
    if constexpr (B32) {
        // blocks of 18 bytes -> the row-major code tile (16 bytes per block) and
        // the f32 scale of each block; from here on the W4A16 G = 32 path
        float *scf = reinterpret_cast<float *>(smem + p.sc_off);
        const uint32_t nun_magic = div_magic((uint32_t)nun);
        for (int i = tid; i < rows * nun; i += nthr) {
            const int r = fast_div(i, nun_magic), b = i - r * nun;
            const uint16_t *blk = reinterpret_cast<const uint16_t *>(smem + p.raw_off + r * p.rawstride + 18 * b);
            uint32_t wd[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) wd[q] = (uint32_t)blk[1 + 2 * q] | ((uint32_t)blk[2 + 2 * q] << 16);
            *reinterpret_cast<uint4 *>(smem + p.w_off + r * p.wstride + 16 * b) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
            scf[r * p.sstride + b] = __half2float(__ushort_as_half(blk[0]));
        }
        __syncthreads();
    }
    // Let the next kernel on the stream start (and begin its weight fetch)
    // once this CTA's tiles are in shared memory.
    griddep_launch_dependents();

    // ---- 4. tensor-core k-reduction.
    using Acc = typename std::conditional<kIntAcc<KIND>, int, float>::type;
    Acc acc[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mt][i] = 0;

    const int rbase = wr * RB;
    const int cpg = CPG > 0 ? CPG : p.cpg;
    const int R128 = p.R * 128;
    const uint8_t *wrow = smem + p.w_off + (rbase + g) * p.wstride;
    const uint8_t *wrow8 = wrow + 8 * p.wstride;
    const uint8_t *xrow[MT];
    bool xvalid[MT];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const int m = g + 8 * mt;
        xvalid[mt] = m < p.M;
        xrow[mt] = smem + p.x_off + (xvalid[mt] ? m : 0) * p.xstride + 16 * t;
    }
    const float *scf = reinterpret_cast<const float *>(smem + p.sc_off);
    const float *sc0 = scf + (rbase + g) * p.sstride;
    const float *sc1 = scf + (rbase + g + 8) * p.sstride;

    const int *zc0 = reinterpret_cast<const int *>(smem + p.zc_off) + (rbase + g) * p.sstride;
    const int *zc1 = reinterpret_cast<const int *>(smem + p.zc_off) + (rbase + g + 8) * p.sstride;
    const int *xsum = reinterpret_cast<const int *>(smem + p.xs_off);
    const bool f32sum = kIntAcc<KIND> && f32_sum_exact<KIND>((nun + p.WK - 1) / p.WK, p.unit_k);
    // fold one unit's partial into acc (units arrive in increasing order)
    auto fold = [&](const float (&part)[MT][4], int u) {
        if constexpr (KIND == KIND_W4A8G) {
            // exact group sum with the zero point: sum x*(u - 8) + (8 - z) * sum x, then * s_g
            const float s0 = sc0[u];
            const float s1 = (RB == 16) ? sc1[u] : 0.0f;
            const int c0 = zc0[u];
            const int c1 = (RB == 16) ? zc1[u] : 0;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const int ma = 8 * mt + 2 * t;
                const int xa = ma < p.M ? xsum[ma * p.upc + u] : 0;
                const int xb = ma + 1 < p.M ? xsum[(ma + 1) * p.upc + u] : 0;
                acc[mt][0] = fmaf(s0, (float)(__float2int_rn(part[mt][0]) + c0 * xa), acc[mt][0]);
                acc[mt][1] = fmaf(s0, (float)(__float2int_rn(part[mt][1]) + c0 * xb), acc[mt][1]);
                acc[mt][2] = fmaf(s1, (float)(__float2int_rn(part[mt][2]) + c1 * xa), acc[mt][2]);
                acc[mt][3] = fmaf(s1, (float)(__float2int_rn(part[mt][3]) + c1 * xb), acc[mt][3]);
            }
        } else if constexpr (KIND == KIND_W8A16) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[mt][i] += part[mt][i];
        } else if constexpr (KIND == KIND_W4A16) {
            const float s0 = sc0[u];
            const float s1 = (RB == 16) ? sc1[u] : 0.0f;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                acc[mt][0] = fmaf(s0, part[mt][0], acc[mt][0]);
                acc[mt][1] = fmaf(s0, part[mt][1], acc[mt][1]);
                acc[mt][2] = fmaf(s1, part[mt][2], acc[mt][2]);
                acc[mt][3] = fmaf(s1, part[mt][3], acc[mt][3]);
            }
        } else {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) add_exact(acc[mt][i], part[mt][i], f32sum);
        }
    };
    auto run_unit = [&](int u, int ul, float (&part)[MT][4]) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) part[mt][i] = 0.0f;
        const uint8_t *xr[MT];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) xr[mt] = xrow[mt] + 64 * cpg * u;
        unit_mma<KIND, false, RB, MT, CPG>(wrow, wrow8, cpg * ul, g, t, R128, xr, xvalid, cpg, part,
                                           p.M * p.xstride);
    };

    // Units are processed in phases (one phase for the row-major layout); a
    // warp always takes units wk, wk + WK, ... in increasing order, so both
    // layouts accumulate every output in the same order.
    const int upp = N64 ? p.upp : nun;
    const int WK = p.WK;
    for (int ph0 = 0; ph0 < nun; ph0 += upp) {
        const int ph1 = min(nun, ph0 + upp);
        const int wbase = N64 ? ph0 : 0;  // unit index of the tile's first unit
        if constexpr (N64) {
            // transpose this phase's columns into the row-major tile
            const int kq = (ph1 - ph0) * p.unit_k / 8;  // 8-column groups in the phase
            const uint8_t *raw = smem + p.raw_off + (size_t)ph0 * p.unit_k * 32;
            for (int j = tid; j < kq * 8; j += nthr) {
                const int dq = j & 7, k8 = j >> 3;
                uint32_t lo[4], hi[4];
                deinterleave8(raw + k8 * 8 * 32, dq, lo, hi);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    *reinterpret_cast<uint32_t *>(smem + p.w_off + (4 * dq + c) * p.wstride + 4 * k8) = lo[c];
                    *reinterpret_cast<uint32_t *>(smem + p.w_off + (4 * dq + c + 32) * p.wstride + 4 * k8) = hi[c];
                }
            }
            __syncthreads();
        }
        // four units at a time, each with its own partial accumulators so the
        // MMA chains overlap, then the remaining units one by one
        int u = ph0 + wk;
        for (; u + 3 * WK < ph1; u += 4 * WK) {
            float part[4][MT][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) run_unit(u + j * WK, u + j * WK - wbase, part[j]);
#pragma unroll
            for (int j = 0; j < 4; ++j) fold(part[j], u + j * WK);
        }
        for (; u < ph1; u += WK) {
            float part[MT][4];
            run_unit(u, u - wbase, part);
            fold(part, u);
        }
        if constexpr (N64) __syncthreads();  // the next phase overwrites the tile
    }
    if constexpr (kIntAcc<KIND>) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) finish_exact(acc[mt][i], f32sum);
    }

    combine_and_store<KIND, RB, MT>(p, acc, wr, wk, lane, g, t, row0 + rbase, smem);
}

// ---------------------------------------------------------------- direct-load kernel
//
// gemv_kernel's arithmetic on the row-major layout -- the same unit -> warp
// assignment, MMA operand order, fold order and K-split combine -- with each
// thread's A fragments loaded straight from global memory into registers
// (one 32-bit word per row per 32-column chunk, issued before the PDL wait)
// instead of through a shared-memory weight tile.  Only activations and
// W4A16 scales pass through shared memory, so there is no tile to store,
// re-read and synchronise on.  Results are bit-identical to gemv_kernel, and
// so to the interleaved layout and across M.
template <int KIND, int RB, int MT, int CPG, int NW>
__global__ void __launch_bounds__(512) gemv_direct_kernel(const __grid_constant__ GemvParams p) {
    static_assert(KIND != KIND_W8A8 && NW % CPG == 0, "int4 kinds, whole units per window");
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wr = warp % p.WR, wk = warp / p.WR;
    const int g = lane >> 2, t = lane & 3;
    const int row0 = blockIdx.x * p.R;
    const int u0 = blockIdx.y * p.upc;
    const int nun = min(p.units, u0 + p.upc) - u0;  // >= 1 (host guarantees)
    const int k0 = u0 * p.unit_k;
    const int span_k = nun * p.unit_k;
    constexpr bool kInt = KIND != KIND_W4A16;
    const int rows = min(p.R, p.N - row0);
    const int nthr = blockDim.x;
    const int WK = p.WK;
    const int rbase = wr * RB;
    // the warp's units: wk, wk + WK, ... of the CTA's span (gemv_kernel's order)
    const int nu_w = wk < nun ? (nun - wk + WK - 1) / WK : 0;
    const bool f32sum = kInt && f32_sum_exact<KIND>((nun + WK - 1) / WK, p.unit_k);
    constexpr int kUW = NW / CPG;  // units held in registers per window
    // rows g and g + 8 of the warp's block, clamped to a valid row (clamped rows are never stored)
    const int rA = min(row0 + rbase + g, p.N - 1);
    const int rB = min(row0 + rbase + g + 8, p.N - 1);
    const uint8_t *wA = p.w + (size_t)rA * p.Kb + (size_t)u0 * p.unit_bytes + 4 * t;
    const uint8_t *wB = p.w + (size_t)rB * p.Kb + (size_t)u0 * p.unit_bytes + 4 * t;
    uint32_t fa[NW], fb[NW];
    // words of units jw .. jw + kUW - 1 of the warp (chunk cc of unit j at byte 16 * cc)
    auto load_window = [&](int jw) {
#pragma unroll
        for (int j = 0; j < kUW; ++j) {
            if (jw + j < nu_w) {
                const size_t off = (size_t)(wk + (jw + j) * WK) * p.unit_bytes;
#pragma unroll
                for (int cc = 0; cc < CPG; ++cc) {
                    fa[j * CPG + cc] = __ldg(reinterpret_cast<const uint32_t *>(wA + off + 16 * cc));
                    if (RB == 16) fb[j * CPG + cc] = __ldg(reinterpret_cast<const uint32_t *>(wB + off + 16 * cc));
                }
            }
        }
    };
    load_window(0);
    constexpr int kMaxSc = 2;
    uint4 sv[kMaxSc];
    const bool svec = prefetch_scales<KIND>(p, row0, rows, u0, nun, nthr, sv, smem);

    griddep_wait();  // x may be written, and y read, by the previous kernel
    stage_x<KIND>(p, k0, span_k, nthr, smem);
    store_scales<KIND>(p, rows, nun, nthr, svec, sv, smem);
    __syncthreads();
    griddep_launch_dependents();

    using Acc = typename std::conditional<kInt, int, float>::type;
    Acc acc[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mt][i] = 0;
    const uint8_t *xrow[MT];
    bool xvalid[MT];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const int m = g + 8 * mt;
        xvalid[mt] = m < p.M;
        xrow[mt] = smem + p.x_off + (xvalid[mt] ? m : 0) * p.xstride + 16 * t;
    }
    const float *scf = reinterpret_cast<const float *>(smem + p.sc_off);
    const float *sc0 = scf + (rbase + g) * p.sstride;
    const float *sc1 = scf + (rbase + g + 8) * p.sstride;

    for (int jw = 0; jw < nu_w; jw += kUW) {
        if (jw > 0) load_window(jw);
#pragma unroll
        for (int j = 0; j < kUW; ++j) {
            if (jw + j < nu_w) {
                const int u = wk + (jw + j) * WK;  // unit, relative to the CTA's span
                float part[MT][4];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) part[mt][i] = 0.0f;
#pragma unroll
                for (int cc = 0; cc < CPG; ++cc) {
                    uint32_t pa[4], pb[4] = {0u, 0u, 0u, 0u};
                    if constexpr (KIND == KIND_W4A16) {
                        unpack_signed_bf16(fa[j * CPG + cc], pa);
                        if (RB == 16) unpack_signed_bf16(fb[j * CPG + cc], pb);
                    } else {
                        unpack_biased_f16(fa[j * CPG + cc], pa);
                        if (RB == 16) unpack_biased_f16(fb[j * CPG + cc], pb);
                    }
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        uint4 xv = make_uint4(0u, 0u, 0u, 0u);
                        if (xvalid[mt]) xv = *reinterpret_cast<const uint4 *>(xrow[mt] + 64 * (CPG * u + cc));
                        if constexpr (KIND == KIND_W4A16) {
                            mma_bf16(part[mt], pa[0], pb[0], pa[1], pb[1], xv.x, xv.y);
                            mma_bf16(part[mt], pa[2], pb[2], pa[3], pb[3], xv.z, xv.w);
                        } else {
                            mma_f16(part[mt], pa[0], pb[0], pa[1], pb[1], xv.x, xv.y);
                            mma_f16(part[mt], pa[2], pb[2], pa[3], pb[3], xv.z, xv.w);
                        }
                    }
                }
                if constexpr (KIND == KIND_W4A16) {
                    const float s0 = sc0[u];
                    const float s1 = (RB == 16) ? sc1[u] : 0.0f;
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        acc[mt][0] = fmaf(s0, part[mt][0], acc[mt][0]);
                        acc[mt][1] = fmaf(s0, part[mt][1], acc[mt][1]);
                        acc[mt][2] = fmaf(s1, part[mt][2], acc[mt][2]);
                        acc[mt][3] = fmaf(s1, part[mt][3], acc[mt][3]);
                    }
                } else {
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                        for (int i = 0; i < 4; ++i) add_exact(acc[mt][i], part[mt][i], f32sum);
                }
            }
        }
    }
    if constexpr (kInt) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) finish_exact(acc[mt][i], f32sum);
    }
    combine_and_store<KIND, RB, MT>(p, acc, wr, wk, lane, g, t, row0 + rbase, smem);
}

// ---------------------------------------------------------------- fused Q8 quantisation


// W4A8 activations straight from f32 ("Q4 weights x Q8 activations"): at
// M = 1 (the only case the host routes here; more rows run the separate
// quantizer kernel first) every CTA quantises the row itself with
// quantize_row_q8's arithmetic
// (amax over the row, sx = fl(amax / 127), codes clamp(rint(fl(v / sx)))),
// and stages the codes as stage_x<KIND_W4A8> would (biased f16 pairs), the
// row scales in shared memory.  CTA 0 also writes the codes and scales out.
// Codes k0..k7 of an 8-column group (lo: k0..k3, hi: k4..k7) -> the staged
// form of the integer-dot kernel: the even columns (k0 k2 k4 k6) then the odd
// ones (k1 k3 k5 k7), matching the low and high nibbles of a weight word.
W4_DEV uint2 even_odd(uint32_t lo, uint32_t hi) { return make_uint2(prmt(lo, hi, 0x6420u), prmt(lo, hi, 0x7531u)); }

// One 16-byte weight chunk (32 columns: word j holds columns 8j..8j+7, low
// nibbles even, high nibbles odd) against the chunk's even / odd codes.
W4_DEV int dot_chunk_dp(uint4 w, uint4 xe, uint4 xo, int acc) {
    const uint32_t m = 0x0F0F0F0Fu;
    acc = __dp4a((int)(w.x & m), (int)xe.x, acc);
    acc = __dp4a((int)((w.x >> 4) & m), (int)xo.x, acc);
    acc = __dp4a((int)(w.y & m), (int)xe.y, acc);
    acc = __dp4a((int)((w.y >> 4) & m), (int)xo.y, acc);
    acc = __dp4a((int)(w.z & m), (int)xe.z, acc);
    acc = __dp4a((int)((w.z >> 4) & m), (int)xo.z, acc);
    acc = __dp4a((int)(w.w & m), (int)xe.w, acc);
    acc = __dp4a((int)((w.w >> 4) & m), (int)xo.w, acc);
    return acc;
}

// Sum of the 32 codes of a chunk.
W4_DEV int sum_chunk_dp(uint4 xe, uint4 xo, int acc) {
    const int one = 0x01010101;
    acc = __dp4a((int)xe.x, one, acc);
    acc = __dp4a((int)xe.y, one, acc);
    acc = __dp4a((int)xe.z, one, acc);
    acc = __dp4a((int)xe.w, one, acc);
    acc = __dp4a((int)xo.x, one, acc);
    acc = __dp4a((int)xo.y, one, acc);
    acc = __dp4a((int)xo.z, one, acc);
    acc = __dp4a((int)xo.w, one, acc);
    return acc;
}

template <bool DP>
W4_DEV void stage_x_q8(const GemvParams &p, int nthr, uint8_t *smem) {
    // The code here runs once per launch: it is kept short (one division and
    // one reciprocal in the common case, loops where unrolling buys nothing),
    // as instruction fetch, not arithmetic, bounds it.
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = nthr >> 5;
    float *sx_s = reinterpret_cast<float *>(smem + p.xq_off);
    float *red = sx_s + 16;  // [warp][m]
    const int K = p.K;
    const bool write_out = blockIdx.x == 0 && p.xq_out != nullptr;
    const uint32_t xsel4[4] = {0x0400u, 0x0501u, 0x0602u, 0x0703u};
    // M = 1 with K % 8 == 0: every 4-column vector held in registers from
    // the max pass to the code pass; lanes 2i, 2i + 1 hold the two halves of
    // one 8-column group.
    constexpr int kV = 4;
    const int n4 = K >> 2;
    const bool regs = p.M == 1 && p.x_vec && (K & 7) == 0 && n4 <= kV * nthr &&
                      (!write_out || (reinterpret_cast<uintptr_t>(p.xq_out) & 7) == 0);
    float4 v[kV];
    if (regs) {
        float am = 0.0f;
#pragma unroll
        for (int i = 0; i < kV; ++i) {
            const int j = tid + i * nthr;
            v[i] = j < n4 ? __ldg(reinterpret_cast<const float4 *>(p.xf) + j) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            am = fmaxf(am, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        if (lane == 0) red[warp * 8] = am;
    } else {
#pragma unroll 1
        for (int m = 0; m < p.M; ++m) {
            const float *xr = p.xf + (size_t)m * K;
            float am = 0.0f;
#pragma unroll 1
            for (int k = tid; k < K; k += nthr) am = fmaxf(am, fabsf(xr[k]));
#pragma unroll
            for (int o = 16; o; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
            if (lane == 0) red[warp * 8 + m] = am;
        }
    }
    __syncthreads();
    if (tid < p.M) {
        float a = red[tid];
#pragma unroll 1
        for (int w2 = 1; w2 < nw; ++w2) a = fmaxf(a, red[w2 * 8 + tid]);
        const float sx = __fdiv_rn(a, 127.0f);
        sx_s[tid] = sx;
        if (blockIdx.x == 0 && p.sx_out) p.sx_out[tid] = sx;
    }
    __syncthreads();
    if (regs) {
        // Codes clamp(rint(fl(v / sx)), -127, 127) by t = fl(v * r), r = fl(1 / sx)
        // finite: t is within 2^-16 + 2^-24 of x = v / sx when |x| < 256 (two
        // correctly rounded operations, each within 2^-24 relative) and fl(x)
        // within ulp(x) / 2 <= 2^-17 of x, so t and fl(x) lie within 2^-15 of
        // each other; when t is farther than 2^-13 from every half-integer,
        // rint(t) == rint(fl(x)).  The other values (or all, when 1 / sx
        // overflows) are redone with the IEEE quotient.
        const float sx = sx_s[0];
        const float r = sx != 0.0f ? __frcp_rn(sx) : 0.0f;
        const bool fast = isfinite(r);
        uint32_t c4[kV];
        uint32_t redo = 0;
#pragma unroll
        for (int i = 0; i < kV; ++i) {
            c4[i] = 0;
            const float e[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float tq = __fmul_rn(e[q], r);
                const float rt = rintf(tq);
                const bool ok = fast && fabsf(tq) < 256.0f && 0.5f - fabsf(tq - rt) > 0x1p-13f;
                const int c = ok ? min(max(__float2int_rn(rt), -127), 127) : 0;
                c4[i] |= (uint32_t)(uint8_t)(int8_t)c << (8 * q);
                if (!ok && sx != 0.0f) redo |= 1u << (4 * i + q);
            }
        }
#pragma unroll 1
        for (uint32_t rd = redo; rd; rd &= rd - 1) {
            const int b = __ffs(rd) - 1, i = b >> 2, q = b & 3;
            const float4 vi = i == 0 ? v[0] : i == 1 ? v[1] : i == 2 ? v[2] : v[3];
            const float e = q == 0 ? vi.x : q == 1 ? vi.y : q == 2 ? vi.z : vi.w;
            const uint32_t c = (uint32_t)(uint8_t)(int8_t)min(max(__float2int_rn(__fdiv_rn(e, sx)), -127), 127);
            const uint32_t bits = c << (8 * q);
            c4[0] |= i == 0 ? bits : 0u;
            c4[1] |= i == 1 ? bits : 0u;
            c4[2] |= i == 2 ? bits : 0u;
            c4[3] |= i == 3 ? bits : 0u;
        }
#pragma unroll
        for (int i = 0; i < kV; ++i) {
            // exchange the 4 codes with the partner lane (the other half of the 8-column group)
            const int j = tid + i * nthr;
            const uint32_t other = __shfl_xor_sync(0xffffffffu, c4[i], 1);
            if (j < n4 && (j & 1) == 0) {
                if (write_out) *reinterpret_cast<uint2 *>(p.xq_out + 4 * j) = make_uint2(c4[i], other);
                if constexpr (DP) {
                    *reinterpret_cast<uint2 *>(smem + p.x_off + 4 * j) = even_odd(c4[i], other);
                } else {
                    uint32_t b[4];
                    s8_to_f16_pairs(c4[i], other, xsel4, b);
                    *reinterpret_cast<uint4 *>(smem + p.x_off + 8 * j) = make_uint4(b[0], b[1], b[2], b[3]);
                }
            }
        }
    } else {
        // one 8-column group per step; zero codes beyond K
        const int per_row = (p.units * p.unit_k) >> 3;
        const uint32_t pr_magic = div_magic((uint32_t)per_row);
#pragma unroll 1
        for (int j = tid; j < p.M * per_row; j += nthr) {
            const int m = fast_div(j, pr_magic), b8 = j - m * per_row;
            const float *xr = p.xf + (size_t)m * K;
            const float sx = sx_s[m];
            uint32_t lohi[2] = {0u, 0u};
#pragma unroll 1
            for (int i = 0; i < 8; ++i) {
                const int k = 8 * b8 + i;
                int c = 0;
                if (k < K && sx != 0.0f) c = min(max(__float2int_rn(__fdiv_rn(xr[k], sx)), -127), 127);
                if (k < K && write_out) p.xq_out[(size_t)m * K + k] = (int8_t)c;
                const uint32_t bits = (uint32_t)(uint8_t)(int8_t)c << (8 * (i & 3));
                if (i < 4) lohi[0] |= bits;
                else lohi[1] |= bits;
            }
            if constexpr (DP) {
                *reinterpret_cast<uint2 *>(smem + p.x_off + m * p.xstride + 8 * b8) = even_odd(lohi[0], lohi[1]);
            } else {
                uint32_t b[4];
                s8_to_f16_pairs(lohi[0], lohi[1], xsel4, b);
                *reinterpret_cast<uint4 *>(smem + p.x_off + m * p.xstride + 16 * b8) =
                    make_uint4(b[0], b[1], b[2], b[3]);
            }
        }
    }
}

// ---------------------------------------------------------------- streaming kernel
//
// gemv_kernel's arithmetic on the row-major layout for large N and M <= 8,
// with the data movement rebuilt around whole-SM row ranges:
//  * each CTA owns ~N / 152 consecutive rows (a whole number of 8-row
//    blocks) over the full K range;
//  * its entire weight range is requested at once, one bulk async copy per
//    row into a padded shared row, each 8-row block completing on its own
//    mbarrier -- all before the PDL wait, and with the PDL trigger at entry:
//    a CTA takes under half of an SM's shared memory, so the next launch's
//    CTA shares the SM and fetches its whole range while this one computes,
//    and no third launch can start before this one ends;
//  * warps walk their row blocks in order as the blocks land, and the K-split
//    warps are combined once at the end.
// The K split (WK warps, one split per row), the unit -> warp assignment, the
// MMA operand order, the fold and the combine order are gemv_kernel's, so the
// results are bit-identical to it (and so across M and layouts).
template <int KIND, int RB, int CPG, int NRBW, bool XQ, int MT = 1>
__global__ void __launch_bounds__(512, MT == 1 ? 2 : 1) gemv_stream_kernel(const __grid_constant__ GemvParams p) {
    static_assert(KIND == KIND_W4A16 || KIND == KIND_W4A8, "row-major int4 kinds");
    static_assert(!XQ || (KIND == KIND_W4A8 && MT == 1), "fused quantisation is W4A8's, one activation tile (the host uses it at M = 1)");
    griddep_launch_dependents();
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr bool kInt = kIntAcc<KIND>;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wr = warp % p.WR, wk = warp / p.WR;
    const int g = lane >> 2, t = lane & 3;
    const int row0 = blockIdx.x * p.R;
    const int rows = min(p.R, p.N - row0);
    const int nrb = (rows + RB - 1) / RB;
    const int nun = p.units;
    const int nthr = blockDim.x;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.bar_off);

    // ---- 1. the whole weight range in flight (no earlier kernel writes weights).
    if (tid == 0) {
        for (int b = 0; b < nrb; ++b) mbar_init(&bars[b], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {
        if (lane == 0)
            for (int b = 0; b < nrb; ++b) mbar_arrive_expect_tx(&bars[b], (uint32_t)(min(RB, rows - b * RB) * p.Kb));
        __syncwarp();
        for (int r = lane; r < rows; r += 32)
            bulk_g2s(smem + p.w_off + r * p.wstride, p.w + (size_t)(row0 + r) * p.Kb, (uint32_t)p.Kb, &bars[r / RB]);
    }
    uint4 sv[2];
    const bool svec = prefetch_scales<KIND>(p, row0, rows, 0, nun, nthr, sv, smem);

    griddep_wait();  // x may be written, and y read, by the previous kernel
    if constexpr (XQ) stage_x_q8<false>(p, nthr, smem);
    else stage_x<KIND>(p, 0, nun * p.unit_k, nthr, smem);
    store_scales<KIND>(p, rows, nun, nthr, svec, sv, smem);
    __syncthreads();

    // ---- 2. the warp's row blocks, in order, as they land.
    using Acc = typename std::conditional<kInt, int, float>::type;
    Acc acc[NRBW][MT][4];
#pragma unroll
    for (int j = 0; j < NRBW; ++j)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[j][mt][i] = 0;
    bool xvalid[MT];
    const uint8_t *xrow[MT];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const int m = g + 8 * mt;
        xvalid[mt] = m < p.M;
        xrow[mt] = smem + p.x_off + (xvalid[mt] ? m : 0) * p.xstride + 16 * t;
    }
    const float *scf = reinterpret_cast<const float *>(smem + p.sc_off);
    const int WK = p.WK;
    const int cpg = CPG > 0 ? CPG : p.cpg;
    const bool f32sum = kInt && f32_sum_exact<KIND>((nun + WK - 1) / WK, p.unit_k);
    bool ok = true;
#pragma unroll
    for (int j = 0; j < NRBW; ++j) {
        const int rb = wr + j * p.WR;
        if (rb >= nrb) break;
        if (!mbar_wait_bounded(&bars[rb], 0)) {
            ok = false;
            continue;
        }
        const uint8_t *wrow = smem + p.w_off + (rb * RB + g) * p.wstride;
        const uint8_t *wrow8 = wrow + 8 * p.wstride;
        const float *sc0 = scf + (rb * RB + g) * p.sstride;
        const float *sc1 = scf + (rb * RB + g + 8) * p.sstride;
        auto fold = [&](const float (&part)[MT][4], int u) {
            if constexpr (KIND == KIND_W4A16) {
                const float s0 = sc0[u];
                const float s1 = (RB == 16) ? sc1[u] : 0.0f;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    acc[j][mt][0] = fmaf(s0, part[mt][0], acc[j][mt][0]);
                    acc[j][mt][1] = fmaf(s0, part[mt][1], acc[j][mt][1]);
                    acc[j][mt][2] = fmaf(s1, part[mt][2], acc[j][mt][2]);
                    acc[j][mt][3] = fmaf(s1, part[mt][3], acc[j][mt][3]);
                }
            } else {
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) add_exact(acc[j][mt][i], part[mt][i], f32sum);
            }
        };
        auto run_unit = [&](int u, float (&part)[MT][4]) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) part[mt][i] = 0.0f;
            const uint8_t *xr[MT];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) xr[mt] = xrow[mt] + 64 * cpg * u;
            unit_mma<KIND, false, RB, MT, CPG>(wrow, wrow8, cpg * u, g, t, 0, xr, xvalid, cpg, part,
                                                p.M * p.xstride);
        };
        int u = wk;
        if (kInt && f32sum) {
            // every partial sum of the warp is an integer below 2^24: the MMA
            // accumulators run across units (four chains), added once at the end
            float chain[4][MT][4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) chain[q][mt][i] = 0.0f;
            for (; u + 3 * WK < nun; u += 4 * WK) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint8_t *xr[MT];
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) xr[mt] = xrow[mt] + 64 * cpg * (u + q * WK);
                    unit_mma<KIND, false, RB, MT, CPG>(wrow, wrow8, cpg * (u + q * WK), g, t, 0, xr, xvalid, cpg,
                                                        chain[q]);
                }
            }
            for (; u < nun; u += WK) {
                const uint8_t *xr[MT];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) xr[mt] = xrow[mt] + 64 * cpg * u;
                unit_mma<KIND, false, RB, MT, CPG>(wrow, wrow8, cpg * u, g, t, 0, xr, xvalid, cpg, chain[0]);
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    acc[j][mt][i] = __float2int_rn((chain[0][mt][i] + chain[1][mt][i]) +
                                                   (chain[2][mt][i] + chain[3][mt][i]));
            continue;
        }
        for (; u + 3 * WK < nun; u += 4 * WK) {
            float part[4][MT][4];
#pragma unroll
            for (int q = 0; q < 4; ++q) run_unit(u + q * WK, part[q]);
#pragma unroll
            for (int q = 0; q < 4; ++q) fold(part[q], u + q * WK);
        }
        for (; u < nun; u += WK) {
            float part[MT][4];
            run_unit(u, part);
            fold(part, u);
        }
        if constexpr (kInt) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) finish_exact(acc[j][mt][i], f32sum);
        }
    }
    if (!ok) {
        if (lane == 0 && p.status) atomicOr(p.status, kStatusCopyTimeout);
        // give copies still in flight one more bounded wait before the CTA's shared memory goes away
        for (int b = wr; b < nrb; b += p.WR) (void)mbar_wait_bounded(&bars[b], 0);
    }

    // ---- 3. combine the K-split warps in index order, then the epilogue.
    constexpr int kVals = MT * 4;
    uint32_t *red = reinterpret_cast<uint32_t *>(smem + p.red_off);
    if (WK > 1) {
        __syncthreads();  // red may alias the weight tile
        if (wk > 0) {
#pragma unroll
            for (int j = 0; j < NRBW; ++j)
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        red[((((wk - 1) * p.WR + wr) * NRBW + j) * 32 + lane) * kVals + mt * 4 + i] =
                            kInt ? (uint32_t)acc[j][mt][i] : __float_as_uint((float)acc[j][mt][i]);
        }
        __syncthreads();
        if (wk != 0) return;
        for (int w2 = 1; w2 < WK; ++w2)
#pragma unroll
            for (int j = 0; j < NRBW; ++j)
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t v = red[((((w2 - 1) * p.WR + wr) * NRBW + j) * 32 + lane) * kVals + mt * 4 + i];
                        if constexpr (kInt) acc[j][mt][i] += (int)v;
                        else acc[j][mt][i] += __uint_as_float(v);
                    }
    }
#pragma unroll
    for (int j = 0; j < NRBW; ++j) {
        const int rb = wr + j * p.WR;
        if (rb >= nrb) break;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (RB == 8 && i >= 2) continue;
                const int m = 8 * mt + 2 * t + (i & 1);
                const int n = row0 + rb * RB + g + 8 * (i >> 1);
                if (m >= p.M || n >= p.N) continue;
                float out;
                if constexpr (kInt) {
                    const float sw = static_cast<const float *>(p.scale)[n];
                    const float sxm = XQ ? reinterpret_cast<const float *>(smem + p.xq_off)[m] : p.sx[m];
                    out = __fmul_rn(__fmul_rn(__int2float_rn((int)acc[j][mt][i]), sxm), sw);
                } else {
                    out = acc[j][mt][i];
                }
                p.y[(size_t)m * p.N + n] = out;
            }
    }
}

// ---------------------------------------------------------------- W4A8, one activation row
//
// linear_q4 at M = 1 by integer dot products ("Q4 weights x Q8
// activations": acc = sum_k xq * u - 8 * sum_k xq, exact in i32).  The data
// movement is the streaming kernel's (whole-SM row ranges by bulk copies
// before the PDL wait, the trigger at entry, two CTAs per SM); the
// arithmetic is integer, so any order gives the same result.  One warp per
// row: each lane takes 16-byte weight chunks (32 columns) and dp4a's the
// low and high nibbles of each word against the even and odd activation
// codes of that chunk, which it holds in registers for all its rows; the
// warp sums its lanes.  At M = 1 the m16n8 MMA would leave 7 of its 8
// columns idle and the f16 unpack would cost the integer pipe three times
// as much.  XQ: the activations arrive as f32 and every CTA quantises them
// (stage_x_q8); otherwise as Q8 codes.
template <bool XQ, int XR>
__global__ void __launch_bounds__(512, 2) gemv_q4dp_kernel(const __grid_constant__ GemvParams p) {
    griddep_launch_dependents();
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int nthr = blockDim.x;
    const int row0 = blockIdx.x * p.R;
    const int rows = min(p.R, p.N - row0);
    const int RB = p.rb;
    const int nrb = (rows + RB - 1) / RB;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.bar_off);

    if (tid == 0) {
        for (int b = 0; b < nrb; ++b) mbar_init(&bars[b], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {
        if (lane == 0)
            for (int b = 0; b < nrb; ++b) mbar_arrive_expect_tx(&bars[b], (uint32_t)(min(RB, rows - b * RB) * p.Kb));
        __syncwarp();
        for (int r = lane; r < rows; r += 32)
            bulk_g2s(smem + p.w_off + r * p.wstride, p.w + (size_t)(row0 + r) * p.Kb, (uint32_t)p.Kb, &bars[r / RB]);
    }

    griddep_wait();  // x may be written, and y read, by the previous kernel
    if constexpr (XQ) {
        stage_x_q8<true>(p, nthr, smem);
    } else {
        const int8_t *xr = static_cast<const int8_t *>(p.x);
        const int groups = p.Kb >> 2;  // 8-column groups (K padded to Kp)
        for (int b8 = tid; b8 < groups; b8 += nthr) {
            const int kk = 8 * b8;
            uint32_t lo = 0, hi = 0;
            if (p.x_vec && kk + 8 <= p.K) {
                const uint2 v = __ldg(reinterpret_cast<const uint2 *>(xr + kk));
                lo = v.x;
                hi = v.y;
            } else {
#pragma unroll 1
                for (int i = 0; i < 8; ++i) {
                    const uint32_t b = kk + i < p.K ? (uint32_t)(uint8_t)xr[kk + i] : 0u;
                    if (i < 4) lo |= b << (8 * i);
                    else hi |= b << (8 * (i - 4));
                }
            }
            *reinterpret_cast<uint2 *>(smem + p.x_off + 8 * b8) = even_odd(lo, hi);
        }
    }
    __syncthreads();

    // the lane's activation chunks (c = lane + 32 i), and the sum of all codes
    const int chunks = p.Kb >> 4;
    uint4 xe[XR], xo[XR];
    int xs = 0;
#pragma unroll
    for (int i = 0; i < XR; ++i) {
        const int c = lane + 32 * i;
        xe[i] = make_uint4(0u, 0u, 0u, 0u);
        xo[i] = xe[i];
        if (c < chunks) {
            const uint4 a = *reinterpret_cast<const uint4 *>(smem + p.x_off + 32 * c);
            const uint4 b = *reinterpret_cast<const uint4 *>(smem + p.x_off + 32 * c + 16);
            xe[i] = make_uint4(a.x, a.z, b.x, b.z);
            xo[i] = make_uint4(a.y, a.w, b.y, b.w);
        }
        xs = sum_chunk_dp(xe[i], xo[i], xs);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) xs += __shfl_xor_sync(0xffffffffu, xs, o);
    const float sx = XQ ? reinterpret_cast<const float *>(smem + p.xq_off)[0] : p.sx[0];
    const float *sw = static_cast<const float *>(p.scale);

    bool ok = true;
    for (int r = warp; r < rows; r += nw) {
        if (!mbar_wait_bounded(&bars[r / RB], 0)) {
            ok = false;
            continue;
        }
        const uint8_t *wrow = smem + p.w_off + r * p.wstride;
        int acc = 0;
#pragma unroll
        for (int i = 0; i < XR; ++i) {
            const int c = lane + 32 * i;
            if (c < chunks) acc = dot_chunk_dp(*reinterpret_cast<const uint4 *>(wrow + 16 * c), xe[i], xo[i], acc);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) {
            const int n = row0 + r;
            p.y[n] = __fmul_rn(__fmul_rn(__int2float_rn(acc - 8 * xs), sx), sw[n]);
        }
    }
    if (!ok) {
        if (lane == 0 && p.status) atomicOr(p.status, kStatusCopyTimeout);
        for (int b = warp; b < nrb; b += nw) (void)mbar_wait_bounded(&bars[b], 0);
    }
}

// ---------------------------------------------------------------- W4A16, one activation row
//
// linear_w4a16_group at M = 1 (the decode step of "Fused int4 and int8
// dequantize-matmul in C", section 4): the streaming kernel's data movement
// -- each CTA's weight rows and f16 scale rows requested by bulk copies at
// entry, before griddepcontrol.wait, with the PDL trigger at entry -- but
// all 16 warps of the CTA at work once the wait returns, and no staging of
// the activations in shared memory:
//  * the activation row (asked into L2 before the wait) arrives in shared
//    memory by one bulk copy issued right after the wait -- a few line
//    requests per CTA instead of one per thread on the same 4 KB;
//  * warp w takes the units (groups) u = w, w + 16, ...; its lanes 0-3 turn
//    the activations of those units into the MMA's B fragments, in the pair
//    order of the unpacked nibbles;
//  * for every 16-row block the warp forms each unit's partial with the
//    streaming kernel's MMA sequence (the same k-slot order, the chunks of
//    the unit in order, from a zero accumulator), so each partial has the
//    same bits, and stores it to shared memory;
//  * after one barrier, thread (row, w') of the WK K-warps of the other M <= 16
//    paths folds its units u = w', w' + WK, ... in order, acc = fma(s_u,
//    part_u, acc), and the WK sums are added in index order -- bit for bit
//    the result of every other M <= 16 path for the same (N, K, G).
// IL: the weights are in the interleaved [N/64][K][32 B] layout and each CTA
// owns one 64-channel block; before the wait its threads turn the block into
// row-major rows in shared memory (4x4 byte transposes and nibble repacking,
// the decode path's deinterleave), after which everything is as above, so
// both layouts give the same bits.
template <int CPG, int NU, int JJ, bool IL = false>
__global__ void __launch_bounds__(512, 2) gemv_m1_w4a16_kernel(const __grid_constant__ GemvParams p) {
    griddep_launch_dependents();
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int NCH = NU * CPG;  // 32-column chunks per warp: NU units of CPG chunks
    constexpr int WK = 4;          // K-warp chains of the other M <= 16 paths
    constexpr bool kPre = NCH <= 4;  // the first row block unpacked before the wait
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int row0 = blockIdx.x * p.R;
    const int rows = min(p.R, p.N - row0);
    const int nrb = (rows + 15) >> 4;
    constexpr int U = WK * JJ;  // units per row (= NU * warps)
    const int sbytes = 2 * p.ng;
    const int ps = p.sstride;  // floats per row of the partial and scale tiles: U + 4
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.bar_off);
    float *part = reinterpret_cast<float *>(smem + p.red_off);
    float *sf = reinterpret_cast<float *>(smem + p.xq_off);

    // ---- 1. weights and scales in flight, the activations toward L2.
    uint64_t *xbar = &bars[nrb];
    if (tid == 0) {
        for (int b = 0; b <= nrb; ++b) mbar_init(&bars[b], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {
        if (lane == 0) {
            for (int b = 0; b < nrb; ++b)
                mbar_arrive_expect_tx(&bars[b], (uint32_t)(min(16, rows - 16 * b) * ((IL ? 0 : p.Kb) + sbytes)));
            prefetch_l2(p.x, (uint32_t)p.x_pref);
        }
        __syncwarp();
        const uint16_t *s16 = static_cast<const uint16_t *>(p.scale);
        for (int r = lane; r < rows; r += 32) {
            if constexpr (!IL)
                bulk_g2s(smem + p.w_off + r * p.wstride, p.w + (size_t)(row0 + r) * p.Kb, (uint32_t)p.Kb,
                         &bars[r >> 4]);
            bulk_g2s(smem + p.sc_off + r * sbytes, s16 + (size_t)(row0 + r) * p.ng, (uint32_t)sbytes, &bars[r >> 4]);
        }
    }
    if constexpr (IL) {
        // the block [K][32 B] -> row-major rows: task (dq, k8) reads bytes
        // 4dq..4dq+3 of rows 8k8..8k8+7 and writes word k8 of channels
        // 4dq..4dq+3 and 4dq+32..4dq+35 (K % 8 == 0, one block per CTA)
        const uint8_t *raw = p.w + (size_t)blockIdx.x * p.K * 32;
        const int ntask = p.K;  // 8 quads x K / 8 column groups
        for (int task = tid; task < ntask; task += nw * 32) {
            const int dq = task & 7, k8 = task >> 3;
            uint32_t v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[i] = __ldg(reinterpret_cast<const uint32_t *>(raw + (size_t)(8 * k8 + i) * 32 + 4 * dq));
            uint32_t lo[4], hi[4];
            deinterleave8_words(v, lo, hi);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                *reinterpret_cast<uint32_t *>(smem + p.w_off + (4 * dq + c) * p.wstride + 4 * k8) = lo[c];
                *reinterpret_cast<uint32_t *>(smem + p.w_off + (4 * dq + c + 32) * p.wstride + 4 * k8) = hi[c];
            }
        }
    }

    // ---- 2. before the wait: the first row block's A fragments, and the
    // scales as f32 in fold order ([row][chain][j], unit = chain + WK j).
    // One warp polls the copies; the others sleep in the CTA barrier rather
    // than take issue slots from the kernel still computing on this SM, and
    // then check each (completed) phase once for the acquire.
    const uint32_t woff = 16 * warp * CPG + 4 * t;  // the lane's word in the warp's first chunk
    bool ok = true;
    if (warp == 0)
        for (int b = 0; b < nrb; ++b) ok = mbar_wait_bounded(&bars[b], 0) && ok;
    __syncthreads();
    for (int b = 0; b < nrb; ++b) ok = mbar_try_wait(&bars[b], 0) && ok;
    uint32_t pre[kPre ? NCH : 1][8];
    if constexpr (kPre) {
        const uint8_t *w0 = smem + p.w_off + g * p.wstride + woff;
        const uint8_t *w8 = rows > 8 ? w0 + 8 * p.wstride : w0;
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
            const int o = 16 * (nw * (i / CPG) * CPG + i % CPG);
            uint32_t a[4], b[4];
            unpack_signed_bf16(*reinterpret_cast<const uint32_t *>(w0 + o), a);
            unpack_signed_bf16(*reinterpret_cast<const uint32_t *>(w8 + o), b);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                pre[i][e] = a[e];
                pre[i][4 + e] = b[e];
            }
        }
    }
    {
        const uint16_t *sc = reinterpret_cast<const uint16_t *>(smem + p.sc_off);
        // U = WK * JJ units per row; thread -> (row, chain, j) with j fastest
        for (int i = tid; i < rows * U; i += nw * 32) {
            const int r = i / U, cj = i - r * U;  // U is a compile-time WK * JJ
            const int c = cj / JJ, j = cj - c * JJ;
            sf[r * ps + cj] = __half2float(__ushort_as_half(sc[r * p.ng + c + WK * j]));
        }
    }

    griddep_wait();  // x may be written, and y read, by the previous kernel
    if (tid == 0) {
        // the 16-byte-aligned part of the row (x_pref bytes); a ragged tail is read below
        mbar_arrive_expect_tx(xbar, (uint32_t)p.x_pref);
        bulk_g2s(smem + p.x_off, p.x, (uint32_t)p.x_pref, xbar);
    }

    // ---- 3. the warp's activation chunks as B fragments (lanes 0-3; zero elsewhere).
    ok = mbar_wait_bounded(xbar, 0) && ok;
    uint4 xb[NCH];
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        xb[i] = make_uint4(0u, 0u, 0u, 0u);
        if (g == 0) {
            const int u = warp + nw * (i / CPG);
            const int kk = u * p.unit_k + 32 * (i % CPG) + 8 * t;
            uint4 v;
            if (2 * (kk + 8) <= p.x_pref) {
                v = *reinterpret_cast<const uint4 *>(smem + p.x_off + 2 * kk);
            } else {
                const uint16_t *xr = static_cast<const uint16_t *>(p.x) + kk;
                uint32_t e[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) e[j] = (kk + j < p.K) ? (uint32_t)__ldcg(xr + j) : 0u;
                v = make_uint4(e[0] | (e[1] << 16), e[2] | (e[3] << 16), e[4] | (e[5] << 16), e[6] | (e[7] << 16));
            }
            // (x0 x4)(x1 x5)(x2 x6)(x3 x7): the pair order of unpack_signed_bf16
            xb[i] = make_uint4(prmt(v.x, v.z, 0x5410), prmt(v.x, v.z, 0x7632), prmt(v.y, v.w, 0x5410),
                               prmt(v.y, v.w, 0x7632));
        }
    }

    // ---- 4. unit partials of every 16-row block.  In a last block of at
    // most 8 rows the MMA rows g + 8 read row g again; those rows are never
    // stored, and each MMA row depends only on its own A row.
    auto store = [&](int rb, int j, const float (&pt)[4]) {
        if (t == 0) {
            const int u = warp + nw * j;
            const int o = (u % WK) * JJ + u / WK;
            part[(16 * rb + g) * ps + o] = pt[0];
            if (16 * rb + 8 < rows) part[(16 * rb + g + 8) * ps + o] = pt[2];
        }
    };
    if constexpr (kPre) {
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            float pt[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int cc = 0; cc < CPG; ++cc) {
                const uint32_t(&a)[8] = pre[j * CPG + cc];
                mma_bf16(pt, a[0], a[4], a[1], a[5], xb[j * CPG + cc].x, xb[j * CPG + cc].y);
                mma_bf16(pt, a[2], a[6], a[3], a[7], xb[j * CPG + cc].z, xb[j * CPG + cc].w);
            }
            store(0, j, pt);
        }
    }
    for (int rb = kPre ? 1 : 0; rb < nrb; ++rb) {
        const uint8_t *w0 = smem + p.w_off + (16 * rb + g) * p.wstride + woff;
        const uint8_t *w8 = 16 * rb + 8 < rows ? w0 + 8 * p.wstride : w0;
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            float pt[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int cc = 0; cc < CPG; ++cc) {
                const int o = 16 * (nw * j * CPG + cc);  // chunk (warp + nw j) CPG + cc, relative to woff
                uint32_t pa[4], pb[4];
                unpack_signed_bf16(*reinterpret_cast<const uint32_t *>(w0 + o), pa);
                unpack_signed_bf16(*reinterpret_cast<const uint32_t *>(w8 + o), pb);
                mma_bf16(pt, pa[0], pb[0], pa[1], pb[1], xb[j * CPG + cc].x, xb[j * CPG + cc].y);
                mma_bf16(pt, pa[2], pb[2], pa[3], pb[3], xb[j * CPG + cc].z, xb[j * CPG + cc].w);
            }
            store(rb, j, pt);
        }
    }
    if (!__syncthreads_and(ok)) {
        if (tid == 0 && p.status) atomicOr(p.status, kStatusCopyTimeout);
        // copies still in flight get one more bounded wait before the CTA's shared memory goes away
        for (int b = 0; b <= nrb; ++b) (void)mbar_wait_bounded(&bars[b], 0);
        return;
    }

    // ---- 5. fold: thread (row, chain c) takes units c, c + WK, ... in order,
    // acc = fma(s_u, part_u, acc); the WK chains are added in index order.
    for (int i = tid; i < ((rows * WK + 31) & ~31); i += nw * 32) {
        const int r = i >> 2, c = i & 3;
        float acc = 0.0f;
        if (r < rows) {
            const float4 *pr = reinterpret_cast<const float4 *>(part + r * ps + c * JJ);
            const float4 *sr = reinterpret_cast<const float4 *>(sf + r * ps + c * JJ);
            float4 pv[JJ / 4], sv[JJ / 4];
#pragma unroll
            for (int j = 0; j < JJ / 4; ++j) {
                pv[j] = pr[j];
                sv[j] = sr[j];
            }
#pragma unroll
            for (int j = 0; j < JJ / 4; ++j) {
                acc = fmaf(sv[j].x, pv[j].x, acc);
                acc = fmaf(sv[j].y, pv[j].y, acc);
                acc = fmaf(sv[j].z, pv[j].z, acc);
                acc = fmaf(sv[j].w, pv[j].w, acc);
            }
        }
        const float a1 = __shfl_down_sync(0xffffffffu, acc, 1);
        const float a2 = __shfl_down_sync(0xffffffffu, acc, 2);
        const float a3 = __shfl_down_sync(0xffffffffu, acc, 3);
        if (c == 0 && r < rows) p.y[row0 + r] = ((acc + a1) + a2) + a3;
    }
}

// ---------------------------------------------------------------- W4A8, one activation row, all warps
//
// linear_q4 at M = 1 under PDL ("Q4 weights x Q8 activations": acc = sum_k
// xq * u - 8 * sum_k xq, exact in i32; y = (f32(acc) * sx) * sw), laid out
// like gemv_m1_w4a16_kernel: each CTA's weight rows arrive by bulk copies
// before griddepcontrol.wait and each warp's first row is loaded into
// registers there; the activation row (f32 for the fused quantize + linear
// call, else Q8 codes) is asked into L2 before the wait and brought into
// shared memory by one bulk copy after it.  XQ: every CTA quantises the row
// with quantize_row_q8's arithmetic (one 4-column vector per thread: amax
// through one CTA barrier, sx = fl(amax / 127), codes rint(fl(v / sx)) by a
// reciprocal with an exact-division fallback near ties) and CTA 0 writes the
// codes and the scale out.  Then warp w takes rows w, w + 16, ...: each lane
// dp4a's the low and high nibbles of its 16-byte chunks against the even and
// odd codes.  The result is an exact integer, so any order gives the same bits.
// IL: interleaved [N/64][K][32 B] weights, one 64-channel block per CTA,
// turned into row-major rows in shared memory before the wait (as in
// gemv_m1_w4a16_kernel); the nibbles are the same, so the sums are.
template <bool XQ, int CH, bool IL = false>
__global__ void __launch_bounds__(512, 2) gemv_m1_q4_kernel(const __grid_constant__ GemvParams p) {
    griddep_launch_dependents();
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int nthr = nw * 32;
    const int row0 = blockIdx.x * p.R;
    const int rows = min(p.R, p.N - row0);
    const int nrb = (rows + 15) >> 4;
    const int chunks = p.Kb >> 4;  // 16-byte weight chunks (32 columns) per row
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.bar_off);
    uint64_t *xbar = &bars[nrb];
    const uint8_t *xq_s = smem + p.xq_off;  // codes as (even, odd) words per 8 columns

    // ---- 1. weight rows in flight, the activations toward L2.
    if (tid == 0) {
        for (int b = 0; b <= nrb; ++b) mbar_init(&bars[b], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {
        if (lane == 0) {
            if constexpr (!IL)
                for (int b = 0; b < nrb; ++b)
                    mbar_arrive_expect_tx(&bars[b], (uint32_t)(min(16, rows - 16 * b) * p.Kb));
            prefetch_l2(XQ ? static_cast<const void *>(p.xf) : p.x, (uint32_t)p.x_pref);
        }
        __syncwarp();
        if constexpr (!IL)
            for (int r = lane; r < rows; r += 32)
                bulk_g2s(smem + p.w_off + r * p.wstride, p.w + (size_t)(row0 + r) * p.Kb, (uint32_t)p.Kb,
                         &bars[r >> 4]);
    }
    if constexpr (IL) {
        // the block [K][32 B] -> row-major rows (K % 8 == 0, one block per CTA)
        const uint8_t *raw = p.w + (size_t)blockIdx.x * p.K * 32;
        for (int task = tid; task < p.K; task += nthr) {
            const int dq = task & 7, k8 = task >> 3;
            uint32_t v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[i] = __ldg(reinterpret_cast<const uint32_t *>(raw + (size_t)(8 * k8 + i) * 32 + 4 * dq));
            uint32_t lo[4], hi[4];
            deinterleave8_words(v, lo, hi);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                *reinterpret_cast<uint32_t *>(smem + p.w_off + (4 * dq + c) * p.wstride + 4 * k8) = lo[c];
                *reinterpret_cast<uint32_t *>(smem + p.w_off + (4 * dq + c + 32) * p.wstride + 4 * k8) = hi[c];
            }
        }
    }
    // one warp polls the copies, the others sleep in the CTA barrier
    bool ok = true;
    if (!IL && warp == 0)
        for (int b = 0; b < nrb; ++b) ok = mbar_wait_bounded(&bars[b], 0) && ok;
    __syncthreads();
    if (!IL)
        for (int b = 0; b < nrb; ++b) ok = mbar_try_wait(&bars[b], 0) && ok;
    uint4 w1[CH];  // the warp's first row
#pragma unroll
    for (int i = 0; i < CH; ++i) {
        const int c = lane + 32 * i;
        w1[i] = make_uint4(0u, 0u, 0u, 0u);
        if (c < chunks && warp < rows) w1[i] = lds_u128(smem_u32(smem + p.w_off + warp * p.wstride + 16 * c));
    }

    griddep_wait();  // x may be written, and y read, by the previous kernel
    if (tid == 0) {
        mbar_arrive_expect_tx(xbar, (uint32_t)p.x_pref);
        bulk_g2s(smem + p.x_off, XQ ? static_cast<const void *>(p.xf) : p.x, (uint32_t)p.x_pref, xbar);
    }
    ok = mbar_wait_bounded(xbar, 0) && ok;
    const int K = p.K;
    const int ncols = 32 * chunks;  // codes staged, zero beyond K

    // ---- 2. the Q8 codes as (even, odd) words of each 8-column group.
    float sx;
    if constexpr (XQ) {
        float *red = reinterpret_cast<float *>(smem + p.red_off);
        const float *xs = reinterpret_cast<const float *>(smem + p.x_off);
        float4 v[2];
        float am = 0.0f;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int k = 4 * (tid + i * nthr);
            v[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (4 * (k + 4) <= p.x_pref) {
                v[i] = *reinterpret_cast<const float4 *>(xs + k);
            } else if (k < K) {
                v[i].x = p.xf[k];
                if (k + 1 < K) v[i].y = p.xf[k + 1];
                if (k + 2 < K) v[i].z = p.xf[k + 2];
                if (k + 3 < K) v[i].w = p.xf[k + 3];
            }
            am = fmaxf(am, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        if (lane == 0) red[warp] = am;
        __syncthreads();
        am = red[0];
        for (int w2 = 1; w2 < nw; ++w2) am = fmaxf(am, red[w2]);
        sx = __fdiv_rn(am, 127.0f);
        // Codes clamp(rint(fl(v / sx)), -127, 127) by t = fl(v * r), r = fl(1 / sx):
        // t lies within 2^-15 of fl(v / sx) when |v / sx| < 256 (two correctly
        // rounded operations), so rint(t) is rint(fl(v / sx)) unless t is within
        // 2^-13 of a half-integer; those values (and all of them when 1 / sx
        // overflows) take the IEEE quotient.
        const float r = sx != 0.0f ? __frcp_rn(sx) : 0.0f;
        const bool fast = isfinite(r);
        const bool out = blockIdx.x == 0 && p.xq_out != nullptr;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int k = 4 * (tid + i * nthr);
            const float e[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            uint32_t c4 = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float tq = __fmul_rn(e[q], r);
                const float rt = rintf(tq);
                int c = 0;
                if (sx != 0.0f) {
                    if (fast && fabsf(tq) < 256.0f && 0.5f - fabsf(tq - rt) > 0x1p-13f) c = __float2int_rn(rt);
                    else c = __float2int_rn(__fdiv_rn(e[q], sx));
                    c = min(max(c, -127), 127);
                }
                c4 |= (uint32_t)(uint8_t)(int8_t)c << (8 * q);
            }
            // the partner lane holds the other half of the 8-column group
            const uint32_t other = __shfl_xor_sync(0xffffffffu, c4, 1);
            if (k < ncols && (tid & 1) == 0)
                *reinterpret_cast<uint2 *>(const_cast<uint8_t *>(xq_s) + k) = even_odd(c4, other);
            if (out) {
                if (k + 3 < K) {
                    *reinterpret_cast<uint32_t *>(p.xq_out + k) = c4;  // k % 4 == 0 and xq_out 4-byte aligned
                } else {
                    for (int q = 0; q < 4 && k + q < K; ++q) p.xq_out[k + q] = (int8_t)(c4 >> (8 * q));
                }
            }
        }
        if (out && tid == 0 && p.sx_out) p.sx_out[0] = sx;
        __syncthreads();
    } else {
        sx = p.sx[0];
    }

    // ---- 3. the lane's activation chunks (c = lane + 32 i) and their code sum.
    uint4 xe[CH], xo[CH];
    int xsum = 0;
#pragma unroll
    for (int i = 0; i < CH; ++i) {
        const int c = lane + 32 * i;
        xe[i] = make_uint4(0u, 0u, 0u, 0u);
        xo[i] = xe[i];
        if (c < chunks) {
            if constexpr (XQ) {
                const uint4 a = lds_u128(smem_u32(xq_s + 32 * c));
                const uint4 b = lds_u128(smem_u32(xq_s + 32 * c + 16));
                xe[i] = make_uint4(a.x, a.z, b.x, b.z);
                xo[i] = make_uint4(a.y, a.w, b.y, b.w);
            } else {
                // raw Q8 codes; zero beyond K
                uint32_t wv[8];
                const int k0 = 32 * c;
                if (k0 + 32 <= p.x_pref) {
                    const uint4 a = lds_u128(smem_u32(smem + p.x_off + k0));
                    const uint4 b = lds_u128(smem_u32(smem + p.x_off + k0 + 16));
                    wv[0] = a.x; wv[1] = a.y; wv[2] = a.z; wv[3] = a.w;
                    wv[4] = b.x; wv[5] = b.y; wv[6] = b.z; wv[7] = b.w;
                } else {
                    const int8_t *xr = static_cast<const int8_t *>(p.x);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint32_t wd = 0;
                        for (int q = 0; q < 4; ++q) {
                            const int k = k0 + 4 * j + q;
                            const uint32_t b8 = k < p.x_pref ? smem[p.x_off + k] : (k < K ? (uint8_t)xr[k] : 0u);
                            wd |= b8 << (8 * q);
                        }
                        wv[j] = wd;
                    }
                }
                const uint2 g0 = even_odd(wv[0], wv[1]), g1 = even_odd(wv[2], wv[3]);
                const uint2 g2 = even_odd(wv[4], wv[5]), g3 = even_odd(wv[6], wv[7]);
                xe[i] = make_uint4(g0.x, g1.x, g2.x, g3.x);
                xo[i] = make_uint4(g0.y, g1.y, g2.y, g3.y);
            }
        }
        xsum = sum_chunk_dp(xe[i], xo[i], xsum);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) xsum += __shfl_xor_sync(0xffffffffu, xsum, o);

    // ---- 4. rows: exact integer dot products, one warp per row.
    const float *sw = static_cast<const float *>(p.scale);
    for (int r = warp; r < rows; r += nw) {
        int acc = 0;
#pragma unroll
        for (int i = 0; i < CH; ++i) {
            const int c = lane + 32 * i;
            if (c < chunks) {
                const uint4 wv = r == warp ? w1[i] : lds_u128(smem_u32(smem + p.w_off + r * p.wstride + 16 * c));
                acc = dot_chunk_dp(wv, xe[i], xo[i], acc);
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0 && ok) {
            const int n = row0 + r;
            p.y[n] = __fmul_rn(__fmul_rn(__int2float_rn(acc - 8 * xsum), sx), sw[n]);
        }
    }
    if (!ok) {
        if (lane == 0 && p.status) atomicOr(p.status, kStatusCopyTimeout);
        for (int b = IL ? nrb : 0; b <= nrb; ++b) (void)mbar_wait_bounded(&bars[b], 0);
    }
}

// ---------------------------------------------------------------- generic fallback

// One warp per output element; any shape, any layout.  Integer kinds are
// exact; W4A16 sums each group across the warp with a fixed butterfly.
template <int KIND>
__global__ void __launch_bounds__(256) generic_kernel(const __grid_constant__ GemvParams p, int layout) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t total = (int64_t)p.M * p.N;
    const int64_t Kb = (p.K + 1) >> 1;
    for (int64_t o = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); o < total; o += warps) {
        const int64_t m = o / p.N, n = o - (o / p.N) * p.N;
        const int64_t nb32 = (p.K + (p.K & 1) + 31) / 32;  // blocks per row (inline-scale layout)
        auto nibble = [&](int64_t k) -> unsigned {
            if (layout == 0) return (p.w[n * Kb + (k >> 1)] >> ((k & 1) * 4)) & 0xFu;
            if (layout == 2) return (p.w[(n * nb32 + (k >> 5)) * 18 + 2 + ((k & 31) >> 1)] >> ((k & 1) * 4)) & 0xFu;
            const uint8_t b = p.w[((n >> 6) * p.K + k) * 32 + ((n & 63) & 31)];
            return ((n & 63) < 32) ? (b & 0xFu) : (b >> 4);
        };
        if constexpr (KIND == KIND_W8A16) {
            const float *xr = static_cast<const float *>(p.x) + m * p.K;
            float acc = 0.0f;
            for (int64_t k = lane; k < p.K; k += 32) acc = fmaf(xr[k], (float)reinterpret_cast<const int8_t *>(p.w)[n * p.K + k], acc);
#pragma unroll
            for (int sft = 16; sft; sft >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sft);
            if (lane == 0) p.y[m * p.N + n] = __fmul_rn(acc, static_cast<const float *>(p.scale)[n]);
        } else if constexpr (KIND == KIND_W4A8G) {
            const int8_t *xr = static_cast<const int8_t *>(p.x) + m * p.K;
            const uint16_t *s16 = static_cast<const uint16_t *>(p.scale);
            const int64_t G = p.unit_k;
            float out = 0.0f;
            for (int64_t gi = 0; gi < p.ng; ++gi) {
                const int z = p.zeros[n * p.ng + gi];
                int acc = 0;
                const int64_t kend = ((gi + 1) * G < p.K) ? (gi + 1) * G : (int64_t)p.K;
                for (int64_t k = gi * G + lane; k < kend; k += 32) acc += (int)xr[k] * ((int)nibble(k) - z);
#pragma unroll
                for (int sft = 16; sft; sft >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sft);
                out = fmaf(__half2float(__ushort_as_half(s16[n * p.ng + gi])), (float)acc, out);
            }
            if (lane == 0) p.y[m * p.N + n] = __fmul_rn(out, p.sx[m]);
        } else if constexpr (KIND != KIND_W4A16) {
            const int8_t *xr = static_cast<const int8_t *>(p.x) + m * p.K;
            int acc = 0;
            for (int64_t k = lane; k < p.K; k += 32) {
                const int wv = (KIND == KIND_W4A8) ? (int)nibble(k) - 8
                                                   : (int)reinterpret_cast<const int8_t *>(p.w)[n * p.K + k];
                acc += (int)xr[k] * wv;
            }
#pragma unroll
            for (int s = 16; s; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
            if (lane == 0) {
                const float sw = static_cast<const float *>(p.scale)[n];
                p.y[m * p.N + n] = __fmul_rn(__fmul_rn(__int2float_rn(acc), p.sx[m]), sw);
            }
        } else {
            const uint16_t *xr = static_cast<const uint16_t *>(p.x) + m * p.K;
            const uint16_t *s16 = static_cast<const uint16_t *>(p.scale);
            const int64_t G = p.unit_k;
            float out = 0.0f;
            for (int64_t gi = 0; gi < p.ng; ++gi) {
                float part = 0.0f;
                const int64_t kend = ((gi + 1) * G < p.K) ? (gi + 1) * G : (int64_t)p.K;
                for (int64_t k = gi * G + lane; k < kend; k += 32) {
                    const unsigned uu = nibble(k);
                    const int q = (int)uu - (int)((uu & 8u) << 1);
                    part = fmaf(__uint_as_float((uint32_t)xr[k] << 16), (float)q, part);
                }
#pragma unroll
                for (int s = 16; s; s >>= 1) part += __shfl_xor_sync(0xffffffffu, part, s);
                const uint16_t sg = (layout == 2) ? (uint16_t)(p.w[(n * nb32 + gi) * 18] | (p.w[(n * nb32 + gi) * 18 + 1] << 8))
                                                  : s16[n * p.ng + gi];
                out = fmaf(__half2float(__ushort_as_half(sg)), part, out);
            }
            if (lane == 0) p.y[m * p.N + n] = out;
        }
    }
}

// ---------------------------------------------------------------- host side

struct Shape {
    int RB, WR, WK, S, MT;
};

template <int KIND, int LAY, int RB, int MT, int CPG>
cudaError_t launch_one(const GemvParams &p, int S, int threads, int smem, cudaStream_t st, bool pdl) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(gemv_kernel<KIND, LAY, RB, MT, CPG>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ceil_div(p.N, p.R), (unsigned)S, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (S > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = 1;
        attrs[na].val.clusterDim.y = (unsigned)S;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = (unsigned)na;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<KIND, LAY, RB, MT, CPG>, p);
}

constexpr int kDirectWords = 16;  // words per row a thread holds (gemv_direct_kernel NW)

template <int KIND, int RB, int MT, int CPG>
cudaError_t launch_direct(const GemvParams &p, int S, int threads, int smem, cudaStream_t st, bool pdl) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    auto *kern = gemv_direct_kernel<KIND, RB, MT, CPG, kDirectWords>;
    std::call_once(once, [kern] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ceil_div(p.N, p.R), (unsigned)S, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (S > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = 1;
        attrs[na].val.clusterDim.y = (unsigned)S;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = (unsigned)na;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int KIND, int RB, int CPG, int NRBW, bool XQ = false, int MT = 1>
cudaError_t launch_stream(const GemvParams &p, int threads, int smem, cudaStream_t st, bool pdl) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    auto *kern = gemv_stream_kernel<KIND, RB, CPG, NRBW, XQ, MT>;
    std::call_once(once, [kern] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ceil_div(p.N, p.R), 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1u : 0u;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int KIND, int RB, int CPG, bool XQ, int MT>
cudaError_t dispatch_stream_nrbw(const GemvParams &p, int nrbw, int threads, int smem, cudaStream_t st, bool pdl) {
    switch (nrbw) {
        case 1: return launch_stream<KIND, RB, CPG, 1, XQ, MT>(p, threads, smem, st, pdl);
        case 2: return launch_stream<KIND, RB, CPG, 2, XQ, MT>(p, threads, smem, st, pdl);
        case 3: return launch_stream<KIND, RB, CPG, 3, XQ, MT>(p, threads, smem, st, pdl);
        default: return launch_stream<KIND, RB, CPG, 4, XQ, MT>(p, threads, smem, st, pdl);
    }
}

template <int KIND, int CPG, bool XQ = false, int MT = 1>
cudaError_t dispatch_stream(const GemvParams &p, int rb, int nrbw, int threads, int smem, cudaStream_t st, bool pdl) {
    if (rb == 16) return dispatch_stream_nrbw<KIND, 16, CPG, XQ, MT>(p, nrbw, threads, smem, st, pdl);
    return dispatch_stream_nrbw<KIND, 8, CPG, XQ, MT>(p, nrbw, threads, smem, st, pdl);
}

template <bool XQ, int XR>
cudaError_t launch_q4dp(const GemvParams &p, int threads, int smem, cudaStream_t st, bool pdl) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    auto *kern = gemv_q4dp_kernel<XQ, XR>;
    std::call_once(once, [kern] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ceil_div(p.N, p.R), 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1u : 0u;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int CPG, int NU, int JJ, bool IL = false>
cudaError_t launch_m1_w4a16(const GemvParams &p, int threads, int smem, cudaStream_t st, bool pdl) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    auto *kern = gemv_m1_w4a16_kernel<CPG, NU, JJ, IL>;
    std::call_once(once, [kern] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ceil_div(p.N, p.R), 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1u : 0u;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <bool XQ, int CH, bool IL = false>
cudaError_t launch_m1_q4(const GemvParams &p, int threads, int smem, cudaStream_t st, bool pdl) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    auto *kern = gemv_m1_q4_kernel<XQ, CH, IL>;
    std::call_once(once, [kern] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ceil_div(p.N, p.R), 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1u : 0u;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <bool XQ>
cudaError_t dispatch_m1_q4(const GemvParams &p, int threads, int smem, cudaStream_t st, bool pdl, bool il = false) {
    const int chunks = p.Kb >> 4;
    if (il) return launch_m1_q4<XQ, 2, true>(p, threads, smem, st, pdl);  // K = 2048: the planner allows only that
    if (chunks <= 32) return launch_m1_q4<XQ, 1>(p, threads, smem, st, pdl);
    if (chunks <= 64) return launch_m1_q4<XQ, 2>(p, threads, smem, st, pdl);
    return launch_m1_q4<XQ, 4>(p, threads, smem, st, pdl);
}

// Warps of the integer-dot kernel: about one per 4 rows of the CTA, 4 to 16
// (measured: 4 warps for 16 rows and 16 for 88 rows beat the other choice).
int q4dp_threads(int R) { return 32 * std::max(4, std::min(16, R / 4)); }

// W4A8, M = 1, row-major, no K split, K <= 4096: the integer-dot kernel.
template <bool XQ>
cudaError_t dispatch_q4dp(const GemvParams &p, int threads, int smem, cudaStream_t st, bool pdl) {
    const int chunks = p.Kb >> 4;
    if (chunks <= 32) return launch_q4dp<XQ, 1>(p, threads, smem, st, pdl);
    if (chunks <= 64) return launch_q4dp<XQ, 2>(p, threads, smem, st, pdl);
    return launch_q4dp<XQ, 4>(p, threads, smem, st, pdl);
}

template <int KIND, int CPG>
cudaError_t dispatch_direct(const GemvParams &p, const Shape &s, int threads, int smem, cudaStream_t st, bool pdl) {
    if (s.RB == 8) {
        if (s.MT == 1) return launch_direct<KIND, 8, 1, CPG>(p, s.S, threads, smem, st, pdl);
        return launch_direct<KIND, 8, 2, CPG>(p, s.S, threads, smem, st, pdl);
    }
    if (s.MT == 1) return launch_direct<KIND, 16, 1, CPG>(p, s.S, threads, smem, st, pdl);
    return launch_direct<KIND, 16, 2, CPG>(p, s.S, threads, smem, st, pdl);
}

template <int KIND, int LAY, int CPG>
cudaError_t dispatch_rb_mt(const GemvParams &p, const Shape &s, int threads, int smem, cudaStream_t st, bool pdl) {
    if (s.RB == 8) {
        if (s.MT == 1) return launch_one<KIND, LAY, 8, 1, CPG>(p, s.S, threads, smem, st, pdl);
        return launch_one<KIND, LAY, 8, 2, CPG>(p, s.S, threads, smem, st, pdl);
    }
    if (s.MT == 1) return launch_one<KIND, LAY, 16, 1, CPG>(p, s.S, threads, smem, st, pdl);
    return launch_one<KIND, LAY, 16, 2, CPG>(p, s.S, threads, smem, st, pdl);
}

template <int KIND, int LAY>
cudaError_t dispatch_grouped(const GemvParams &p, const Shape &s, int threads, int smem, cudaStream_t st, bool pdl) {
    switch (p.cpg) {
        case 1: return dispatch_rb_mt<KIND, LAY, 1>(p, s, threads, smem, st, pdl);
        case 4: return dispatch_rb_mt<KIND, LAY, 4>(p, s, threads, smem, st, pdl);
        default: return dispatch_rb_mt<KIND, LAY, 0>(p, s, threads, smem, st, pdl);
    }
}

constexpr int kSmemLimit = 227 * 1024;
constexpr int kMinTiles = 128;  // CTAs (of 8 rows) below which K is split across a cluster

// Fills the unit geometry of p for the call; false when the fast path cannot describe it.
bool geometry(const LinearArgs &a, GemvParams &p) {
    const int64_t Kp = a.K + (a.K & 1);
    p.Kb = (int)((a.kind == KIND_W8A8 || a.kind == KIND_W8A16) ? a.K : (a.K + 1) / 2);
    if (a.kind == KIND_W8A8 || a.kind == KIND_W8A16) {
        if (a.K % 32) return false;
        p.cpg = 1; p.unit_k = 32; p.unit_bytes = 32; p.units = (int)(a.K / 32); p.ng = 0;
    } else if (a.kind == KIND_W4A8) {
        if (Kp % 32) return false;
        p.cpg = 1; p.unit_k = 32; p.unit_bytes = 16; p.units = (int)(Kp / 32); p.ng = 0;
    } else if (a.layout == W4_LAYOUT_B32) {  // inline-scale blocks: a unit is one 18-byte block
        if (a.kind != KIND_W4A16 || a.G != 32 || Kp % 256) return false;  // rows of whole 16-byte chunks
        p.cpg = 1; p.unit_k = 32; p.unit_bytes = 18; p.units = (int)(Kp / 32); p.ng = p.units;
        p.Kb = 18 * p.units;
    } else {  // group-wise kinds: a unit is one group
        if (Kp % 32 || a.G % 32) return false;
        p.cpg = (int)(a.G / 32); p.unit_k = (int)a.G; p.unit_bytes = (int)(a.G / 2);
        p.units = (int)(Kp / a.G); p.ng = p.units;
    }
    return true;
}

int pad_to(int bytes, int target) { return bytes + ((target - bytes % 128) + 256) % 128; }

// Shared-memory carve-up for a given shape (p.upc, p.upp set); returns total bytes.
int plan_smem(const LinearArgs &a, const Shape &s, GemvParams &p, bool weight_tile = true) {
    const bool n64 = a.layout == W4_LAYOUT_N64;
    p.R = n64 ? 64 : s.RB * s.WR;
    p.WR = n64 ? 64 / s.RB : s.WR;
    p.WK = s.WK;
    const int span_k = p.upc * p.unit_k;
    const int tile_units = n64 ? p.upp : p.upc;
    const bool w8 = a.kind == KIND_W8A8 || a.kind == KIND_W8A16;
    const bool b32 = a.layout == W4_LAYOUT_B32;
    p.wstride = pad_to(tile_units * (b32 ? 16 : p.unit_bytes), w8 ? 32 : 16);  // b32: codes only
    p.rawstride = (int)round_up((int64_t)p.upc * p.unit_bytes, 16);
    p.xstride = pad_to(span_k * 2, 64);  // staged as 16-bit pairs for every kind
    p.sstride = p.upc | 1;  // f32 scales per row, odd so the 8 rows of a warp hit 8 banks
    int off = 0;
    p.raw_off = off;
    if (n64) off += (int)round_up((int64_t)span_k * 32, 128);
    if (b32) off += (int)round_up((int64_t)p.R * p.rawstride, 128);
    p.w_off = off;
    if (weight_tile) off += (int)round_up((int64_t)p.R * p.wstride, 128);
    p.x_off = off;
    off += (int)round_up((int64_t)a.M * p.xstride * (a.kind == KIND_W8A16 ? 2 : 1), 128);
    p.sc_off = off;
    const bool grouped = a.kind == KIND_W4A16 || a.kind == KIND_W4A8G;
    if (grouped) off += (int)round_up((int64_t)p.R * p.sstride * 4, 128);
    p.zc_off = off;
    p.xs_off = off;
    if (a.kind == KIND_W4A8G) {
        off += (int)round_up((int64_t)p.R * p.sstride * 4, 128);
        p.xs_off = off;
        off += (int)round_up((int64_t)a.M * p.upc * 4, 128);
    }
    p.red_off = off;
    const int warps = p.WR * p.WK;
    off += (int)round_up((int64_t)warps * 32 * ((a.M > 8) ? 8 : 4) * 4, 128);
    return off;
}

constexpr int kStreamSmemPerCta = 112 * 1024;  // two CTAs (and their reserved 1 KB each) per SM
constexpr int kStreamMaxBlocks = 16;            // row blocks per CTA (4 warps along rows x NRBW <= 4)
constexpr int kStreamMinSmem = 80 * 1024;               // dynamic shared memory requested at least

// Plans the streaming kernel for a call; false when it does not apply.
// p must hold the call's geometry, upc = units (no K split) and WK.
// MT = 2 (9 to 16 activation rows): one CTA per SM (the staged rows take
// 2 x 4 KB per 2048 columns), so the cap on shared memory is the SM's.
bool plan_stream(const LinearArgs &a, GemvParams &p, int &rb_out, int &nrbw_out, int &threads, int &smem,
                 int MT = 1) {
    if (a.layout != W4_LAYOUT_ROWMAJOR || a.M > 8 * MT || (a.kind != KIND_W4A16 && a.kind != KIND_W4A8)) return false;
    const int cap = MT == 1 ? kStreamSmemPerCta : 220 * 1024;
    if (p.Kb % 16 != 0 || p.upc != p.units) return false;
    const int span_k = p.units * p.unit_k;
    p.wstride = pad_to(p.Kb, 16);
    p.xstride = pad_to(span_k * 2, 64);
    p.sstride = p.upc | 1;
    const int xbytes = (int)round_up((int64_t)a.M * p.xstride, 128);
    const int per_row = p.wstride + (a.kind == KIND_W4A16 ? 4 * p.sstride : 0);
    const int fixed = 128 + xbytes + 2 * 128 + (a.xf ? 640 : 0);
    // rows per CTA: the fewest waves of 152 CTAs, rows spread evenly, a whole number of RB-row blocks
    auto rows_for = [&](int RB) -> int {
        const int rmax = std::min((cap - fixed) / per_row / RB * RB, kStreamMaxBlocks * RB);
        if (rmax < RB) return 0;
        const int64_t waves = ceil_div(a.N, (int64_t)152 * rmax);
        return (int)std::min<int64_t>(rmax, round_up(ceil_div(a.N, 152 * waves), RB));
    };
    const int R8 = rows_for(8), R16 = rows_for(16);
    if (R8 == 0) return false;
    const int RB = (R16 > 0 && R16 * 100 <= R8 * 103) ? 16 : 8;
    const int R = RB == 16 ? R16 : R8;
    const int nrb = R / RB;
    const int WR = std::min(4, nrb);
    const int nrbw = (int)ceil_div(nrb, WR);
    if (nrbw > 4) return false;
    p.R = R;
    p.WR = WR;
    int off = 0;
    p.bar_off = off;
    off += (int)round_up((int64_t)nrb * 8, 128);
    p.w_off = off;
    off += (int)round_up((int64_t)R * p.wstride, 128);
    p.x_off = off;
    off += xbytes;
    p.sc_off = off;
    if (a.kind == KIND_W4A16) off += (int)round_up((int64_t)R * p.sstride * 4, 128);
    p.xq_off = off;
    if (a.xf) off += 640;  // 16 row scales + 16 warps x 8 row maxima (f32)
    // the K-split combine reuses the weight tile once every warp is done with it
    const int red = (p.WK - 1) * WR * nrbw * 32 * 16 * MT;
    p.red_off = p.w_off;
    if (red > R * p.wstride) {
        p.red_off = off;
        off += red;
    }
    if (off > cap) return false;
    rb_out = RB;
    nrbw_out = nrbw;
    threads = 32 * WR * p.WK;
    smem = std::max(off, kStreamMinSmem);
    return true;
}

// Plans gemv_m1_w4a16_kernel (W4A16, M = 1, row-major, no K split); false
// when it does not apply.  p holds the call's geometry with upc = units and
// the call's WK.  Rows per CTA: a multiple of 8, spread over the fewest
// waves of 152 CTAs, within two CTAs' worth of shared memory per SM.
bool plan_m1_w4a16(const LinearArgs &a, GemvParams &p, int &threads, int &smem) {
    const bool il = a.layout == W4_LAYOUT_N64;
    if (a.kind != KIND_W4A16 || a.M != 1 || p.upc != p.units) return false;
    if (a.layout != W4_LAYOUT_ROWMAJOR && !il) return false;
    // interleaved: one 64-channel block per CTA, transposed from K % 8 == 0 rows
    if (il && (a.K % 8 != 0 || a.N / 64 < 120)) return false;
    if (p.WK != 1 && p.WK != 2 && p.WK != 4) return false;
    if (p.Kb % 16 != 0 || (2 * p.ng) % 16 != 0 || reinterpret_cast<uintptr_t>(a.scale) % 16 != 0) return false;
    if (p.cpg != 1 && p.cpg != 2 && p.cpg != 4) return false;
    // every warp takes the same number of units, 4 or 8 chunks: 8 to 16 warps;
    // the fold reads chains of units/4 in 16-byte vectors
    const int chunks = p.units * p.cpg;
    const int nch = chunks <= 64 ? 4 : 8;
    if (chunks % nch != 0 || chunks / nch > 16 || chunks / nch < 4 || (nch / p.cpg) * (chunks / nch) != p.units)
        return false;
    if (p.WK != 4 || p.units % 16 != 0 || p.units > 64) return false;
    if (reinterpret_cast<uintptr_t>(a.x) % 16 != 0 || a.K < 8) return false;
    const int cap = kStreamSmemPerCta;
    p.wstride = pad_to(p.Kb, 16);
    p.sstride = p.units + 4;  // f32 partials / scales per row: 16-byte rows, the 8 rows a warp stores on distinct banks
    p.x_al = 1;
    p.x_pref = (int)((a.K * 2) & ~(int64_t)15);  // bytes of x in the bulk copy
    auto layout = [&](int R) -> int {
        int off = 0;
        p.bar_off = off;
        off += (int)round_up((int64_t)(ceil_div(R, 16) + 1) * 8, 128);
        p.w_off = off;
        off += (int)round_up((int64_t)R * p.wstride, 128);
        p.sc_off = off;
        off += (int)round_up((int64_t)R * 2 * p.ng, 128);
        p.red_off = off;
        off += (int)round_up((int64_t)R * p.sstride * 4, 128);
        p.xq_off = off;
        off += (int)round_up((int64_t)R * p.sstride * 4, 128);
        p.x_off = off;
        off += (int)round_up(p.x_pref, 128);
        return off;
    };
    int rmax = 256;
    while (rmax >= 8 && layout(rmax) > cap) rmax -= 8;
    if (rmax < 8 || (il && rmax < 64)) return false;
    const int64_t waves = ceil_div(a.N, (int64_t)152 * rmax);
    const int R = il ? 64 : (int)std::min<int64_t>(rmax, round_up(ceil_div(a.N, 152 * waves), 8));
    p.R = R;
    const int off = layout(R);
    threads = 32 * (chunks / nch);
    smem = std::max(off, kStreamMinSmem);
    return true;
}

// Plans gemv_m1_q4_kernel (W4A8, M = 1, row-major, K <= 4096); false when it
// does not apply.  xq: the fused call (f32 activations quantised in the CTAs).
bool plan_m1_q4(const LinearArgs &a, GemvParams &p, bool xq, int &threads, int &smem) {
    const bool il = a.layout == W4_LAYOUT_N64;
    if (a.kind != KIND_W4A8 || a.M != 1 || a.N < 1024) return false;
    if (a.layout != W4_LAYOUT_ROWMAJOR && !il) return false;
    // interleaved: one 64-channel block per CTA, K = 2048 (two chunks per lane), at least 120 blocks
    if (il && (a.K != 2048 || a.N / 64 < 120)) return false;
    if (p.Kb % 16 != 0 || (p.Kb >> 4) > 128) return false;
    const void *x = xq ? static_cast<const void *>(a.xf) : a.x;
    if (reinterpret_cast<uintptr_t>(x) % 16 != 0) return false;
    if (xq && a.xq_out && reinterpret_cast<uintptr_t>(a.xq_out) % 4 != 0) return false;
    const int cap = kStreamSmemPerCta;
    p.wstride = pad_to(p.Kb, 16);
    p.x_pref = (int)((a.K * (xq ? 4 : 1)) & ~(int64_t)15);
    const int ncols = 2 * p.Kb;
    const int R = il ? 64 : (int)ceil_div(a.N, 152);
    int off = 0;
    p.bar_off = off;
    off += (int)round_up((ceil_div(R, 16) + 1) * 8, 128);
    p.w_off = off;
    off += (int)round_up((int64_t)R * p.wstride, 128);
    p.x_off = off;
    off += (int)round_up(std::max(p.x_pref, 16), 128);
    p.xq_off = off;
    if (xq) off += (int)round_up(ncols, 128);
    p.red_off = off;
    off += 128;
    if (off > cap) return false;
    p.R = R;
    threads = 512;
    smem = std::max(off, kStreamMinSmem);
    return true;
}

}  // namespace

bool gemv_supported(const LinearArgs &a) {
    if (a.M > 16 || a.M < 1) return false;
    if (a.N > 0x3FFFFFFF || a.K > 0x7FFFFFF) return false;
    if ((a.kind == KIND_W8A8 || a.kind == KIND_W8A16) && a.layout != W4_LAYOUT_ROWMAJOR) return false;
    if (a.layout == W4_LAYOUT_B32 && a.kind != KIND_W4A16) return false;
    GemvParams p = {};
    if (!geometry(a, p)) return false;
    if ((reinterpret_cast<uintptr_t>(a.w) % 16) != 0) return false;
    return true;
}

cudaError_t launch_gemv(const LinearArgs &a, cudaStream_t st) {
    GemvParams p = {};
    geometry(a, p);
    p.x = a.x;
    p.w = a.w;
    p.scale = a.scale;
    p.sx = a.sx;
    p.zeros = a.zeros;
    p.y = a.y;
    p.status = a.status;
    p.M = (int)a.M;
    p.N = (int)a.N;
    p.K = (int)a.K;
    const int esize = (a.kind == KIND_W4A16) ? 2 : (a.kind == KIND_W8A16) ? 4 : 1;
    const bool n64 = a.layout == W4_LAYOUT_N64;

    // The K split (warps per CTA along K, cluster ranks along K) depends only
    // on (N, K, G): every M and both layouts then sum each output in the same
    // order, so W4A16 results are bit-identical across batch sizes and layouts.
    Shape s;
    s.MT = a.M > 8 ? 2 : 1;
    s.WK = std::max(1, std::min(4, p.units));
    const int64_t tiles8 = ceil_div(a.N, 8);
    int S = tiles8 >= kMinTiles ? 1 : (int)std::min<int64_t>(8, ceil_div(kMinTiles, tiles8));
    S = std::max(1, std::min(S, p.units / s.WK));
    // units per interleave phase: ~512 packed bytes per row, a multiple of WK
    p.upp = std::max(s.WK, (512 / p.unit_bytes) / s.WK * s.WK);
    // A split starts on a 128-byte column boundary: units per split are a
    // multiple of lcm(unit, 128) / unit.
    const int ualign = std::lcm(p.unit_bytes, 128) / p.unit_bytes;
    {
        // size the split for the largest tile any M or layout uses
        LinearArgs worst = a;
        worst.M = 16;
        Shape sw = s;
        sw.RB = 16;
        sw.WR = 4;
        GemvParams q = p;
        for (;;) {
            q.upc = (int)round_up(ceil_div(p.units, S), ualign);
            S = (int)ceil_div(p.units, q.upc);  // no empty splits
            worst.layout = (a.layout == W4_LAYOUT_B32) ? W4_LAYOUT_B32 : W4_LAYOUT_N64;
            const int a1 = plan_smem(worst, sw, q);
            worst.layout = W4_LAYOUT_ROWMAJOR;
            const int a2 = plan_smem(worst, sw, q);
            if (std::max(a1, a2) <= kSmemLimit || S >= 8 || q.upc <= ualign) break;
            ++S;
        }
    }
    p.upc = (int)round_up(ceil_div(p.units, S), ualign);
    S = (int)ceil_div(p.units, p.upc);
    if (n64) {
        s.RB = 16;
        s.WR = 4;
    } else {
        s.RB = (a.N >= 16 * 2 * 152 || a.M > 4) ? 16 : 8;
        s.WR = 1;
        if (a.M >= 4)
            while (s.WR < 4 && a.N / (s.RB * s.WR * 2) >= 2 * 152) s.WR *= 2;
    }
    // Fused W4A8 (f32 activations quantised in every CTA, M = 1): the
    // streaming kernels when they apply, else the row quantizer and then
    // this path.
    if (a.xf) {
        GemvParams q = p;
        q.WK = s.WK;
        int mthreads = 0, msmem = 0;
        if (plan_m1_q4(a, q, true, mthreads, msmem)) {
            q.xf = a.xf;
            q.xq_out = a.xq_out;
            q.sx_out = a.sx_out;
            return dispatch_m1_q4<true>(q, mthreads, msmem, st, (a.flags & W4_FLAG_PDL) != 0, n64);
        }
        q = p;
        q.WK = s.WK;
        int rb = 0, nrbw = 0, sthreads = 0, ssmem = 0;
        // M = 1 only: more rows take the per-element quantiser path, slower
        // inside every CTA than the separate quantizer kernel
        if (a.kind == KIND_W4A8 && a.M == 1 && S == 1 && plan_stream(a, q, rb, nrbw, sthreads, ssmem) &&
            ceil_div(a.N, (int64_t)q.R) >= 120) {
            q.xf = a.xf;
            q.xq_out = a.xq_out;
            q.sx_out = a.sx_out;
            q.x_vec = (a.K % 4 == 0 && reinterpret_cast<uintptr_t>(a.xf) % 16 == 0) ? 1 : 0;
            q.rb = rb;
            const bool qpdl = (a.flags & W4_FLAG_PDL) != 0;
            if (a.M == 1 && (q.Kb >> 4) <= 128) return dispatch_q4dp<true>(q, q4dp_threads(q.R), ssmem, st, qpdl);
            return dispatch_stream<KIND_W4A8, 1, true>(q, rb, nrbw, sthreads, ssmem, st, qpdl);
        }
        const cudaError_t e = launch_quantize_rows(a.xf, a.M, a.K, 127, a.xq_out, a.sx_out, nullptr, st);
        if (e != cudaSuccess) return e;
    }
    const int smem = plan_smem(a, s, p);
    if (smem > kSmemLimit) return launch_generic(a, st);

    p.x_vec = ((a.K * esize) % 16 == 0 && reinterpret_cast<uintptr_t>(a.x) % 16 == 0) ? 1 : 0;
    p.s_vec = ((a.kind == KIND_W4A16 || a.kind == KIND_W4A8G) && p.ng % 8 == 0 && p.upc % 8 == 0 &&
               reinterpret_cast<uintptr_t>(a.scale) % 16 == 0) ? 1 : 0;
    s.S = S;
    const int threads = 32 * p.WR * p.WK;
    const bool pdl = (a.flags & W4_FLAG_PDL) != 0;
    // W4A8, M = 1, PDL: the all-warp integer-dot kernel, else the streaming one.
    if (pdl && a.kind == KIND_W4A8 && a.M == 1) {
        GemvParams q = p;
        int mthreads = 0, msmem = 0;
        if (plan_m1_q4(a, q, false, mthreads, msmem)) return dispatch_m1_q4<false>(q, mthreads, msmem, st, pdl, n64);
    }
    if (pdl && a.kind == KIND_W4A8 && a.M == 1 && a.layout == W4_LAYOUT_ROWMAJOR && S == 1 && (p.Kb >> 4) <= 128) {
        GemvParams q = p;
        int rb = 0, nrbw = 0, sthreads = 0, ssmem = 0;
        if (plan_stream(a, q, rb, nrbw, sthreads, ssmem) && ceil_div(a.N, (int64_t)q.R) >= 120) {
            q.rb = rb;
            return dispatch_q4dp<false>(q, q4dp_threads(q.R), ssmem, st, pdl);
        }
    }
    // Large N, 9 <= M <= 16, no K split, PDL: the streaming kernel with two
    // activation tiles, one CTA per SM (same arithmetic).
    if (pdl && (a.kind == KIND_W4A16 || a.kind == KIND_W4A8) && a.M > 8 && S == 1) {
        GemvParams q = p;
        int rb = 0, nrbw = 0, sthreads = 0, ssmem = 0;
        if (plan_stream(a, q, rb, nrbw, sthreads, ssmem, 2) && ceil_div(a.N, (int64_t)q.R) >= 120) {
            if (a.kind == KIND_W4A8) return dispatch_stream<KIND_W4A8, 1, false, 2>(q, rb, nrbw, sthreads, ssmem, st, pdl);
            switch (p.cpg) {
                case 1: return dispatch_stream<KIND_W4A16, 1, false, 2>(q, rb, nrbw, sthreads, ssmem, st, pdl);
                case 4: return dispatch_stream<KIND_W4A16, 4, false, 2>(q, rb, nrbw, sthreads, ssmem, st, pdl);
                default: return dispatch_stream<KIND_W4A16, 0, false, 2>(q, rb, nrbw, sthreads, ssmem, st, pdl);
            }
        }
    }
    // W4A16, M = 1, no K split, PDL: every warp of the CTA after the wait (same bits).
    if (pdl && a.kind == KIND_W4A16 && a.M == 1 && S == 1 && a.N >= 1024 && a.layout != W4_LAYOUT_B32) {
        GemvParams q = p;
        q.WK = s.WK;
        q.upc = p.units;
        int mthreads = 0, msmem = 0;
        if (plan_m1_w4a16(a, q, mthreads, msmem)) {
            // (chunks per unit, units per warp, units per fold chain)
            const int nu = (p.units * p.cpg > 64 ? 8 : 4) / p.cpg, jj = p.units / 4;
            cudaError_t (*fn)(const GemvParams &, int, int, cudaStream_t, bool) = nullptr;
            if (n64) {
                // interleaved: the gate_up / down shapes of the decode set (G = 128 or 32)
                if (p.cpg == 4 && nu == 1 && jj == 4) fn = launch_m1_w4a16<4, 1, 4, true>;
                if (p.cpg == 1 && nu == 4 && jj == 16) fn = launch_m1_w4a16<1, 4, 16, true>;
            } else {
                if (p.cpg == 1 && nu == 4 && jj == 16) fn = launch_m1_w4a16<1, 4, 16>;
                if (p.cpg == 1 && nu == 4 && jj == 8) fn = launch_m1_w4a16<1, 4, 8>;
                if (p.cpg == 2 && nu == 2 && jj == 8) fn = launch_m1_w4a16<2, 2, 8>;
                if (p.cpg == 2 && nu == 2 && jj == 4) fn = launch_m1_w4a16<2, 2, 4>;
                if (p.cpg == 2 && nu == 4 && jj == 16) fn = launch_m1_w4a16<2, 4, 16>;
                if (p.cpg == 4 && nu == 1 && jj == 4) fn = launch_m1_w4a16<4, 1, 4>;
                if (p.cpg == 4 && nu == 2 && jj == 8) fn = launch_m1_w4a16<4, 2, 8>;
            }
            if (fn) return fn(q, mthreads, msmem, st, pdl);
        }
    }
    // Large N, M <= 8, no K split, PDL: the streaming kernel (same arithmetic).
    // Without PDL its per-row bulk copies have nothing to overlap with, and
    // the staged kernel's register loads reach HBM sooner.
    {
        GemvParams q = p;
        int rb = 0, nrbw = 0, sthreads = 0, ssmem = 0;
        if (pdl && (a.kind == KIND_W4A16 || a.kind == KIND_W4A8) && S == 1 &&
            plan_stream(a, q, rb, nrbw, sthreads, ssmem) && ceil_div(a.N, (int64_t)q.R) >= 120) {
            if (a.kind == KIND_W4A8) return dispatch_stream<KIND_W4A8, 1>(q, rb, nrbw, sthreads, ssmem, st, pdl);
            switch (p.cpg) {
                case 1: return dispatch_stream<KIND_W4A16, 1>(q, rb, nrbw, sthreads, ssmem, st, pdl);
                case 4: return dispatch_stream<KIND_W4A16, 4>(q, rb, nrbw, sthreads, ssmem, st, pdl);
                default: return dispatch_stream<KIND_W4A16, 0>(q, rb, nrbw, sthreads, ssmem, st, pdl);
            }
        }
    }
    // Row-major int4 with two activation tiles (M > 8): fragments straight
    // from global memory, so shared memory holds only x and the scales and
    // more CTAs fit per SM (the same arithmetic, so the same bits).  For
    // M <= 8 the 128-bit staged tile streams HBM better.
    if (a.layout == W4_LAYOUT_ROWMAJOR && a.M > 8 && (a.kind == KIND_W4A16 || a.kind == KIND_W4A8) &&
        (p.cpg == 1 || p.cpg == 2 || p.cpg == 4) &&
        (a.kind == KIND_W4A16 || p.cpg == 1)) {
        GemvParams q = p;
        const int dsmem = plan_smem(a, s, q, false);
        if (a.kind == KIND_W4A8) return dispatch_direct<KIND_W4A8, 1>(q, s, threads, dsmem, st, pdl);
        switch (p.cpg) {
            case 1: return dispatch_direct<KIND_W4A16, 1>(q, s, threads, dsmem, st, pdl);
            case 2: return dispatch_direct<KIND_W4A16, 2>(q, s, threads, dsmem, st, pdl);
            default: return dispatch_direct<KIND_W4A16, 4>(q, s, threads, dsmem, st, pdl);
        }
    }
    switch (a.kind) {
        case KIND_W4A8:
            return n64 ? dispatch_rb_mt<KIND_W4A8, 1, 1>(p, s, threads, smem, st, pdl)
                       : dispatch_rb_mt<KIND_W4A8, 0, 1>(p, s, threads, smem, st, pdl);
        case KIND_W8A8:
            return dispatch_rb_mt<KIND_W8A8, 0, 1>(p, s, threads, smem, st, pdl);
        case KIND_W8A16:
            return dispatch_rb_mt<KIND_W8A16, 0, 1>(p, s, threads, smem, st, pdl);
        case KIND_W4A8G:
            return n64 ? dispatch_grouped<KIND_W4A8G, 1>(p, s, threads, smem, st, pdl)
                       : dispatch_grouped<KIND_W4A8G, 0>(p, s, threads, smem, st, pdl);
        default:
            if (a.layout == W4_LAYOUT_B32) return dispatch_rb_mt<KIND_W4A16, 2, 1>(p, s, threads, smem, st, pdl);
            return n64 ? dispatch_grouped<KIND_W4A16, 1>(p, s, threads, smem, st, pdl)
                       : dispatch_grouped<KIND_W4A16, 0>(p, s, threads, smem, st, pdl);
    }
}

cudaError_t launch_generic(const LinearArgs &a, cudaStream_t st) {
    GemvParams p = {};
    p.x = a.x;
    p.w = a.w;
    p.scale = a.scale;
    p.sx = a.sx;
    p.zeros = a.zeros;
    p.y = a.y;
    p.status = a.status;
    p.M = (int)a.M;
    p.N = (int)a.N;
    p.K = (int)a.K;
    if (a.kind == KIND_W4A16 || a.kind == KIND_W4A8G) {
        const int64_t Kp = a.K + (a.K & 1);
        p.ng = (int)(Kp / a.G);
        p.unit_k = (int)a.G;
    }
    const int64_t total = a.M * a.N;
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(ceil_div(total, 8), 152 * 16));
    switch (a.kind) {
        case KIND_W4A8: generic_kernel<KIND_W4A8><<<(unsigned)blocks, 256, 0, st>>>(p, a.layout); break;
        case KIND_W8A8: generic_kernel<KIND_W8A8><<<(unsigned)blocks, 256, 0, st>>>(p, a.layout); break;
        case KIND_W4A8G: generic_kernel<KIND_W4A8G><<<(unsigned)blocks, 256, 0, st>>>(p, a.layout); break;
        case KIND_W8A16: generic_kernel<KIND_W8A16><<<(unsigned)blocks, 256, 0, st>>>(p, a.layout); break;
        default: generic_kernel<KIND_W4A16><<<(unsigned)blocks, 256, 0, st>>>(p, a.layout); break;
    }
    return cudaGetLastError();
}

}  // namespace w4
