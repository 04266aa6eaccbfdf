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
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "../../include/w4.h"
#include "common.cuh"
#include "internal.h"

namespace w4 {
namespace {

struct GemvParams {
    const void *x;
    const uint8_t *w;
    const void *scale;
    const float *sx;
    float *y;
    uint32_t *status;
    int M, N, K;
    int Kb;          // bytes per packed row (row-major)
    int ng;          // W4A16: scale groups per row
    int cpg;         // 32-column chunks per unit (a unit is one group for W4A16, one chunk otherwise)
    int units;       // units per row
    int upc;         // units per CTA (split-K granularity)
    int R, WR, WK;   // rows per CTA, warps along rows, warps along K
    int unit_k;      // columns per unit
    int unit_bytes;  // packed bytes per unit per row
    int wstride;     // shared row stride of the weight tile (bytes)
    int xstride;     // shared row stride of the activation tile (bytes)
    int raw_off, w_off, x_off, sc_off, red_off, xsum_off, flag_off;
    int x_vec;       // activation rows can be read with aligned vector loads
};

// ---------------------------------------------------------------- MMA wrappers

W4_DEV void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

W4_DEV void mma_s8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Signed nibbles k0..k7 of a word -> four bf16x2 pairs of exact integers:
// P0 = (k0, k4), P1 = (k1, k5), P2 = (k2, k6), P3 = (k3, k7).
// 0x4300 | v is the bf16 128 + v (v < 128); with v = u ^ 8 = q + 8 the value
// is 136 + q, and subtracting 136 is exact.
W4_DEV void unpack_signed_bf16(uint32_t w, uint32_t (&p)[4]) {
    const __nv_bfloat162 off = __halves2bfloat162(__ushort_as_bfloat16((unsigned short)0x4308),
                                                  __ushort_as_bfloat16((unsigned short)0x4308));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t v = ((w >> (4 * i)) & 0x000F000Fu) ^ 0x43084308u;
        __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&v);
        h = __hsub2(h, off);
        p[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
}

// ---------------------------------------------------------------- kernel

template <int KIND, bool N64, int RB, int MT>
__global__ void __launch_bounds__(512) gemv_kernel(const __grid_constant__ GemvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    int *flag = reinterpret_cast<int *>(smem + p.flag_off);
    int *xsum = reinterpret_cast<int *>(smem + p.xsum_off);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wr = warp % p.WR, wk = warp / p.WR;
    const int g = lane >> 2, t = lane & 3;
    const int row0 = blockIdx.x * p.R;
    const int u0 = blockIdx.y * p.upc;
    const int nun = min(p.units, u0 + p.upc) - u0;  // >= 1 (host guarantees)
    const int k0 = u0 * p.unit_k;
    const int span_k = nun * p.unit_k;
    const int span_bytes = nun * p.unit_bytes;
    constexpr bool kInt = KIND != KIND_W4A16;

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        *flag = 1;
    }
    if (tid < 16) xsum[tid] = 0;
    __syncthreads();

    // ---- weight tile: bulk async copies, issued before the PDL wait.
    if (tid == 0) {
        if constexpr (!N64) {
            const int rows = min(p.R, p.N - row0);
            mbar_arrive_expect_tx(bar, (uint32_t)(rows * span_bytes));
            const uint8_t *src = p.w + (size_t)row0 * p.Kb + (size_t)u0 * p.unit_bytes;
            for (int r = 0; r < rows; ++r)
                bulk_g2s(smem + p.w_off + r * p.wstride, src + (size_t)r * p.Kb, (uint32_t)span_bytes, bar);
        } else {
            const int kend = min(p.K, k0 + span_k);
            const uint32_t bytes = (uint32_t)(kend - k0) * 32u;
            mbar_arrive_expect_tx(bar, bytes);
            bulk_g2s(smem + p.raw_off, p.w + ((size_t)blockIdx.x * p.K + k0) * 32, bytes, bar);
        }
    }
    // ---- W4A16 group scales (also weight-side data): f16 -> f32 into shared.
    if constexpr (KIND == KIND_W4A16) {
        float *sc = reinterpret_cast<float *>(smem + p.sc_off);
        const uint16_t *s16 = static_cast<const uint16_t *>(p.scale);
        for (int i = tid; i < p.R * nun; i += blockDim.x) {
            const int r = i / nun, gi = i - r * nun;
            const int n = row0 + r;
            sc[r * nun + gi] = n < p.N ? __half2float(__ushort_as_half(s16[(size_t)n * p.ng + u0 + gi])) : 0.0f;
        }
    }

    griddep_launch_dependents();
    griddep_wait();  // x may be written, and y read, by the previous kernel

    // ---- activations: permuted copy of the CTA's K range, zero beyond K.
    {
        const int blocks8 = span_k >> 3;
        const int jobs = p.M * blocks8;
        for (int j = tid; j < jobs; j += blockDim.x) {
            const int m = j / blocks8, b8 = j - m * blocks8;
            const int kk = k0 + 8 * b8;
            if constexpr (kInt) {
                const int8_t *xr = static_cast<const int8_t *>(p.x) + (size_t)m * p.K;
                uint32_t lo = 0, hi = 0;
                if (p.x_vec && kk + 8 <= p.K) {
                    const uint2 v = *reinterpret_cast<const uint2 *>(xr + kk);
                    lo = v.x;
                    hi = v.y;
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t b = (kk + i < p.K) ? (uint32_t)(uint8_t)xr[kk + i] : 0u;
                        if (i < 4) lo |= b << (8 * i);
                        else hi |= b << (8 * (i - 4));
                    }
                }
                uint8_t *dst = smem + p.x_off + m * p.xstride + 8 * b8;
                if constexpr (KIND == KIND_W4A8) {
                    // [x0 x2 x4 x6 | x1 x3 x5 x7]: bytes of the low/high nibble planes
                    *reinterpret_cast<uint2 *>(dst) = make_uint2(prmt(lo, hi, 0x6420), prmt(lo, hi, 0x7531));
                    int s = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) s += (int)(int8_t)(lo >> (8 * i)) + (int)(int8_t)(hi >> (8 * i));
                    atomicAdd(&xsum[m], s);
                } else {
                    *reinterpret_cast<uint2 *>(dst) = make_uint2(lo, hi);
                }
            } else {
                const uint16_t *xr = static_cast<const uint16_t *>(p.x) + (size_t)m * p.K;
                uint32_t i0 = 0, i1 = 0, i2 = 0, i3 = 0;
                if (p.x_vec && kk + 8 <= p.K) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(xr + kk);
                    i0 = v.x; i1 = v.y; i2 = v.z; i3 = v.w;
                } else {
                    uint32_t e[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) e[i] = (kk + i < p.K) ? (uint32_t)xr[kk + i] : 0u;
                    i0 = e[0] | (e[1] << 16); i1 = e[2] | (e[3] << 16);
                    i2 = e[4] | (e[5] << 16); i3 = e[6] | (e[7] << 16);
                }
                // [x0 x4 | x1 x5 | x2 x6 | x3 x7] as bf16 pairs
                uint4 o;
                o.x = prmt(i0, i2, 0x5410);
                o.y = prmt(i0, i2, 0x7632);
                o.z = prmt(i1, i3, 0x5410);
                o.w = prmt(i1, i3, 0x7632);
                *reinterpret_cast<uint4 *>(smem + p.x_off + m * p.xstride + 16 * b8) = o;
            }
        }
    }

    // ---- wait for the weight tile (bounded).
    if (tid == 0) {
        if (!mbar_wait_bounded(bar, 0)) {
            atomicOr(p.status, kStatusCopyTimeout);
            mbar_wait_bounded(bar, 0);  // give copies still in flight one more bounded chance
            *flag = 0;
        }
    }
    __syncthreads();
    const bool ok = *flag != 0;
    if (ok) mbar_wait_bounded(bar, 0);  // completed: acquire for every thread

    // ---- interleaved layout: transpose [k][32 B] into the row-major tile.
    if constexpr (N64) {
        if (ok) {
            const uint8_t *raw = smem + p.raw_off;
            const int jobs = (span_k >> 3) * 8;
            for (int j = tid; j < jobs; j += blockDim.x) {
                const int dq = j & 7, k8 = j >> 3;
                uint32_t v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = *reinterpret_cast<const uint32_t *>(raw + (8 * k8 + i) * 32 + 4 * dq);
                uint32_t T[2][4];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t a01 = prmt(v[4 * h + 0], v[4 * h + 1], 0x5140);
                    const uint32_t b01 = prmt(v[4 * h + 0], v[4 * h + 1], 0x7362);
                    const uint32_t a23 = prmt(v[4 * h + 2], v[4 * h + 3], 0x5140);
                    const uint32_t b23 = prmt(v[4 * h + 2], v[4 * h + 3], 0x7362);
                    T[h][0] = prmt(a01, a23, 0x5410);  // byte i = column 4h+i of channel 4dq+0
                    T[h][1] = prmt(a01, a23, 0x7632);
                    T[h][2] = prmt(b01, b23, 0x5410);
                    T[h][3] = prmt(b01, b23, 0x7632);
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t la = T[0][c] & 0x0F0F0F0Fu, lb = T[1][c] & 0x0F0F0F0Fu;
                    const uint32_t ha = (T[0][c] >> 4) & 0x0F0F0F0Fu, hb = (T[1][c] >> 4) & 0x0F0F0F0Fu;
                    const uint32_t lo = prmt(la | (la >> 4), lb | (lb >> 4), 0x6420);
                    const uint32_t hi = prmt(ha | (ha >> 4), hb | (hb >> 4), 0x6420);
                    *reinterpret_cast<uint32_t *>(smem + p.w_off + (4 * dq + c) * p.wstride + 4 * k8) = lo;
                    *reinterpret_cast<uint32_t *>(smem + p.w_off + (4 * dq + c + 32) * p.wstride + 4 * k8) = hi;
                }
            }
        }
        __syncthreads();
    }

    // ---- tensor-core k-reduction.
    using Acc = typename std::conditional<kInt, int, float>::type;
    Acc acc[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mt][i] = 0;

    const int rbase = wr * RB;
    if (ok) {
        constexpr int kWordBytes = (KIND == KIND_W8A8) ? 8 : 4;
        const uint8_t *wrow = smem + p.w_off + (rbase + g) * p.wstride + kWordBytes * t;
        const uint8_t *wrow8 = wrow + 8 * p.wstride;
        const uint8_t *xrow[MT];
        bool xvalid[MT];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int m = g + 8 * mt;
            xvalid[mt] = m < p.M;
            xrow[mt] = smem + p.x_off + (xvalid[mt] ? m : 0) * p.xstride + (kInt ? 8 : 16) * t;
        }
        for (int u = wk; u < nun; u += p.WK) {
            if constexpr (KIND == KIND_W4A16) {
                float part[MT][4];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) part[mt][i] = 0.0f;
                for (int c = 0; c < p.cpg; ++c) {
                    const int chunk = u * p.cpg + c;
                    uint32_t pa[4], pb[4] = {0u, 0u, 0u, 0u};
                    unpack_signed_bf16(*reinterpret_cast<const uint32_t *>(wrow + 16 * chunk), pa);
                    if (RB == 16) unpack_signed_bf16(*reinterpret_cast<const uint32_t *>(wrow8 + 16 * chunk), pb);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        uint4 xv = make_uint4(0u, 0u, 0u, 0u);
                        if (xvalid[mt]) xv = *reinterpret_cast<const uint4 *>(xrow[mt] + 64 * chunk);
                        mma_bf16(part[mt], pa[0], pb[0], pa[1], pb[1], xv.x, xv.y);
                        mma_bf16(part[mt], pa[2], pb[2], pa[3], pb[3], xv.z, xv.w);
                    }
                }
                const float *sc = reinterpret_cast<const float *>(smem + p.sc_off);
                const float s0 = sc[(rbase + g) * nun + u];
                const float s1 = (RB == 16) ? sc[(rbase + g + 8) * nun + u] : 0.0f;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    acc[mt][0] = fmaf(s0, part[mt][0], acc[mt][0]);
                    acc[mt][1] = fmaf(s0, part[mt][1], acc[mt][1]);
                    acc[mt][2] = fmaf(s1, part[mt][2], acc[mt][2]);
                    acc[mt][3] = fmaf(s1, part[mt][3], acc[mt][3]);
                }
            } else if constexpr (KIND == KIND_W4A8) {
                const int chunk = u;
                const uint32_t wa = *reinterpret_cast<const uint32_t *>(wrow + 16 * chunk);
                const uint32_t wb = (RB == 16) ? *reinterpret_cast<const uint32_t *>(wrow8 + 16 * chunk) : 0u;
                // biased codes u in [0, 15] are non-negative int8 values
                const uint32_t a0 = wa & 0x0F0F0F0Fu, a2 = (wa >> 4) & 0x0F0F0F0Fu;
                const uint32_t a1 = wb & 0x0F0F0F0Fu, a3 = (wb >> 4) & 0x0F0F0F0Fu;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    uint2 xv = make_uint2(0u, 0u);
                    if (xvalid[mt]) xv = *reinterpret_cast<const uint2 *>(xrow[mt] + 32 * chunk);
                    mma_s8(acc[mt], a0, a1, a2, a3, xv.x, xv.y);
                }
            } else {  // W8A8
                const int chunk = u;
                const uint2 wa = *reinterpret_cast<const uint2 *>(wrow + 32 * chunk);
                uint2 wb = make_uint2(0u, 0u);
                if (RB == 16) wb = *reinterpret_cast<const uint2 *>(wrow8 + 32 * chunk);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    uint2 xv = make_uint2(0u, 0u);
                    if (xvalid[mt]) xv = *reinterpret_cast<const uint2 *>(xrow[mt] + 32 * chunk);
                    mma_s8(acc[mt], wa.x, wb.x, wa.y, wb.y, xv.x, xv.y);
                }
            }
        }
    }

    // ---- combine the K-split warps in index order.
    uint32_t *red = reinterpret_cast<uint32_t *>(smem + p.red_off);
    constexpr int kVals = MT * 4;
    if (p.WK > 1) {
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
            for (int w2 = 1; w2 < p.WK; ++w2)
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
    // W4A8: this CTA's share of the bias correction, -8 * sum of its x columns.
    if constexpr (KIND == KIND_W4A8) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = 8 * mt + 2 * t + (i & 1);
                if (m < p.M) acc[mt][i] -= 8 * xsum[m];
            }
    }

    // ---- combine the cluster's K splits in rank order (distributed shared memory).
    const int S = gridDim.y;
    bool all_ok = ok;
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
                all_ok = all_ok && dsmem_ld_u32(dsmem_map(flag, (uint32_t)r)) != 0;
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
    if (blockIdx.y != 0 || wk != 0 || !all_ok) return;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (RB == 8 && i >= 2) continue;
            const int m = 8 * mt + 2 * t + (i & 1);
            const int n = row0 + rbase + g + 8 * (i >> 1);
            if (m >= p.M || n >= p.N) continue;
            float out;
            if constexpr (kInt) {
                const float sw = static_cast<const float *>(p.scale)[n];
                out = __fmul_rn(__fmul_rn(__int2float_rn((int)acc[mt][i]), p.sx[m]), sw);
            } else {
                out = (float)acc[mt][i];
            }
            p.y[(size_t)m * p.N + n] = out;
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
        auto nibble = [&](int64_t k) -> unsigned {
            if (layout == 0) return (p.w[n * Kb + (k >> 1)] >> ((k & 1) * 4)) & 0xFu;
            const uint8_t b = p.w[((n >> 6) * p.K + k) * 32 + ((n & 63) & 31)];
            return ((n & 63) < 32) ? (b & 0xFu) : (b >> 4);
        };
        if constexpr (KIND != KIND_W4A16) {
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
                out = fmaf(__half2float(__ushort_as_half(s16[n * p.ng + gi])), part, out);
            }
            if (lane == 0) p.y[m * p.N + n] = out;
        }
    }
}

// ---------------------------------------------------------------- host side

struct Shape {
    int RB, WR, WK, S, MT;
};

template <int KIND, bool N64, int RB, int MT>
cudaError_t launch_one(const GemvParams &p, int S, int threads, int smem, cudaStream_t st, bool pdl) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(gemv_kernel<KIND, N64, RB, MT>,
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
    return cudaLaunchKernelEx(&cfg, gemv_kernel<KIND, N64, RB, MT>, p);
}

template <int KIND, bool N64>
cudaError_t dispatch_rb_mt(const GemvParams &p, const Shape &s, int threads, int smem, cudaStream_t st, bool pdl) {
    if (s.RB == 8) {
        if (s.MT == 1) return launch_one<KIND, N64, 8, 1>(p, s.S, threads, smem, st, pdl);
        return launch_one<KIND, N64, 8, 2>(p, s.S, threads, smem, st, pdl);
    }
    if (s.MT == 1) return launch_one<KIND, N64, 16, 1>(p, s.S, threads, smem, st, pdl);
    return launch_one<KIND, N64, 16, 2>(p, s.S, threads, smem, st, pdl);
}

constexpr int kTargetCtas = 2 * 152;
constexpr int kSmemLimit = 227 * 1024;

// Fills the unit geometry of p for the call; false when the fast path cannot describe it.
bool geometry(const LinearArgs &a, GemvParams &p) {
    const int64_t Kp = a.K + (a.K & 1);
    p.Kb = (int)((a.kind == KIND_W8A8) ? a.K : (a.K + 1) / 2);
    if (a.kind == KIND_W8A8) {
        if (a.K % 32) return false;
        p.cpg = 1; p.unit_k = 32; p.unit_bytes = 32; p.units = (int)(a.K / 32); p.ng = 0;
    } else if (a.kind == KIND_W4A8) {
        if (Kp % 32) return false;
        p.cpg = 1; p.unit_k = 32; p.unit_bytes = 16; p.units = (int)(Kp / 32); p.ng = 0;
    } else {
        if (Kp % 32 || a.G % 32) return false;
        p.cpg = (int)(a.G / 32); p.unit_k = (int)a.G; p.unit_bytes = (int)(a.G / 2);
        p.units = (int)(Kp / a.G); p.ng = p.units;
    }
    return true;
}

// Shared-memory carve-up for a given shape; returns total bytes.
int plan_smem(const LinearArgs &a, const Shape &s, GemvParams &p) {
    const bool n64 = a.layout == W4_LAYOUT_N64;
    p.R = n64 ? 64 : s.RB * s.WR;
    p.WR = n64 ? 64 / s.RB : s.WR;
    p.WK = s.WK;
    const int span_k = p.upc * p.unit_k;
    const int span_bytes = p.upc * p.unit_bytes;
    const int wtarget = (a.kind == KIND_W8A8) ? 32 : 16;
    p.wstride = span_bytes + ((wtarget - span_bytes % 128) + 256) % 128;
    const int esize = (a.kind == KIND_W4A16) ? 2 : 1;
    const int xtarget = (a.kind == KIND_W4A16) ? 64 : 32;
    const int xbytes = span_k * esize;
    p.xstride = xbytes + ((xtarget - xbytes % 128) + 256) % 128;
    int off = 128;  // mbarrier + flag live in the first 128 bytes
    p.flag_off = 16;
    p.xsum_off = 64;
    p.raw_off = off;
    if (n64) off += (int)round_up((int64_t)span_k * 32, 128);
    p.w_off = off;
    off += (int)round_up((int64_t)p.R * p.wstride, 128);
    p.x_off = off;
    off += (int)round_up((int64_t)a.M * p.xstride, 128);
    p.sc_off = off;
    if (a.kind == KIND_W4A16) off += (int)round_up((int64_t)p.R * p.upc * 4, 128);
    p.red_off = off;
    const int warps = p.WR * p.WK;
    off += (int)round_up((int64_t)warps * 32 * ((a.M > 8) ? 8 : 4) * 4, 128);
    return off;
}

}  // namespace

bool gemv_supported(const LinearArgs &a) {
    if (a.M > 16 || a.M < 1) return false;
    if (a.N > 0x7FFFFFFF / 2 || a.K > 0x7FFFFFF) return false;
    if (a.kind == KIND_W8A8 && a.layout != W4_LAYOUT_ROWMAJOR) return false;
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
    p.y = a.y;
    p.status = a.status;
    p.M = (int)a.M;
    p.N = (int)a.N;
    p.K = (int)a.K;
    const int esize = (a.kind == KIND_W4A16) ? 2 : 1;
    p.x_vec = ((a.K * esize) % 16 == 0 && reinterpret_cast<uintptr_t>(a.x) % 16 == 0) ? 1 : 0;
    const bool n64 = a.layout == W4_LAYOUT_N64;

    // The K split (warps per CTA along K, cluster ranks along K) depends only
    // on (N, K, G): every M and both layouts then sum each output in the same
    // order, so W4A16 results are bit-identical across batch sizes and layouts.
    Shape s;
    s.MT = a.M > 8 ? 2 : 1;
    s.WK = std::max(1, std::min(4, p.units));
    int S = (int)std::min<int64_t>(8, ceil_div(kTargetCtas, ceil_div(a.N, 8)));
    S = std::max(1, std::min(S, p.units / s.WK));
    {
        LinearArgs worst = a;  // size the split for the largest tile any M or layout uses
        worst.M = 16;
        worst.layout = W4_LAYOUT_N64;
        Shape sw = s;
        sw.RB = 16;
        sw.WR = 4;
        GemvParams q = p;
        for (;;) {
            q.upc = (int)ceil_div(p.units, S);
            S = (int)ceil_div(p.units, q.upc);  // no empty splits
            if (plan_smem(worst, sw, q) <= kSmemLimit || S >= 8 || S >= p.units) break;
            ++S;
        }
    }
    p.upc = (int)ceil_div(p.units, S);
    if (n64) {
        s.RB = 16;
        s.WR = 4;
    } else {
        s.RB = (a.N >= 16 * kTargetCtas || a.M > 4) ? 16 : 8;
        s.WR = 1;
        if (a.M >= 4)
            while (s.WR < 4 && a.N / (s.RB * s.WR * 2) >= kTargetCtas) s.WR *= 2;
    }
    const int smem = plan_smem(a, s, p);
    if (smem > kSmemLimit) return launch_generic(a, st);
    s.S = S;
    const int threads = 32 * p.WR * p.WK;
    const bool pdl = (a.flags & W4_FLAG_PDL) != 0;
    switch (a.kind) {
        case KIND_W4A8:
            return n64 ? dispatch_rb_mt<KIND_W4A8, true>(p, s, threads, smem, st, pdl)
                       : dispatch_rb_mt<KIND_W4A8, false>(p, s, threads, smem, st, pdl);
        case KIND_W8A8:
            return dispatch_rb_mt<KIND_W8A8, false>(p, s, threads, smem, st, pdl);
        default:
            return n64 ? dispatch_rb_mt<KIND_W4A16, true>(p, s, threads, smem, st, pdl)
                       : dispatch_rb_mt<KIND_W4A16, false>(p, s, threads, smem, st, pdl);
    }
}

cudaError_t launch_generic(const LinearArgs &a, cudaStream_t st) {
    GemvParams p = {};
    p.x = a.x;
    p.w = a.w;
    p.scale = a.scale;
    p.sx = a.sx;
    p.y = a.y;
    p.status = a.status;
    p.M = (int)a.M;
    p.N = (int)a.N;
    p.K = (int)a.K;
    if (a.kind == KIND_W4A16) {
        const int64_t Kp = a.K + (a.K & 1);
        p.ng = (int)(Kp / a.G);
        p.unit_k = (int)a.G;
    }
    const int64_t total = a.M * a.N;
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(ceil_div(total, 8), 152 * 16));
    switch (a.kind) {
        case KIND_W4A8: generic_kernel<KIND_W4A8><<<(unsigned)blocks, 256, 0, st>>>(p, a.layout); break;
        case KIND_W8A8: generic_kernel<KIND_W8A8><<<(unsigned)blocks, 256, 0, st>>>(p, a.layout); break;
        default: generic_kernel<KIND_W4A16><<<(unsigned)blocks, 256, 0, st>>>(p, a.layout); break;
    }
    return cudaGetLastError();
}

}  // namespace w4
