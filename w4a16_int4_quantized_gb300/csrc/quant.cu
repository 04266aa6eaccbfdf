// quant.cu -- quantizers, the single-row biased-Q4 dot, and the interleave packer.
//
// quantize_row_q8 / quantize_matrix_q8 / quantize_matrix_q4 follow the
// canonical symmetric recipe of docs.rs ftts_kernels::int8 (module summary,
// quantize_row_q8) and its Q4 counterpart in ftts_kernels::int4 ("The
// quantization contract", "Packing"): s = max|row| / Q by one IEEE f32
// division, codes = clamp(rint(v / s), -Q, Q) with ties to even.  The
// kernels use __fdiv_rn and __float2int_rn (IEEE round-to-nearest-even) and
// max via fmaxf, which is exact and order-free, so their codes and scales
// are bit-identical to the CPU definition.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

#include <algorithm>

namespace w4 {
namespace {

constexpr int kThreads = 256;

W4_DEV float block_max(float v, float *red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.0f;
#pragma unroll
        for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0) red[0] = v;
    }
    __syncthreads();
    const float r = red[0];
    __syncthreads();
    return r;
}

W4_DEV int block_sum_i32(int v, int *red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0;
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[0] = v;
    }
    __syncthreads();
    const int r = red[0];
    __syncthreads();
    return r;
}

// One code of the symmetric recipe (s > 0).
W4_DEV int quant_code(float v, float s, int Q) {
    int q = __float2int_rn(__fdiv_rn(v, s));
    return min(max(q, -Q), Q);
}

// One CTA per row: max|v|, the scale, the codes, and (optionally) their sum.
// Launched with programmatic stream serialization: it touches memory only
// after griddepcontrol.wait (the previous kernel may write x or read q), and
// lets the next kernel start at once, so a linear after it fetches its
// weights while the rows are quantised.
__global__ void __launch_bounds__(kThreads) quantize_rows_kernel(const float *__restrict__ x, int64_t K, int Q,
                                                                 int8_t *__restrict__ q, float *__restrict__ s,
                                                                 int32_t *__restrict__ rowsum) {
    __shared__ float redf[32];
    __shared__ int redi[32];
    griddep_launch_dependents();
    griddep_wait();
    const int64_t row = blockIdx.x;
    const float *xr = x + row * K;
    float amax = 0.0f;
    for (int64_t k = threadIdx.x; k < K; k += blockDim.x) amax = fmaxf(amax, fabsf(xr[k]));
    amax = block_max(amax, redf);
    const float sc = __fdiv_rn(amax, (float)Q);
    if (threadIdx.x == 0) s[row] = sc;
    int8_t *qr = q + row * K;
    int sum = 0;
    if (sc == 0.0f) {
        for (int64_t k = threadIdx.x; k < K; k += blockDim.x) qr[k] = 0;
    } else {
        for (int64_t k = threadIdx.x; k < K; k += blockDim.x) {
            const int c = quant_code(xr[k], sc, Q);
            qr[k] = (int8_t)c;
            sum += c;
        }
    }
    if (rowsum) {
        sum = block_sum_i32(sum, redi);
        if (threadIdx.x == 0) rowsum[row] = sum;
    }
}

// quantize_row_q8 for the prefill path, one warp per row, and the exact f16
// image of the codes that the tensor-core GEMM reads (its activation
// operand), in the same pass.  K % 8 == 0.  Rows of up to 2048 columns stay
// in registers (16 four-column vectors per lane); longer rows are read a
// second time for the codes.  Codes are clamp(rint(fl(v / sx)), -127, 127)
// with sx = fl(amax / 127): t = fl(v * fl(1 / sx)) lies within 2^-15 of
// fl(v / sx) when |v / sx| < 256, so rint(t) decides unless t is within
// 2^-13 of a half-integer, where the IEEE quotient is taken (and for every
// value when 1 / sx overflows).
constexpr int kQF16Warps = 8;
constexpr int kQF16Vec = 16;  // float4 per lane held in registers

W4_DEV int code_of(float v, float sx, float r, bool fast) {
    if (sx == 0.0f) return 0;
    const float t = __fmul_rn(v, r);
    const float rt = rintf(t);
    const int c = (fast && fabsf(t) < 256.0f && 0.5f - fabsf(t - rt) > 0x1p-13f) ? __float2int_rn(rt)
                                                                                  : __float2int_rn(__fdiv_rn(v, sx));
    return min(max(c, -127), 127);
}

W4_DEV void store_codes(int8_t *qr, uint16_t *hr, int k, const float4 &v, float sx, float r, bool fast) {
    const int c0 = code_of(v.x, sx, r, fast), c1 = code_of(v.y, sx, r, fast);
    const int c2 = code_of(v.z, sx, r, fast), c3 = code_of(v.w, sx, r, fast);
    *reinterpret_cast<uint32_t *>(qr + k) = (uint32_t)(uint8_t)c0 | ((uint32_t)(uint8_t)c1 << 8) |
                                            ((uint32_t)(uint8_t)c2 << 16) | ((uint32_t)(uint8_t)c3 << 24);
    const uint32_t h0 = __half_as_ushort(__int2half_rn(c0)), h1 = __half_as_ushort(__int2half_rn(c1));
    const uint32_t h2 = __half_as_ushort(__int2half_rn(c2)), h3 = __half_as_ushort(__int2half_rn(c3));
    *reinterpret_cast<uint2 *>(hr + k) = make_uint2(h0 | (h1 << 16), h2 | (h3 << 16));
}

__global__ void __launch_bounds__(32 * kQF16Warps) quantize_rows_f16_kernel(const float *__restrict__ x, int64_t M,
                                                                            int64_t K, int8_t *__restrict__ q,
                                                                            float *__restrict__ s,
                                                                            uint16_t *__restrict__ xh) {
    griddep_launch_dependents();
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kQF16Warps + (threadIdx.x >> 5);
    if (row >= M) return;
    const float4 *xr = reinterpret_cast<const float4 *>(x + row * K);
    const int n4 = (int)(K >> 2);
    const bool regs = n4 <= 32 * kQF16Vec;
    float4 v[kQF16Vec];
    float amax = 0.0f;
    if (regs) {
#pragma unroll
        for (int i = 0; i < kQF16Vec; ++i) {
            const int j = lane + 32 * i;
            v[i] = j < n4 ? __ldg(xr + j) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
        }
    } else {
        for (int j = lane; j < n4; j += 32) {
            const float4 a = __ldg(xr + j);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))));
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sx = __fdiv_rn(amax, 127.0f);
    if (lane == 0) s[row] = sx;
    const float r = sx != 0.0f ? __frcp_rn(sx) : 0.0f;
    const bool fast = isfinite(r);
    int8_t *qr = q + row * K;
    uint16_t *hr = xh + row * K;
    if (regs) {
#pragma unroll
        for (int i = 0; i < kQF16Vec; ++i) {
            const int j = lane + 32 * i;
            if (j < n4) store_codes(qr, hr, 4 * j, v[i], sx, r, fast);
        }
    } else {
        for (int j = lane; j < n4; j += 32) store_codes(qr, hr, 4 * j, __ldg(xr + j), sx, r, fast);
    }
}

// One CTA per output channel: Q4 codes stored u = q + 8, two per byte, low
// nibble = even column; odd K pads the last high nibble with 8.
__global__ void __launch_bounds__(kThreads) quantize_q4_kernel(const float *__restrict__ W, int64_t K,
                                                               uint8_t *__restrict__ packed, float *__restrict__ sw) {
    __shared__ float redf[32];
    const int64_t row = blockIdx.x;
    const float *wr = W + row * K;
    const int64_t Kb = (K + 1) >> 1;
    float amax = 0.0f;
    for (int64_t k = threadIdx.x; k < K; k += blockDim.x) amax = fmaxf(amax, fabsf(wr[k]));
    amax = block_max(amax, redf);
    const float sc = __fdiv_rn(amax, 7.0f);
    if (threadIdx.x == 0) sw[row] = sc;
    uint8_t *pr = packed + row * Kb;
    for (int64_t b = threadIdx.x; b < Kb; b += blockDim.x) {
        const int64_t k = 2 * b;
        int lo = 8, hi = 8;
        if (sc != 0.0f) {
            lo = quant_code(wr[k], sc, 7) + 8;
            if (k + 1 < K) hi = quant_code(wr[k + 1], sc, 7) + 8;
        }
        pr[b] = (uint8_t)(lo | (hi << 4));
    }
}

// dot_i32_q4: sum xq*u - 8 * sum xq over one row, exact in i32.
__global__ void __launch_bounds__(kThreads) dot_q4_kernel(const int8_t *__restrict__ xq,
                                                          const uint8_t *__restrict__ w, int64_t K,
                                                          int32_t *__restrict__ out) {
    __shared__ int redi[32];
    int sxu = 0, sx = 0;
    for (int64_t k = threadIdx.x; k < K; k += blockDim.x) {
        const int x = xq[k];
        const int u = (w[k >> 1] >> ((k & 1) * 4)) & 0xF;
        sxu += x * u;
        sx += x;
    }
    sxu = block_sum_i32(sxu, redi);
    sx = block_sum_i32(sx, redi);
    if (threadIdx.x == 0) *out = sxu - 8 * sx;
}

// [N/64][K][32]: byte d of (block b, column k) = nib(64b+d, k) | nib(64b+d+32, k) << 4.
__global__ void pack_n64_kernel(const uint8_t *__restrict__ w, uint8_t *__restrict__ il, int64_t N, int64_t K) {
    const int64_t total = (N / 64) * K * 32;
    const int64_t Kb = (K + 1) >> 1;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i / (K * 32);
        const int64_t rem = i - b * K * 32;
        const int64_t k = rem >> 5;
        const int d = (int)(rem & 31);
        const int64_t n0 = 64 * b + d;
        const int sh = (int)(k & 1) * 4;
        const unsigned lo = (w[n0 * Kb + (k >> 1)] >> sh) & 0xFu;
        const unsigned hi = (w[(n0 + 32) * Kb + (k >> 1)] >> sh) & 0xFu;
        il[i] = (uint8_t)(lo | (hi << 4));
    }
}

}  // namespace

cudaError_t launch_quantize_rows(const float *x, int64_t rows, int64_t K, int Q, int8_t *q, float *s,
                                 int32_t *rowsum, cudaStream_t st) {
    if (rows > 0x7FFFFFFF) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_rows_kernel, x, K, Q, q, s, rowsum);
}

cudaError_t launch_quantize_rows_f16(const float *x, int64_t M, int64_t K, int8_t *q, float *s, uint16_t *xh,
                                     cudaStream_t st) {
    if (K % 8 != 0 || M > 0x3FFFFFFF) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ceil_div(M, kQF16Warps), 1, 1);
    cfg.blockDim = dim3(32 * kQF16Warps, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_rows_f16_kernel, x, M, K, q, s, xh);
}

cudaError_t launch_quantize_matrix_q4(const float *W, int64_t N, int64_t K, uint8_t *packed, float *sw,
                                      cudaStream_t st) {
    if (N > 0x7FFFFFFF) return cudaErrorInvalidValue;
    quantize_q4_kernel<<<(unsigned)N, kThreads, 0, st>>>(W, K, packed, sw);
    return cudaGetLastError();
}

cudaError_t launch_dot_i32_q4(const int8_t *xq, const uint8_t *wrow, int64_t K, int32_t *out, cudaStream_t st) {
    dot_q4_kernel<<<1, kThreads, 0, st>>>(xq, wrow, K, out);
    return cudaGetLastError();
}

cudaError_t launch_pack_n64(const uint8_t *w, uint8_t *il, int64_t N, int64_t K, cudaStream_t st) {
    const int64_t total = (N / 64) * K * 32;
    const int64_t blocks = std::min<int64_t>(ceil_div(total, 256), 152 * 32);
    pack_n64_kernel<<<(unsigned)blocks, 256, 0, st>>>(w, il, N, K);
    return cudaGetLastError();
}

// pack_block32: one thread per 18-byte block: the f16 scale, then the
// block's 16 code bytes (W4A16 planes -> inline-scale blocks of 32).
__global__ void pack_block32_kernel(const uint8_t *__restrict__ w, const uint16_t *__restrict__ s,
                                    uint8_t *__restrict__ blocks, int64_t N, int64_t nb) {
    const int64_t total = N * nb;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / nb, b = i - n * nb;
        uint8_t *blk = blocks + i * 18;
        const uint16_t sc = s[i];
        blk[0] = (uint8_t)(sc & 0xFF);
        blk[1] = (uint8_t)(sc >> 8);
        const uint8_t *src = w + n * (nb * 16) + 16 * b;
#pragma unroll
        for (int j = 0; j < 16; ++j) blk[2 + j] = src[j];
    }
}

cudaError_t launch_pack_block32(const uint8_t *w, const uint16_t *s, uint8_t *blocks, int64_t N, int64_t K,
                                cudaStream_t st) {
    const int64_t nb = (K + (K & 1)) / 32;
    const int64_t total = N * nb;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, 152 * 16));
    pack_block32_kernel<<<(unsigned)grid, 256, 0, st>>>(w, s, blocks, N, nb);
    return cudaGetLastError();
}

}  // namespace w4
