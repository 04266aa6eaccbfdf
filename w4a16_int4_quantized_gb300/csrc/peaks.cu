// peaks.cu -- tensor-core throughput probes used as roofline denominators.
//
// The measured peaks cover HBM copy bandwidth and bf16 GEMM; the
// metric of the W4A8 prefill is quoted against the int8 tensor rate, which
// on this part is only reachable through the legacy mma.sync path (tcgen05
// has no integer kind for sm_103a in this toolchain).  These kernels issue
// independent chains of one MMA shape back to back on every SM so the host
// can time them: a microbenchmark, not part of any linear.
#include <cuda_runtime.h>

#include <cstdint>

#include "w4.h"

namespace {

constexpr int kChains = 8;

__global__ void __launch_bounds__(256) mma_s8_loop(int *out, int iters) {
    int d[kChains][4] = {};
    const uint32_t a = 0x01010101u + threadIdx.x, b = 0x01010101u;
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < kChains; ++c)
            asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                         : "+r"(d[c][0]), "+r"(d[c][1]), "+r"(d[c][2]), "+r"(d[c][3])
                         : "r"(a), "r"(a), "r"(a), "r"(a), "r"(b), "r"(b));
    }
    int s = 0;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += d[c][0] + d[c][1] + d[c][2] + d[c][3];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void __launch_bounds__(256) mma_bf16_loop(int *out, int iters) {
    float d[kChains][4] = {};
    const uint32_t a = 0x3f803f80u + threadIdx.x, b = 0x3f803f80u;
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < kChains; ++c)
            asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                         : "+f"(d[c][0]), "+f"(d[c][1]), "+f"(d[c][2]), "+f"(d[c][3])
                         : "r"(a), "r"(a), "r"(a), "r"(a), "r"(b), "r"(b));
    }
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += d[c][0] + d[c][1] + d[c][2] + d[c][3];
    out[blockIdx.x * blockDim.x + threadIdx.x] = (int)s;
}

}  // namespace

extern "C" w4_status w4_probe_mma_peak(int32_t kind, int32_t *scratch, int64_t scratch_ints, double *tera_ops,
                                       void *stream) {
    if (!scratch || !tera_ops || (kind != 0 && kind != 1)) return W4_EINVAL;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return W4_ECUDA;
    const int blocks = 4 * sms, threads = 256, iters = 4096;
    if (scratch_ints < (int64_t)blocks * threads) return W4_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess) return W4_ECUDA;
    if (cudaEventCreate(&e1) != cudaSuccess) {
        cudaEventDestroy(e0);
        return W4_ECUDA;
    }
    float best = 1e30f;
    for (int rep = 0; rep < 3; ++rep) {
        cudaEventRecord(e0, st);
        if (kind == 0) mma_s8_loop<<<blocks, threads, 0, st>>>(scratch, iters);
        else mma_bf16_loop<<<blocks, threads, 0, st>>>(scratch, iters);
        cudaEventRecord(e1, st);
        if (cudaEventSynchronize(e1) != cudaSuccess) break;
        float ms = 0.f;
        cudaEventElapsedTime(&ms, e0, e1);
        if (rep > 0 && ms < best) best = ms;  // first launch warms up
    }
    const cudaError_t e = cudaGetLastError();
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (e != cudaSuccess || best >= 1e30f) return W4_ECUDA;
    const double mnk = (kind == 0) ? 16.0 * 8 * 32 : 16.0 * 8 * 16;
    const double ops = 2.0 * mnk * kChains * iters * ((double)blocks * threads / 32);
    *tera_ops = ops / (best * 1e-3) / 1e12;
    return W4_OK;
}
