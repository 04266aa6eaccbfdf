// chain.cu -- a chain of M = 1 W4A8 linears run as one persistent kernel.
//
// The microdecoder of docs.rs ftts_kernels::int4 ("Why the microdecoder"):
// a small decoder body whose int4 weights are re-read many times per frame,
// each linear reading the per-row Q8 quantisation (ftts_kernels::int8,
// quantize_row_q8) of an earlier linear's f32 output.  Launched one call at
// a time that is hundreds of launches per frame of ~1 MB each, bound by
// launch latency; here the whole chain, all passes, is one cooperative grid
// (one CTA per SM) that keeps its working set in L2:
//
//   - linears are grouped into stages by depth (a linear reading the pass
//     input is depth 0, one reading linear j is depth(j) + 1); all linears
//     of a stage read the same vector and run together;
//   - between stages a grid barrier (one global counter, release/acquire,
//     bounded wait);
//   - each CTA re-quantises the stage's input vector itself (the redundant
//     copy is ~4-12 KB from L2), with exactly the arithmetic of
//     quantize_row_q8: s = max|v| / 127 by one IEEE division, codes
//     clamp(rint(v / s), -127, 127);
//   - rows of the stage are dealt out over all warps of the grid; one lane
//     holds 16 bytes (32 nibbles) of a row per chunk, dot products by dp4a
//     on the biased nibbles, acc = sum xq*u - 8 * sum xq, exact in i32, then
//     y = (f32(acc) * sx) * sw[n] as two rounded multiplies;
//   - each warp loads its rows of the NEXT stage into registers before it
//     waits at the barrier, so the weight reads overlap the barrier.
// Every value is the one the per-call path (and the CPU definition) gives.
#include "common.cuh"
#include "internal.h"
#include "w4.h"

#include <algorithm>
#include <vector>

namespace w4 {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kPF = 8;  // 16-byte weight chunks a lane holds in registers across a barrier
constexpr int kVR = kChainMaxK / (4 * kThreads);  // float4s of the input vector per thread
static_assert(kChainMaxK % (4 * kThreads) == 0, "input vector must tile the CTA");

struct ChainLin {
    const uint4 *w;  // packed row-major, K/2 bytes per row (16-byte chunks)
    const float *sw;
    float *y;
    int32_t N;
    int32_t row0;  // first row of this linear in its stage's row space
};

struct ChainStage {
    int32_t lin0, nlin;  // linears [lin0, lin0 + nlin) of the sorted table
    int32_t input;       // -1: the pass input; else the sorted index of the linear whose y is read
    int32_t R;           // rows of the stage (sum of N)
    int32_t K;           // input length (multiple of 32)
};

struct ChainParams {
    ChainLin lin[kChainMaxLinears];
    ChainStage st[kChainMaxLinears];
    const float *x0;
    uint32_t *bar;     // workspace: [0] arrival counter (bit 31: abort)
    uint32_t *status;  // device status word
    int32_t n_stage;
    int32_t passes;
    int32_t pass_output;  // sorted index
};

constexpr uint32_t kAbortBit = 0x80000000u;

W4_DEV uint4 ldg_nc_128(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

W4_DEV uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

W4_DEV void red_release_gpu_add(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Row r of the stage -> its linear (stages hold few linears).
W4_DEV int lin_of_row(const ChainParams &p, const ChainStage &S, int r) {
    int l = S.lin0;
    while (l + 1 < S.lin0 + S.nlin && r >= p.lin[l + 1].row0) ++l;
    return l;
}

// Sum over one 16-byte chunk (32 biased nibbles, k = 32c .. 32c + 31) of
// xq[k] * u[k]; xe / xo hold the chunk's even / odd-k activations.
W4_DEV int dot_chunk(uint4 w, uint4 xe, uint4 xo, int acc) {
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

W4_DEV int warp_sum(int v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Loads (row i, round t) slots 0..kPF-1 of this warp's share of stage S.
W4_DEV void prefetch_stage(const ChainParams &p, const ChainStage &S, int gw, int nw, int lane, uint4 (&pf)[kPF]) {
    const int Kc = S.K >> 5;
    const int rounds = (Kc + 31) >> 5;
    int i = 0, t = 0;
#pragma unroll
    for (int j = 0; j < kPF; ++j) {
        const int r = gw + i * nw;
        const int c = lane + 32 * t;
        if (r < S.R && c < Kc) {
            const ChainLin &L = p.lin[lin_of_row(p, S, r)];
            pf[j] = ldg_nc_128(L.w + (size_t)(r - L.row0) * Kc + c);
        }
        if (++t == rounds) { t = 0; ++i; }
    }
}

// Grid barrier number `gen` (1-based).  Returns false when the grid aborts
// (a barrier wait ran out somewhere).
W4_DEV bool grid_barrier(const ChainParams &p, uint32_t gen, int *abort_flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        red_release_gpu_add(p.bar, 1u);
        const uint32_t target = gen * gridDim.x;
        uint32_t v = ld_acquire_gpu(p.bar);
        if ((v & ~kAbortBit) < target && !(v & kAbortBit)) {
            const uint64_t t0 = globaltimer_ns();
            while (true) {
                v = ld_acquire_gpu(p.bar);
                if ((v & ~kAbortBit) >= target || (v & kAbortBit)) break;
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    atomicOr(p.bar, kAbortBit);
                    atomicOr(p.status, kStatusBarrierTimeout);
                    v = kAbortBit;
                    break;
                }
            }
        }
        *abort_flag = (v & kAbortBit) ? 1 : 0;
    }
    __syncthreads();
    return *abort_flag == 0;
}

__global__ void __launch_bounds__(kThreads, 1) chain_q4_kernel(const __grid_constant__ ChainParams p) {
    __shared__ __align__(16) int8_t xs[kChainMaxK];  // [K/2] even-k codes, then [K/2] odd-k codes
    __shared__ float red_max[kWarps];
    __shared__ int red_sum[kWarps];
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kWarps + warp;
    const int nw = gridDim.x * kWarps;
    const int total = p.passes * p.n_stage;

    uint4 pf[kPF];
#pragma unroll
    for (int j = 0; j < kPF; ++j) pf[j] = make_uint4(0, 0, 0, 0);
    prefetch_stage(p, p.st[0], gw, nw, lane, pf);

    for (int gs = 0; gs < total; ++gs) {
        const int pass = gs / p.n_stage;
        const ChainStage &S = p.st[gs - pass * p.n_stage];
        const int K = S.K, Kc = K >> 5, rounds = (Kc + 31) >> 5;
        const float *in = S.input >= 0 ? p.lin[S.input].y : (pass == 0 ? p.x0 : p.lin[p.pass_output].y);

        // ---- quantize_row_q8 of the input vector into shared memory
        const int n4 = K >> 2;
        float4 v[kVR];
        float amax = 0.0f;
#pragma unroll
        for (int u = 0; u < kVR; ++u) {
            const int j = threadIdx.x + u * kThreads;
            v[u] = j < n4 ? __ldcg(reinterpret_cast<const float4 *>(in) + j) : make_float4(0.f, 0.f, 0.f, 0.f);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[u].x), fabsf(v[u].y)), fmaxf(fabsf(v[u].z), fabsf(v[u].w))));
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) red_max[warp] = amax;
        __syncthreads();
        amax = red_max[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) amax = fmaxf(amax, red_max[w]);
        const float sx = __fdiv_rn(amax, 127.0f);
        int qsum = 0;
#pragma unroll
        for (int u = 0; u < kVR; ++u) {
            const int j = threadIdx.x + u * kThreads;
            if (j < n4) {
                int c0 = 0, c1 = 0, c2 = 0, c3 = 0;
                if (sx != 0.0f) {
                    c0 = min(max(__float2int_rn(__fdiv_rn(v[u].x, sx)), -127), 127);
                    c1 = min(max(__float2int_rn(__fdiv_rn(v[u].y, sx)), -127), 127);
                    c2 = min(max(__float2int_rn(__fdiv_rn(v[u].z, sx)), -127), 127);
                    c3 = min(max(__float2int_rn(__fdiv_rn(v[u].w, sx)), -127), 127);
                }
                qsum += c0 + c1 + c2 + c3;
                // k = 4j .. 4j+3: even-k codes to xs[2j], xs[2j+1]; odd-k codes to xs[K/2 + 2j], xs[K/2 + 2j + 1]
                reinterpret_cast<uint16_t *>(xs)[j] = (uint16_t)((c0 & 0xFF) | ((c2 & 0xFF) << 8));
                reinterpret_cast<uint16_t *>(xs + (K >> 1))[j] = (uint16_t)((c1 & 0xFF) | ((c3 & 0xFF) << 8));
            }
        }
        qsum = warp_sum(qsum);
        if (lane == 0) red_sum[warp] = qsum;
        __syncthreads();
        qsum = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) qsum += red_sum[w];

        // ---- this warp's rows: registers first, then direct loads
        const int nrows = gw < S.R ? (S.R - gw + nw - 1) / nw : 0;
        const uint4 *xe4 = reinterpret_cast<const uint4 *>(xs);
        const uint4 *xo4 = reinterpret_cast<const uint4 *>(xs + (K >> 1));
        int i = 0, t = 0, acc = 0;
        auto finish_row = [&](int row_i, int a) {
            a = warp_sum(a);
            if (lane == 0) {
                const int r = gw + row_i * nw;
                const ChainLin &L = p.lin[lin_of_row(p, S, r)];
                const int n = r - L.row0;
                const float v = __fmul_rn(__fmul_rn(__int2float_rn(a - 8 * qsum), sx), __ldg(L.sw + n));
                L.y[n] = v;
            }
        };
#pragma unroll
        for (int j = 0; j < kPF; ++j) {
            if (i < nrows) {
                const int c = lane + 32 * t;
                if (c < Kc) acc = dot_chunk(pf[j], xe4[c], xo4[c], acc);
                if (++t == rounds) {
                    finish_row(i, acc);
                    acc = 0;
                    t = 0;
                    ++i;
                }
            }
        }
        while (i < nrows) {
            const int r = gw + i * nw;
            const ChainLin &L = p.lin[lin_of_row(p, S, r)];
            const uint4 *wr = L.w + (size_t)(r - L.row0) * Kc;
            for (; t < rounds; ++t) {
                const int c = lane + 32 * t;
                if (c < Kc) acc = dot_chunk(ldg_nc_128(wr + c), xe4[c], xo4[c], acc);
            }
            finish_row(i, acc);
            acc = 0;
            t = 0;
            ++i;
        }

        if (gs + 1 < total) {
            const int ns = (gs + 1) % p.n_stage;
            prefetch_stage(p, p.st[ns], gw, nw, lane, pf);
            if (!grid_barrier(p, (uint32_t)(gs + 1), &abort_flag)) return;
        }
    }
}

}  // namespace

bool chain_stages_ok(const w4_chain_linear *lin, int32_t n_lin, int32_t passes, int32_t pass_output) {
    // depth of each linear; all linears of one depth must read the same vector
    std::vector<int> depth(n_lin);
    for (int i = 0; i < n_lin; ++i) depth[i] = lin[i].input < 0 ? 0 : depth[lin[i].input] + 1;
    const int n_stage = *std::max_element(depth.begin(), depth.end()) + 1;
    std::vector<int> stage_input(n_stage, -2);
    std::vector<int64_t> rows(n_stage, 0);
    for (int i = 0; i < n_lin; ++i) {
        int &si = stage_input[depth[i]];
        if (si == -2) si = lin[i].input;
        else if (si != lin[i].input) return false;
        rows[depth[i]] += lin[i].N;
        if (rows[depth[i]] > kChainMaxStageRows) return false;
    }
    return !(passes > 1 && depth[pass_output] == 0);
}

int chain_plan_launch(const float *x0, int32_t K0, const w4_chain_linear *lin, int32_t n_lin, int32_t passes,
                      int32_t pass_output, void *workspace, uint32_t *status, cudaStream_t st, cudaError_t *err) {
    *err = cudaSuccess;
    if (!chain_stages_ok(lin, n_lin, passes, pass_output)) return W4_ESHAPE;
    std::vector<int> depth(n_lin);
    for (int i = 0; i < n_lin; ++i) depth[i] = lin[i].input < 0 ? 0 : depth[lin[i].input] + 1;
    const int n_stage = *std::max_element(depth.begin(), depth.end()) + 1;
    std::vector<int> stage_input(n_stage, -1);
    for (int i = 0; i < n_lin; ++i) stage_input[depth[i]] = lin[i].input;

    ChainParams p;
    std::vector<int> sorted_of(n_lin);
    int pos = 0;
    for (int s = 0; s < n_stage; ++s) {
        ChainStage &S = p.st[s];
        S.lin0 = pos;
        S.nlin = 0;
        S.R = 0;
        for (int i = 0; i < n_lin; ++i) {
            if (depth[i] != s) continue;
            sorted_of[i] = pos;
            ChainLin &L = p.lin[pos++];
            L.w = reinterpret_cast<const uint4 *>(lin[i].w);
            L.sw = lin[i].sw;
            L.y = lin[i].y;
            L.N = lin[i].N;
            L.row0 = S.R;
            S.R += lin[i].N;
            S.K = lin[i].K;
            ++S.nlin;
        }
    }
    for (int s = 0; s < n_stage; ++s) {
        const int in = stage_input[s];
        p.st[s].input = in < 0 ? -1 : sorted_of[in];
    }
    p.x0 = x0;
    p.bar = static_cast<uint32_t *>(workspace);
    p.status = status;
    p.n_stage = n_stage;
    p.passes = passes;
    p.pass_output = sorted_of[pass_output];
    (void)K0;

    int dev = 0, sms = 0, occ = 0;
    if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return W4_ECUDA;
    if ((*err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return W4_ECUDA;
    if ((*err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, chain_q4_kernel, kThreads, 0)) != cudaSuccess)
        return W4_ECUDA;
    if (occ < 1) {
        *err = cudaErrorLaunchOutOfResources;
        return W4_ECUDA;
    }
    if ((int64_t)passes * n_stage * sms >= (int64_t)kAbortBit) return W4_ESHAPE;
    if ((*err = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), st)) != cudaSuccess) return W4_ECUDA;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((*err = cudaLaunchKernelEx(&cfg, chain_q4_kernel, p)) != cudaSuccess) return W4_ECUDA;
    return W4_OK;
}

}  // namespace w4
