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
//   - dataflow without barriers inside a pass: the output of a linear that
//     a later stage reads is also stored as (value, stage tag) pairs, one
//     64-bit store per element, in the workspace; a consumer spins on the
//     pairs it needs until they carry the producing stage's tag (one
//     store-to-load hop instead of fence + atomic + poll + read);
//   - one grid barrier per pass boundary keeps a buffer from being
//     rewritten (next pass) while a slow CTA may still read it; the pass
//     output goes to a buffer double-buffered by pass parity;
//   - each CTA re-quantises the stage's input vector itself (the redundant
//     copy is 4-12 KB from L2) with exactly quantize_row_q8's results;
//   - rows of the stage are dealt out over all warps of the grid; one lane
//     holds 16 bytes (32 nibbles) of a row per chunk, dot products by dp4a
//     on the biased nibbles, acc = sum xq*u - 8 * sum xq, exact in i32, then
//     y = (f32(acc) * sx) * sw[n] as two rounded multiplies;
//   - each warp loads its rows of the NEXT stage into registers before it
//     waits for that stage's input, so the weight reads overlap the wait.
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
constexpr int kPF = 8;  // 16-byte weight chunks a lane holds in registers while it waits
constexpr int kVPerRound = 1024 / (2 * kThreads);  // float2 of the input per thread per 1024 of K
static_assert(kChainMaxK == 8 * 1024, "K <= 8192: at most 8 rounds of 32 chunks");

struct ChainLin {
    const uint4 *w;  // packed row-major, K/2 bytes per row (16-byte chunks)
    const float *sw;
    float *y;
    uint64_t *tag;  // (value | stage tag << 32) copy when a later stage reads y; else null
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
    uint32_t *bar;      // workspace: [0] pass-barrier arrival counter (bit 31: abort)
    uint32_t *status;   // device status word
    uint64_t *pbuf;     // workspace: tagged pass output, [2][K0] by pass parity
    int32_t n_lin;
    int32_t n_stage;
    int32_t passes;
    int32_t pass_output;  // sorted index
    int32_t s_out;        // stage of the pass output
    int32_t K0;
    int32_t hold_stage;   // test of the failure path: this global stage never publishes its outputs (-1: none)
    uint64_t wait_ns;     // limit of every wait (kWaitLimitNs; shorter in the failure-path test)
};
static_assert(sizeof(ChainParams) <= 4096, "kernel parameters");

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

W4_DEV ulonglong2 ld_relaxed_gpu_v2(const uint64_t *p) {
    ulonglong2 v;
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p) : "memory");
    return v;
}

W4_DEV void st_relaxed_gpu(uint64_t *p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

W4_DEV uint64_t tagged(float v, uint32_t tag) { return (uint64_t)__float_as_uint(v) | ((uint64_t)tag << 32); }

// Q8 code of v for scale sx > 0 (quantize_row_q8: clamp(rint(fl(v / sx)), -127, 127)),
// given r = fl(1 / sx) (finite).  t = fl(v * r) is within 2^-16 + 2^-24 of
// x = v / sx when |x| < 256 (two correctly rounded operations, each within
// 2^-24 relative), and fl(x) within ulp(x) / 2 <= 2^-17 of x, so t and fl(x)
// lie within 2^-15 of each other.  When t is farther than 2^-13 from every
// half-integer, rint(t) == rint(fl(x)); otherwise (about 1 value in 4000)
// the IEEE quotient itself is rounded.
W4_DEV int q8_code(float v, float sx, float r) {
    const float t = __fmul_rn(v, r);
    const float rt = rintf(t);
    int q;
    if (fabsf(t) < 256.0f && 0.5f - fabsf(t - rt) > 0x1p-13f) q = __float2int_rn(rt);
    else q = __float2int_rn(__fdiv_rn(v, sx));
    return min(max(q, -127), 127);
}

// Row r of the stage -> its linear (stages hold few linears).
W4_DEV int lin_of_row(const ChainLin *lin, const ChainStage &S, int r) {
    int l = S.lin0;
    while (l + 1 < S.lin0 + S.nlin && r >= lin[l + 1].row0) ++l;
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

// Sum of the 32 activation codes of one chunk.
W4_DEV int sum_chunk(uint4 xe, uint4 xo, int acc) {
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

W4_DEV int warp_sum(int v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Rows a warp holds in registers across a barrier when a row takes ROUNDS
// 16-byte chunks per lane (a power of two, for the transposed reduction).
template <int ROUNDS>
struct RowsInRegs {
    static constexpr int n = kPF / ROUNDS;
    static constexpr int value = n >= 8 ? 8 : n >= 4 ? 4 : n >= 2 ? 2 : 1;  // at most 8 (lanes 4i hold row i)
};

// Sums v[i] over the 32 lanes for NR rows at once (NR a power of two <= 8):
// each exchange step halves the rows a lane carries, so NR rows cost
// NR - 1 + 5 - log2(NR) shuffles instead of 5 * NR.  Afterwards lane L holds
// the total of row L / (32 / NR) in v[0].
template <int NR>
W4_DEV void transposed_warp_sum(int (&v)[NR], int lane) {
    int o = 16;
#pragma unroll
    for (int half = NR / 2; half >= 1; half >>= 1, o >>= 1) {
        const bool hi = (lane & o) != 0;
#pragma unroll
        for (int r = 0; r < half; ++r) {
            const int send = hi ? v[r] : v[r + half];
            const int keep = hi ? v[r + half] : v[r];
            v[r] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
#pragma unroll
    for (; o; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
}

// Per-warp state carried across a barrier: the next stage's weight chunks,
// and for the lane that will write row i, that row's scale and output.
struct Prefetched {
    uint4 w[kPF];
    float sw;
    float *y;
    uint64_t *t;    // the row's tagged copy, or null
    int32_t pn;     // the row's index in the pass output, or -1
    int32_t nrows;  // rows of the stage this warp owns
};

// Rows of stage S this warp owns (rows gw, gw + nw, ...).
W4_DEV int rows_of_warp(const ChainStage &S, int gw, int nw) { return gw < S.R ? (S.R - gw + nw - 1) / nw : 0; }

// Loads this warp's first RowsInRegs<ROUNDS> rows of stage S (row i = gw + i * nw).
template <int ROUNDS>
W4_DEV void prefetch_stage(const ChainLin *lin, const ChainStage &S, int pass_output, int gw, int nw, int lane,
                           Prefetched &pf) {
    constexpr int NR = RowsInRegs<ROUNDS>::value;
    const int Kc = S.K >> 5;
    const int nrows = rows_of_warp(S, gw, nw);
    pf.nrows = nrows;
    const int lend = S.lin0 + S.nlin;
    int l = S.lin0;
#pragma unroll
    for (int i = 0; i < NR; ++i) {
        if (i < nrows) {
            const int r = gw + i * nw;
            while (l + 1 < lend && r >= lin[l + 1].row0) ++l;  // rows only grow with i
            const ChainLin &L = lin[l];
            const int n = r - L.row0;
            const uint4 *wr = L.w + (size_t)n * Kc;
#pragma unroll
            for (int t = 0; t < ROUNDS; ++t) {
                const int c = lane + 32 * t;
                if (c < Kc) pf.w[i * ROUNDS + t] = ldg_nc_128(wr + c);
            }
            if (lane == i * (32 / NR)) {
                pf.sw = __ldg(L.sw + n);
                pf.y = L.y + n;
                pf.t = L.tag ? L.tag + n : nullptr;
                pf.pn = l == pass_output ? n : -1;
            }
        }
    }
}

W4_DEV void prefetch_any(int rounds, const ChainLin *lin, const ChainStage &S, int pass_output, int gw, int nw,
                         int lane, Prefetched &pf) {
    switch (rounds) {
        case 1: prefetch_stage<1>(lin, S, pass_output, gw, nw, lane, pf); break;
        case 2: prefetch_stage<2>(lin, S, pass_output, gw, nw, lane, pf); break;
        case 3: prefetch_stage<3>(lin, S, pass_output, gw, nw, lane, pf); break;
        case 4: prefetch_stage<4>(lin, S, pass_output, gw, nw, lane, pf); break;
        case 5: prefetch_stage<5>(lin, S, pass_output, gw, nw, lane, pf); break;
        case 6: prefetch_stage<6>(lin, S, pass_output, gw, nw, lane, pf); break;
        case 7: prefetch_stage<7>(lin, S, pass_output, gw, nw, lane, pf); break;
        default: prefetch_stage<8>(lin, S, pass_output, gw, nw, lane, pf); break;
    }
}

// Where a finished row goes: y, its tagged copy, and the tagged pass output.
struct RowSink {
    uint64_t *pout;  // pass output buffer of this pass, or null (last pass)
    uint32_t tag;    // this stage's tag (global stage index + 1)
};

W4_DEV void store_row(float v, float *y, uint64_t *t, int pn, const RowSink &k) {
    *y = v;
    if (t || (pn >= 0 && k.pout)) {
        const uint64_t pk = tagged(v, k.tag);
        if (t) st_relaxed_gpu(t, pk);
        if (pn >= 0 && k.pout) st_relaxed_gpu(k.pout + pn, pk);
    }
}

// y[n] = (f32(acc) * sx) * sw[n], two rounded multiplies (the linear_q4 epilogue).
W4_DEV float epilogue(int acc, float sx, float sw) {
    return __fmul_rn(__fmul_rn(__int2float_rn(acc), sx), sw);
}

// This warp's rows of stage S against the quantized input in shared memory.
template <int ROUNDS>
W4_DEV void compute_stage(const ChainLin *lin, const ChainStage &S, int pass_output, int gw, int nw, int lane,
                          const Prefetched &pf, const int8_t *xs, float sx, const RowSink &k) {
    constexpr int NR = RowsInRegs<ROUNDS>::value;
    const int K = S.K, Kc = K >> 5;
    const uint4 *xe4 = reinterpret_cast<const uint4 *>(xs);
    const uint4 *xo4 = reinterpret_cast<const uint4 *>(xs + (K >> 1));
    const int nrows = pf.nrows;
    // acc = sum xq*u - 8 * sum xq; each lane subtracts 8x its own chunks' code sum
    int xsum = 0;
#pragma unroll
    for (int t = 0; t < ROUNDS; ++t) {
        const int c = lane + 32 * t;
        if (c < Kc) xsum = sum_chunk(xe4[c], xo4[c], xsum);
    }
    int v[NR];
#pragma unroll
    for (int i = 0; i < NR; ++i) v[i] = 0;
#pragma unroll
    for (int t = 0; t < ROUNDS; ++t) {
        const int c = lane + 32 * t;
        if (c < Kc) {
            const uint4 xe = xe4[c], xo = xo4[c];
#pragma unroll
            for (int i = 0; i < NR; ++i)
                if (i < nrows) v[i] = dot_chunk(pf.w[i * ROUNDS + t], xe, xo, v[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < NR; ++i) v[i] = i < nrows ? v[i] - 8 * xsum : 0;
    transposed_warp_sum<NR>(v, lane);
    if ((lane & (32 / NR - 1)) == 0 && lane / (32 / NR) < nrows)
        store_row(epilogue(v[0], sx, pf.sw), pf.y, pf.t, pf.pn, k);
    // rows beyond the registers (stages with more rows than warps x NR)
    for (int i = NR; i < nrows; ++i) {
        const int r = gw + i * nw;
        const ChainLin &L = lin[lin_of_row(lin, S, r)];
        const uint4 *wr = L.w + (size_t)(r - L.row0) * Kc;
        int a = 0;
        for (int c = lane; c < Kc; c += 32) a = dot_chunk(ldg_nc_128(wr + c), xe4[c], xo4[c], a);
        a = warp_sum(a - 8 * xsum);
        if (lane == 0) {
            const int n = r - L.row0;
            store_row(epilogue(a, sx, __ldg(L.sw + n)), L.y + n, L.tag ? L.tag + n : nullptr,
                      (&L - lin) == pass_output ? n : -1, k);
        }
    }
}

// Input pair j (elements 2j, 2j+1) from a tagged buffer: spins until both
// carry `want`; false if that takes longer than the wait limit.
W4_DEV bool wait_pair(const uint64_t *src, uint32_t want, ulonglong2 &a, uint64_t limit_ns) {
    const auto ok = [&]() { return (uint32_t)(a.x >> 32) == want && (uint32_t)(a.y >> 32) == want; };
    if (ok()) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        __nanosleep(64);  // fewer requests on the lines every CTA polls: measured best of 0-512 ns
        a = ld_relaxed_gpu_v2(src);
        if (ok()) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// One stage on this CTA: quantize_row_q8 of the stage's input into shared
// memory (ROUNDS * kVPerRound float2 per thread covers K <= 1024 * ROUNDS),
// then this warp's rows.  False when a wait for an input element ran out.
template <int ROUNDS>
W4_DEV bool run_stage(const ChainParams &p, const ChainLin *lin, const ChainStage &S, int gs, int pass, int gw,
                      int nw, int warp, int lane, const Prefetched &pf, int8_t *xs, float *red_max, int *fail_flag) {
    const int K = S.K;
    // the stage's input: x0, or the tagged copy of the vector it reads
    const float *plain = nullptr;
    const uint64_t *tin = nullptr;
    uint32_t want = 0;
    if (S.input >= 0) {
        tin = lin[S.input].tag;
        want = (uint32_t)gs;  // written by the previous stage, tag (gs - 1) + 1
    } else if (pass == 0) {
        plain = p.x0;
    } else {
        tin = p.pbuf + (size_t)((pass - 1) & 1) * p.K0;
        want = (uint32_t)((pass - 1) * p.n_stage + p.s_out + 1);
    }

    constexpr int KV = ROUNDS * kVPerRound;  // float2 of the input per thread
    const int n2 = K >> 1;
    float2 v[KV];
    if (plain) {
#pragma unroll
        for (int u = 0; u < KV; ++u) {
            const int j = threadIdx.x + u * kThreads;
            v[u] = j < n2 ? __ldg(reinterpret_cast<const float2 *>(plain) + j) : make_float2(0.f, 0.f);
        }
    } else {
        ulonglong2 a[KV];
#pragma unroll
        for (int u = 0; u < KV; ++u) {
            const int j = threadIdx.x + u * kThreads;
            a[u] = j < n2 ? ld_relaxed_gpu_v2(tin + 2 * j) : make_ulonglong2(0, 0);
        }
        bool good = true;
#pragma unroll
        for (int u = 0; u < KV; ++u) {
            const int j = threadIdx.x + u * kThreads;
            if (j < n2) good = good && wait_pair(tin + 2 * j, want, a[u], p.wait_ns);
            v[u] = make_float2(__uint_as_float((uint32_t)a[u].x), __uint_as_float((uint32_t)a[u].y));
        }
        if (!good) {
            *fail_flag = 1;
            atomicOr(p.status, kStatusBarrierTimeout);
        }
    }
    float amax = 0.0f;
#pragma unroll
    for (int u = 0; u < KV; ++u) amax = fmaxf(amax, fmaxf(fabsf(v[u].x), fabsf(v[u].y)));
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) red_max[warp] = amax;
    __syncthreads();
    if (*fail_flag) return false;  // a wait ran out: the whole CTA leaves
    amax = red_max[lane & (kWarps - 1)];
#pragma unroll
    for (int o = kWarps / 2; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sx = __fdiv_rn(amax, 127.0f);
    const float r = sx != 0.0f ? __frcp_rn(sx) : 0.0f;
    const bool fast = isfinite(r);
#pragma unroll
    for (int u = 0; u < KV; ++u) {
        const int j = threadIdx.x + u * kThreads;
        if (j < n2) {
            int c0 = 0, c1 = 0;
            if (sx != 0.0f) {
                if (fast) {
                    c0 = q8_code(v[u].x, sx, r);
                    c1 = q8_code(v[u].y, sx, r);
                } else {
                    c0 = min(max(__float2int_rn(__fdiv_rn(v[u].x, sx)), -127), 127);
                    c1 = min(max(__float2int_rn(__fdiv_rn(v[u].y, sx)), -127), 127);
                }
            }
            xs[j] = (int8_t)c0;             // k = 2j (even)
            xs[(K >> 1) + j] = (int8_t)c1;  // k = 2j + 1 (odd)
        }
    }
    __syncthreads();

    RowSink k;
    // tag 0 is what the cleared workspace holds: a held stage's outputs never appear
    k.tag = gs == p.hold_stage ? 0u : (uint32_t)(gs + 1);
    k.pout = pass + 1 < p.passes ? p.pbuf + (size_t)(pass & 1) * p.K0 : nullptr;
    compute_stage<ROUNDS>(lin, S, p.pass_output, gw, nw, lane, pf, xs, sx, k);
    return true;
}

W4_DEV bool run_stage_any(int rounds, const ChainParams &p, const ChainLin *lin, const ChainStage &S, int gs,
                          int pass, int gw, int nw, int warp, int lane, const Prefetched &pf, int8_t *xs,
                          float *red_max, int *fail_flag) {
    switch (rounds) {
        case 1: return run_stage<1>(p, lin, S, gs, pass, gw, nw, warp, lane, pf, xs, red_max, fail_flag);
        case 2: return run_stage<2>(p, lin, S, gs, pass, gw, nw, warp, lane, pf, xs, red_max, fail_flag);
        case 3: return run_stage<3>(p, lin, S, gs, pass, gw, nw, warp, lane, pf, xs, red_max, fail_flag);
        case 4: return run_stage<4>(p, lin, S, gs, pass, gw, nw, warp, lane, pf, xs, red_max, fail_flag);
        case 5: return run_stage<5>(p, lin, S, gs, pass, gw, nw, warp, lane, pf, xs, red_max, fail_flag);
        case 6: return run_stage<6>(p, lin, S, gs, pass, gw, nw, warp, lane, pf, xs, red_max, fail_flag);
        case 7: return run_stage<7>(p, lin, S, gs, pass, gw, nw, warp, lane, pf, xs, red_max, fail_flag);
        default: return run_stage<8>(p, lin, S, gs, pass, gw, nw, warp, lane, pf, xs, red_max, fail_flag);
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
                if (globaltimer_ns() - t0 > p.wait_ns) {
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
    __shared__ ChainLin lin[kChainMaxLinears];
    __shared__ ChainStage st[kChainMaxLinears];
    __shared__ float red_max[kWarps];
    __shared__ int fail_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kWarps + warp;
    const int nw = gridDim.x * kWarps;
    for (int i = threadIdx.x; i < p.n_lin; i += kThreads) lin[i] = p.lin[i];
    for (int i = threadIdx.x; i < p.n_stage; i += kThreads) st[i] = p.st[i];
    if (threadIdx.x == 0) fail_flag = 0;
    __syncthreads();

    Prefetched pf;
#pragma unroll
    for (int j = 0; j < kPF; ++j) pf.w[j] = make_uint4(0, 0, 0, 0);
    pf.sw = 0.0f;
    pf.y = nullptr;
    pf.t = nullptr;
    pf.pn = -1;
    prefetch_any((st[0].K + 1023) >> 10, lin, st[0], p.pass_output, gw, nw, lane, pf);

    int s = 0, pass = 0;
    const int total = p.passes * p.n_stage;
    for (int gs = 0; gs < total; ++gs) {
        const ChainStage S = st[s];
        if (blockIdx.x * kWarps < S.R &&  // this CTA has rows in the stage
            !run_stage_any((S.K + 1023) >> 10, p, lin, S, gs, pass, gw, nw, warp, lane, pf, xs, red_max, &fail_flag))
            return;
        if (++s == p.n_stage) {
            s = 0;
            ++pass;
        }
        if (gs + 1 < total) {
            prefetch_any((st[s].K + 1023) >> 10, lin, st[s], p.pass_output, gw, nw, lane, pf);
            // pass boundary: every read of this pass's buffers is done before the next pass rewrites them
            if (s == 0 && !grid_barrier(p, (uint32_t)pass, &fail_flag)) return;
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

size_t chain_workspace_bytes(const w4_chain_linear *lin, int32_t n_lin, int32_t K0) {
    std::vector<bool> consumed(n_lin, false);
    for (int i = 0; i < n_lin; ++i)
        if (lin[i].input >= 0 && lin[i].input < n_lin) consumed[lin[i].input] = true;
    size_t elems = 2 * (size_t)K0;  // the pass output, by pass parity
    for (int i = 0; i < n_lin; ++i)
        if (consumed[i]) elems += (size_t)lin[i].N;
    return kChainHeaderBytes + 8 * elems;
}

int chain_plan_launch(const float *x0, int32_t K0, const w4_chain_linear *lin, int32_t n_lin, int32_t passes,
                      int32_t pass_output, void *workspace, uint32_t *status, cudaStream_t st, cudaError_t *err,
                      uint64_t wait_ns, int32_t hold_stage) {
    *err = cudaSuccess;
    if (!chain_stages_ok(lin, n_lin, passes, pass_output)) return W4_ESHAPE;
    std::vector<int> depth(n_lin);
    for (int i = 0; i < n_lin; ++i) depth[i] = lin[i].input < 0 ? 0 : depth[lin[i].input] + 1;
    const int n_stage = *std::max_element(depth.begin(), depth.end()) + 1;
    std::vector<int> stage_input(n_stage, -1);
    for (int i = 0; i < n_lin; ++i) stage_input[depth[i]] = lin[i].input;
    std::vector<bool> consumed(n_lin, false);
    for (int i = 0; i < n_lin; ++i)
        if (lin[i].input >= 0) consumed[lin[i].input] = true;

    // workspace: header | pass output [2][K0] | tagged copies of consumed linears
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint64_t *pbuf = reinterpret_cast<uint64_t *>(ws + kChainHeaderBytes);
    uint64_t *next_tag = pbuf + 2 * (size_t)K0;

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
            L.tag = nullptr;
            if (consumed[i]) {
                L.tag = next_tag;
                next_tag += lin[i].N;
            }
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
    p.bar = reinterpret_cast<uint32_t *>(ws);
    p.status = status;
    p.pbuf = pbuf;
    p.n_lin = n_lin;
    p.n_stage = n_stage;
    p.passes = passes;
    p.pass_output = sorted_of[pass_output];
    p.s_out = depth[pass_output];
    p.K0 = K0;
    p.hold_stage = hold_stage;
    p.wait_ns = wait_ns;
    const size_t ws_used = (size_t)(reinterpret_cast<uint8_t *>(next_tag) - ws);

    int dev = 0, sms = 0, occ = 0;
    if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return W4_ECUDA;
    if ((*err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return W4_ECUDA;
    if ((*err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, chain_q4_kernel, kThreads, 0)) != cudaSuccess)
        return W4_ECUDA;
    if (occ < 1) {
        *err = cudaErrorLaunchOutOfResources;
        return W4_ECUDA;
    }
    if ((int64_t)passes * sms >= (int64_t)kAbortBit || (int64_t)passes * n_stage >= (int64_t)kAbortBit)
        return W4_ESHAPE;
    // barrier counter and every tag to 0 (no stage has tag 0)
    if ((*err = cudaMemsetAsync(workspace, 0, ws_used, st)) != cudaSuccess) return W4_ECUDA;

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

