// gemm_tc.cu -- prefill linears (M > 16) on the 5th-generation tensor cores.
//
// y[m][n] = sum_k x[m][k] W[n][k], W never stored in float in global memory.
//
// Persistent: one CTA per SM walks the 128 (output channels n) x 256
// (activation rows m) tiles of y (n fastest, so concurrent CTAs share the
// activation tiles in L2), accumulating each in tensor memory over K in steps
// of 64 columns; the stage pipeline runs on across tile boundaries:
//   warp 0       TMA producer: the packed weight tile [128 rows][32|64 B] and
//                the 16-bit activation tile [256 rows][64] (128-byte swizzle)
//                of each stage, both on one transaction-count mbarrier;
//   warp 1       allocates 512 TMEM columns (two 256-column accumulators) and
//                issues tcgen05.mma (one thread): kind::f16, A = weights
//                (M = 128), B = activations (N = 256), K-major shared-memory
//                descriptors, f32 accumulator; tcgen05.commit releases each
//                stage, and each finished tile's accumulator;
//   warps 2-9    convert the packed weights of a stage into the A operand tile
//                (128B-swizzled, K-major);
//   warps 10-17  epilogue of tile i (tcgen05.ld of the accumulator, scales,
//                coalesced stores) while the MMA warp accumulates tile i + 1
//                into the other accumulator.
// Weight conversion (the dequantisation happens only in shared memory):
//   W4A16  w = bf16_rne(f32(q) * f32(s)): q * s is exact in f32 and rounded
//          once to bf16 ("Fused int4 ..." sections 2.2-2.3 dequantised once per
//          tile, as vllm-omni "The 4-bit CPU path" does for large batches);
//   W4A8   f16(q), q = u - 8 in [-8, 7]: exact;
//   W8A8   f16(q), q in [-128, 127]: exact.
// For the integer kinds the activations are the exact f16 images of the int8
// codes, every product is an exact integer and every partial sum an integer
// of magnitude <= 127 * max|q| * K, below 2^24 for W4A8 (|q| <= 8) up to
// K = 16384 and for W8A8 (|q| <= 128) up to K = 1024 -- the shapes this path
// accepts -- so the f32 accumulator holds the exact i32 dot product; the
// epilogue applies y = (f32(acc) * sx[m]) * sw[n] like the decode path.
//
// Every mbarrier wait is bounded (about one second of %globaltimer); a wait
// that runs out sets the status word, raises a CTA-wide abort flag that ends
// every other wait at once, and the tile is not stored.  TMEM is always
// released before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "w4.h"

namespace w4 {
namespace {

constexpr int kBM = 128;   // weight rows per tile (UMMA M)
constexpr int kBN = 256;   // activation rows per tile (UMMA N)
constexpr int kBK = 64;    // columns per stage (128 bytes of 16-bit values)
constexpr int kStages = 4;
constexpr int kConvWarps = 8;
constexpr int kEpiWarps = 8;  // two per TMEM lane quadrant, one per column half
constexpr int kThreads = 64 + 32 * (kConvWarps + kEpiWarps);
constexpr int kTmemCols = 512;  // two accumulators of kBN columns

struct GemmParams {
    CUtensorMap xmap;  // 16-bit activations [M][Kx], box {64, 256}, 128B swizzle
    CUtensorMap wmap;  // packed weights [N][Kb] bytes, box {32|64, 128}
    CUtensorMap smap;  // W4A16 row-major, s_tma: f16 scales [N][ng], box {8 groups, 128 rows}
    const uint16_t *scales;  // W4A16, W4A8G: f16 [N][ng]
    const uint8_t *zeros;    // W4A8G: zero points [N][ng]
    const float *sx;         // int kinds: [M]
    const float *sw;         // int kinds: [N]
    float *y;                // [M][N]
    uint32_t *status;
    int M, N, K, G, ng;
    int s_tma;  // the group scales of each stage arrive by TMA with the packed weights
    int nk;   // k-blocks of 64 columns
    int ntn;  // tiles along N (n fastest)
    int ntiles;
};

struct Smem {
    uint64_t tma_full[kStages];  // the activation tile of a stage
    uint64_t w_full[kStages];    // the packed weight tile (and its group scales) of a stage
    uint64_t conv_full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint32_t tmem_base;
    int abort;
};

// ---------------------------------------------------------------- tcgen05 wrappers

W4_DEV void tmem_alloc(uint32_t *dst_smem, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
W4_DEV void tmem_dealloc(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}
W4_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
W4_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, K-major operand, 128-byte swizzle:
// 8-row atoms of 1024 bytes (stride byte offset 1024), start address >> 4.
W4_DEV uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;             // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset: next 8-row atom
    d |= (uint64_t)1 << 46;             // descriptor version
    d |= (uint64_t)2 << 61;             // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16: f32 accumulator, A/B f16 (0) or bf16 (1),
// both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t ab_fmt, uint32_t M, uint32_t N) {
    return (1u << 4) | (ab_fmt << 7) | (ab_fmt << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

W4_DEV void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

W4_DEV void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 consecutive accumulator columns of the warp's 32 TMEM lanes.
W4_DEV void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Bounded wait that also ends as soon as another role has aborted.
W4_DEV bool wait_or_abort(uint64_t *bar, uint32_t parity, Smem *sh, uint32_t *status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile int *>(&sh->abort)) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(status, kStatusPipeTimeout);
            *reinterpret_cast<volatile int *>(&sh->abort) = 1;
            return false;
        }
    }
}

// ---------------------------------------------------------------- weight conversion

// 8 packed signed nibbles (columns c..c+7) -> 8 bf16 = bf16_rne(q * s), as 16 bytes.
// u' = u ^ 8 = q + 8 of each nibble goes under the exponent byte 0x4B by one
// PRMT (the float 2^23 + u', exact); q * s = (that - (2^23 + 8)) * s is
// exact in f32, formed two columns at a time with packed f32x2 arithmetic,
// and rounded once to bf16.
W4_DEV uint4 conv_w4a16(uint32_t w, float s) {
    const uint32_t v = w ^ 0x88888888u;
    const uint32_t lo = v & 0x0F0F0F0Fu, hi = (v >> 4) & 0x0F0F0F0Fu;
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t fl = prmt(lo, 0x4B000000u, 0x7540u | e), fh = prmt(hi, 0x4B000000u, 0x7540u | e);
        asm("{\n\t.reg .b64 v, c, m, r;\n\t.reg .f32 r0, r1;\n\t"
            "mov.b64 v, {%1, %2};\n\t"
            "mov.b64 c, {%3, %3};\n\t"
            "mov.b64 m, {%4, %4};\n\t"
            "add.rn.f32x2 r, v, c;\n\t"
            "mul.rn.f32x2 r, r, m;\n\t"
            "mov.b64 {r0, r1}, r;\n\t"
            "cvt.rn.bf16x2.f32 %0, r1, r0;\n\t}"
            : "=r"(o[e])
            : "r"(fl), "r"(fh), "f"(-8388616.0f), "f"(s));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// W4A8G: 8 packed nibbles (columns c..c+7) -> 8 f16 = f16_rne((u - z) * s):
// (u - z) * s is exact in f32 and rounded once to f16.
W4_DEV uint4 conv_w4a8g(uint32_t w, float s, float zb) {
    // zb = 2^23 + z: (2^23 + u) - (2^23 + z) = u - z exactly
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t lo = (w >> (8 * e)) & 0xFu, hi = (w >> (8 * e + 4)) & 0xFu;
        const float ql = __int_as_float(0x4B000000 | lo) - zb;
        const float qh = __int_as_float(0x4B000000 | hi) - zb;
        __half2 h = __floats2half2_rn(ql * s, qh * s);
        o[e] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// 8 packed biased nibbles -> 8 f16 of q = u - 8 (exact), natural column order.
W4_DEV uint4 conv_w4a8(uint32_t w) {
    const __half2 mul = __halves2half2(__float2half(1.0f), __float2half(0.0625f));
    const __half2 add = __halves2half2(__float2half(-1032.0f), __float2half(-72.0f));
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        // byte e in both halves: low half 0x6400 | lo = 1024 + lo, high half 0x6400 | (hi << 4) = 1024 + 16 hi
        const uint32_t t = prmt(w, 0u, 0x4040u | ((uint32_t)e * 0x0101u));
        const uint32_t v = (t & 0x00F0000Fu) | 0x64006400u;
        __half2 h = __hfma2(*reinterpret_cast<const __half2 *>(&v), mul, add);
        o[e] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// 8 int8 (two words) -> 8 bf16 of the same integers (exact), natural order.
W4_DEV uint4 conv_w8a16(uint32_t lo, uint32_t hi) {
    const uint32_t wd[2] = {lo, hi};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t w = wd[e >> 1];
        const int a = (int)(int8_t)((w >> (16 * (e & 1))) & 0xFFu);
        const int b = (int)(int8_t)((w >> (16 * (e & 1) + 8)) & 0xFFu);
        __nv_bfloat162 h = __floats2bfloat162_rn((float)a, (float)b);
        o[e] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// 8 int8 (two words) -> 8 f16 of the same integers, natural order.
W4_DEV uint4 conv_w8a8(uint32_t lo, uint32_t hi) {
    const __half2 off = __halves2half2(__ushort_as_half((unsigned short)0x6480), __ushort_as_half((unsigned short)0x6480));
    lo ^= 0x80808080u;
    hi ^= 0x80808080u;
    const uint32_t sel[4] = {0x0100u, 0x0302u, 0x0504u, 0x0706u};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t v = (prmt(lo, hi, sel[e]) & 0x00FF00FFu) | 0x64006400u;
        __half2 h = __hsub2(*reinterpret_cast<const __half2 *>(&v), off);
        o[e] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// ---------------------------------------------------------------- kernel

// IL: the weights are in the interleaved [N/64][K][32 B] layout (vllm-omni
// "The 4-bit CPU path"): the TMA brings two 64-channel blocks x 64 columns
// per stage (the same 4 KB as the row-major tile) and the converters undo
// the interleave with 4x4 byte transposes before the same dequantisation.
template <int KIND, bool IL>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
    constexpr bool kW4 = KIND != KIND_W8A8 && KIND != KIND_W8A16;
    static_assert(!IL || kW4, "the interleaved layout holds int4 only");
    constexpr int kPRow = kW4 ? 32 : 64;             // packed bytes per weight row per stage
    constexpr int kATile = kBM * 128;                // 16 KB
    constexpr int kBTile = kBN * 128;                // 32 KB
    constexpr int kPTile = kBM * kPRow;              // 4 | 8 KB
    constexpr uint32_t kSTile = kBM * 16;                // 2 KB: 8 f16 group scales per weight row
    constexpr uint32_t kIdesc = idesc_f16((KIND == KIND_W4A16 || KIND == KIND_W8A16) ? 1u : 0u, kBM, kBN);

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Smem *sh = reinterpret_cast<Smem *>(smem);
    uint8_t *a_tiles = smem + 1024;
    uint8_t *b_tiles = a_tiles + kStages * kATile;
    uint8_t *p_tiles = b_tiles + kStages * kBTile;
    uint8_t *s_tiles = p_tiles + kStages * kPTile;  // s_tma: [stage][128 rows][8 f16 scales]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // this CTA's tiles: blockIdx.x, blockIdx.x + gridDim.x, ...; tile t -> (n-tile t % ntn, m-tile t / ntn)
    const int my_tiles = blockIdx.x < (unsigned)p.ntiles ? (p.ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    auto tile_of = [&](int i, int &m0, int &n0) {
        const int t = (int)blockIdx.x + i * (int)gridDim.x;
        n0 = (t % p.ntn) * kBM;
        m0 = (t / p.ntn) * kBN;
    };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sh->tma_full[s], 1);
            mbar_init(&sh->w_full[s], 1);
            mbar_init(&sh->conv_full[s], 32 * kConvWarps);
            mbar_init(&sh->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh->acc_full[b], 1);
            mbar_init(&sh->acc_empty[b], kEpiWarps);
        }
        sh->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&sh->tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    const int total = my_tiles * p.nk;  // stages this CTA runs (the pipeline spans tiles)

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            for (int g = 0; g < total; ++g) {
                const int s = g % kStages, kb = g % p.nk;
                int m0, n0;
                tile_of(g / p.nk, m0, n0);
                if (g >= kStages && !wait_or_abort(&sh->empty[s], ((g / kStages) - 1) & 1, sh, p.status)) break;
                // the weights first: the converters need them before the MMA needs the activations
                mbar_arrive_expect_tx(&sh->w_full[s], kPTile + (p.s_tma ? kSTile : 0u));
                if constexpr (IL) tma_load_3d(p_tiles + s * kPTile, &p.wmap, 0, kb * kBK, n0 / 64, &sh->w_full[s]);
                else tma_load_2d(p_tiles + s * kPTile, &p.wmap, kb * kPRow, n0, &sh->w_full[s]);
                if (p.s_tma)
                    tma_load_2d(s_tiles + s * kSTile, &p.smap, (kb * kBK / p.G) & ~7, n0, &sh->w_full[s]);
                mbar_arrive_expect_tx(&sh->tma_full[s], kBTile);
                tma_load_2d(b_tiles + s * kBTile, &p.xmap, kb * kBK, m0, &sh->tma_full[s]);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            bool ok = true;
            int g = 0;
            for (int i = 0; i < my_tiles && ok; ++i) {
                const int b = i & 1;
                if (i >= 2) ok = wait_or_abort(&sh->acc_empty[b], ((i >> 1) - 1) & 1, sh, p.status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)(kBN * b);
                for (int kb = 0; kb < p.nk; ++kb, ++g) {
                    const int s = g % kStages;
                    const uint32_t ph = (g / kStages) & 1;
                    ok = wait_or_abort(&sh->tma_full[s], ph, sh, p.status) &&
                         wait_or_abort(&sh->conv_full[s], ph, sh, p.status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(a_tiles + s * kATile);
                    const uint32_t b_addr = smem_u32(b_tiles + s * kBTile);
#pragma unroll
                    for (int j = 0; j < kBK / 16; ++j)  // 16 columns (32 bytes) per MMA
                        umma_f16(acc, smem_desc_sw128(a_addr + 32 * j), smem_desc_sw128(b_addr + 32 * j), kIdesc,
                                 (kb > 0 || j > 0) ? 1u : 0u);
                    umma_commit(&sh->empty[s]);
                }
                if (ok) umma_commit(&sh->acc_full[b]);
            }
        }
    } else if (warp < 2 + kConvWarps && IL) {
        // ---------------- weight conversion from the interleaved layout (256 threads)
        // Thread: 64-channel block ib, 8-column group k8 of the stage, channel
        // quad dq, low (channels 4dq+c) or high (4dq+c+32) half: four rows of A.
        const int ct = tid - 64;
        const int ib = ct >> 7, r = ct & 127, k8 = r >> 4, dq = (r >> 1) & 7, sel = r & 1;
        // W4A16 scales of the four rows at this thread's columns, cached per
        // (tile, group) and fetched one stage ahead (G % 32 == 0: one group per 8 columns)
        float s_cur[4] = {0.f, 0.f, 0.f, 0.f}, s_nxt[4] = {0.f, 0.f, 0.f, 0.f};
        int key_last = -1;
        auto load_il_scales = [&](int g, float (&dst)[4]) {
            if constexpr (KIND == KIND_W4A16) {
                int m0, n0;
                tile_of(g / p.nk, m0, n0);
                const int col = (g % p.nk) * kBK + 8 * k8, grp = col / p.G;
                const int key = (g / p.nk) * p.ng + grp;
                if (key != key_last) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int n = n0 + 64 * ib + 4 * dq + c + 32 * sel;
                        dst[c] = (n < p.N && col < p.K)
                                     ? __half2float(__ushort_as_half(__ldg(p.scales + (size_t)n * p.ng + grp)))
                                     : 0.0f;
                    }
                    key_last = key;
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) dst[c] = s_cur[c];
                }
            }
        };
        if (total > 0) {
            key_last = -1;
            load_il_scales(0, s_cur);
        }
        for (int g = 0; g < total; ++g) {
            const int s = g % kStages;
            if (g + 1 < total) load_il_scales(g + 1, s_nxt);
            if (!wait_or_abort(&sh->w_full[s], (g / kStages) & 1, sh, p.status)) break;
            uint32_t lo[4], hi[4];
            deinterleave8(p_tiles + s * kPTile + ib * 2048 + k8 * 8 * 32, dq, lo, hi);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int row = 64 * ib + 4 * dq + c + 32 * sel, rr = row & 7;
                const uint32_t wd = sel ? hi[c] : lo[c];
                uint4 v;
                if constexpr (KIND == KIND_W4A16) v = conv_w4a16(wd, s_cur[c]);
                else v = conv_w4a8(wd);
                *reinterpret_cast<uint4 *>(a_tiles + s * kATile + (row >> 3) * 1024 + rr * 128 + ((k8 ^ rr) << 4)) = v;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(&sh->conv_full[s]);
#pragma unroll
            for (int c = 0; c < 4; ++c) s_cur[c] = s_nxt[c];
        }
    } else if (warp < 2 + kConvWarps) {
        // ---------------- weight conversion, row-major layout (256 threads)
        const int ct = tid - 64;
        const int row = ct & (kBM - 1), half = ct >> 7;  // row of the tile, columns [32 half, 32 half + 32)
        const int rr = row & 7;
        uint8_t *a_row = a_tiles + (row >> 3) * 1024 + rr * 128;
        // W4A16 group scales of this thread's 4 chunks, fetched one stage
        // ahead.  The chunks of a thread share a group when G >= 32 and
        // consecutive stages share it when G > 64: each distinct scale is
        // loaded once (these row-strided loads cost a sector lookup per lane).
        float sc_cur[4] = {0.f, 0.f, 0.f, 0.f}, sc_nxt[4] = {0.f, 0.f, 0.f, 0.f};
        float zb_cur = 8388608.0f, zb_nxt = 8388608.0f;  // W4A8G: 2^23 + zero point of the thread's group
        int grp_last = -1, n_last = -1;
        float s_last = 0.0f, zb_last = 8388608.0f;
        auto load_scales = [&](int g, float (&dst)[4]) {
            if constexpr (KIND == KIND_W4A16 || KIND == KIND_W4A8G) {
                int m0, n0;
                tile_of(g / p.nk, m0, n0);
                const int n = n0 + row, kb = g % p.nk;
                const int kc0 = kb * kBK + 8 * (4 * half), kc3 = kc0 + 24;
                if (kc0 / p.G == kc3 / p.G) {
                    const int grp = kc0 / p.G;
                    if (grp != grp_last || n != n_last) {
                        const bool in = n < p.N && kc0 < p.K;
                        s_last = in ? __half2float(__ushort_as_half(__ldg(p.scales + (size_t)n * p.ng + grp))) : 0.0f;
                        if constexpr (KIND == KIND_W4A8G)
                            zb_last = 8388608.0f + (in ? (float)__ldg(p.zeros + (size_t)n * p.ng + grp) : 0.0f);
                        grp_last = grp;
                        n_last = n;
                    }
                    zb_nxt = zb_last;
#pragma unroll
                    for (int c = 0; c < 4; ++c) dst[c] = (kc0 + 8 * c < p.K) ? s_last : 0.0f;
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int kcol = kc0 + 8 * c;
                        dst[c] = (n < p.N && kcol < p.K)
                                     ? __half2float(__ushort_as_half(__ldg(p.scales + (size_t)n * p.ng + kcol / p.G)))
                                     : 0.0f;
                    }
                    grp_last = -1;
                }
            }
        };
        if (total > 0 && !p.s_tma) load_scales(0, sc_cur);
        zb_cur = zb_nxt;
        for (int g = 0; g < total; ++g) {
            const int s = g % kStages;
            if (g + 1 < total && !p.s_tma) load_scales(g + 1, sc_nxt);
            if (!wait_or_abort(&sh->w_full[s], (g / kStages) & 1, sh, p.status)) break;
            if (KIND == KIND_W4A16 && p.s_tma) {
                // the stage's scales came with its weights: one group for the thread's
                // 32 columns (G is a multiple of 32), at its place in the 8-group box
                const int c0 = (g % p.nk) * kBK;
                const int gi = (c0 + 32 * half) / p.G - ((c0 / p.G) & ~7);
                const float sv = __half2float(__ushort_as_half(
                    *reinterpret_cast<const uint16_t *>(s_tiles + s * kSTile + row * 16 + 2 * gi)));
#pragma unroll
                for (int c = 0; c < 4; ++c) sc_cur[c] = sv;
            }
            const uint8_t *prow = p_tiles + s * kPTile + row * kPRow;
            uint8_t *arow = a_row + s * kATile;
            if constexpr (!kW4) {
                const uint4 q0 = *reinterpret_cast<const uint4 *>(prow + 32 * half);
                const uint4 q1 = *reinterpret_cast<const uint4 *>(prow + 32 * half + 16);
                const uint32_t wds[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int chunk = 4 * half + c;
                    *reinterpret_cast<uint4 *>(arow + ((chunk ^ rr) << 4)) =
                        KIND == KIND_W8A16 ? conv_w8a16(wds[2 * c], wds[2 * c + 1]) : conv_w8a8(wds[2 * c], wds[2 * c + 1]);
                }
            } else {
                const uint4 pk = *reinterpret_cast<const uint4 *>(prow + 16 * half);
                const uint32_t wds[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int chunk = 4 * half + c;  // columns kb*64 + 8*chunk .. +7
                    uint4 v;
                    if constexpr (KIND == KIND_W4A16) {
                        v = conv_w4a16(wds[c], sc_cur[c]);
                    } else if constexpr (KIND == KIND_W4A8G) {
                        v = conv_w4a8g(wds[c], sc_cur[c], zb_cur);
                    } else {
                        v = conv_w4a8(wds[c]);
                    }
                    *reinterpret_cast<uint4 *>(arow + ((chunk ^ rr) << 4)) = v;
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(&sh->conv_full[s]);
#pragma unroll
            for (int c = 0; c < 4; ++c) sc_cur[c] = sc_nxt[c];
            zb_cur = zb_nxt;
        }
    } else {
        // ---------------- epilogue (warps 2 + kConvWarps ..): TMEM -> registers -> y
        const int q = warp & 3;                         // TMEM lane quadrant this warp may access
        const int hc = (warp - 2 - kConvWarps) >> 2;    // column half
        for (int i = 0; i < my_tiles; ++i) {
            const int b = i & 1;
            int m0, n0;
            tile_of(i, m0, n0);
            // the tile's scales, loaded while its accumulator is still being formed
            const int nrow = n0 + 32 * q + lane;
            float swn = 1.0f;
            if constexpr (KIND == KIND_W4A8 || KIND == KIND_W8A8 || KIND == KIND_W8A16)
                swn = (nrow < p.N) ? p.sw[nrow] : 0.0f;
            float sx_pre[kBN / 64];
#pragma unroll
            for (int cc = 0; cc < kBN / 64; ++cc) {
                const int mm = m0 + (kBN / 2) * hc + 32 * cc + lane;
                sx_pre[cc] = 0.0f;
                if constexpr (KIND != KIND_W4A16 && KIND != KIND_W8A16) sx_pre[cc] = mm < p.M ? p.sx[mm] : 0.0f;
            }
            bool ok = wait_or_abort(&sh->acc_full[b], (i >> 1) & 1, sh, p.status);
            ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld is warp-collective
            if (!ok) break;
            tc_fence_after();
#pragma unroll 1
            for (int cc = 0; cc < kBN / 64; ++cc) {
                const int col0 = (kBN / 2) * hc + 32 * cc;
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(kBN * b + col0), v);
                if (cc == kBN / 64 - 1) {
                    // the accumulator is in registers: the MMA warp may reuse it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh->acc_empty[b]);
                }
                // sx of the chunk's 32 activation rows (loaded above), then shuffles
                static_assert(kBN / 64 == 4, "four 32-column chunks per epilogue warp");
                const float sxl = cc == 0 ? sx_pre[0] : cc == 1 ? sx_pre[1] : cc == 2 ? sx_pre[2] : sx_pre[3];
#pragma unroll
                for (int j = 0; j < 32; ++j) {  // every lane takes part in the shuffles
                    const int m = m0 + col0 + j;
                    float out = __uint_as_float(v[j]);
                    if constexpr (KIND == KIND_W4A8G)
                        out = __fmul_rn(out, __shfl_sync(0xffffffffu, sxl, j));  // sx * sum_g acc_g * s_g
                    else if constexpr (KIND == KIND_W8A16)
                        out = __fmul_rn(out, swn);  // sw * sum x q
                    else if constexpr (KIND != KIND_W4A16)
                        out = __fmul_rn(__fmul_rn(out, __shfl_sync(0xffffffffu, sxl, j)), swn);
                    // streaming store: y is written once, the operand tiles stay in L2
                    if (nrow < p.N && m < p.M) __stcs(p.y + (size_t)m * p.N + nrow, out);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// int8 codes [M][K] -> f16 [M][Kx] (Kx = K rounded up to 8, zero padded): exact.
__global__ void s8_to_f16_kernel(const int8_t *__restrict__ x, uint16_t *__restrict__ out, int64_t M, int64_t K,
                                 int64_t Kx) {
    const int64_t groups = M * (Kx / 8);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < groups; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / (Kx / 8), k = (i - m * (Kx / 8)) * 8;
        uint16_t h[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int v = (k + e < K) ? (int)x[m * K + k + e] : 0;
            h[e] = __half_as_ushort(__int2half_rn(v));
        }
        *reinterpret_cast<uint4 *>(out + m * Kx + k) =
            make_uint4(h[0] | ((uint32_t)h[1] << 16), h[2] | ((uint32_t)h[3] << 16), h[4] | ((uint32_t)h[5] << 16),
                       h[6] | ((uint32_t)h[7] << 16));
    }
}

// f32 activations [M][K] -> bf16 [M][Kx] (round to nearest even, zero padded).
__global__ void f32_to_bf16_kernel(const float *__restrict__ x, uint16_t *__restrict__ out, int64_t M, int64_t K,
                                   int64_t Kx) {
    const int64_t groups = M * (Kx / 8);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < groups; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / (Kx / 8), k = (i - m * (Kx / 8)) * 8;
        uint32_t h[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float a = (k + 2 * e < K) ? x[m * K + k + 2 * e] : 0.0f;
            const float b = (k + 2 * e + 1 < K) ? x[m * K + k + 2 * e + 1] : 0.0f;
            __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
            h[e] = *reinterpret_cast<uint32_t *>(&v);
        }
        *reinterpret_cast<uint4 *>(out + m * Kx + k) = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

constexpr int smem_bytes(int kind) {
    return 1024 +
           kStages * (kBM * 128 + kBN * 128 + kBM * ((kind == KIND_W8A8 || kind == KIND_W8A16) ? 64 : 32) +
                      (kind == KIND_W4A16 ? kBM * 16 : 0)) +
           1024;
}

template <int KIND, bool IL>
cudaError_t launch_kernel(const GemmParams &p, cudaStream_t st) {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(gemm_kernel<KIND, IL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    smem_bytes(KIND));
    });
    if (attr != cudaSuccess) return attr;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int grid = std::max(1, std::min(p.ntiles, sms));  // one persistent CTA per SM
    gemm_kernel<KIND, IL><<<grid, kThreads, smem_bytes(KIND), st>>>(p);
    return cudaGetLastError();
}

int64_t kx_of(int64_t K) { return round_up(K, 8); }

}  // namespace

bool gemm_supported(const LinearArgs &a) {
    if (a.M <= 16) return false;
    if (a.layout == W4_LAYOUT_B32) return false;  // inline-scale blocks: 16-row decode slices
    if (a.N > 0x7FFFFFFF || a.M > 0x7FFFFFFF) return false;
    if (reinterpret_cast<uintptr_t>(a.w) % 16) return false;
    if (a.kind == KIND_W4A8G && (a.layout != W4_LAYOUT_ROWMAJOR || a.G % 32)) return false;
    if (a.layout == W4_LAYOUT_N64) {
        // [N/64][K][32 B]: rows of 32 bytes, any K; W4A16 groups of whole 32-column chunks
        if (a.kind == KIND_W8A8 || a.kind == KIND_W8A16 || a.N % 64) return false;
        if (a.kind == KIND_W4A16 && a.G % 32) return false;
    } else {
        const int64_t Kb = (a.kind == KIND_W8A8 || a.kind == KIND_W8A16) ? a.K : (a.K + 1) / 2;
        if (Kb % 16) return false;  // TMA row stride
    }
    if (a.kind == KIND_W4A16) {
        if (a.K % 8 || a.G % 8) return false;  // bf16 rows for TMA; one scale per 8 columns
        if (reinterpret_cast<uintptr_t>(a.x) % 16) return false;
    } else if (a.kind == KIND_W4A8 || a.kind == KIND_W8A8) {
        // exact integer accumulation in f32 needs 127 * max|q| * K < 2^24
        if (a.K > (a.kind == KIND_W4A8 ? 16384 : 1024)) return false;
    }
    return true;
}

size_t gemm_workspace_bytes(int kind, int64_t M, int64_t N, int64_t K, int64_t G) {
    (void)N;
    (void)G;
    if (kind == KIND_W4A16 || M <= 16) return 0;
    return (size_t)(M * kx_of(K) * 2);
}

cudaError_t launch_gemm(const LinearArgs &a, cudaStream_t st) {
    GemmParams p = {};
    p.M = (int)a.M;
    p.N = (int)a.N;
    p.K = (int)a.K;
    p.G = (int)a.G;
    p.ng = (a.kind == KIND_W4A16 || a.kind == KIND_W4A8G) ? (int)((a.K + (a.K & 1)) / a.G) : 0;
    p.zeros = a.zeros;
    p.y = a.y;
    p.status = a.status;
    p.scales = static_cast<const uint16_t *>(a.scale);
    p.sx = a.sx;
    p.sw = static_cast<const float *>(a.scale);
    const void *xsrc = a.x;
    int64_t Kx = a.K;
    if (a.kind != KIND_W4A16) {
        // exact f16 images of the int8 activation codes, in the caller's workspace
        Kx = kx_of(a.K);
        const size_t need = (size_t)(a.M * Kx * 2);
        if (!a.workspace || a.ws_bytes < need) return cudaErrorInvalidValue;
        const int64_t groups = a.M * (Kx / 8);
        const int64_t blocks = std::min<int64_t>(ceil_div(groups, 256), 152 * 8);
        if (a.x16_ready)  // the row quantizer already wrote the f16 image
            ;
        else if (a.kind == KIND_W8A16)  // f32 activations -> bf16 (the prefill's one rounding of x)
            f32_to_bf16_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const float *>(a.x),
                                                                 static_cast<uint16_t *>(a.workspace), a.M, a.K, Kx);
        else
            s8_to_f16_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const int8_t *>(a.x),
                                                               static_cast<uint16_t *>(a.workspace), a.M, a.K, Kx);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        xsrc = a.workspace;
    }
    p.nk = (int)ceil_div(Kx, kBK);
    p.ntn = (int)ceil_div(a.N, kBM);
    p.ntiles = p.ntn * (int)ceil_div(a.M, kBN);
    {
        const uint64_t dims[2] = {(uint64_t)Kx, (uint64_t)a.M};
        const uint64_t strides[1] = {(uint64_t)Kx * 2};
        const uint32_t box[2] = {(uint32_t)kBK, (uint32_t)kBN};
        if (!encode_tmap(&p.xmap, (a.kind == KIND_W4A16 || a.kind == KIND_W8A16) ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                         2, xsrc, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    const bool il = a.layout == W4_LAYOUT_N64;
    if (il) {
        // [N/64][K][32 B] as a 3-D tensor: box of 32 bytes x 64 columns x 2 blocks (128 channels)
        const uint64_t dims[3] = {32, (uint64_t)a.K, (uint64_t)(a.N / 64)};
        const uint64_t strides[2] = {32, (uint64_t)a.K * 32};
        const uint32_t box[3] = {32, (uint32_t)kBK, (uint32_t)(kBM / 64)};
        if (!encode_tmap(&p.wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.w, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else {
        const bool w8 = a.kind == KIND_W8A8 || a.kind == KIND_W8A16;
        const int64_t Kb = w8 ? a.K : (a.K + 1) / 2;
        const uint64_t dims[2] = {(uint64_t)Kb, (uint64_t)a.N};
        const uint64_t strides[1] = {(uint64_t)Kb};
        const uint32_t box[2] = {(uint32_t)(w8 ? 64 : 32), (uint32_t)kBM};
        if (!encode_tmap(&p.wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.w, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    // W4A16 row-major: each stage's group scales by TMA beside its weights
    // (8 groups x 128 rows per box; rows of whole 16-byte multiples).
    p.s_tma = 0;
    if (a.kind == KIND_W4A16 && !il && a.G % 32 == 0 && p.ng % 8 == 0 &&
        reinterpret_cast<uintptr_t>(a.scale) % 16 == 0) {
        const uint64_t dims[2] = {(uint64_t)p.ng, (uint64_t)a.N};
        const uint64_t strides[1] = {(uint64_t)p.ng * 2};
        const uint32_t box[2] = {8, (uint32_t)kBM};
        if (!encode_tmap(&p.smap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, a.scale, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
        p.s_tma = 1;
    }
    switch (a.kind) {
        case KIND_W4A16: return il ? launch_kernel<KIND_W4A16, true>(p, st) : launch_kernel<KIND_W4A16, false>(p, st);
        case KIND_W4A8: return il ? launch_kernel<KIND_W4A8, true>(p, st) : launch_kernel<KIND_W4A8, false>(p, st);
        case KIND_W4A8G: return launch_kernel<KIND_W4A8G, false>(p, st);
        case KIND_W8A16: return launch_kernel<KIND_W8A16, false>(p, st);
        default: return launch_kernel<KIND_W8A8, false>(p, st);
    }
}

}  // namespace w4
