// common.cuh -- device helpers shared by the kernels of libw4gb300 (sm_103a).
//
// Inline-PTX wrappers for the Blackwell memory path used by the kernels:
// mbarriers with transaction counts, bulk async global->shared copies,
// programmatic dependent launch, cluster barriers and distributed shared
// memory, and a bounded wait built on %globaltimer.  Every wait in the
// library has a time limit; a wait that runs out sets a bit in the caller's
// status word and the kernel returns without touching its outputs.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#define W4_DEV __device__ __forceinline__
#define W4_HD __host__ __device__ __forceinline__

namespace w4 {

// Status-word bits (mirrored in include/w4.h, w4_device_status).
constexpr uint32_t kStatusCopyTimeout = 1u;
constexpr uint32_t kStatusPipeTimeout = 2u;
constexpr uint32_t kStatusBarrierTimeout = 4u;

// Bounded waits give up after this many nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

W4_DEV uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

W4_DEV uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier

W4_DEV void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async proxy and the cluster.
W4_DEV void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

W4_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

W4_DEV void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

W4_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete; false after the limit.
W4_DEV bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------- bulk copy

// 1-D bulk async copy global -> this CTA's shared memory, completing `bytes`
// transactions on `bar`.  dst, src 16-byte aligned; bytes a multiple of 16.
W4_DEV void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 2-D tiled TMA load of box (c0, c1) of `map` into shared memory, completing
// the box's bytes on `bar`.  c0 * element size must be a multiple of 16.
W4_DEV void tma_load_2d(void *dst, const void *map, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// 3-D tiled TMA load of box (c0, c1, c2); c0 * element size must be a multiple of 16.
W4_DEV void tma_load_3d(void *dst, const void *map, int c0, int c1, int c2, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// Bulk prefetch of [src, src + bytes) from global memory into L2 (a hint:
// nothing is written to shared memory).  src 16-byte aligned, bytes a
// multiple of 16.
W4_DEV void prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 16 bytes from global memory through L2 only (not cached in L1).
W4_DEV uint4 ldg_cg_u128(const void *p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ---------------------------------------------------------------- PDL

W4_DEV void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
W4_DEV void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- cluster

W4_DEV uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

W4_DEV void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
W4_DEV uint32_t dsmem_map(const void *p, uint32_t rank) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
    return out;
}

W4_DEV uint32_t dsmem_ld_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// ---------------------------------------------------------------- misc

W4_DEV uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

W4_DEV uint32_t lds_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

W4_DEV uint2 lds_u64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

W4_DEV uint4 lds_u128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// 4x4 byte transpose + nibble repack of the interleaved layout: raw rows
// [k][32 B] (byte d = channel d | channel d+32 << 4) of 8 consecutive k for
// channels 4*dq..4*dq+3 -> one packed row-major word (8 nibbles, low first)
// for each of the channels 4*dq+c (lo[c]) and 4*dq+c+32 (hi[c]).
// The same, from the 8 words (bytes 4dq..4dq+3 of the 8 rows) already in registers.
W4_DEV void deinterleave8_words(const uint32_t (&v)[8], uint32_t (&lo)[4], uint32_t (&hi)[4]) {
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
        lo[c] = prmt(la | (la >> 4), lb | (lb >> 4), 0x6420);
        hi[c] = prmt(ha | (ha >> 4), hb | (hb >> 4), 0x6420);
    }
}

W4_DEV void deinterleave8(const uint8_t *raw, int dq, uint32_t (&lo)[4], uint32_t (&hi)[4]) {
    uint32_t v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = *reinterpret_cast<const uint32_t *>(raw + i * 32 + 4 * dq);
    deinterleave8_words(v, lo, hi);
}

W4_HD int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
W4_HD int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

}  // namespace w4
