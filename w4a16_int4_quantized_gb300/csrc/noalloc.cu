// noalloc.cu -- w4_linear_q4_noalloc: the W4A8 linear for callers that may not
// allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) once they are
// running: a serving process that reserves its whole memory budget at start
// and treats any later allocation as a failure, a host framework whose own
// allocator owns the device and must not be bypassed, or a latency-critical
// loop where an allocation could block or fragment memory.  w4_linear_q4
// needs caller-provided device scratch for large batches (the f16 copy of the
// activation codes that feeds the tensor cores); this entry point uses a
// fixed scratch array that lives in the library's device image instead.
//
// The array is a file-scope static __device__ object of W4_NOALLOC_SCRATCH_BYTES
// bytes: every GPU that loads the library holds it until the process exits.
// Host code cannot use the array's name as a device address (it names a
// host-side stand-in), so the first call on each device resolves the real
// address with cudaGetSymbolAddress while that device is current, checks the
// result, and caches it per device.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "internal.h"
#include "w4.h"

namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[W4_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device, resolved once per device.
cudaError_t scratch_address(void **out) {
    constexpr int kMaxDev = 64;
    static std::atomic<void *> cache[kMaxDev];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    void *p = cache[dev].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lk(mu);
        p = cache[dev].load(std::memory_order_relaxed);
        if (!p) {
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess) return e;
            cache[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" w4_status w4_linear_q4_noalloc(const int8_t *xq, const float *sx, const uint8_t *w, const float *sw,
                                          float *y, int64_t M, int64_t N, int64_t K, int32_t layout, void *stream) {
    // w4_linear_q4's own argument checks come first, so an invalid call gets
    // the same error from both entry points; the scratch size is computed
    // only for arguments inside those limits.
    if (M < 0 || N < 0 || K < 0) return W4_EINVAL;
    if (layout != W4_LAYOUT_ROWMAJOR && layout != W4_LAYOUT_N64) return W4_EINVAL;
    if (K > 1000000 || M >= ((int64_t)1 << 31) || N >= ((int64_t)1 << 31)) return W4_ESHAPE;
    if (layout == W4_LAYOUT_N64 && N % 64) return W4_ESHAPE;
    if (M == 0 || N == 0) return W4_OK;
    if (!y || !sx || !sw || (K > 0 && (!xq || !w))) return W4_EINVAL;
    const size_t need = w4_workspace_bytes(W4_OP_LINEAR_Q4, M, N, K, 0);
    if (need > (size_t)W4_NOALLOC_SCRATCH_BYTES) return W4_ESHAPE;  // batch too large for the fixed scratch
    void *scratch = nullptr;
    if (need > 0) {
        const cudaError_t e = scratch_address(&scratch);
        if (e != cudaSuccess) return w4::record_cuda_error(e);
    }
    // The prepass writes every byte of the scratch it uses (zero padding
    // included) before the GEMM reads it, so nothing has to start at zero.
    return w4_linear_q4(xq, sx, w, sw, y, M, N, K, layout, scratch, need > 0 ? (size_t)W4_NOALLOC_SCRATCH_BYTES : 0,
                        0u, stream);
}
