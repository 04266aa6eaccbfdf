// capi.cu -- the extern "C" boundary of libw4gb300 (declared in include/w4.h).
//
// Host-side validation happens here, before anything is launched or read,
// in the order the header documents; then each call is routed to one CUDA
// path: the quantizers, the decode GEMV (M <= 16), the tcgen05 prefill GEMM
// (M > 16, shapes it can tile) or the generic kernel (anything else).  There
// is no CPU fallback: every result comes from a kernel.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "w4.h"
#include "common.cuh"
#include "internal.h"

namespace {

__device__ uint32_t g_status_word;

thread_local int32_t t_last_cuda_error = 0;

w4_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return W4_OK;
    t_last_cuda_error = (int32_t)e;
    return W4_ECUDA;
}

// Device address of the status word on the current device (resolved once per device).
cudaError_t status_ptr(uint32_t **out) {
    constexpr int kMaxDev = 64;
    static std::atomic<uint32_t *> cache[kMaxDev];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    uint32_t *p = cache[dev].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lk(mu);
        p = cache[dev].load(std::memory_order_relaxed);
        if (!p) {
            void *addr = nullptr;
            e = cudaGetSymbolAddress(&addr, g_status_word);
            if (e != cudaSuccess) return e;
            p = static_cast<uint32_t *>(addr);
            cache[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return cudaSuccess;
}

inline cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

constexpr int64_t kMaxKQ4 = 1000000;        // |sum xq*u| < 2^31 needs K <= 1,127,288
constexpr int64_t kMaxKQ8 = 131072;         // |sum xq*w| < 2^31 for any int8 weights needs K <= 133,144
constexpr int64_t kMaxKDot = 1127288;
constexpr int64_t kMaxDim = (int64_t)1 << 31;

w4_status run_linear(w4::LinearArgs &a, cudaStream_t st) {
    uint32_t *status = nullptr;
    cudaError_t e = status_ptr(&status);
    if (e != cudaSuccess) return cuda_status(e);
    a.status = status;
    if (a.M <= 16 && w4::gemv_supported(a)) return cuda_status(w4::launch_gemv(a, st));
    if (a.M > 16 && w4::gemm_supported(a)) return cuda_status(w4::launch_gemm(a, st));
    // M > 16 shapes the tensor-core GEMM does not take (interleaved layout,
    // odd K, W8A8 with K > 1024): slices of 16 activation rows through the
    // decode kernel, which handles them exactly.
    w4::LinearArgs s16 = a;
    s16.M = 16;
    if (a.M > 16 && w4::gemv_supported(s16)) {
        const size_t xrow = (size_t)a.K * (a.kind == w4::KIND_W4A16 ? 2 : a.kind == w4::KIND_W8A16 ? 4 : 1);
        for (int64_t m0 = 0; m0 < a.M; m0 += 16) {
            w4::LinearArgs sl = a;
            sl.M = std::min<int64_t>(16, a.M - m0);
            sl.x = static_cast<const uint8_t *>(a.x) + (size_t)m0 * xrow;
            sl.sx = a.sx ? a.sx + m0 : nullptr;
            sl.y = a.y + (size_t)m0 * a.N;
            sl.flags = 0;
            const cudaError_t e = w4::launch_gemv(sl, st);
            if (e != cudaSuccess) return cuda_status(e);
        }
        return W4_OK;
    }
    return cuda_status(w4::launch_generic(a, st));
}

w4_status check_workspace(int32_t op, int64_t M, int64_t N, int64_t K, int64_t G, void *ws, size_t ws_bytes) {
    const size_t need = w4_workspace_bytes(op, M, N, K, G);
    if (need > ws_bytes) return W4_EINVAL;
    if (need > 0 && ws == nullptr) return W4_EINVAL;
    return W4_OK;
}

}  // namespace

namespace w4 {
w4_status record_cuda_error(cudaError_t e) { return cuda_status(e); }
}  // namespace w4

extern "C" {

w4_status w4_quantize_row_q8(const float *x, int64_t M, int64_t K, int8_t *q, float *sx, int32_t *rowsum,
                             void *stream) {
    if (M < 0 || K < 0) return W4_EINVAL;
    if (M >= kMaxDim || K >= kMaxDim) return W4_ESHAPE;
    if (M == 0) return W4_OK;
    if (!sx || (K > 0 && (!x || !q))) return W4_EINVAL;
    return cuda_status(w4::launch_quantize_rows(x, M, K, 127, q, sx, rowsum, as_stream(stream)));
}

w4_status w4_quantize_matrix_q4(const float *W, int64_t N, int64_t K, uint8_t *packed, float *sw, void *stream) {
    if (N < 0 || K < 0) return W4_EINVAL;
    if (N >= kMaxDim || K >= kMaxDim) return W4_ESHAPE;
    if (N == 0) return W4_OK;
    if (!sw || (K > 0 && (!W || !packed))) return W4_EINVAL;
    return cuda_status(w4::launch_quantize_matrix_q4(W, N, K, packed, sw, as_stream(stream)));
}

w4_status w4_quantize_matrix_q8(const float *W, int64_t N, int64_t K, int8_t *q, float *sw, void *stream) {
    if (N < 0 || K < 0) return W4_EINVAL;
    if (N >= kMaxDim || K >= kMaxDim) return W4_ESHAPE;
    if (N == 0) return W4_OK;
    if (!sw || (K > 0 && (!W || !q))) return W4_EINVAL;
    return cuda_status(w4::launch_quantize_rows(W, N, K, 127, q, sw, nullptr, as_stream(stream)));
}

w4_status w4_dot_i32_q4(const int8_t *xq, const uint8_t *wrow, int64_t K, int32_t *out, void *stream) {
    if (K < 0) return W4_EINVAL;
    if (K > kMaxKDot) return W4_ESHAPE;
    if (!out || (K > 0 && (!xq || !wrow))) return W4_EINVAL;
    if (K == 0) return cuda_status(cudaMemsetAsync(out, 0, sizeof(int32_t), as_stream(stream)));
    return cuda_status(w4::launch_dot_i32_q4(xq, wrow, K, out, as_stream(stream)));
}

w4_status w4_linear_q4(const int8_t *xq, const float *sx, const uint8_t *w, const float *sw, float *y, int64_t M,
                       int64_t N, int64_t K, int32_t layout, void *workspace, size_t ws_bytes, uint32_t flags,
                       void *stream) {
    if (M < 0 || N < 0 || K < 0) return W4_EINVAL;
    if (layout != W4_LAYOUT_ROWMAJOR && layout != W4_LAYOUT_N64) return W4_EINVAL;
    if (K > kMaxKQ4 || M >= kMaxDim || N >= kMaxDim) return W4_ESHAPE;
    if (layout == W4_LAYOUT_N64 && N % 64) return W4_ESHAPE;
    if (M == 0 || N == 0) return W4_OK;
    if (!y || !sx || !sw || (K > 0 && (!xq || !w))) return W4_EINVAL;
    const w4_status ws = check_workspace(W4_OP_LINEAR_Q4, M, N, K, 0, workspace, ws_bytes);
    if (ws != W4_OK) return ws;
    if (K == 0) return cuda_status(cudaMemsetAsync(y, 0, (size_t)(M * N) * sizeof(float), as_stream(stream)));
    w4::LinearArgs a = {};
    a.kind = w4::KIND_W4A8;
    a.x = xq; a.w = w; a.scale = sw; a.sx = sx; a.y = y;
    a.M = M; a.N = N; a.K = K; a.G = 0; a.layout = layout; a.flags = flags;
    a.workspace = workspace; a.ws_bytes = ws_bytes;
    return run_linear(a, as_stream(stream));
}

w4_status w4_linear_q4_f32(const float *x, const uint8_t *w, const float *sw, float *y, int8_t *xq, float *sx,
                           int64_t M, int64_t N, int64_t K, int32_t layout, void *workspace, size_t ws_bytes,
                           uint32_t flags, void *stream) {
    if (M < 0 || N < 0 || K < 0) return W4_EINVAL;
    if (layout != W4_LAYOUT_ROWMAJOR && layout != W4_LAYOUT_N64) return W4_EINVAL;
    if (K > kMaxKQ4 || M >= kMaxDim || N >= kMaxDim) return W4_ESHAPE;
    if (layout == W4_LAYOUT_N64 && N % 64) return W4_ESHAPE;
    if (M == 0) return W4_OK;
    if (!sx || (K > 0 && (!x || !xq))) return W4_EINVAL;
    if (N > 0 && (!y || !sw || (K > 0 && !w))) return W4_EINVAL;
    const w4_status ws = check_workspace(W4_OP_LINEAR_Q4, M, N, K, 0, workspace, ws_bytes);
    if (ws != W4_OK) return ws;
    cudaStream_t st = as_stream(stream);
    w4::LinearArgs a = {};
    a.kind = w4::KIND_W4A8;
    a.x = xq; a.w = w; a.scale = sw; a.sx = sx; a.y = y;
    a.M = M; a.N = N; a.K = K; a.G = 0; a.layout = layout; a.flags = flags;
    a.workspace = workspace; a.ws_bytes = ws_bytes;
    if (N > 0 && K > 0 && M <= 8 && layout == W4_LAYOUT_ROWMAJOR && w4::gemv_supported(a)) {
        uint32_t *status = nullptr;
        const cudaError_t e = status_ptr(&status);
        if (e != cudaSuccess) return cuda_status(e);
        a.status = status;
        a.xf = x; a.xq_out = xq; a.sx_out = sx;
        return cuda_status(w4::launch_gemv(a, st));  // fused, or the quantizer then the linear
    }
    // Prefill on the tensor cores: one pass writes the codes, the scales and
    // the f16 image of the codes the GEMM reads (no separate prepass).
    if (N > 0 && K > 0 && M > 16 && K % 8 == 0 && w4::gemm_supported(a) &&
        reinterpret_cast<uintptr_t>(x) % 16 == 0 && reinterpret_cast<uintptr_t>(xq) % 4 == 0 &&
        reinterpret_cast<uintptr_t>(workspace) % 16 == 0) {
        const cudaError_t e = w4::launch_quantize_rows_f16(x, M, K, xq, sx, static_cast<uint16_t *>(workspace), st);
        if (e != cudaSuccess) return cuda_status(e);
        a.x16_ready = true;
        return run_linear(a, st);
    }
    const cudaError_t e = w4::launch_quantize_rows(x, M, K, 127, xq, sx, nullptr, st);
    if (e != cudaSuccess) return cuda_status(e);
    if (N == 0) return W4_OK;
    if (K == 0) return cuda_status(cudaMemsetAsync(y, 0, (size_t)(M * N) * sizeof(float), st));
    return run_linear(a, st);
}

w4_status w4_linear_q8(const int8_t *xq, const float *sx, const int8_t *w, const float *sw, float *y, int64_t M,
                       int64_t N, int64_t K, void *workspace, size_t ws_bytes, uint32_t flags, void *stream) {
    if (M < 0 || N < 0 || K < 0) return W4_EINVAL;
    if (K > kMaxKQ8 || M >= kMaxDim || N >= kMaxDim) return W4_ESHAPE;
    if (M == 0 || N == 0) return W4_OK;
    if (!y || !sx || !sw || (K > 0 && (!xq || !w))) return W4_EINVAL;
    const w4_status ws = check_workspace(W4_OP_LINEAR_Q8, M, N, K, 0, workspace, ws_bytes);
    if (ws != W4_OK) return ws;
    if (K == 0) return cuda_status(cudaMemsetAsync(y, 0, (size_t)(M * N) * sizeof(float), as_stream(stream)));
    w4::LinearArgs a = {};
    a.kind = w4::KIND_W8A8;
    a.x = xq; a.w = reinterpret_cast<const uint8_t *>(w); a.scale = sw; a.sx = sx; a.y = y;
    a.M = M; a.N = N; a.K = K; a.G = 0; a.layout = W4_LAYOUT_ROWMAJOR; a.flags = flags;
    a.workspace = workspace; a.ws_bytes = ws_bytes;
    return run_linear(a, as_stream(stream));
}

w4_status w4_linear_w4a16_group(const uint16_t *x_bf16, const uint8_t *w, const uint16_t *scales_f16, float *y,
                                int64_t M, int64_t N, int64_t K, int64_t G, int32_t layout, void *workspace,
                                size_t ws_bytes, uint32_t flags, void *stream) {
    if (M < 0 || N < 0 || K < 0) return W4_EINVAL;
    if (layout != W4_LAYOUT_ROWMAJOR && layout != W4_LAYOUT_N64 && layout != W4_LAYOUT_B32) return W4_EINVAL;
    const int64_t Kp = K + (K & 1);
    if (G <= 0 || (G & 1) || (Kp % G) != 0) return W4_ESHAPE;
    if (layout == W4_LAYOUT_B32 && G != 32) return W4_ESHAPE;
    if (M >= kMaxDim || N >= kMaxDim || K >= kMaxDim) return W4_ESHAPE;
    if (layout == W4_LAYOUT_N64 && N % 64) return W4_ESHAPE;
    if (M == 0 || N == 0) return W4_OK;
    if (!y || (K > 0 && (!x_bf16 || !w || (layout != W4_LAYOUT_B32 && !scales_f16)))) return W4_EINVAL;
    const w4_status ws = check_workspace(W4_OP_LINEAR_W4A16, M, N, K, G, workspace, ws_bytes);
    if (ws != W4_OK) return ws;
    if (K == 0) return cuda_status(cudaMemsetAsync(y, 0, (size_t)(M * N) * sizeof(float), as_stream(stream)));
    w4::LinearArgs a = {};
    a.kind = w4::KIND_W4A16;
    a.x = x_bf16; a.w = w; a.scale = scales_f16; a.sx = nullptr; a.y = y;
    a.M = M; a.N = N; a.K = K; a.G = G; a.layout = layout; a.flags = flags;
    a.workspace = workspace; a.ws_bytes = ws_bytes;
    return run_linear(a, as_stream(stream));
}

w4_status w4_linear_w8a16(const float *x, const int8_t *w, const float *sw, float *y, int64_t M, int64_t N,
                          int64_t K, void *workspace, size_t ws_bytes, uint32_t flags, void *stream) {
    if (M < 0 || N < 0 || K < 0) return W4_EINVAL;
    if (M >= kMaxDim || N >= kMaxDim || K >= kMaxDim) return W4_ESHAPE;
    if (M == 0 || N == 0) return W4_OK;
    if (!y || !sw || (K > 0 && (!x || !w))) return W4_EINVAL;
    const w4_status ws = check_workspace(W4_OP_LINEAR_W8A16, M, N, K, 0, workspace, ws_bytes);
    if (ws != W4_OK) return ws;
    if (K == 0) return cuda_status(cudaMemsetAsync(y, 0, (size_t)(M * N) * sizeof(float), as_stream(stream)));
    w4::LinearArgs a = {};
    a.kind = w4::KIND_W8A16;
    a.x = x; a.w = reinterpret_cast<const uint8_t *>(w); a.scale = sw; a.sx = nullptr; a.y = y;
    a.M = M; a.N = N; a.K = K; a.G = 0; a.layout = W4_LAYOUT_ROWMAJOR; a.flags = flags;
    a.workspace = workspace; a.ws_bytes = ws_bytes;
    return run_linear(a, as_stream(stream));
}

w4_status w4_linear_q4_group(const int8_t *xq, const float *sx, const uint8_t *w, const uint16_t *scales_f16,
                             const uint8_t *zeros, float *y, int64_t M, int64_t N, int64_t K, int64_t G,
                             int32_t layout, void *workspace, size_t ws_bytes, uint32_t flags, void *stream) {
    if (M < 0 || N < 0 || K < 0) return W4_EINVAL;
    if (layout != W4_LAYOUT_ROWMAJOR && layout != W4_LAYOUT_N64) return W4_EINVAL;
    const int64_t Kp = K + (K & 1);
    if (G <= 0 || (G & 1) || (Kp % G) != 0) return W4_ESHAPE;
    if (M >= kMaxDim || N >= kMaxDim || K >= kMaxDim) return W4_ESHAPE;
    if (layout == W4_LAYOUT_N64 && N % 64) return W4_ESHAPE;
    if (M == 0 || N == 0) return W4_OK;
    if (!y || !sx || (K > 0 && (!xq || !w || !scales_f16 || !zeros))) return W4_EINVAL;
    const w4_status ws = check_workspace(W4_OP_LINEAR_Q4_GROUP, M, N, K, G, workspace, ws_bytes);
    if (ws != W4_OK) return ws;
    if (K == 0) return cuda_status(cudaMemsetAsync(y, 0, (size_t)(M * N) * sizeof(float), as_stream(stream)));
    w4::LinearArgs a = {};
    a.kind = w4::KIND_W4A8G;
    a.x = xq; a.w = w; a.scale = scales_f16; a.zeros = zeros; a.sx = sx; a.y = y;
    a.M = M; a.N = N; a.K = K; a.G = G; a.layout = layout; a.flags = flags;
    a.workspace = workspace; a.ws_bytes = ws_bytes;
    return run_linear(a, as_stream(stream));
}

w4_status w4_pack_interleaved_n64(const uint8_t *w_rowmajor, uint8_t *w_il, int64_t N, int64_t K, void *stream) {
    if (N < 0 || K < 0) return W4_EINVAL;
    if (N % 64) return W4_ESHAPE;
    if (N >= kMaxDim || K >= kMaxDim) return W4_ESHAPE;
    if (N == 0 || K == 0) return W4_OK;
    if (!w_rowmajor || !w_il) return W4_EINVAL;
    return cuda_status(w4::launch_pack_n64(w_rowmajor, w_il, N, K, as_stream(stream)));
}

static w4_status chain_q4_impl(const float *x0, int32_t K0, const w4_chain_linear *lin, int32_t n_lin, int32_t passes,
                               int32_t pass_output, void *workspace, size_t ws_bytes, void *stream, uint64_t wait_ns,
                               int32_t hold_stage) {
    if (n_lin < 1 || n_lin > W4_CHAIN_MAX_LINEARS || passes < 0 || K0 <= 0 || !lin) return W4_EINVAL;
    if (pass_output < 0 || pass_output >= n_lin) return W4_EINVAL;
    for (int32_t i = 0; i < n_lin; ++i) {
        const w4_chain_linear &L = lin[i];
        if (L.N <= 0 || L.K <= 0 || L.input < -1 || L.input >= i || L.reserved != 0) return W4_EINVAL;
    }
    if (K0 % 32 || K0 > W4_CHAIN_MAX_K) return W4_ESHAPE;
    for (int32_t i = 0; i < n_lin; ++i) {
        const w4_chain_linear &L = lin[i];
        if (L.K % 32 || L.K > W4_CHAIN_MAX_K) return W4_ESHAPE;
        if (L.K != (L.input < 0 ? K0 : lin[L.input].N)) return W4_ESHAPE;
    }
    if (passes > 1 && lin[pass_output].N != K0) return W4_ESHAPE;
    if (!w4::chain_stages_ok(lin, n_lin, passes, pass_output)) return W4_ESHAPE;
    if (passes == 0) return W4_OK;
    auto misaligned = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) != 0; };
    if (!x0 || misaligned(x0)) return W4_EINVAL;
    for (int32_t i = 0; i < n_lin; ++i) {
        const w4_chain_linear &L = lin[i];
        if (!L.w || !L.sw || !L.y || misaligned(L.w) || misaligned(L.y)) return W4_EINVAL;
    }
    if (!workspace || misaligned(workspace) || ws_bytes < w4::chain_workspace_bytes(lin, n_lin, K0))
        return W4_EINVAL;
    uint32_t *status = nullptr;
    cudaError_t e = status_ptr(&status);
    if (e != cudaSuccess) return cuda_status(e);
    const int rc = w4::chain_plan_launch(x0, K0, lin, n_lin, passes, pass_output, workspace, status,
                                         as_stream(stream), &e, wait_ns, hold_stage);
    if (rc == W4_ECUDA) return cuda_status(e);
    return (w4_status)rc;
}

w4_status w4_chain_q4(const float *x0, int32_t K0, const w4_chain_linear *lin, int32_t n_lin, int32_t passes,
                      int32_t pass_output, void *workspace, size_t ws_bytes, void *stream) {
    return chain_q4_impl(x0, K0, lin, n_lin, passes, pass_output, workspace, ws_bytes, stream, w4::kWaitLimitNs, -1);
}

w4_status w4_chain_q4_test_timeout(const float *x0, int32_t K0, const w4_chain_linear *lin, int32_t n_lin,
                                   int32_t passes, int32_t pass_output, void *workspace, size_t ws_bytes,
                                   uint64_t wait_limit_ns, int32_t hold_stage, void *stream) {
    if (wait_limit_ns == 0 || wait_limit_ns > w4::kWaitLimitNs || hold_stage < -1) return W4_EINVAL;
    return chain_q4_impl(x0, K0, lin, n_lin, passes, pass_output, workspace, ws_bytes, stream, wait_limit_ns,
                         hold_stage);
}

w4_status w4_pack_block32(const uint8_t *w_rowmajor, const uint16_t *scales_f16, uint8_t *blocks, int64_t N,
                          int64_t K, void *stream) {
    if (N < 0 || K < 0) return W4_EINVAL;
    if ((K + (K & 1)) % 32) return W4_ESHAPE;
    if (N >= kMaxDim || K >= kMaxDim) return W4_ESHAPE;
    if (N == 0 || K == 0) return W4_OK;
    if (!w_rowmajor || !scales_f16 || !blocks) return W4_EINVAL;
    return cuda_status(w4::launch_pack_block32(w_rowmajor, scales_f16, blocks, N, K, as_stream(stream)));
}

size_t w4_chain_workspace_bytes(const w4_chain_linear *lin, int32_t n_lin, int32_t K0) {
    if (!lin || n_lin < 1 || n_lin > W4_CHAIN_MAX_LINEARS || K0 < 0) return 0;
    return w4::chain_workspace_bytes(lin, n_lin, K0);
}

size_t w4_workspace_bytes(int32_t op, int64_t M, int64_t N, int64_t K, int64_t G) {
    if (M <= 16 || N <= 0 || K <= 0) return 0;
    if (M >= kMaxDim || N >= kMaxDim || K >= kMaxDim) return SIZE_MAX;  // beyond every call's limits
    switch (op) {
        case W4_OP_LINEAR_Q4: return w4::gemm_workspace_bytes(w4::KIND_W4A8, M, N, K, G);
        case W4_OP_LINEAR_Q8: return w4::gemm_workspace_bytes(w4::KIND_W8A8, M, N, K, G);
        case W4_OP_LINEAR_W4A16: return w4::gemm_workspace_bytes(w4::KIND_W4A16, M, N, K, G);
        case W4_OP_LINEAR_Q4_GROUP: return w4::gemm_workspace_bytes(w4::KIND_W4A8G, M, N, K, G);
        case W4_OP_LINEAR_W8A16: return w4::gemm_workspace_bytes(w4::KIND_W8A16, M, N, K, G);
        default: return 0;
    }
}

w4_status w4_device_status(uint32_t *out, int32_t clear) {
    if (!out) return W4_EINVAL;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_status_word, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_status(e);
    if (clear) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(uint32_t));
        if (e != cudaSuccess) return cuda_status(e);
    }
    return W4_OK;
}

int32_t w4_last_cuda_error(void) { return t_last_cuda_error; }

const char *w4_status_string(w4_status s) {
    switch (s) {
        case W4_OK: return "W4_OK";
        case W4_EINVAL: return "W4_EINVAL: invalid argument";
        case W4_ESHAPE: return "W4_ESHAPE: shape not supported by the layout";
        case W4_ECUDA: return "W4_ECUDA: CUDA call failed";
        default: return "unknown w4_status";
    }
}

int32_t w4_version(void) { return 100; }

}  // extern "C"
