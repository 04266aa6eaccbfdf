// internal.h -- launchers shared between the kernel translation units and the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "w4.h"

namespace w4 {

// W4A8G: grouped asymmetric W4A8 (per-group f16 scales and zero points).
// W8A16: int8 weights with f32 channel scales, f32 activations.
enum Kind : int { KIND_W4A8 = 0, KIND_W8A8 = 1, KIND_W4A16 = 2, KIND_W4A8G = 3, KIND_W8A16 = 4 };

// One linear call after host validation (shapes legal, pointers non-NULL,
// M, N, K > 0).
struct LinearArgs {
    int kind;
    const void *x;       // int8 [M][K] (W4A8, W8A8, W4A8G), bf16 [M][K] (W4A16) or f32 [M][K] (W8A16)
    const uint8_t *w;    // packed int4 (layout) or int8 [N][K]
    const void *scale;   // f32 sw [N] (W4A8, W8A8) or f16 [N][Kp/G] (W4A16, W4A8G)
    const uint8_t *zeros;  // W4A8G: zero points [N][Kp/G]
    const float *sx;     // f32 [M] (int kinds)
    float *y;            // f32 [M][N]
    int64_t M, N, K, G;  // G: W4A16 only
    int layout;          // 0 row-major, 1 interleaved [N/64][K][32]
    uint32_t flags;      // W4_FLAG_PDL
    void *workspace;
    size_t ws_bytes;
    uint32_t *status;    // device status word
    // fused W4A8 (w4_linear_q4_f32): f32 activations quantised inside the
    // linear; x / sx then name the buffers that receive the codes and scales
    const float *xf;
    int8_t *xq_out;
    float *sx_out;
    // prefill of the int kinds: the workspace already holds the f16 image of the activation codes
    bool x16_ready;
};

// capi.cu -- W4_OK for cudaSuccess; otherwise records e for w4_last_cuda_error and returns W4_ECUDA.
w4_status record_cuda_error(cudaError_t e);

// tmap.cu -- TMA tensor map of a tiled box (rank <= 5); strides of dims 1..rank-1 in bytes.
bool encode_tmap(CUtensorMap *map, CUtensorMapDataType type, int rank, const void *base, const uint64_t *dims,
                 const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle swizzle);

// quant.cu
cudaError_t launch_quantize_rows(const float *x, int64_t rows, int64_t K, int Q, int8_t *q, float *s,
                                 int32_t *rowsum, cudaStream_t st);
cudaError_t launch_quantize_matrix_q4(const float *W, int64_t N, int64_t K, uint8_t *packed, float *sw,
                                      cudaStream_t st);
// quantize_row_q8 of M rows (K % 8 == 0) plus the f16 image of the codes, [M][K], for the prefill GEMM.
cudaError_t launch_quantize_rows_f16(const float *x, int64_t M, int64_t K, int8_t *q, float *s, uint16_t *xh,
                                     cudaStream_t st);
cudaError_t launch_dot_i32_q4(const int8_t *xq, const uint8_t *wrow, int64_t K, int32_t *out, cudaStream_t st);
cudaError_t launch_pack_n64(const uint8_t *w, uint8_t *il, int64_t N, int64_t K, cudaStream_t st);
cudaError_t launch_pack_block32(const uint8_t *w, const uint16_t *s, uint8_t *blocks, int64_t N, int64_t K,
                                cudaStream_t st);

// gemv.cu -- small-M tensor-core GEMV (M <= 16) and the generic fallback.
bool gemv_supported(const LinearArgs &a);
cudaError_t launch_gemv(const LinearArgs &a, cudaStream_t st);
cudaError_t launch_generic(const LinearArgs &a, cudaStream_t st);

// gemm_tc.cu -- tcgen05 prefill GEMM (M > 16).
bool gemm_supported(const LinearArgs &a);
size_t gemm_workspace_bytes(int kind, int64_t M, int64_t N, int64_t K, int64_t G);
cudaError_t launch_gemm(const LinearArgs &a, cudaStream_t st);

// chain.cu -- a chain of M = 1 W4A8 linears as one persistent cooperative kernel.
constexpr int kChainMaxLinears = W4_CHAIN_MAX_LINEARS;
constexpr int kChainMaxK = W4_CHAIN_MAX_K;
constexpr int64_t kChainMaxStageRows = (int64_t)1 << 24;
constexpr size_t kChainHeaderBytes = 256;
// Workspace of a chain: header + tagged pass output [2][K0] + tagged copies of read linears.
size_t chain_workspace_bytes(const w4_chain_linear *lin, int32_t n_lin, int32_t K0);
// Host check: linears of one depth read one vector, stage rows bounded, and
// with passes > 1 the pass output is not of depth 0.
bool chain_stages_ok(const w4_chain_linear *lin, int32_t n_lin, int32_t passes, int32_t pass_output);
// Plans (stages by depth) and launches a validated chain; returns a w4_status
// (W4_ESHAPE when the chain has no stage structure), *err the CUDA error.
// wait_ns bounds every wait of the kernel; hold_stage >= 0 (the failure-path
// test only) keeps that global stage's outputs from ever being published.
int chain_plan_launch(const float *x0, int32_t K0, const w4_chain_linear *lin, int32_t n_lin, int32_t passes,
                      int32_t pass_output, void *workspace, uint32_t *status, cudaStream_t st, cudaError_t *err,
                      uint64_t wait_ns, int32_t hold_stage);

}  // namespace w4
