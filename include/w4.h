/*
 * w4.h -- C ABI of libw4gb300: fused int4 dequantize-matmul on GB300 (sm_103a).
 *
 * y = x . W^T with a 4-bit W that is never materialised in float.  Two
 * contracts:
 *   W4A8 (docs.rs ftts_kernels::int4): symmetric per-output-channel Q4
 *     codes q in [-7, 7] stored biased u = q + 8, two per byte, low nibble
 *     first along k, odd K padded with the biased zero 8; activations
 *     quantized per row to Q8; exact i32 accumulation; two f32 scales
 *     applied once per element in a fixed order.
 *   Group-wise W4A16 ("Fused int4 and int8 dequantize-matmul in C",
 *     sections 2.2-2.3): signed two's-complement nibbles in [-8, 7], one IEEE
 *     f16 scale per group of G columns, bf16 activations, fp32 accumulation:
 *     y = sum_g s_g * sum_{k in g} x_k q_k.
 * and the interleaved [N/64][K][32 B] weight layout of vllm-omni "The 4-bit
 * CPU path" ("The weight layout, measured"), read in-kernel.
 *
 * Conventions shared by every call
 *   - Pointers are DEVICE pointers owned by the caller, unless stated
 *     otherwise.  Tensors are dense and row-major.  The library never
 *     allocates device memory and never frees caller memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call is asynchronous on that stream; results are
 *     visible after the stream is synchronised.
 *   - Validation happens on the host before anything is launched or read.
 *     On any error return nothing is read and every output is left untouched
 *     ("Fused int4 ..." section 4: errors before any read).  Order of checks:
 *       1. a negative dimension                          -> W4_EINVAL
 *       2. a shape the layout cannot describe            -> W4_ESHAPE
 *       3. M == 0 or N == 0 (rows == 0)                  -> W4_OK, no launch
 *       4. a required pointer is NULL                    -> W4_EINVAL
 *       5. K == 0: outputs that are sums are zero-filled -> W4_OK
 *     A pointer to a buffer that would hold zero elements may be NULL.
 *   - W4_ECUDA: a CUDA launch or copy failed (the CUDA error is returned by
 *     w4_last_cuda_error()).
 *   - Kernels never spin without a bound.  A wait that runs out (about one
 *     second) sets a bit in the device status word and the kernel returns
 *     early; read it with w4_device_status().
 *   - Odd K is accepted for both contracts: a packed row then has
 *     Kp/2 bytes (Kp = K + 1) and its last high nibble is a pad that is never
 *     multiplied by a real activation (the kernels treat x[K] as 0).
 */
#ifndef W4_H
#define W4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W4_OK = 0,
    W4_EINVAL = 1, /* NULL pointer, negative dimension, unknown layout/op, workspace too small */
    W4_ESHAPE = 2, /* shape the layout cannot describe ("Fused int4 ..." section 4: TL_ESHAPE) */
    W4_ECUDA = 3   /* a CUDA call failed */
} w4_status;

/* Weight layouts accepted by the linears. */
enum {
    W4_LAYOUT_ROWMAJOR = 0,  /* packed [N][ceil(K/2)] (int4) or [N][K] (int8) */
    W4_LAYOUT_N64 = 1,       /* int4 only: [N/64][K][32 B], byte d = channel d (low) | channel d+32 (high);
                                requires N % 64 == 0 (vllm-omni "The 4-bit CPU path": the block must tile N) */
    W4_LAYOUT_B32 = 2        /* w4_linear_w4a16_group only, G = 32: inline-scale blocks ("Fused int4 ...",
                                Going further: blocks of 32 with the scale beside the codes); row n is Kp/32
                                blocks of 18 bytes, [f16 scale, little-endian][16 bytes: the signed nibbles of
                                columns 32b .. 32b+31, low nibble = even column]; scales_f16 is not read */
};

/* Launch flags of the linears. */
enum {
    /* Programmatic dependent launch: the kernel may start, and begin reading
     * the weights and scales, while the previous kernel on `stream` is still
     * running; it waits for that kernel before it reads x or writes y.  Only
     * set it when no earlier work on the stream that may still be running
     * writes the weight or scale buffers of this call.  The library's kernels
     * let the next kernel on the stream start early, as PDL allows: a kernel
     * of the caller's launched after them with programmatic stream
     * serialization must execute griddepcontrol.wait before it reads their
     * outputs (the CUDA rule for any such kernel). */
    W4_FLAG_PDL = 1u
};

/* Operation ids for w4_workspace_bytes. */
enum { W4_OP_LINEAR_Q4 = 0, W4_OP_LINEAR_Q8 = 1, W4_OP_LINEAR_W4A16 = 2, W4_OP_LINEAR_Q4_GROUP = 3,
       W4_OP_LINEAR_W8A16 = 4 };

/* ---- quantizers ------------------------------------------------------------ */

/* quantize_row_q8 (docs.rs ftts_kernels::int8, module summary and
 * quantize_row_q8): per row m of x [M][K] (f32), the canonical symmetric Q8
 * recipe: sx[m] = max_k |x[m][k]| / 127 (one f32 IEEE division);
 * q[m][k] = clamp(rint(x[m][k] / sx[m]), -127, 127), ties to even; -128 is
 * never emitted.  A row whose sx is 0 (all zero, or an underflowing max)
 * gets all-zero codes.  rowsum[m] = sum_k q[m][k] (i32), the activation sum
 * of the bias correction of dot_i32_q4 (NULL: not written).
 * Outputs: q [M][K] int8, sx [M] f32, rowsum [M] i32.  NaN/Inf inputs are
 * unsupported (not checked: checking would read data before validation).
 * Bit-exact with the CPU definition: same division, same rounding. */
w4_status w4_quantize_row_q8(const float *x, int64_t M, int64_t K, int8_t *q, float *sx,
                             int32_t *rowsum, void *stream);

/* quantize_matrix_q4 (docs.rs ftts_kernels::int4, "The quantization
 * contract" and "Packing"): per output channel n of W [N][K] (f32),
 * sw[n] = max_k |W[n][k]| / 7, q = clamp(rint(W / sw), -7, 7) (ties to
 * even; -8 never emitted), stored u = q + 8 in packed [N][ceil(K/2)]:
 * byte b holds column 2b in bits 0-3 and column 2b+1 in bits 4-7; for odd
 * K the last high nibble is 8 (the biased zero, which decodes to 0).
 * A channel with sw == 0 stores all u = 8. */
w4_status w4_quantize_matrix_q4(const float *W, int64_t N, int64_t K, uint8_t *packed, float *sw,
                                void *stream);

/* quantize_matrix_q8 (docs.rs ftts_kernels::int8, QuantizedMatrix): the
 * Q8 recipe of w4_quantize_row_q8 per output channel: q [N][K] int8 in
 * [-127, 127], sw [N] f32.  Weights for w4_linear_q8. */
w4_status w4_quantize_matrix_q8(const float *W, int64_t N, int64_t K, int8_t *q, float *sw,
                                void *stream);

/* ---- dot ------------------------------------------------------------------- */

/* dot_i32_q4 (docs.rs ftts_kernels::int4, dot_i32_q4 and "Packing"):
 * exact i32 dot of one Q8 activation row xq [K] with one packed biased-Q4
 * weight row wrow [ceil(K/2)]:  sum_k xq[k]*u[k] - 8 * sum_k xq[k]
 * (= sum_k xq[k]*(u[k]-8)).  `out` is a device pointer to one int32.
 * K > 1,127,288 -> W4_ESHAPE (|sum xq*u| could leave i32). */
w4_status w4_dot_i32_q4(const int8_t *xq, const uint8_t *wrow, int64_t K, int32_t *out, void *stream);

/* ---- linears --------------------------------------------------------------- */

/* linear_q4, W4A8 (docs.rs ftts_kernels::int4, linear_q4; scale order:
 * docs.rs ftts_kernels::int8 module summary):
 *   acc[m][n] = sum_k xq[m][k] * (u[n][k] - 8)          exact i32
 *   y[m][n]   = (f32(acc) * sx[m]) * sw[n]               two f32 multiplies,
 *                                                        round to nearest even,
 *                                                        no fused multiply-add
 * xq [M][K] int8 and sx [M] from w4_quantize_row_q8; w packed biased
 * nibbles in `layout` (W4_LAYOUT_ROWMAJOR: [N][ceil(K/2)]; W4_LAYOUT_N64:
 * [N/64][K][32]); sw [N]; y [M][N] f32.  Bit-exact with the CPU oracle for
 * every M.  Every nibble value decodes (0 -> -8) even though the quantizer
 * never emits it.
 * workspace: device scratch of at least w4_workspace_bytes(W4_OP_LINEAR_Q4,
 * M, N, K, 0) bytes (may be NULL when that is 0); it must not be used by
 * concurrently running work.  flags: 0 or W4_FLAG_PDL.
 * ESHAPE: K > 1,000,000; layout N64 with N % 64 != 0.  EINVAL: unknown layout. */
w4_status w4_linear_q4(const int8_t *xq, const float *sx, const uint8_t *w, const float *sw,
                       float *y, int64_t M, int64_t N, int64_t K, int32_t layout,
                       void *workspace, size_t ws_bytes, uint32_t flags, void *stream);

/* quantize_row_q8 followed by linear_q4, as one call (docs.rs
 * ftts_kernels::int4 and ::int8: activations are quantised per row before
 * the W4A8 linear).  x [M][K] f32 device; xq [M][K] int8 and sx [M] f32
 * receive exactly what w4_quantize_row_q8 writes; y [M][N] what
 * w4_linear_q4 writes for them -- bit for bit.  For M = 1 on the row-major
 * layout with N >= 1024 the quantisation runs inside the linear (every
 * thread block quantises the row itself; one launch); otherwise the two
 * kernels run in order.  Other arguments, limits and errors: those of
 * w4_linear_q4 and w4_quantize_row_q8. */
w4_status w4_linear_q4_f32(const float *x, const uint8_t *w, const float *sw, float *y, int8_t *xq, float *sx,
                           int64_t M, int64_t N, int64_t K, int32_t layout, void *workspace, size_t ws_bytes,
                           uint32_t flags, void *stream);

/* linear_q8, W8A8 (docs.rs ftts_kernels::int8, linear_q8): the same
 * epilogue over acc[m][n] = sum_k xq[m][k] * w[n][k] (exact i32), w [N][K]
 * int8 (from w4_quantize_matrix_q8), sw [N].  Bit-exact with the oracle.
 * ESHAPE: K > 131,072 (|acc| could leave i32 for arbitrary int8 weights).
 * linear_q8_dynamic is the composition w4_quantize_row_q8 + w4_linear_q8. */
w4_status w4_linear_q8(const int8_t *xq, const float *sx, const int8_t *w, const float *sw,
                       float *y, int64_t M, int64_t N, int64_t K,
                       void *workspace, size_t ws_bytes, uint32_t flags, void *stream);

/* linear_w4a16_group ("Fused int4 and int8 dequantize-matmul in C",
 * sections 2.2-2.3):
 *   y[m][n] = sum_g s[n][g] * sum_{k in group g} x[m][k] * q[n][k]
 * x [M][K] bf16 bit patterns; w signed two's-complement nibbles
 * (q = u - 16 when u >= 8) in `layout`; scales [N][Kp/G] IEEE f16 bit
 * patterns (Kp = K rounded up to even); y [M][N] f32; fp32 accumulation.
 * Accuracy (against the exact-product sum):
 *   |y - y_exact| <= 1e-5 * sum_k |x_k W_nk| + 1e-6        for M <= 16,
 *   |y - y_exact| <= 4e-3 * sum_k |x_k W_nk| + 1e-6        for M > 16, where
 * the weight is dequantised once to bf16(q * s) in shared memory and fed to
 * bf16 tensor-core MMA (vllm-omni "The 4-bit CPU path": large batches
 * dequantize once and run a dense GEMM).
 * ESHAPE: G <= 0, G odd, Kp % G != 0 ("Fused int4 ..." section 2.2: G even
 * and positive, whole groups); layout N64 with N % 64 != 0. */
w4_status w4_linear_w4a16_group(const uint16_t *x_bf16, const uint8_t *w, const uint16_t *scales_f16,
                                float *y, int64_t M, int64_t N, int64_t K, int64_t G, int32_t layout,
                                void *workspace, size_t ws_bytes, uint32_t flags, void *stream);

/* linear_q4 without caller-provided scratch.  No counterpart in the pages
 * this library follows: it exists for callers that cannot allocate device
 * memory while they run -- a serving process that reserves its whole memory
 * budget up front, a host framework whose own allocator owns the device, a
 * latency-critical loop where an allocation could block.  Same arguments,
 * result and errors as w4_linear_q4 (flags 0), but the scratch a large batch
 * needs (M * round_up(K, 8) * 2 bytes when M > 16, see w4_workspace_bytes)
 * comes from a fixed array inside the library's device image, of
 * W4_NOALLOC_SCRATCH_BYTES bytes; every GPU that loads the library keeps it
 * until the process exits.  The function itself calls no allocator.
 *   - Batches that need more scratch than that return W4_ESHAPE before
 *     anything is launched.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  W4_ECUDA if the lookup fails.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents (every call rewrites what it uses before reading it).  Calls
 *     that can run at the same time on the GPU -- different streams, or
 *     different host threads -- race on it: order them on one stream. */
#define W4_NOALLOC_SCRATCH_BYTES (8u << 20)
w4_status w4_linear_q4_noalloc(const int8_t *xq, const float *sx, const uint8_t *w, const float *sw, float *y,
                               int64_t M, int64_t N, int64_t K, int32_t layout, void *stream);

/* linear_w8a16 (docs.rs ftts_kernels::int8, linear_w8a16): f32 activations
 * times the per-channel Q8 matrix of w4_quantize_matrix_q8:
 *   y[m][n] = sw[n] * sum_k x[m][k] * q[n][k]   (f32, summation order not fixed)
 * |y - y_ref| <= 1e-5 * sum_k |x * q * sw| + 1e-6 for M <= 16 (x enters the
 * tensor cores as two bf16 terms, hi = bf16(x) and lo = bf16(x - hi), within
 * 2^-18 of x; the products with the int8 codes are exact); the tensor-core
 * path for M > 16 rounds x to bf16 once and is held to 4e-3.
 * x f32 [M][K]; w int8 [N][K]; sw [N]; y [M][N].
 * workspace: w4_workspace_bytes(W4_OP_LINEAR_W8A16, M, N, K, 0) bytes (the
 * bf16 image of x when M > 16).  EINVAL: a NULL pointer. */
w4_status w4_linear_w8a16(const float *x, const int8_t *w, const float *sw, float *y, int64_t M, int64_t N,
                          int64_t K, void *workspace, size_t ws_bytes, uint32_t flags, void *stream);

/* ---- grouped asymmetric W4A8 ------------------------------------------------ */

/* linear_q4_group: the GPTQ-style W4A8 of vllm-omni "The 4-bit CPU path"
 * ("W4A8 -- _C::int4_scaled_mm_cpu": weights with per-group scales and the
 * checkpoint's zero points, the constant 8 only when none are given; int8
 * activations).  With u the stored nibble (low nibble = even column, the
 * same packing as linear_q4):
 *   acc[m][n][g] = sum_{k in group g} xq[m][k] * (u[n][k] - z[n][g])   exact in i32
 *   y[m][n]      = sx[m] * sum_g acc * s[n][g]                        f32
 * The sum over groups is in f32, order not fixed: |y - y_ref| <=
 * 1e-5 * sum_k |xq * sx * (u - z) * s| + 1e-6 at M <= 16; the tensor-core
 * path for M > 16 multiplies the f16 rounding of (u - z) * s (exact in f32)
 * and is held to 4e-3 of the same sum.  Zero points all 8 with one scale per
 * row give linear_q4 (to rounding).
 * xq [M][K], sx [M] as for linear_q4; w packed [N][ceil(K/2)] (row-major) or
 * [N/64][K][32] (W4_LAYOUT_N64); scales_f16 and zeros [N][Kp/G] (zero points
 * 0..15, one byte each); y [M][N].
 * workspace: w4_workspace_bytes(W4_OP_LINEAR_Q4_GROUP, M, N, K, G) bytes.
 * ESHAPE: G <= 0, G odd or Kp % G != 0; layout N64 with N % 64 != 0.
 * EINVAL: unknown layout; a NULL pointer. */
w4_status w4_linear_q4_group(const int8_t *xq, const float *sx, const uint8_t *w, const uint16_t *scales_f16,
                             const uint8_t *zeros, float *y, int64_t M, int64_t N, int64_t K, int64_t G,
                             int32_t layout, void *workspace, size_t ws_bytes, uint32_t flags, void *stream);

/* ---- weight-resident chains -------------------------------------------------- */

/* The microdecoder of docs.rs ftts_kernels::int4 ("Why the microdecoder"): a
 * small decoder body whose int4 weights are re-read many times per frame,
 * each linear fed by the per-row Q8 quantisation of an earlier linear's
 * output.  w4_chain_q4 runs such a chain -- every linear, every pass -- as
 * ONE persistent kernel (one CTA per SM; inside a pass each step waits only
 * for the tagged elements it reads, a grid barrier separates passes), in
 * place of one quantize_row_q8 + linear_q4 launch per step. */
#define W4_CHAIN_MAX_LINEARS 64
#define W4_CHAIN_MAX_K 8192

/* One W4A8 linear of a chain at M = 1. */
typedef struct w4_chain_linear {
    const uint8_t *w; /* packed biased Q4 [N][K/2], row-major (quantize_matrix_q4), 16-byte aligned */
    const float *sw;  /* [N] per-channel scales */
    float *y;         /* [N] f32 output, 16-byte aligned; after the call it holds the last pass's value */
    int32_t N;        /* output channels, >= 1 */
    int32_t K;        /* input length: K0 when input == -1, else N of the input linear; K % 32 == 0 */
    int32_t input;    /* -1: the pass input; else the index (< this one's) of the linear whose y is read */
    int32_t reserved; /* must be 0 */
} w4_chain_linear;

/* chain_q4: h = x0 (length K0); for each of `passes` passes, for i = 0 ..
 * n_lin - 1 in order:
 *     in_i = (lin[i].input < 0) ? h : lin[lin[i].input].y
 *     (q, sx) = quantize_row_q8(in_i)           -- as w4_quantize_row_q8
 *     lin[i].y = linear_q4(q, sx, lin[i].w, lin[i].sw)   -- as w4_linear_q4, M = 1
 * and at the end of the pass h = lin[pass_output].y.  Every output is bit-
 * identical to that sequence of w4_quantize_row_q8 / w4_linear_q4 calls.
 *   lin: HOST array of n_lin descriptors (1 <= n_lin <= W4_CHAIN_MAX_LINEARS),
 *     read during the call only.  x0, w, sw, y: device pointers; the y
 *     buffers must not overlap each other, x0, or any weights.
 *   Linears are grouped by depth (depth 0 reads the pass input; a linear
 *   reading linear j has depth(j) + 1); all linears of one depth must read the
 *   same vector (W4_ESHAPE otherwise).
 *   workspace: at least w4_chain_workspace_bytes(lin, n_lin, K0) bytes of
 *   device scratch (a barrier counter and tagged copies of the vectors the
 *   chain passes along), 16-byte aligned, not used by concurrent work; the
 *   call clears it on `stream` before the kernel.
 * Errors (before any launch): n_lin out of range, passes < 0, K0 <= 0, a
 * descriptor with N <= 0, K <= 0, input outside [-1, i) or reserved != 0,
 * pass_output outside [0, n_lin) -> W4_EINVAL; K0 or a K not a multiple of
 * 32 or above W4_CHAIN_MAX_K, a K that is not its input's length, passes > 1
 * with lin[pass_output].N != K0 or pass_output of depth 0, or the depth rule
 * broken -> W4_ESHAPE; passes == 0 -> W4_OK, nothing launched; a NULL
 * pointer, x0 / w / y / workspace not 16-byte aligned, or workspace too
 * small -> W4_EINVAL; the device cannot keep one CTA per SM resident ->
 * W4_ECUDA.  A wait (for an input element or at a pass barrier) that runs
 * out, about one second, sets status bit 4 and the kernel returns. */
w4_status w4_chain_q4(const float *x0, int32_t K0, const w4_chain_linear *lin, int32_t n_lin, int32_t passes,
                      int32_t pass_output, void *workspace, size_t ws_bytes, void *stream);

/* Test entry point of the failure path of w4_chain_q4 (the pages have no
 * counterpart).  The same chain and arguments, with every wait of the kernel
 * limited to wait_limit_ns (1 .. 1e9) instead of about one second, and, when
 * hold_stage >= 0, global stage hold_stage (stage index + pass * stages per
 * pass; the stages are the linears grouped by depth) computing its outputs
 * without ever publishing them, so the waits of the stages that read them run
 * out.  The kernel then sets status bit 4 (w4_device_status) and returns;
 * outputs of the stages after the held one are left unspecified.  With
 * hold_stage = -1 the call is w4_chain_q4 with a shorter limit.  For tests of
 * the timeout path; not part of a production call sequence.
 * EINVAL: wait_limit_ns out of range or hold_stage < -1; otherwise as w4_chain_q4. */
w4_status w4_chain_q4_test_timeout(const float *x0, int32_t K0, const w4_chain_linear *lin, int32_t n_lin,
                                   int32_t passes, int32_t pass_output, void *workspace, size_t ws_bytes,
                                   uint64_t wait_limit_ns, int32_t hold_stage, void *stream);

/* Bytes of workspace w4_chain_q4 needs for this chain: 256 + 8 * (2 * K0 +
 * the N of every linear some other linear reads).  Host only; 0 when lin is
 * NULL or n_lin is out of range. */
size_t w4_chain_workspace_bytes(const w4_chain_linear *lin, int32_t n_lin, int32_t K0);

/* ---- layout ---------------------------------------------------------------- */

/* pack_interleaved_n64 (vllm-omni "The 4-bit CPU path", "The weight layout,
 * measured"): row-major packed int4 [N][ceil(K/2)] -> [N/64][K][32]:
 * w_il[b][k][d] = nib(64b+d, k) | nib(64b+d+32, k) << 4.  A pure
 * permutation of nibbles (either encoding).  ESHAPE: N % 64 != 0. */
w4_status w4_pack_interleaved_n64(const uint8_t *w_rowmajor, uint8_t *w_il, int64_t N, int64_t K,
                                  void *stream);

/* pack_block32: W4A16 planes (packed signed nibbles [N][Kp/2], f16 scales
 * [N][Kp/32]) -> the W4_LAYOUT_B32 blocks [N][Kp/32][18].  ESHAPE: Kp % 32. */
w4_status w4_pack_block32(const uint8_t *w_rowmajor, const uint16_t *scales_f16, uint8_t *blocks, int64_t N,
                          int64_t K, void *stream);

/* ---- host queries ---------------------------------------------------------- */

/* Bytes of device scratch the op needs at this shape (0: pass NULL).
 * SIZE_MAX when M, N or K is 2^31 or more (no call accepts such a shape). */
size_t w4_workspace_bytes(int32_t op, int64_t M, int64_t N, int64_t K, int64_t G);

/* Reads (and when clear != 0, clears) the device status word of the
 * current device: 0 when no kernel has given up on a bounded wait.  Bits:
 * 1 = a weight-tile copy wait timed out, 2 = a tensor-core pipeline wait
 * timed out, 4 = a chain_q4 wait (input element or pass barrier) timed out.  Synchronous (a small device-to-host copy). */
w4_status w4_device_status(uint32_t *out, int32_t clear);

/* The cudaError_t (as int) behind the last W4_ECUDA of this thread. */
int32_t w4_last_cuda_error(void);

/* Static string for a status code. */
const char *w4_status_string(w4_status s);

/* Measurement utility (roofline denominators): times a loop of legacy
 * mma.sync tensor-core instructions on every SM -- kind 0: m16n8k32 s8
 * (the int8 rate), kind 1: m16n8k16 bf16 -- and returns their throughput in
 * tera-ops per second.  scratch: device buffer of at least 4 * SMs * 256
 * int32 (written with junk).  Synchronous.  Not part of any linear. */
w4_status w4_probe_mma_peak(int32_t kind, int32_t *scratch, int64_t scratch_ints, double *tera_ops, void *stream);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t w4_version(void);

#ifdef __cplusplus
}
#endif
#endif /* W4_H */
