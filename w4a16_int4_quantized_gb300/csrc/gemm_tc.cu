// gemm_tc.cu -- prefill (M > 16) tensor-core GEMM.  Filled in by the tcgen05 path.
#include "internal.h"

namespace w4 {

bool gemm_supported(const LinearArgs &) { return false; }

size_t gemm_workspace_bytes(int, int64_t, int64_t, int64_t, int64_t) { return 0; }

cudaError_t launch_gemm(const LinearArgs &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace w4
