// Internal interfaces of the 2:4-sparse offline steps (sparse24.cu) used by the C ABI.
// The 2:4 GEMM itself is the streaming kernel's SP24 variant (gemm_mma.cu, planned by
// make_plan24 and launched by run_gemm).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"

namespace w4a16 {

// Dense codes uint8[K][N] (at most two codes != 8 in each group of four rows of a
// column) -> packed 2:4 stream; a group with more flags kDevErrValue.
cudaError_t launch_repack24(const uint8_t* q, int K, int N, uint32_t* packed24, cudaStream_t stream);
// Packed 2:4 stream -> dense codes (8 at the pruned positions); invalid positions flag kDevErrValue.
cudaError_t launch_unpack24(const uint32_t* packed24, int K, int N, uint8_t* q, cudaStream_t stream);
// FP16 scales s[K/G][N] -> the permuted order the GEMMs read (defined in repack.cu).
cudaError_t launch_permute_scales(const uint16_t* s, int K, int N, int G, uint16_t* scales_p, cudaStream_t stream);
cudaError_t read_and_clear_sparse_flag(unsigned int* flag, cudaStream_t stream);

}  // namespace w4a16
