// Internal interfaces of the 2:4-sparse W4A16 path (sparse24.cu) used by the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"

namespace w4a16 {

// Packed 2:4 stream: 32-bit words per 64-row piece of one 128-column strip
// (codes: 8 column blocks x 32 lanes x 2 words; metadata: 8 x 32 x 1 word).
constexpr int kPiece24Words = 768;

// Dense codes uint8[K][N] (at most two codes != 8 in each group of four rows of a
// column) -> packed 2:4 stream; a group with more flags kDevErrValue.
cudaError_t launch_repack24(const uint8_t* q, int K, int N, uint32_t* packed24, cudaStream_t stream);
// Packed 2:4 stream -> dense codes (8 at the pruned positions); invalid positions flag kDevErrValue.
cudaError_t launch_unpack24(const uint32_t* packed24, int K, int N, uint8_t* q, cudaStream_t stream);
// FP16 scales s[K/G][N] -> the permuted order the GEMMs read (defined in repack.cu).
cudaError_t launch_permute_scales(const uint16_t* s, int K, int N, int G, uint16_t* scales_p, cudaStream_t stream);
cudaError_t read_and_clear_sparse_flag(unsigned int* flag, cudaStream_t stream);

struct Plan24 {
  MmaConfig cfg;
  MmaLayout lay;
  int srows, KU, strips, units, T, grid, m_chunk;
  size_t workspace;
};

Plan24 make_plan24(int M, int K, int N, int G, int sms, int smem_optin, int ablate);
// c.packed is the packed 2:4 stream; zeros and bias are not used.  Returns a W4A16 status.
int run_gemm24(const Plan24& pl, const GemmCall& c);

}  // namespace w4a16
