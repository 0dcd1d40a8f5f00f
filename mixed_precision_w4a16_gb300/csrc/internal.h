// Internal interfaces between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace w4a16 {

// status bits recorded in the workspace status word / the repack flag
enum : uint32_t {
  kDevErrCodeRange = 1u << 0,
  kDevErrTimeout = 1u << 1,
};

// Parameters of one launch of the streaming (mma.sync) GEMM kernel.
struct GemmParams {
  const uint32_t* packed;   // uint32[N/16][K/64][32][4]
  const uint16_t* scales;   // permuted fp16[K/G][N]
  uint16_t* C;              // fp16[M][N]
  uint32_t* status;         // workspace status word
  uint32_t* counters;       // one arrival counter per column tile
  float* slots;             // 2 * grid partial-sum slots of n_tile * 8 * m_tiles floats
  int M;                    // rows of A / C
  int m0;                   // first row handled by this launch
  int K, N, G;              // G: effective group size (128 or K)
  int KU;                   // K / 128 work units per column tile
  int units;                // (N / n_tile) * KU
  int T;                    // units per CTA
  int grid;                 // CTAs
  int stages;               // pipeline depth
  long long wait_limit;     // clock cycles a pipeline wait may take
  int debug_stall;          // 1: never fill the first stage (failure-detection test)
};

struct MmaConfig {
  int m_tiles;      // 8-row token tiles (1, 2, 4, 8)
  int nbw;          // 16-column blocks per consumer warp (1, 2, 4)
  int n_tile;       // 64 * nbw
  int stages;
  int smem_bytes;
  int threads;
};

// shared-memory footprint of one kernel configuration
int mma_stage_bytes(int m_tiles, int nbw);
int mma_smem_bytes(int m_tiles, int nbw, int stages);
constexpr int kMmaThreads = 288;  // 8 consumer warps + 1 producer warp
constexpr int kKTile = 128;

cudaError_t launch_gemm_mma(const MmaConfig& cfg, const CUtensorMap& tmA, const GemmParams& p, cudaStream_t stream);

cudaError_t launch_repack(const uint8_t* q, const uint16_t* s, int K, int N, int G, uint32_t* packed,
                          uint16_t* scales_p, cudaStream_t stream);
cudaError_t launch_unpack(const uint32_t* packed, const uint16_t* scales_p, int K, int N, int G, uint8_t* q,
                          uint16_t* s, cudaStream_t stream);
cudaError_t launch_dequant(const uint32_t* packed, const uint16_t* scales_p, int K, int N, int G, uint16_t* bhat,
                           cudaStream_t stream);
cudaError_t read_and_clear_repack_flag(unsigned int* flag, cudaStream_t stream);

}  // namespace w4a16
