// Internal interfaces between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace w4a16 {

// Launch of a GEMM kernel that may overlap the tail of the previous kernel in its stream
// (programmatic dependent launch; the kernel waits with griddepcontrol.wait before any global
// memory access).  Captured into a CUDA graph it becomes a programmatic edge.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kern)(KArgs...), int grid, int block, int smem, cudaStream_t stream,
                              Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(block));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Raise a kernel's dynamic shared-memory limit to `bytes` once per device (the attribute
// call costs a driver round trip; later launches that need no more skip it).  `cache` is
// the kernel's own table of the largest limit set per device.
template <typename Kern>
cudaError_t ensure_smem(Kern kern, int bytes, int (&cache)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (__atomic_load_n(&cache[dev], __ATOMIC_ACQUIRE) >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  int cur = __atomic_load_n(&cache[dev], __ATOMIC_RELAXED);
  while (cur < bytes && !__atomic_compare_exchange_n(&cache[dev], &cur, bytes, true, __ATOMIC_RELEASE,
                                                     __ATOMIC_RELAXED)) {
  }
  return cudaSuccess;
}

// status bits recorded in the workspace status word / the repack flag
enum : uint32_t {
  kDevErrCodeRange = 1u << 0,
  kDevErrTimeout = 1u << 1,
  kDevErrValue = 1u << 2,
};

// Ablation switches (the MARLIN paper's Figure 12, re-run on these kernels): each
// removes one design choice; they combine as a bit mask.
enum : int {
  kAblateNoEvictFirst = 1,  // weight stream without the L2 evict-first hint (evict-normal)
  kAblateStages2 = 2,       // weight pipeline depth 2
  kAblateNoSwizzle = 4,     // activation tile without the 128-byte XOR swizzle (streaming kernel)
};

// Shared-memory layout of one streaming-kernel configuration (byte offsets
// from the 1024-aligned base; one stage = activation pieces, weight chunk,
// scale rows).
struct MmaLayout {
  int w_off, s_off, z_off, stage_bytes, tx_bytes;  // z_off: zero-point rows (with zero points only)
  int red_off, bar_off, flag_off, moe_off, smem_bytes;  // moe_off: expert tables of the grouped GEMM
};

// moe_E: experts of a grouped GEMM (0 for a plain GEMM); their tables take shared memory.
// piece_bytes: packed weights per 64-row piece of a strip (4096 dense, 3072 for 2:4).
MmaLayout mma_layout(int m_tiles, int kq, int srows, int stages, bool zp, int moe_E = 0, int piece_bytes = 4096);

// 2:4-sparse packed stream: 32-bit words per 64-row piece of one 128-column strip
// (codes: 8 column blocks x 32 lanes x 2 words; positions: 8 x 32 x 1 word).
constexpr int kPiece24Words = 768;

// Parameters of one launch of the streaming (mma.sync) GEMM kernel.
struct GemmParams {
  const uint32_t* packed;   // uint32[N/128][K/64][8][32][4]
  const uint16_t* scales;   // permuted fp16[N/128][K/G][128]
  const uint8_t* zeros;     // permuted zero codes uint8[N/128][K/G][128], or null (z = 8)
  const uint16_t* bias;     // fp16[N] added to C, or null
  uint16_t* C;              // fp16[M][N]
  uint32_t* status;         // workspace status word
  uint32_t* counters;       // one arrival counter per 128-column strip
  float* slots;             // 2 * grid partial-sum slots of 128 * 8 * m_tiles floats
  int M;                    // rows of A / C
  int m0;                   // first row handled by this launch
  int K, N, G;              // G: effective group size (128 or K)
  int kq;                   // 64-row pieces per work unit (KT = 64 * kq)
  int srows;                // scale rows per work unit
  int KU;                   // K / KT work units per strip
  int units;                // (N / 128) * KU
  int T;                    // units per CTA
  int grid;                 // CTAs
  int stages;               // pipeline depth
  int w_off, s_off, z_off, stage_bytes, tx_bytes, red_off, bar_off, flag_off;
  long long wait_limit;     // clock cycles a pipeline wait may take
  int debug_stall;          // 1: never fill the first stage (failure-detection test)
  int ablate;               // kAblate* bits
  // grouped expert GEMM only (the kernel derives units and T from the offsets; grid = gridDim.x):
  const int* expert_off;    // device int32[E + 1]: rows of expert e are [off[e], off[e + 1])
  int E;                    // experts
  int strips;               // N / 128
  int max_seg;              // row segments the counters were sized for
  long long w_stride;       // packed words per expert (K * N / 8)
  long long s_stride;       // permuted scales per expert ((K / G) * N)
  int moe_off;              // shared-memory offset of the expert tables
};

constexpr int kMoeMaxExperts = 2048;

struct MmaConfig {
  int m_tiles;      // 8-row token tiles (1, 2, 4)
  int kq;           // 64-row pieces per unit (2, 4, 8, 12, 16)
  int stages;
  int smem_bytes;
  int threads;
  bool final8;      // build with the eight-warp last split-strip sum (see gemm_mma.cu)
};

constexpr int kMmaThreads = 288;  // 8 consumer warps + 1 producer warp
constexpr int kStrip = 128;       // output columns per strip / work unit

cudaError_t launch_gemm_mma(const MmaConfig& cfg, const CUtensorMap& tmA, const GemmParams& p, cudaStream_t stream);
// grouped expert GEMM: one launch over all experts (p.expert_off set, p.M = rows of A)
cudaError_t launch_moe_mma(const MmaConfig& cfg, const CUtensorMap& tmA, const GemmParams& p, cudaStream_t stream);
// 2:4-sparse weights (p.packed is the packed 2:4 stream; m_tiles 1, 2 or 4)
cudaError_t launch_gemm_sp24(const MmaConfig& cfg, const CUtensorMap& tmA, const GemmParams& p, cudaStream_t stream);
// with zero points (p.zeros != null) the kernels are built with the per-row zero decode

// ---- tensor-memory (tcgen05) GEMM ----------------------------------------
// 2 single-thread copy producers, 2 MMA issuers (one per strip of a unit), 16 dequant warps
constexpr int kTcThreads = 640;
constexpr int kTcStrips = 2;      // 128-column strips per work unit (pair mode; the wide mode has one)
constexpr int kTcMaxNA = 7;       // A buffers per strip in tensor memory
constexpr int kTcMaxNS = 8;       // activation stages
constexpr int kTcMaxSW = 8;       // weight stages

// Shared-memory layout of one tensor-memory-kernel configuration (byte offsets from the
// 1024-aligned base): activation stages, then weight stages (each: both strips' packed
// chunks, their scale rows at s_off, their zero-code rows at z_off), barriers, flags.
struct TcLayout {
  int a_stage_bytes, w_stage_bytes, w_base, s_off, z_off, bar_off, flag_off, moe_off, smem_bytes;
};
TcLayout tc_layout(int us, int mb, int ch, int srows, int a_stages, int w_stages, bool zp, int moe_E = 0);
uint32_t tc_idesc(int m, int n);

struct TcParams {
  const uint32_t* packed;
  const uint16_t* scales;
  const uint8_t* zeros;     // permuted zero codes, or null (z = 8)
  const uint16_t* bias;     // fp16[N], or null
  uint16_t* C;
  uint32_t* status;
  uint32_t* counters;       // one per unit column (strip pair, or strip in the wide mode)
  float* slots;             // 2 * grid slots of us * 128 * mb floats ([strip][token][column])
  int M, m0, K, N, G;
  int strips;               // N / 128 (the last pair has one strip when odd)
  int us;                   // strips per unit: 2 (pair mode) or 1 (wide mode)
  int mb;                   // token rows of this launch padded to 16 (the MMA's N)
  int ch;                   // 128-row chunks per work unit (KT = 128 * ch)
  int na;                   // A buffers per strip (64 tensor-memory columns each): 2..3, or 4 wide
  int srows;                // scale rows per strip and unit
  int KU, units, T, grid;   // units per unit column (strip pair or strip), units, units per CTA, CTAs
  int a_stages, w_stages;   // activation ring / weight ring depths
  int a_stage_bytes, w_stage_bytes, w_base, s_off, z_off, bar_off, flag_off;
  uint32_t idesc;
  long long wait_limit;
  int debug_stall;
  int ablate;               // kAblate* bits (no-swizzle does not apply to this kernel)
  // grouped expert GEMM only (pair mode; the kernel derives units and T from the offsets, grid =
  // gridDim.x; counters are per (row segment, strip pair)):
  const int* expert_off;    // device int32[E + 1], or null for the plain GEMM
  int E;                    // experts
  int max_seg;              // row segments the counters were sized for
  long long w_stride;       // packed words per expert (K * N / 8)
  long long s_stride;       // permuted scales per expert ((K / G) * N)
  int moe_off;              // shared-memory offset of the expert tables
};

cudaError_t launch_gemm_tc(int smem_bytes, const CUtensorMap& tmA, const TcParams& p, cudaStream_t stream);

// sms: the device's SM count (the tile walkers are persistent)
cudaError_t launch_repack(const uint8_t* q, const uint16_t* s, int K, int N, int G, uint32_t* packed,
                          uint16_t* scales_p, int sms, cudaStream_t stream);
cudaError_t launch_quantize_repack(const uint16_t* w, const uint16_t* s, const uint8_t* z, int K, int N, int G,
                                   uint32_t* packed, uint16_t* scales_p, int sms, cudaStream_t stream);
cudaError_t launch_minmax_scales(const uint16_t* w, int K, int N, int G, uint16_t* s, uint8_t* z,
                                 cudaStream_t stream);
cudaError_t launch_repack_zeros(const uint8_t* z, int K, int N, int G, uint8_t* zeros_p, cudaStream_t stream);
cudaError_t launch_unpack(const uint32_t* packed, const uint16_t* scales_p, int K, int N, int G, uint8_t* q,
                          uint16_t* s, cudaStream_t stream);
cudaError_t launch_dequant(const uint32_t* packed, const uint16_t* scales_p, const uint8_t* zeros_p, int K, int N,
                           int G, uint16_t* bhat, cudaStream_t stream);
cudaError_t read_and_clear_repack_flag(unsigned int* flag, cudaStream_t stream);

// ---- work planning and launch of one GEMM (gemm_launch.cu) ------------------
constexpr size_t kStatusBytes = 256;  // workspace head: the status word
// bytes of the per-strip arrival counters that follow the status word
inline size_t counter_bytes(int strips) { return (static_cast<size_t>(strips) * 4 + 255) / 256 * 256; }

// Which kernel runs and how it splits (M, K, N) over `sms` SMs with `smem_optin`
// bytes of shared memory per CTA.
struct Plan {
  int path;          // 1 = streaming mma.sync kernel, 2 = tensor-memory (tcgen05) kernel
  MmaConfig cfg;     // path 1
  MmaLayout lay;     // path 1
  TcLayout tlay;     // path 2
  int mb, ch;        // path 2: token rows per launch (multiple of 16), 128-row chunks per unit
  int us;            // path 2: strips per unit (2 = pair mode, 1 = wide mode)
  int a_stages, w_stages;  // path 2: activation / weight ring depths
  int ni, na;        // path 2: MMA issuers (accumulators), A chunks in tensor memory (= a_stages)
  int m_chunk;       // token rows per launch
  int k_tile;        // reduction rows per work unit
  int srows;
  int KU, strips, units, T, grid, stages, smem_bytes, threads;
  int moe_E, max_seg;  // grouped expert GEMM: experts, row segments the counters are sized for
  bool sp24;           // path 1 on the 2:4-sparse packed stream
  size_t workspace;
};

// Tensor map of the activations A fp16[M][K] viewed as [K/64][M][64]: box {64, box_rows, kq}
// fetches kq 64-column pieces of box_rows rows (128-byte swizzle unless `swizzle` is false);
// rows beyond M read as zero.
int encode_a_map(CUtensorMap* map, const uint16_t* A, int M, int K, int box_rows, int kq, bool swizzle = true);

// forced_path: 0 = by M, 1 = streaming kernel, 2 = tensor-memory kernel (mode by M), 3 = tensor-memory
// kernel in pair mode only, 4 = tensor-memory kernel in wide mode where K allows it; zp: the GEMM reads
// zero points (their rows take shared-memory stage space next to the scales)
Plan make_plan(int M, int K, int N, int G, int sms, int smem_optin, bool zp, int forced_path, int ablate = 0);

struct GemmCall {
  const uint16_t* A;
  const uint32_t* packed;
  const uint16_t* scales;  // permuted
  const uint8_t* zeros;    // permuted, or null
  const uint16_t* bias;    // or null
  uint16_t* C;
  int M, K, N, G;
  void* workspace;         // >= plan.workspace bytes; status word and counters zero
  long long wait_limit;
  int debug_stall;
  int ablate;              // kAblate* bits; the plan must have been made with the same bits
  cudaStream_t stream;
};
// Launches the planned kernels over all token-row chunks; returns a W4A16 status.
int run_gemm(const Plan& pl, const GemmCall& c);

// Grouped expert GEMM over M expert-sorted rows.  max_rows bounds the rows of any one expert and
// picks the kernel and the row-segment height: the streaming kernel with 8 or 16 rows up to 16,
// the tensor-memory kernel (pair mode) with up to 128 rows from 17 (forced_path as for make_plan).
Plan make_plan_moe(int E, int M, int max_rows, int K, int N, int G, int sms, int smem_optin, int ablate = 0,
                   int forced_path = 0);
// c.M = rows of A and C, c.packed / c.scales = E stacked layers; zeros and bias unused.
int run_moe_gemm(const Plan& pl, const GemmCall& c, const int* expert_off);

// 2:4-sparse GEMM on the streaming kernel (run with run_gemm; c.packed = the packed 2:4 stream).
Plan make_plan24(int M, int K, int N, int G, int sms, int smem_optin, int ablate);

}  // namespace w4a16
