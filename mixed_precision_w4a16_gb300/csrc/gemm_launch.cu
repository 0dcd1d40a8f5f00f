// Work planning and launch of the GEMM kernels: which kernel runs for a given
// (M, K, N, G), how the work splits over the SMs, the shared- and tensor-memory
// layouts, the activation tensor map, and the launches over token-row chunks.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>

#include "../../include/w4a16.h"
#include "internal.h"

namespace w4a16 {

namespace {

constexpr int kTcMinRows = 17;   // from 17 token rows on, the tensor-memory kernel runs
constexpr int kTcWideRows = 129; // from 129 on, in its wide mode (one strip per unit, 256 rows per launch)

void finish_split(Plan& pl, int K, int sms, size_t slot_floats) {
  pl.KU = K / pl.k_tile;
  pl.units = pl.strips * pl.KU;
  pl.T = (pl.units + sms - 1) / sms;
  pl.grid = (pl.units + pl.T - 1) / pl.T;
  pl.workspace = kStatusBytes + counter_bytes(pl.strips) + 2ull * pl.grid * slot_floats * sizeof(float);
}

// moe_E > 0: the grouped expert GEMM (its expert tables take shared memory), with up
// to moe_cols row segments sharing the SMs.  sp24: the 2:4-sparse stream (3 KB per piece).
// Up to 32 token rows per launch.
Plan make_plan_mma(int M, int K, int N, int G, int sms, int smem_optin, bool zp, int moe_E = 0, int moe_cols = 1,
                   int ablate = 0, bool sp24 = false) {
  Plan pl{};
  pl.path = 1;
  pl.sp24 = sp24;
  const int piece_bytes = sp24 ? kPiece24Words * 4 : 4096;
  const int mc = std::min(std::max(M, 1), 32);
  const int mt = mc <= 8 ? 1 : mc <= 16 ? 2 : 4;
  pl.strips = N / kStrip;
  // Unit depth KT = 64 * kq (kq up to 16: each of the 4 K-split warps takes every
  // fourth piece).  Per-SM time of a unit is modelled from copy-engine measurements
  // on GB300: ~89 ns per 4 KB of weights streamed plus ~80 ns of fixed cost for the
  // unit's three copy operations; each strip segment a CTA's range touches adds ~1 us
  // (the split-strip epilogue: slots, fence, arrival count).  Pick the kq minimising
  // T * unit time + segments * 1 us among those that keep >= 2 pipeline stages in
  // shared memory (measured: two 64 KB stages beat three 48 KB and five 32 KB ones,
  // with fewer bytes in flight -- the per-unit costs weigh more than the pipeline depth).
  const long long piece_ns = 89LL * piece_bytes / 4096;
  int best_kq = 0;
  long long best_cost = 0;
  const int cands[5] = {16, 12, 8, 4, 2};
  for (int c = 0; c < 5; ++c) {
    const int kq = cands[c];
    if (K % (64 * kq) != 0) continue;
    const int srows = (G <= 64 * kq) ? (64 * kq) / G : 1;
    const MmaLayout l0 = mma_layout(mt, kq, srows, 0, zp, moe_E, piece_bytes);
    const int stages = (smem_optin - l0.smem_bytes) / (l0.stage_bytes + 16);
    if (stages < 2) continue;
    const long long KU = K / (64 * kq);
    const long long units = static_cast<long long>(pl.strips) * moe_cols * KU;
    const long long T = (units + sms - 1) / sms;
    // strip segments in a range of T units over strips of KU units, at most
    const long long segs = (KU % T == 0) ? 1 : (T % KU == 0) ? T / KU : (T - 1) / KU + 2;
    const long long cost = T * (piece_ns * kq + 80) + segs * 1000;
    if (best_kq == 0 || cost < best_cost) {
      best_kq = kq;
      best_cost = cost;
    }
  }
  if (!best_kq) best_kq = 2;
  const int kq = best_kq;
  const int KT = 64 * kq;
  pl.srows = (G <= KT) ? KT / G : 1;
  const MmaLayout l0 = mma_layout(mt, kq, pl.srows, 0, zp, moe_E, piece_bytes);
  int stages = (smem_optin - l0.smem_bytes) / (l0.stage_bytes + 16);
  stages = std::max(2, std::min(stages, 8));
  if (ablate & kAblateStages2) stages = 2;
  pl.lay = mma_layout(mt, kq, pl.srows, stages, zp, moe_E, piece_bytes);
  pl.cfg.m_tiles = mt;
  pl.cfg.kq = kq;
  pl.cfg.stages = stages;
  pl.cfg.smem_bytes = pl.lay.smem_bytes;
  pl.cfg.threads = kMmaThreads;
  pl.m_chunk = 8 * mt;
  pl.k_tile = KT;
  pl.stages = stages;
  pl.smem_bytes = pl.lay.smem_bytes;
  pl.threads = kMmaThreads;
  finish_split(pl, K, sms, static_cast<size_t>(kStrip) * 8 * mt);
  // The build whose last split-strip sum all eight consumer warps share (dense layers only):
  // measured as fast or faster for two token tiles at every layer size (1-5 %), and for one tile
  // only where a CTA has at most two units (its larger epilogue costs the one-tile main loop
  // 0.3-1.7 % through code generation, which the shorter sum repays only on the smallest layers).
  pl.cfg.final8 = moe_E == 0 && !sp24 && (mt == 2 || (mt == 1 && pl.T <= 2));
  return pl;
}

GemmParams mma_params(const Plan& pl, const GemmCall& c, uint32_t* status, uint32_t* counters, float* slots) {
  GemmParams p{};
  p.packed = c.packed;
  p.scales = c.scales;
  p.zeros = c.zeros;
  p.bias = c.bias;
  p.C = c.C;
  p.status = status;
  p.counters = counters;
  p.slots = slots;
  p.M = c.M;
  p.K = c.K;
  p.N = c.N;
  p.G = c.G;
  p.kq = pl.cfg.kq;
  p.srows = pl.srows;
  p.KU = pl.KU;
  p.units = pl.units;
  p.T = pl.T;
  p.grid = pl.grid;
  p.stages = pl.cfg.stages;
  p.w_off = pl.lay.w_off;
  p.s_off = pl.lay.s_off;
  p.z_off = pl.lay.z_off;
  p.stage_bytes = pl.lay.stage_bytes;
  p.tx_bytes = pl.lay.tx_bytes;
  p.red_off = pl.lay.red_off;
  p.bar_off = pl.lay.bar_off;
  p.flag_off = pl.lay.flag_off;
  p.moe_off = pl.lay.moe_off;
  p.wait_limit = c.wait_limit;
  p.debug_stall = c.debug_stall;
  p.ablate = c.ablate;
  return p;
}

// wide: one strip per unit and up to 256 token rows per launch (needs K % 512 == 0), else the
// strip-pair mode with up to 128.
Plan make_plan_tc(int M, int K, int N, int G, int sms, int smem_optin, bool zp, int ablate, bool wide, int moe_E = 0) {
  Plan pl{};
  pl.path = 2;
  wide = wide && K % 512 == 0;
  pl.us = wide ? 1 : kTcStrips;
  pl.strips = N / kStrip;
  const int cols = (pl.strips + pl.us - 1) / pl.us;  // unit columns: strip pairs, or strips
  // Tensor memory (512 columns): per strip an accumulator of mb columns and a ring of A
  // buffers of 64 columns (128 k of FP16) each.
  pl.ni = pl.us;  // one MMA issuer per strip
  if (wide) {
    // An accumulator of up to 256 token columns (the token rows are dealt evenly to the
    // launches) and as many A buffers as the rest of tensor memory holds: four (one per
    // dequant warpgroup) at 256 tokens, up to seven for fewer.
    const int launches = (std::max(M, 1) + 255) / 256;
    pl.mb = std::min(256, ((std::max(M, 1) + launches - 1) / launches + 15) / 16 * 16);
    pl.na = std::min(kTcMaxNA, (512 - pl.mb) / 64);
    pl.ch = 4;
  } else {
    pl.mb = std::min(128, (std::max(M, 1) + 15) / 16 * 16);
    pl.na = std::min(3, (512 / kTcStrips - pl.mb) / 64);
    // Unit depth: four 128-row chunks per strip when K allows (each dequant warpgroup then
    // decodes two chunks per unit and pays the unit's stage wait and loop work once for both),
    // else two (a unit still feeds all four warpgroups), one when K is an odd multiple of 128.
    pl.ch = (K % 512 == 0) ? 4 : (K % 256 == 0) ? 2 : 1;
  }
  pl.srows = (G == 128) ? pl.ch : 1;
  // Rings: the weight ring keeps about 100 KB of weights in flight for the HBM latency; the
  // activation ring takes the rest (up to 8 stages: it hides the L2 latency of the tiles).
  // Activation tiles of 128 tokens and more are 32 KB and up: there the activation ring gets
  // the larger share.
  const TcLayout l0 = tc_layout(pl.us, pl.mb, pl.ch, pl.srows, 0, 0, zp, moe_E);
  const int budget = smem_optin - l0.smem_bytes;
  int sw = std::max(2, std::min(kTcMaxSW, (100 * 1024 + l0.w_stage_bytes - 1) / l0.w_stage_bytes));
  if (pl.mb > 64) sw = 2;
  if (ablate & kAblateStages2) sw = 2;
  if (pl.ch == 1) sw &= ~1;  // one-chunk units: an even weight ring (each warpgroup meets every unit of a stage)
  int ns = std::min(kTcMaxNS, (budget - sw * l0.w_stage_bytes) / l0.a_stage_bytes);
  while (ns < 2 && sw > 2) {
    sw -= (pl.ch == 1) ? 2 : 1;
    ns = std::min(kTcMaxNS, (budget - sw * l0.w_stage_bytes) / l0.a_stage_bytes);
  }
  pl.w_stages = sw;
  pl.a_stages = std::max(2, ns);
  pl.tlay = tc_layout(pl.us, pl.mb, pl.ch, pl.srows, pl.a_stages, pl.w_stages, zp, moe_E);
  pl.m_chunk = pl.mb;
  pl.k_tile = 128 * pl.ch;
  pl.stages = pl.w_stages;
  pl.smem_bytes = pl.tlay.smem_bytes;
  pl.threads = kTcThreads;
  pl.KU = K / pl.k_tile;
  pl.units = cols * pl.KU;
  pl.T = (pl.units + sms - 1) / sms;
  pl.grid = (pl.units + pl.T - 1) / pl.T;
  pl.workspace = kStatusBytes + counter_bytes(pl.strips) +
                 2ull * pl.grid * (static_cast<size_t>(pl.us) * kStrip * pl.mb) * sizeof(float);
  return pl;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  // looked up once; a function-local static is initialised exactly once even with concurrent callers
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return nullptr;
  }();
  return fn;
}

}  // namespace

// 3-D view of A (fp16[M][K]) as [K/64][M][64]: box {64, box_rows, kq} fetches the
// kq 64-column pieces of one work unit in one copy, each piece box_rows x 128 bytes
// (128-byte swizzle unless the no-swizzle ablation asks otherwise); rows beyond M are zero-filled.
int encode_a_map(CUtensorMap* map, const uint16_t* A, int M, int K, int box_rows, int kq, bool swizzle) {
  auto enc = get_encoder();
  if (!enc) return W4A16_ERR_CUDA;
  const cuuint64_t dims[3] = {64u, static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128u};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(kq)};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<uint16_t*>(A), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? W4A16_OK : W4A16_ERR_CUDA;
}

Plan make_plan_moe(int E, int M, int max_rows, int K, int N, int G, int sms, int smem_optin, int ablate,
                   int forced_path) {
  // experts that can own rows, and the row segments (m_chunk rows of one expert) they can need
  const int active = std::max(1, std::min(E, M));
  if (forced_path >= 2 || (forced_path != 1 && max_rows >= kTcMinRows)) {
    // From 17 rows per expert: the tensor-memory kernel in pair mode, row segments of up to 128
    // rows (the expert's rows padded to 16, so an expert of up to 128 rows streams its weights once).
    Plan pl = make_plan_tc(std::min(max_rows, 128), K, N, G, sms, smem_optin, false, ablate, false, E);
    pl.moe_E = E;
    pl.max_seg = active + (M + pl.m_chunk - 1) / pl.m_chunk;
    pl.grid = sms;  // persistent: the kernel spreads the segments it finds over all CTAs
    pl.units = 0;   // decided on the device
    pl.T = 0;
    const size_t counters = static_cast<size_t>(pl.max_seg) * ((pl.strips + kTcStrips - 1) / kTcStrips);
    pl.workspace = kStatusBytes + (counters * 4 + 255) / 256 * 256 +
                   2ull * pl.grid * (static_cast<size_t>(kTcStrips) * kStrip * pl.mb) * sizeof(float);
    return pl;
  }
  // Segment height: 8 rows when no expert has more, else 16.  Measured on GB300 (8 experts
  // K=4096 N=14336; 128 x K=2048 N=1536; 256 x K=7168 N=4096), 16-row segments beat 32-row
  // ones even at 32 rows per expert on average: an expert streamed twice at the 16-row
  // rate costs less than once at the 32-row rate of this kernel.
  Plan pl = make_plan_mma(max_rows <= 8 ? 8 : 16, K, N, G, sms, smem_optin, false, E, active, ablate);
  pl.moe_E = E;
  pl.max_seg = active + (M + pl.m_chunk - 1) / pl.m_chunk;
  pl.grid = sms;  // persistent: the kernel spreads the segments it finds over all CTAs
  pl.units = 0;   // decided on the device
  pl.T = 0;
  const size_t counters = static_cast<size_t>(pl.max_seg) * pl.strips;
  pl.workspace = kStatusBytes + (counters * 4 + 255) / 256 * 256 +
                 2ull * pl.grid * (static_cast<size_t>(kStrip) * pl.m_chunk) * sizeof(float);
  return pl;
}

Plan make_plan24(int M, int K, int N, int G, int sms, int smem_optin, int ablate) {
  return make_plan_mma(M, K, N, G, sms, smem_optin, false, 0, 1, ablate, true);
}

Plan make_plan(int M, int K, int N, int G, int sms, int smem_optin, bool zp, int forced_path, int ablate) {
  const bool tc = forced_path >= 2 || (forced_path != 1 && M >= kTcMinRows);
  const bool wide = forced_path == 4 || (forced_path != 3 && M >= kTcWideRows);
  return tc ? make_plan_tc(M, K, N, G, sms, smem_optin, zp, ablate, wide)
            : make_plan_mma(M, K, N, G, sms, smem_optin, zp, 0, 1, ablate);
}

int run_gemm(const Plan& pl, const GemmCall& c) {
  uint8_t* ws = static_cast<uint8_t*>(c.workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  uint32_t* counters = reinterpret_cast<uint32_t*>(ws + kStatusBytes);
  float* slots = reinterpret_cast<float*>(ws + kStatusBytes + counter_bytes(pl.strips));

  CUtensorMap map;
  // activation box depth: one 128-row chunk (2 pieces) per copy on path 2, one unit (kq pieces) on path 1
  // the no-swizzle ablation applies to the streaming kernel only
  const bool swz = pl.path == 2 || !(c.ablate & kAblateNoSwizzle);
  const int er = encode_a_map(&map, c.A, c.M, c.K, pl.m_chunk, pl.path == 2 ? 2 : pl.cfg.kq, swz);
  if (er != W4A16_OK) return er;

  if (pl.path == 2) {
    TcParams p{};
    p.packed = c.packed;
    p.scales = c.scales;
    p.zeros = c.zeros;
    p.bias = c.bias;
    p.C = c.C;
    p.status = status;
    p.counters = counters;
    p.slots = slots;
    p.M = c.M;
    p.K = c.K;
    p.N = c.N;
    p.G = c.G;
    p.strips = pl.strips;
    p.us = pl.us;
    p.mb = pl.mb;
    p.ch = pl.ch;
    p.na = pl.na;
    p.srows = pl.srows;
    p.KU = pl.KU;
    p.units = pl.units;
    p.T = pl.T;
    p.grid = pl.grid;
    p.a_stages = pl.a_stages;
    p.w_stages = pl.w_stages;
    p.a_stage_bytes = pl.tlay.a_stage_bytes;
    p.w_stage_bytes = pl.tlay.w_stage_bytes;
    p.w_base = pl.tlay.w_base;
    p.s_off = pl.tlay.s_off;
    p.z_off = pl.tlay.z_off;
    p.bar_off = pl.tlay.bar_off;
    p.flag_off = pl.tlay.flag_off;
    p.idesc = tc_idesc(128, pl.mb);
    p.wait_limit = c.wait_limit;
    p.debug_stall = c.debug_stall;
    p.ablate = c.ablate & ~kAblateNoSwizzle;
    for (int m0 = 0; m0 < c.M; m0 += pl.m_chunk) {
      p.m0 = m0;
      if (launch_gemm_tc(pl.smem_bytes, map, p, c.stream) != cudaSuccess)
        return W4A16_ERR_CUDA;
    }
    return W4A16_OK;
  }

  GemmParams p = mma_params(pl, c, status, counters, slots);
  for (int m0 = 0; m0 < c.M; m0 += pl.m_chunk) {
    p.m0 = m0;
    const cudaError_t e =
        pl.sp24 ? launch_gemm_sp24(pl.cfg, map, p, c.stream) : launch_gemm_mma(pl.cfg, map, p, c.stream);
    if (e != cudaSuccess) return W4A16_ERR_CUDA;
  }
  return W4A16_OK;
}

int run_moe_gemm(const Plan& pl, const GemmCall& c, const int* expert_off) {
  uint8_t* ws = static_cast<uint8_t*>(c.workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  uint32_t* counters = reinterpret_cast<uint32_t*>(ws + kStatusBytes);
  const int cols = pl.path == 2 ? (pl.strips + kTcStrips - 1) / kTcStrips : pl.strips;  // unit columns per segment
  const size_t ncount = static_cast<size_t>(pl.max_seg) * cols;
  float* slots = reinterpret_cast<float*>(ws + kStatusBytes + (ncount * 4 + 255) / 256 * 256);
  CUtensorMap map;
  if (pl.path == 2) {
    const int er = encode_a_map(&map, c.A, c.M, c.K, pl.m_chunk, 2, true);
    if (er != W4A16_OK) return er;
    TcParams p{};
    p.packed = c.packed;
    p.scales = c.scales;
    p.C = c.C;
    p.status = status;
    p.counters = counters;
    p.slots = slots;
    p.M = c.M;
    p.m0 = 0;
    p.K = c.K;
    p.N = c.N;
    p.G = c.G;
    p.strips = pl.strips;
    p.us = pl.us;
    p.mb = pl.mb;
    p.ch = pl.ch;
    p.na = pl.na;
    p.srows = pl.srows;
    p.KU = pl.KU;
    p.units = 0;
    p.T = 0;
    p.grid = pl.grid;
    p.a_stages = pl.a_stages;
    p.w_stages = pl.w_stages;
    p.a_stage_bytes = pl.tlay.a_stage_bytes;
    p.w_stage_bytes = pl.tlay.w_stage_bytes;
    p.w_base = pl.tlay.w_base;
    p.s_off = pl.tlay.s_off;
    p.z_off = pl.tlay.z_off;
    p.bar_off = pl.tlay.bar_off;
    p.flag_off = pl.tlay.flag_off;
    p.idesc = tc_idesc(128, pl.mb);
    p.wait_limit = c.wait_limit;
    p.debug_stall = c.debug_stall;
    p.ablate = c.ablate & ~kAblateNoSwizzle;
    p.expert_off = expert_off;
    p.E = pl.moe_E;
    p.max_seg = pl.max_seg;
    p.w_stride = static_cast<long long>(c.K) * c.N / 8;
    p.s_stride = static_cast<long long>(c.K / c.G) * c.N;
    p.moe_off = pl.tlay.moe_off;
    return launch_gemm_tc(pl.smem_bytes, map, p, c.stream) == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
  }
  const int er = encode_a_map(&map, c.A, c.M, c.K, pl.m_chunk, pl.cfg.kq, !(c.ablate & kAblateNoSwizzle));
  if (er != W4A16_OK) return er;
  GemmParams p = mma_params(pl, c, status, counters, slots);
  p.m0 = 0;
  p.expert_off = expert_off;
  p.E = pl.moe_E;
  p.strips = pl.strips;
  p.max_seg = pl.max_seg;
  p.w_stride = static_cast<long long>(c.K) * c.N / 8;
  p.s_stride = static_cast<long long>(c.K / c.G) * c.N;
  return launch_moe_mma(pl.cfg, map, p, c.stream) == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

}  // namespace w4a16
