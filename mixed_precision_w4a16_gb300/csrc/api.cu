// C ABI of the W4A16 library: argument checks, work planning, launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>

#include "../../include/w4a16.h"
#include "internal.h"

namespace {

using namespace w4a16;

constexpr int kMaxDevices = 64;
constexpr long long kDefaultWaitCycles = 2000000000LL;  // ~1 s at GB300 clocks
constexpr size_t kStatusBytes = 256;

std::atomic<long long> g_wait_cycles{0};
std::atomic<int> g_stall{0};

struct DeviceInfo {
  int ready = 0;
  int major = 0, minor = 0;
  int sms = 0;
  int smem_optin = 0;
};
DeviceInfo g_dev[kMaxDevices];

int current_device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return W4A16_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return W4A16_ERR_CUDA;
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return W4A16_ERR_CUDA;
    d.ready = 1;
  }
  *out = &d;
  return (d.major == 10 && d.minor == 3) ? W4A16_OK : W4A16_ERR_ARCH;
}

int effective_group(int K, int groupsize) {
  if (groupsize == -1 || groupsize == K) return K;
  if (groupsize == 128) return 128;
  return 0;
}

int check_shape(int K, int N, int groupsize) {
  if (K <= 0 || N <= 0 || K % 128 != 0 || N % 128 != 0) return W4A16_ERR_SHAPE;
  const int G = effective_group(K, groupsize);
  if (G == 0 || K % G != 0) return W4A16_ERR_GROUP;
  return W4A16_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Work plan: which kernel runs and how it splits (M, K, N) over `sms` SMs with
// `smem_optin` bytes of shared memory per CTA.
constexpr int kTcMinRows = 17;  // from 17 token rows on, the tensor-memory kernel runs

struct Plan {
  int path;          // 1 = streaming mma.sync kernel, 2 = tensor-memory (tcgen05) kernel
  MmaConfig cfg;     // path 1
  MmaLayout lay;     // path 1
  TcLayout tlay;     // path 2
  int mb, ch;        // path 2: token rows per launch (multiple of 16), 128-row chunks per unit
  int a_stages, w_stages;  // path 2: activation / weight ring depths
  int ni, na;        // path 2: MMA issuers (accumulators), A chunks in tensor memory (= a_stages)
  int m_chunk;       // token rows per launch
  int k_tile;        // reduction rows per work unit
  int srows;
  int KU, strips, units, T, grid, stages, smem_bytes, threads;
  size_t workspace;
};

void finish_split(Plan& pl, int K, int sms, size_t slot_floats) {
  pl.KU = K / pl.k_tile;
  pl.units = pl.strips * pl.KU;
  pl.T = (pl.units + sms - 1) / sms;
  pl.grid = (pl.units + pl.T - 1) / pl.T;
  const size_t counters = (static_cast<size_t>(pl.strips) * 4 + 255) / 256 * 256;
  pl.workspace = kStatusBytes + counters + 2ull * pl.grid * slot_floats * sizeof(float);
}

Plan make_plan_mma(int M, int K, int N, int G, int sms, int smem_optin, bool zp) {
  Plan pl{};
  pl.path = 1;
  const int mc = std::min(std::max(M, 1), 32);
  const int mt = mc <= 8 ? 1 : mc <= 16 ? 2 : 4;
  pl.strips = N / kStrip;
  // Unit depth KT = 64 * kq.  Per-SM time of a unit is modelled from copy-engine
  // measurements on GB300: ~89 ns per 4 KB of weights streamed plus ~80 ns of
  // fixed cost for the unit's three copy operations.  Pick the kq minimising
  // T * unit time among those that keep >= 3 pipeline stages in shared memory.
  int best_kq = 0;
  long long best_cost = 0;
  const int cands[3] = {8, 4, 2};
  for (int c = 0; c < 3; ++c) {
    const int kq = cands[c];
    if (K % (64 * kq) != 0) continue;
    const int srows = (G <= 64 * kq) ? (64 * kq) / G : 1;
    const MmaLayout l0 = mma_layout(mt, kq, srows, 0, zp);
    const int stages = (smem_optin - l0.smem_bytes) / (l0.stage_bytes + 16);
    if (stages < 3 && kq != 2) continue;
    const long long units = static_cast<long long>(pl.strips) * (K / (64 * kq));
    const long long T = (units + sms - 1) / sms;
    const long long cost = T * (89LL * kq + 80);
    if (best_kq == 0 || cost < best_cost) {
      best_kq = kq;
      best_cost = cost;
    }
  }
  if (!best_kq) best_kq = 2;
  const int kq = best_kq;
  const int KT = 64 * kq;
  pl.srows = (G <= KT) ? KT / G : 1;
  const MmaLayout l0 = mma_layout(mt, kq, pl.srows, 0, zp);
  int stages = (smem_optin - l0.smem_bytes) / (l0.stage_bytes + 16);
  stages = std::max(2, std::min(stages, 8));
  pl.lay = mma_layout(mt, kq, pl.srows, stages, zp);
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
  return pl;
}

Plan make_plan_tc(int M, int K, int N, int G, int sms, int smem_optin, bool zp) {
  Plan pl{};
  pl.path = 2;
  pl.mb = std::min(128, (std::max(M, 1) + 15) / 16 * 16);
  pl.strips = N / kStrip;
  // Tensor memory (512 columns): ni accumulators of mb columns (ni * mb <= 256),
  // the rest for the ring of 64-column A chunks.  Activation stages pair with the
  // A buffers (one per chunk in flight).
  pl.ni = 1;  // a power of two: issuer i takes the chunks gc = i mod ni
  while (2 * pl.ni <= std::min(kTcMaxIssuers, 256 / pl.mb)) pl.ni *= 2;
  pl.na = std::min(6, (512 - pl.ni * pl.mb) / 64) & ~1;  // even: two activation producers take alternate chunks
  // Unit depth KT = 128 * ch for the weight ring (one copy per unit, released by
  // the dequant warps).  Keep >= 8 chunks of weights in flight; among the
  // candidates, minimise T * unit time (memory time as for the streaming kernel
  // vs tensor time, ~2.1 ns per mb * ch).
  int best = 0, best_w = 0;
  long long best_cost = 0;
  const int cands[3] = {4, 2, 1};
  for (int c = 0; c < 3; ++c) {
    const int ch = cands[c];
    if (K % (128 * ch) != 0) continue;
    const int srows = (G == 128) ? ch : 1;
    const TcLayout l0 = tc_layout(pl.mb, ch, srows, pl.na, 0, zp);
    const int w_st = std::min(12, (smem_optin - l0.smem_bytes) / (l0.w_stage_bytes + 16));
    if (w_st < 2 || w_st * ch < 8) continue;
    const long long units = static_cast<long long>(pl.strips) * (K / (128 * ch));
    const long long T = (units + sms - 1) / sms;
    const long long cost = T * (std::max(178LL * ch, (21LL * pl.mb * ch) / 10) + 200);  // + per-unit sync and copy issue
    if (best == 0 || cost < best_cost) {
      best = ch;
      best_w = w_st;
      best_cost = cost;
    }
  }
  if (!best) {
    best = 1;
    const TcLayout l0 = tc_layout(pl.mb, 1, 1, pl.na, 0, zp);
    best_w = std::max(2, std::min(12, (smem_optin - l0.smem_bytes) / (l0.w_stage_bytes + 16)));
  }
  pl.ch = best;
  pl.srows = (G == 128) ? pl.ch : 1;
  pl.tlay = tc_layout(pl.mb, pl.ch, pl.srows, pl.na, best_w, zp);
  pl.a_stages = pl.na;
  pl.w_stages = best_w;
  pl.m_chunk = pl.mb;
  pl.k_tile = 128 * pl.ch;
  pl.stages = best_w;
  pl.smem_bytes = pl.tlay.smem_bytes;
  pl.threads = kTcThreads;
  finish_split(pl, K, sms, static_cast<size_t>(kStrip) * pl.mb);
  return pl;
}

std::atomic<int> g_force_path{0};

// zp: the GEMM reads zero points (their rows take shared-memory stage space next to the scales)
Plan make_plan(int M, int K, int N, int G, int sms, int smem_optin, bool zp = false) {
  const int forced = g_force_path.load();
  const bool tc = forced == 2 || (forced == 0 && M >= kTcMinRows);
  return tc ? make_plan_tc(M, K, N, G, sms, smem_optin, zp) : make_plan_mma(M, K, N, G, sms, smem_optin, zp);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 3-D view of A (fp16[M][K]) as [K/64][M][64]: box {64, box_rows, kq} fetches the
// kq 64-column pieces of one work unit in one copy, each piece box_rows x 128 bytes
// with the 128-byte swizzle; rows beyond M are zero-filled.
int encode_a_map(CUtensorMap* map, const uint16_t* A, int M, int K, int box_rows, int kq) {
  auto enc = get_encoder();
  if (!enc) return W4A16_ERR_CUDA;
  const cuuint64_t dims[3] = {64u, static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128u};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(kq)};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<uint16_t*>(A), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? W4A16_OK : W4A16_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* w4a16_status_string(int status) {
  switch (status) {
    case W4A16_OK: return "W4A16_OK";
    case W4A16_ERR_NULL: return "W4A16_ERR_NULL";
    case W4A16_ERR_SHAPE: return "W4A16_ERR_SHAPE";
    case W4A16_ERR_GROUP: return "W4A16_ERR_GROUP";
    case W4A16_ERR_CODE_RANGE: return "W4A16_ERR_CODE_RANGE";
    case W4A16_ERR_WORKSPACE: return "W4A16_ERR_WORKSPACE";
    case W4A16_ERR_CUDA: return "W4A16_ERR_CUDA";
    case W4A16_ERR_TIMEOUT: return "W4A16_ERR_TIMEOUT";
    case W4A16_ERR_ARCH: return "W4A16_ERR_ARCH";
    case W4A16_ERR_ALIGN: return "W4A16_ERR_ALIGN";
    case W4A16_ERR_VALUE: return "W4A16_ERR_VALUE";
    default: return "W4A16_ERR_UNKNOWN";
  }
}

int w4a16_abi_version(void) { return 1; }

size_t w4a16_packed_bytes(int K, int N) {
  if (K <= 0 || N <= 0 || K % 128 != 0 || N % 128 != 0) return 0;
  return static_cast<size_t>(K) * static_cast<size_t>(N) / 2;
}

size_t w4a16_scales_count(int K, int N, int groupsize) {
  if (check_shape(K, N, groupsize) != W4A16_OK) return 0;
  return static_cast<size_t>(K / effective_group(K, groupsize)) * static_cast<size_t>(N);
}

int w4a16_plan(int M, int K, int N, int groupsize, int num_sms, w4a16_plan_t* out) {
  if (!out) return W4A16_ERR_NULL;
  if (M < 0) return W4A16_ERR_SHAPE;
  const int st = check_shape(K, N, groupsize);
  if (st != W4A16_OK) return st;
  int sms = num_sms;
  int smem = 232448;  // sm_100-class opt-in shared memory per block
  if (sms <= 0) {
    DeviceInfo* d = nullptr;
    const int r = current_device_info(&d);
    if (r != W4A16_OK) return r;
    sms = d->sms;
    smem = d->smem_optin;
  }
  const Plan pl = make_plan(M, K, N, effective_group(K, groupsize), sms, smem);
  out->path = pl.path;
  out->m_tiles = pl.m_chunk / 8;
  out->m_chunk = pl.m_chunk;
  out->n_tile = kStrip;
  out->k_tile = pl.k_tile;
  out->units = pl.units;
  out->units_per_cta = pl.T;
  out->grid = pl.grid;
  out->stages = pl.stages;
  out->smem_bytes = pl.smem_bytes;
  out->threads = pl.threads;
  return W4A16_OK;
}

size_t w4a16_workspace_bytes(int M, int K, int N, int groupsize) {
  if (M < 0 || check_shape(K, N, groupsize) != W4A16_OK) return 0;
  DeviceInfo* d = nullptr;
  if (current_device_info(&d) != W4A16_OK) return 0;
  // enough for the GEMM with and without zero points
  const int G = effective_group(K, groupsize);
  return std::max(make_plan(M, K, N, G, d->sms, d->smem_optin, false).workspace,
                  make_plan(M, K, N, G, d->sms, d->smem_optin, true).workspace);
}

void w4a16_debug_set_wait_cycles(long long cycles) { g_wait_cycles.store(cycles > 0 ? cycles : 0); }

void w4a16_debug_inject_stall(int enable) { g_stall.store(enable ? 1 : 0); }

void w4a16_debug_force_path(int path) { g_force_path.store(path == 1 || path == 2 ? path : 0); }

int w4a16_repack(const uint8_t* q, const uint16_t* s, int K, int N, int groupsize, uint32_t* packed,
                 uint16_t* scales_p, void* stream) {
  const int st = check_shape(K, N, groupsize);
  if (st != W4A16_OK) return st;
  if (!q || !s || !packed || !scales_p) return W4A16_ERR_NULL;
  if (!aligned16(q) || !aligned16(s) || !aligned16(packed) || !aligned16(scales_p)) return W4A16_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  const int r = current_device_info(&d);
  if (r != W4A16_OK) return r;
  const cudaError_t e = launch_repack(q, s, K, N, effective_group(K, groupsize), packed, scales_p,
                                      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

int w4a16_quantize_repack(const uint16_t* w, const uint16_t* s, int K, int N, int groupsize, uint32_t* packed,
                          uint16_t* scales_p, void* stream) {
  const int st = check_shape(K, N, groupsize);
  if (st != W4A16_OK) return st;
  if (!w || !s || !packed || !scales_p) return W4A16_ERR_NULL;
  if (!aligned16(w) || !aligned16(s) || !aligned16(packed) || !aligned16(scales_p)) return W4A16_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  const int r = current_device_info(&d);
  if (r != W4A16_OK) return r;
  const cudaError_t e = launch_quantize_repack(w, s, K, N, effective_group(K, groupsize), packed, scales_p,
                                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

int w4a16_unpack(const uint32_t* packed, const uint16_t* scales_p, int K, int N, int groupsize, uint8_t* q,
                 uint16_t* s, void* stream) {
  const int st = check_shape(K, N, groupsize);
  if (st != W4A16_OK) return st;
  if (!q || !s || !packed || !scales_p) return W4A16_ERR_NULL;
  if (!aligned16(q) || !aligned16(s) || !aligned16(packed) || !aligned16(scales_p)) return W4A16_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  const int r = current_device_info(&d);
  if (r != W4A16_OK) return r;
  const cudaError_t e = launch_unpack(packed, scales_p, K, N, effective_group(K, groupsize), q, s,
                                      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

int w4a16_dequant(const uint32_t* packed, const uint16_t* scales_p, int K, int N, int groupsize, uint16_t* Bhat,
                  void* stream) {
  const int st = check_shape(K, N, groupsize);
  if (st != W4A16_OK) return st;
  if (!packed || !scales_p || !Bhat) return W4A16_ERR_NULL;
  if (!aligned16(packed) || !aligned16(scales_p) || !aligned16(Bhat)) return W4A16_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  const int r = current_device_info(&d);
  if (r != W4A16_OK) return r;
  const cudaError_t e = launch_dequant(packed, scales_p, nullptr, K, N, effective_group(K, groupsize), Bhat,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

}  // extern "C"

namespace {

// The GEMM behind w4a16_gemm and w4a16_gemm_zp (zeros_p and bias may be null).
int gemm_impl(const uint16_t* A, const uint32_t* packed, const uint16_t* scales_p, const uint8_t* zeros_p,
              const uint16_t* bias, uint16_t* C, int M, int K, int N, int groupsize, void* workspace,
              size_t workspace_bytes, void* stream) {
  if (M < 0) return W4A16_ERR_SHAPE;
  const int st = check_shape(K, N, groupsize);
  if (st != W4A16_OK) return st;
  if (M == 0) return W4A16_OK;
  if (!A || !packed || !scales_p || !C) return W4A16_ERR_NULL;
  if (!workspace) return W4A16_ERR_WORKSPACE;
  if (!aligned16(A) || !aligned16(packed) || !aligned16(scales_p) || !aligned16(C) || !aligned16(workspace) ||
      (zeros_p && !aligned16(zeros_p)) || (bias && !aligned16(bias)))
    return W4A16_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  const int r = current_device_info(&d);
  if (r != W4A16_OK) return r;
  const int G = effective_group(K, groupsize);
  const Plan pl = make_plan(M, K, N, G, d->sms, d->smem_optin, zeros_p != nullptr);
  if (workspace_bytes < pl.workspace) return W4A16_ERR_WORKSPACE;

  const long long wc = g_wait_cycles.load();
  const long long wait_limit = wc > 0 ? wc : kDefaultWaitCycles;
  const int stall = g_stall.load();
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  uint32_t* counters = reinterpret_cast<uint32_t*>(ws + kStatusBytes);
  float* slots = reinterpret_cast<float*>(ws + kStatusBytes + (static_cast<size_t>(pl.strips) * 4 + 255) / 256 * 256);

  CUtensorMap map;
  // activation box depth: one 128-row chunk (2 pieces) per copy on path 2, one unit (kq pieces) on path 1
  const int er = encode_a_map(&map, A, M, K, pl.m_chunk, pl.path == 2 ? 2 : pl.cfg.kq);
  if (er != W4A16_OK) return er;

  if (pl.path == 2) {
    TcParams p{};
    p.packed = packed;
    p.scales = scales_p;
    p.zeros = zeros_p;
    p.bias = bias;
    p.C = C;
    p.status = status;
    p.counters = counters;
    p.slots = slots;
    p.M = M;
    p.K = K;
    p.N = N;
    p.G = G;
    p.mb = pl.mb;
    p.ch = pl.ch;
    p.ni = pl.ni;
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
    p.z_off = pl.tlay.z_off;
    p.bar_off = pl.tlay.bar_off;
    p.flag_off = pl.tlay.flag_off;
    p.idesc = tc_idesc(128, pl.mb);
    p.wait_limit = wait_limit;
    p.debug_stall = stall;
    for (int m0 = 0; m0 < M; m0 += pl.m_chunk) {
      p.m0 = m0;
      if (launch_gemm_tc(pl.smem_bytes, map, p, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return W4A16_ERR_CUDA;
    }
    return W4A16_OK;
  }

  GemmParams p{};
  p.packed = packed;
  p.scales = scales_p;
  p.zeros = zeros_p;
  p.bias = bias;
  p.C = C;
  p.status = status;
  p.counters = counters;
  p.slots = slots;
  p.M = M;
  p.K = K;
  p.N = N;
  p.G = G;
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
  p.wait_limit = wait_limit;
  p.debug_stall = stall;
  for (int m0 = 0; m0 < M; m0 += pl.m_chunk) {
    p.m0 = m0;
    const cudaError_t e = launch_gemm_mma(pl.cfg, map, p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return W4A16_ERR_CUDA;
  }
  return W4A16_OK;
}

}  // namespace

extern "C" {

int w4a16_gemm(const uint16_t* A, const uint32_t* packed, const uint16_t* scales_p, uint16_t* C, int M, int K, int N,
               int groupsize, void* workspace, size_t workspace_bytes, void* stream) {
  return gemm_impl(A, packed, scales_p, nullptr, nullptr, C, M, K, N, groupsize, workspace, workspace_bytes, stream);
}

int w4a16_gemm_zp(const uint16_t* A, const uint32_t* packed, const uint16_t* scales_p, const uint8_t* zeros_p,
                  const uint16_t* bias, uint16_t* C, int M, int K, int N, int groupsize, void* workspace,
                  size_t workspace_bytes, void* stream) {
  return gemm_impl(A, packed, scales_p, zeros_p, bias, C, M, K, N, groupsize, workspace, workspace_bytes, stream);
}

int w4a16_repack_zeros(const uint8_t* z, int K, int N, int groupsize, uint8_t* zeros_p, void* stream) {
  const int st = check_shape(K, N, groupsize);
  if (st != W4A16_OK) return st;
  if (!z || !zeros_p) return W4A16_ERR_NULL;
  if (!aligned16(z) || !aligned16(zeros_p)) return W4A16_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  const int r = current_device_info(&d);
  if (r != W4A16_OK) return r;
  const cudaError_t e =
      launch_repack_zeros(z, K, N, effective_group(K, groupsize), zeros_p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

int w4a16_dequant_zp(const uint32_t* packed, const uint16_t* scales_p, const uint8_t* zeros_p, int K, int N,
                     int groupsize, uint16_t* Bhat, void* stream) {
  const int st = check_shape(K, N, groupsize);
  if (st != W4A16_OK) return st;
  if (!packed || !scales_p || !zeros_p || !Bhat) return W4A16_ERR_NULL;
  if (!aligned16(packed) || !aligned16(scales_p) || !aligned16(zeros_p) || !aligned16(Bhat)) return W4A16_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  const int r = current_device_info(&d);
  if (r != W4A16_OK) return r;
  const cudaError_t e = launch_dequant(packed, scales_p, zeros_p, K, N, effective_group(K, groupsize), Bhat,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant: the scratch is a file-scope device array of the
// library, looked up once per device with cudaGetSymbolAddress.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[W4A16_NOALLOC_SCRATCH_BYTES];
void* g_noalloc_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device

}  // namespace

extern "C" {

int w4a16_gemm_noalloc(const uint16_t* A, const uint32_t* packed, const uint16_t* scales_p, uint16_t* C, int M, int K,
                       int N, int groupsize, void* stream) {
  if (M < 0) return W4A16_ERR_SHAPE;
  const int st = check_shape(K, N, groupsize);
  if (st != W4A16_OK) return st;
  if (M == 0) return W4A16_OK;
  if (!A || !packed || !scales_p || !C) return W4A16_ERR_NULL;
  DeviceInfo* d = nullptr;
  const int r = current_device_info(&d);
  if (r != W4A16_OK) return r;
  const Plan pl = make_plan(M, K, N, effective_group(K, groupsize), d->sms, d->smem_optin);
  if (pl.workspace > W4A16_NOALLOC_SCRATCH_BYTES) return W4A16_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return W4A16_ERR_CUDA;
  if (!g_noalloc_addr[dev]) {
    void* addr = nullptr;  // set-up on this device's first call (must precede any stream capture)
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || !addr) return W4A16_ERR_CUDA;
    g_noalloc_addr[dev] = addr;
  }
  void* ws = g_noalloc_addr[dev];
  // the status word and the arrival counters must start at zero; the partial-sum slots need not
  const size_t clear = kStatusBytes + (static_cast<size_t>(pl.strips) * 4 + 255) / 256 * 256;
  if (cudaMemsetAsync(ws, 0, clear, static_cast<cudaStream_t>(stream)) != cudaSuccess) return W4A16_ERR_CUDA;
  return w4a16_gemm(A, packed, scales_p, C, M, K, N, groupsize, ws, W4A16_NOALLOC_SCRATCH_BYTES, stream);
}

int w4a16_get_status(void* workspace, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return W4A16_ERR_CUDA;
  unsigned int flag = 0;
  if (read_and_clear_repack_flag(&flag, s) != cudaSuccess) return W4A16_ERR_CUDA;
  uint32_t word = 0;
  if (workspace) {
    if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return W4A16_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return W4A16_ERR_CUDA;
    if (word && cudaMemsetAsync(workspace, 0, sizeof(word), s) != cudaSuccess) return W4A16_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return W4A16_ERR_CUDA;
  }
  if (flag & kDevErrCodeRange) return W4A16_ERR_CODE_RANGE;
  if (flag & kDevErrValue) return W4A16_ERR_VALUE;
  if (word & kDevErrTimeout) return W4A16_ERR_TIMEOUT;
  if (word) return W4A16_ERR_CUDA;
  return W4A16_OK;
}

}  // extern "C"
