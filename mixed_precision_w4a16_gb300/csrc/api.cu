// C ABI of the W4A16 library: argument checks, workspace handling, status.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/w4a16.h"
#include "internal.h"
#include "sparse24.h"

namespace {

using namespace w4a16;

constexpr int kMaxDevices = 64;
constexpr long long kDefaultWaitCycles = 2000000000LL;  // ~1 s at GB300 clocks

std::atomic<long long> g_wait_cycles{0};
std::atomic<int> g_stall{0};

// Per-device attributes, filled on the device's first use.  Host threads may call
// the library concurrently: the fields are written once under g_dev_mutex and
// published by the release store of `ready`; readers acquire it first.
struct DeviceInfo {
  std::atomic<int> ready{0};
  int major = 0, minor = 0;
  int sms = 0;
  int smem_optin = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

int current_device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return W4A16_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return W4A16_ERR_CUDA;
  DeviceInfo& d = g_dev[dev];
  if (!d.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!d.ready.load(std::memory_order_relaxed)) {
      int major = 0, minor = 0, sms = 0, smem = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return W4A16_ERR_CUDA;
      d.major = major;
      d.minor = minor;
      d.sms = sms;
      d.smem_optin = smem;
      d.ready.store(1, std::memory_order_release);
    }
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

std::atomic<int> g_force_path{0};
std::atomic<int> g_ablate{0};

Plan plan_for(int M, int K, int N, int G, const DeviceInfo* d, bool zp) {
  return make_plan(M, K, N, G, d->sms, d->smem_optin, zp, g_force_path.load(), g_ablate.load());
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
  const Plan pl =
      make_plan(M, K, N, effective_group(K, groupsize), sms, smem, false, g_force_path.load(), g_ablate.load());
  out->path = pl.path;
  out->m_tiles = pl.m_chunk / 8;
  out->m_chunk = pl.m_chunk;
  out->n_tile = pl.path == 2 ? pl.us * kStrip : kStrip;  // tensor-memory kernel: a strip pair, or one strip (wide)
  out->k_tile = pl.k_tile;
  out->units = pl.units;
  out->units_per_cta = pl.T;
  out->grid = pl.grid;
  out->stages = pl.stages;
  out->smem_bytes = pl.smem_bytes;
  out->threads = pl.threads;
  out->final_sum_warps = pl.path == 2 ? 16 : (pl.cfg.final8 ? 8 : 2);
  return W4A16_OK;
}

size_t w4a16_workspace_bytes(int M, int K, int N, int groupsize) {
  if (M < 0 || check_shape(K, N, groupsize) != W4A16_OK) return 0;
  DeviceInfo* d = nullptr;
  if (current_device_info(&d) != W4A16_OK) return 0;
  // enough for the GEMM with and without zero points
  const int G = effective_group(K, groupsize);
  return std::max(plan_for(M, K, N, G, d, false).workspace, plan_for(M, K, N, G, d, true).workspace);
}

void w4a16_debug_set_wait_cycles(long long cycles) { g_wait_cycles.store(cycles > 0 ? cycles : 0); }

void w4a16_debug_inject_stall(int enable) { g_stall.store(enable ? 1 : 0); }

void w4a16_debug_force_path(int path) { g_force_path.store(path >= 1 && path <= 4 ? path : 0); }

void w4a16_debug_ablate(int flags) { g_ablate.store(flags & (kAblateNoEvictFirst | kAblateStages2 | kAblateNoSwizzle)); }

int w4a16_repack(const uint8_t* q, const uint16_t* s, int K, int N, int groupsize, uint32_t* packed,
                 uint16_t* scales_p, void* stream) {
  const int st = check_shape(K, N, groupsize);
  if (st != W4A16_OK) return st;
  if (!q || !s || !packed || !scales_p) return W4A16_ERR_NULL;
  if (!aligned16(q) || !aligned16(s) || !aligned16(packed) || !aligned16(scales_p)) return W4A16_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  const int r = current_device_info(&d);
  if (r != W4A16_OK) return r;
  const cudaError_t e = launch_repack(q, s, K, N, effective_group(K, groupsize), packed, scales_p, d->sms,
                                      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

int w4a16_quantize_repack(const uint16_t* w, const uint16_t* s, int K, int N, int groupsize, uint32_t* packed,
                          uint16_t* scales_p, void* stream) {
  return w4a16_quantize_repack_zp(w, s, nullptr, K, N, groupsize, packed, scales_p, stream);
}

int w4a16_quantize_repack_zp(const uint16_t* w, const uint16_t* s, const uint8_t* z, int K, int N, int groupsize,
                             uint32_t* packed, uint16_t* scales_p, void* stream) {
  const int st = check_shape(K, N, groupsize);
  if (st != W4A16_OK) return st;
  if (!w || !s || !packed || !scales_p) return W4A16_ERR_NULL;
  if (!aligned16(w) || !aligned16(s) || !aligned16(packed) || !aligned16(scales_p) || (z && !aligned16(z)))
    return W4A16_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  const int r = current_device_info(&d);
  if (r != W4A16_OK) return r;
  const cudaError_t e = launch_quantize_repack(w, s, z, K, N, effective_group(K, groupsize), packed, scales_p,
                                               d->sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

int w4a16_minmax_scales(const uint16_t* w, int K, int N, int groupsize, uint16_t* s, uint8_t* z, void* stream) {
  const int st = check_shape(K, N, groupsize);
  if (st != W4A16_OK) return st;
  if (!w || !s) return W4A16_ERR_NULL;
  if (!aligned16(w) || !aligned16(s) || (z && !aligned16(z))) return W4A16_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  const int r = current_device_info(&d);
  if (r != W4A16_OK) return r;
  const cudaError_t e = launch_minmax_scales(w, K, N, effective_group(K, groupsize), s, z,
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
  const int ablate = g_ablate.load();  // one read: the plan and the launch see the same switches
  const Plan pl = make_plan(M, K, N, G, d->sms, d->smem_optin, zeros_p != nullptr, g_force_path.load(), ablate);
  if (workspace_bytes < pl.workspace) return W4A16_ERR_WORKSPACE;

  const long long wc = g_wait_cycles.load();
  GemmCall c{};
  c.A = A;
  c.packed = packed;
  c.scales = scales_p;
  c.zeros = zeros_p;
  c.bias = bias;
  c.C = C;
  c.M = M;
  c.K = K;
  c.N = N;
  c.G = G;
  c.workspace = workspace;
  c.wait_limit = wc > 0 ? wc : kDefaultWaitCycles;
  c.debug_stall = g_stall.load();
  c.ablate = ablate;
  c.stream = static_cast<cudaStream_t>(stream);
  return run_gemm(pl, c);
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
// Grouped expert GEMM
// ---------------------------------------------------------------------------
namespace {

constexpr int kMoeMaxRows = 1 << 24;

// Checks the grouped GEMM's sizes and plans it on this device (status in *st).
Plan moe_plan(int E, int M, int max_rows, int K, int N, int groupsize, int ablate, int* st) {
  Plan pl{};
  *st = check_shape(K, N, groupsize);
  if (*st != W4A16_OK) return pl;
  if (E < 1 || E > kMoeMaxExperts || M < 0 || M > kMoeMaxRows) {
    *st = W4A16_ERR_SHAPE;
    return pl;
  }
  DeviceInfo* d = nullptr;
  *st = current_device_info(&d);
  if (*st != W4A16_OK) return pl;
  const int rows = (max_rows <= 0 || max_rows > M) ? std::max(M, 1) : max_rows;
  pl = make_plan_moe(E, std::max(M, 1), rows, K, N, effective_group(K, groupsize), d->sms, d->smem_optin, ablate,
                     g_force_path.load());
  // the counters (one per segment and strip) and the unit count stay well inside int
  if (static_cast<long long>(pl.max_seg) * pl.strips * pl.KU > (1LL << 30)) *st = W4A16_ERR_SHAPE;
  return pl;
}

}  // namespace

extern "C" {

size_t w4a16_moe_workspace_bytes(int E, int M, int max_rows, int K, int N, int groupsize) {
  int st = 0;
  const Plan pl = moe_plan(E, M, max_rows, K, N, groupsize, 0, &st);
  return st == W4A16_OK ? pl.workspace : 0;
}

int w4a16_moe_gemm(const uint16_t* A, const uint32_t* packed, const uint16_t* scales_p, const int32_t* expert_offsets,
                   uint16_t* C, int E, int M, int max_rows, int K, int N, int groupsize, void* workspace,
                   size_t workspace_bytes, void* stream) {
  int st = 0;
  const int ablate = g_ablate.load();
  const Plan pl = moe_plan(E, M, max_rows, K, N, groupsize, ablate, &st);
  if (st != W4A16_OK) return st;
  if (M == 0) return W4A16_OK;
  if (!A || !packed || !scales_p || !expert_offsets || !C) return W4A16_ERR_NULL;
  if (!workspace) return W4A16_ERR_WORKSPACE;
  if (!aligned16(A) || !aligned16(packed) || !aligned16(scales_p) || !aligned16(C) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(expert_offsets) & 3u) != 0)
    return W4A16_ERR_ALIGN;
  if (workspace_bytes < pl.workspace) return W4A16_ERR_WORKSPACE;
  const long long wc = g_wait_cycles.load();
  GemmCall c{};
  c.A = A;
  c.packed = packed;
  c.scales = scales_p;
  c.C = C;
  c.M = M;
  c.K = K;
  c.N = N;
  c.G = effective_group(K, groupsize);
  c.workspace = workspace;
  c.wait_limit = wc > 0 ? wc : kDefaultWaitCycles;
  c.debug_stall = g_stall.load();
  c.ablate = ablate;
  c.stream = static_cast<cudaStream_t>(stream);
  return run_moe_gemm(pl, c, expert_offsets);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// 2:4-sparse W4A16
// ---------------------------------------------------------------------------
extern "C" {

size_t w4a16_packed24_bytes(int K, int N) {
  if (K <= 0 || N <= 0 || K % 128 != 0 || N % 128 != 0) return 0;
  return static_cast<size_t>(K) * static_cast<size_t>(N) * 3 / 8;
}

int w4a16_repack_24(const uint8_t* q, const uint16_t* s, int K, int N, int groupsize, uint32_t* packed24,
                    uint16_t* scales_p, void* stream) {
  const int st = check_shape(K, N, groupsize);
  if (st != W4A16_OK) return st;
  if (!q || !s || !packed24 || !scales_p) return W4A16_ERR_NULL;
  if (!aligned16(q) || !aligned16(s) || !aligned16(packed24) || !aligned16(scales_p)) return W4A16_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  const int r = current_device_info(&d);
  if (r != W4A16_OK) return r;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (launch_repack24(q, K, N, packed24, cs) != cudaSuccess) return W4A16_ERR_CUDA;
  return launch_permute_scales(s, K, N, effective_group(K, groupsize), scales_p, cs) == cudaSuccess
             ? W4A16_OK
             : W4A16_ERR_CUDA;
}

int w4a16_unpack_24(const uint32_t* packed24, int K, int N, uint8_t* q, void* stream) {
  if (K <= 0 || N <= 0 || K % 128 != 0 || N % 128 != 0) return W4A16_ERR_SHAPE;
  if (!packed24 || !q) return W4A16_ERR_NULL;
  if (!aligned16(packed24) || !aligned16(q)) return W4A16_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  const int r = current_device_info(&d);
  if (r != W4A16_OK) return r;
  return launch_unpack24(packed24, K, N, q, static_cast<cudaStream_t>(stream)) == cudaSuccess ? W4A16_OK
                                                                                              : W4A16_ERR_CUDA;
}

size_t w4a16_workspace_bytes_24(int M, int K, int N, int groupsize) {
  if (M < 0 || check_shape(K, N, groupsize) != W4A16_OK) return 0;
  DeviceInfo* d = nullptr;
  if (current_device_info(&d) != W4A16_OK) return 0;
  return make_plan24(M, K, N, effective_group(K, groupsize), d->sms, d->smem_optin, g_ablate.load()).workspace;
}

int w4a16_gemm_24(const uint16_t* A, const uint32_t* packed24, const uint16_t* scales_p, uint16_t* C, int M, int K,
                  int N, int groupsize, void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 0) return W4A16_ERR_SHAPE;
  const int st = check_shape(K, N, groupsize);
  if (st != W4A16_OK) return st;
  if (M == 0) return W4A16_OK;
  if (!A || !packed24 || !scales_p || !C) return W4A16_ERR_NULL;
  if (!workspace) return W4A16_ERR_WORKSPACE;
  if (!aligned16(A) || !aligned16(packed24) || !aligned16(scales_p) || !aligned16(C) || !aligned16(workspace))
    return W4A16_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  const int r = current_device_info(&d);
  if (r != W4A16_OK) return r;
  const int G = effective_group(K, groupsize);
  const int ablate = g_ablate.load();
  const Plan pl = make_plan24(M, K, N, G, d->sms, d->smem_optin, ablate);
  if (workspace_bytes < pl.workspace) return W4A16_ERR_WORKSPACE;
  const long long wc = g_wait_cycles.load();
  GemmCall c{};
  c.A = A;
  c.packed = packed24;
  c.scales = scales_p;
  c.C = C;
  c.M = M;
  c.K = K;
  c.N = N;
  c.G = G;
  c.workspace = workspace;
  c.wait_limit = wc > 0 ? wc : kDefaultWaitCycles;
  c.debug_stall = g_stall.load();
  c.ablate = ablate;
  c.stream = static_cast<cudaStream_t>(stream);
  return run_gemm(pl, c);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant: the scratch is a file-scope device array of the
// library, looked up once per device with cudaGetSymbolAddress.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[W4A16_NOALLOC_SCRATCH_BYTES];
// Device address of g_noalloc_scratch, per device; null until that device's first call.
// Concurrent first calls may both look it up; they store the same address.
std::atomic<void*> g_noalloc_addr[kMaxDevices];

// The scratch array of the current device, or null if no call has set it up yet.
void* noalloc_scratch_if_ready() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  return g_noalloc_addr[dev].load(std::memory_order_acquire);
}

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
  const Plan pl = plan_for(M, K, N, effective_group(K, groupsize), d, false);
  if (pl.workspace > W4A16_NOALLOC_SCRATCH_BYTES) return W4A16_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return W4A16_ERR_CUDA;
  void* ws = g_noalloc_addr[dev].load(std::memory_order_acquire);
  if (!ws) {
    void* addr = nullptr;  // set-up on this device's first call (must precede any stream capture)
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || !addr) return W4A16_ERR_CUDA;
    g_noalloc_addr[dev].store(addr, std::memory_order_release);
    ws = addr;
  }
  // The arrival counters must start at zero (a timed-out call can leave them set); the
  // partial-sum slots need not.  The status word at the head is left alone: it is
  // sticky until w4a16_get_status(NULL, stream) reads and clears it, so a timeout in
  // one call stays visible however many calls follow.
  if (cudaMemsetAsync(static_cast<uint8_t*>(ws) + kStatusBytes, 0, counter_bytes(pl.strips),
                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return W4A16_ERR_CUDA;
  return w4a16_gemm(A, packed, scales_p, C, M, K, N, groupsize, ws, W4A16_NOALLOC_SCRATCH_BYTES, stream);
}

int w4a16_get_status(void* workspace, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return W4A16_ERR_CUDA;
  unsigned int flag = 0, flag24 = 0;
  if (read_and_clear_repack_flag(&flag, s) != cudaSuccess) return W4A16_ERR_CUDA;
  if (read_and_clear_sparse_flag(&flag24, s) != cudaSuccess) return W4A16_ERR_CUDA;
  flag |= flag24;
  uint32_t word = 0;
  // Without a workspace, the allocation-free GEMM's status word (in the library's
  // scratch array, if a call has set it up on this device) is the one reported.
  if (!workspace) workspace = noalloc_scratch_if_ready();
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
  if (word & kDevErrValue) return W4A16_ERR_VALUE;
  if (word) return W4A16_ERR_CUDA;
  return W4A16_OK;
}

}  // extern "C"
