// Offline repack of 4-bit codes and FP16 scales into the GEMM's fragment
// order, the quantiser in front of it (min-max scales, codes from FP16
// weights), plus the two diagnostic inverses (unpack, dequantise).
//
// Layout (see include/w4a16.h): packed uint32[N/128][K/64][8][32][4] --
// 128-column strips stored contiguously along K; inside a strip, for each
// 64-row block, the 8 tiles of 16 columns x 64 rows follow each other.  Word
// j of lane L in a tile covers the 16x16 block with reduction rows 16j ..;
// nibble slot i < 4 / i + 4 = low / high half of register i.  Register i
// holds block row g + 8*(i & 1) and reduction indices 4t + 2*(i >> 1) + {0, 1},
// with g = L / 4 and t = L % 4: four consecutive k of rows g and g + 8, the
// per-thread fragment of a 16-lane x 256-bit tensor-memory store, and (with k
// permuted inside the block) the m16n8k16 A-operand fragment.  Permuted
// scales: fp16[N/128][K/G][128],
// within each 16-column block fragment rows r and r + 8 side by side.
//
// Kernels here walk the layout from the word side (word -> positions); one
// thread owns one lane's 16-byte vector (four words), so every store of the
// packed stream is a coalesced 16-byte store.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"
#include "sparse24.h"

namespace w4a16 {

// Repack error flag (code-range violations), read and cleared by w4a16_get_status.
__device__ unsigned int g_repack_flag;

namespace {

struct VecCoord {
  int nb, kb, lane;  // nb: global 16-column block
};

__device__ __forceinline__ VecCoord vec_coord(long long v, int K) {
  const int kTiles = K / 64;
  VecCoord c;
  c.lane = static_cast<int>(v & 31);
  long long t = v >> 5;
  const int b = static_cast<int>(t & 7);
  t >>= 3;
  c.kb = static_cast<int>(t % kTiles);
  const long long strip = t / kTiles;
  c.nb = static_cast<int>(strip * 8 + b);
  return c;
}

// (row, reduction index) inside the 16x16 block of nibble slot `slot` for lane (g, t)
__device__ __forceinline__ void slot_rc(int slot, int g, int t, int& r, int& c) {
  const int reg = slot & 3, e = slot >> 2;
  r = g + 8 * (reg & 1);
  c = 4 * t + 2 * (reg >> 1) + e;
}

// One CTA of 256 threads per 64-row x 128-column tile (one strip, one 64-row block):
// the tile's codes are read row by row into shared memory (coalesced 16-byte loads),
// then thread (block b, lane) assembles its four words from there and writes its
// 16-byte vector; the CTA's 256 vectors are consecutive in the packed stream.  The
// rows are padded so that the four lanes t of a quad, which read rows 4 apart, hit
// different banks.
constexpr int kTileThreads = 256;
constexpr int kCodeRow = 136;  // bytes per shared row of codes (128 + 8)
constexpr int kHalfRow = 132;  // halves per shared row of FP16 weights (128 + 4)

__global__ void __launch_bounds__(kTileThreads) repack_codes_kernel(const uint8_t* __restrict__ q, int K, int N,
                                                                    uint4* __restrict__ packed) {
  __shared__ __align__(16) uint8_t tile[64][kCodeRow];
  const int kTiles = K / 64;
  const int kb = static_cast<int>(blockIdx.x % kTiles);
  const long long strip = blockIdx.x / kTiles;
  for (int i = threadIdx.x; i < 64 * 8; i += kTileThreads) {  // 64 rows x 8 16-byte pieces
    const int r = i >> 3, c16 = i & 7;
    const uint4 v = *reinterpret_cast<const uint4*>(q + (kb * 64LL + r) * N + strip * 128 + 16 * c16);
    *reinterpret_cast<uint2*>(&tile[r][16 * c16]) = make_uint2(v.x, v.y);
    *reinterpret_cast<uint2*>(&tile[r][16 * c16 + 8]) = make_uint2(v.z, v.w);
  }
  __syncthreads();
  const int b = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  uint32_t words[4];
  uint32_t bad = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t w = 0;
#pragma unroll
    for (int slot = 0; slot < 8; ++slot) {
      int r, c;
      slot_rc(slot, g, t, r, c);
      const uint32_t code = tile[16 * j + c][16 * b + r];
      bad |= code > 15u;
      w |= (code & 15u) << (4 * slot);
    }
    words[j] = w;
  }
  if (bad) atomicOr(&g_repack_flag, kDevErrCodeRange);
  packed[static_cast<long long>(blockIdx.x) * kTileThreads + threadIdx.x] = make_uint4(words[0], words[1], words[2], words[3]);
}

// Quantise FP16 weights with their FP16 scales straight into the packed layout
// (the original Layer.pack step, deep-dive article section "可复现的调用链"):
// q = clamp(rint(w / s) + 8, 0, 15), the quotient an IEEE float32 division,
// rint rounding half to even.  Same word-side walk as repack_codes_kernel.
// z: zero codes uint8[K/G][N] row-major, or null for the symmetric offset 8.  Tiled like
// repack_codes_kernel: the 64-row tile lies inside one group (G is 128 or K), so its 128
// scales (and zero codes) are one row.
__global__ void __launch_bounds__(kTileThreads) quantize_codes_kernel(const uint16_t* __restrict__ w,
                                                                      const uint16_t* __restrict__ s,
                                                                      const uint8_t* __restrict__ z, int K, int N,
                                                                      int G, uint4* __restrict__ packed) {
  __shared__ __align__(16) uint16_t tile[64][kHalfRow];
  __shared__ float scale[128];
  __shared__ float recip[128];
  __shared__ float offset[128];
  const int kTiles = K / 64;
  const int kb = static_cast<int>(blockIdx.x % kTiles);
  const long long strip = blockIdx.x / kTiles;
  for (int i = threadIdx.x; i < 64 * 16; i += kTileThreads) {  // 64 rows x 16 16-byte pieces
    const int r = i >> 4, c8 = i & 15;
    const uint4 v = *reinterpret_cast<const uint4*>(w + (kb * 64LL + r) * N + strip * 128 + 8 * c8);
    *reinterpret_cast<uint2*>(&tile[r][8 * c8]) = make_uint2(v.x, v.y);
    *reinterpret_cast<uint2*>(&tile[r][8 * c8 + 4]) = make_uint2(v.z, v.w);
  }
  if (threadIdx.x < 128) {
    const long long gi = ((kb * 64LL) / G) * N + strip * 128 + threadIdx.x;
    const float sf = __half2float(__ushort_as_half(s[gi]));
    scale[threadIdx.x] = sf;
    recip[threadIdx.x] = __frcp_rn(sf);
    offset[threadIdx.x] = z ? static_cast<float>(z[gi]) : 8.0f;
  }
  __syncthreads();
  const int b = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  uint32_t words[4];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t word = 0;
#pragma unroll
    for (int slot = 0; slot < 8; ++slot) {
      int r, c;
      slot_rc(slot, g, t, r, c);
      const int col = 16 * b + r;
      const float wf = __half2float(__ushort_as_half(tile[16 * j + c][col]));
      // w * RN(1/s) is within 1.5 ulp of w / s; away from the half-integers it rounds to the
      // same integer as the correctly rounded quotient, which is taken only near them
      const float approx = wf * recip[col];
      const float frac = fabsf(approx - truncf(approx));
      const bool near_tie = fabsf(frac - 0.5f) <= 0x1p-22f * fabsf(approx);  // twice the error bound 2^-23 |w/s|
      const float quot = (isfinite(approx) && !near_tie) ? approx : __fdiv_rn(wf, scale[col]);
      uint32_t code = 8u;
      if (isfinite(quot)) {
        const float qf = fminf(fmaxf(rintf(quot) + offset[col], 0.0f), 15.0f);
        code = static_cast<uint32_t>(qf);
      } else {
        bad = true;
      }
      word |= code << (4 * slot);
    }
    words[j] = word;
  }
  if (bad) atomicOr(&g_repack_flag, kDevErrValue);
  packed[static_cast<long long>(blockIdx.x) * kTileThreads + threadIdx.x] = make_uint4(words[0], words[1], words[2], words[3]);
}

// permuted position p inside a 16-column block -> fragment row r
__device__ __forceinline__ int perm_row(int p) { return (p >> 1) + 8 * (p & 1); }

// sp index i -> (g, n): i = (strip * NG + g) * 128 + p, n = strip * 128 + 16 * (p / 16) + row(p % 16)
// Scales (and zero codes) by the min-max rule: one thread per group and pair
// of adjacent columns walks the group's G rows (a 4-byte load per row; the
// warp's loads of one row are 128 contiguous bytes).  The arithmetic is the
// rule's, one IEEE float32 rounding per step: span = hi - lo (or 2 max|v|),
// s = RNE_fp16(span / 15), z = clamp(rint(-lo / s), 0, 15).  A scale that
// rounds to 0 becomes 1; a non-finite weight flags kDevErrValue and leaves
// s = 1 (and z = 0) for its group.
__global__ void minmax_scales_kernel(const uint16_t* __restrict__ w, int N, int G, uint16_t* __restrict__ s,
                                     uint8_t* __restrict__ z) {
  const int c2 = blockIdx.x * blockDim.x + threadIdx.x;  // column pair
  if (2 * c2 >= N) return;
  const int g = blockIdx.y;
  const uint32_t* col = reinterpret_cast<const uint32_t*>(w + static_cast<size_t>(g) * G * N) + c2;
  const size_t stride = static_cast<size_t>(N / 2);
  float lo0 = INFINITY, lo1 = INFINITY, hi0 = -INFINITY, hi1 = -INFINITY;
  bool bad0 = false, bad1 = false;
#pragma unroll 8
  for (int r = 0; r < G; ++r) {
    const uint32_t v = __ldg(col + r * stride);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v));
    bad0 |= !isfinite(f.x);
    bad1 |= !isfinite(f.y);
    lo0 = fminf(lo0, f.x);
    hi0 = fmaxf(hi0, f.x);
    lo1 = fminf(lo1, f.y);
    hi1 = fmaxf(hi1, f.y);
  }
  const float los[2] = {lo0, lo1}, his[2] = {hi0, hi1};
  const bool bads[2] = {bad0, bad1};
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float lo = los[j], hi = his[j];
    const bool bad = bads[j];
    float span;
    if (z) {
      lo = fminf(lo, 0.0f);
      hi = fmaxf(hi, 0.0f);
      span = __fsub_rn(hi, lo);
    } else {
      span = 2.0f * fmaxf(fabsf(lo), fabsf(hi));  // exact
    }
    __half sh = __float2half_rn(__fdiv_rn(span, 15.0f));
    if (bad || __half2float(sh) == 0.0f) sh = __float2half_rn(1.0f);
    const size_t o = static_cast<size_t>(g) * N + 2 * c2 + j;
    s[o] = __half_as_ushort(sh);
    if (z) {
      const float zq = __fdiv_rn(-lo, __half2float(sh));
      z[o] = bad ? 0 : static_cast<uint8_t>(fminf(fmaxf(rintf(zq), 0.0f), 15.0f));
    }
  }
  if (bad0 || bad1) atomicOr(&g_repack_flag, kDevErrValue);
}

__global__ void permute_scales_kernel(const uint16_t* __restrict__ s, uint16_t* __restrict__ sp, int N, int NG,
                                      long long count, int inverse) {
  const long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (i >= count) return;
  const int p = static_cast<int>(i & 127);
  const long long t = i >> 7;
  const int g = static_cast<int>(t % NG);
  const long long strip = t / NG;
  const long long n = strip * 128 + (p & ~15) + perm_row(p & 15);
  if (!inverse)
    sp[i] = s[g * static_cast<long long>(N) + n];  // forward: natural -> permuted
  else
    sp[g * static_cast<long long>(N) + n] = s[i];  // inverse: permuted -> natural
}

__global__ void unpack_codes_kernel(const uint4* __restrict__ packed, int K, int N, uint8_t* __restrict__ q,
                                    long long nvec) {
  const long long v = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (v >= nvec) return;
  const VecCoord vc = vec_coord(v, K);
  const int g = vc.lane >> 2, t = vc.lane & 3;
  const uint4 pv = packed[v];
  const uint32_t words[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int slot = 0; slot < 8; ++slot) {
      int r, c;
      slot_rc(slot, g, t, r, c);
      const long long k = vc.kb * 64LL + 16 * j + c;
      const long long n = vc.nb * 16LL + r;
      q[k * N + n] = static_cast<uint8_t>((words[j] >> (4 * slot)) & 15u);
    }
  }
}

// Bhat[k][n] = RNE(s * (q - 8)): the exact decode of the GEMM, then one FP16 multiply.
// zero codes uint8[K/G][N] -> the scales' permuted order (uint8[N/128][K/G][128]); codes above 15 flag
__global__ void permute_zeros_kernel(const uint8_t* __restrict__ z, uint8_t* __restrict__ zp, int N, int NG,
                                     long long count) {
  const long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (i >= count) return;
  const int p = static_cast<int>(i & 127);
  const long long t = i >> 7;
  const int g = static_cast<int>(t % NG);
  const long long strip = t / NG;
  const long long n = strip * 128 + (p & ~15) + perm_row(p & 15);
  const uint8_t code = z[g * static_cast<long long>(N) + n];
  if (code > 15) atomicOr(&g_repack_flag, kDevErrCodeRange);
  zp[i] = code & 15;
}

// Bhat[k][n] = RNE(s * (q - z)): the exact decode of the GEMM (z = 8 without zero points), then one
// FP16 multiply.
__global__ void dequant_kernel(const uint4* __restrict__ packed, const uint16_t* __restrict__ sp,
                               const uint8_t* __restrict__ zp, int K, int N, int G, uint16_t* __restrict__ bhat,
                               long long nvec) {
  const long long v = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (v >= nvec) return;
  const VecCoord vc = vec_coord(v, K);
  const int g = vc.lane >> 2, t = vc.lane & 3;
  const int grp = (vc.kb * 64) / G;  // G is a multiple of 64: one group per 64-row tile
  const int NG = K / G;
  const long long sidx = (static_cast<long long>(vc.nb >> 3) * NG + grp) * 128 + (vc.nb & 7) * 16 + 2 * g;
  const uint32_t spair = *reinterpret_cast<const uint32_t*>(sp + sidx);
  const uint32_t s_row_g = (spair & 0xffffu) * 0x10001u;      // scale of fragment row g, both halves
  const uint32_t s_row_g8 = (spair >> 16) * 0x10001u;         // scale of fragment row g + 8
  uint32_t c_lo = 0, c_hi = 0;
  if (zp) {
    const uint32_t zpair = *reinterpret_cast<const uint16_t*>(zp + sidx);  // zero codes of rows g, g + 8
    c_lo = zp_const_lo(zpair & 15u);
    c_hi = zp_const_hi((zpair >> 8) & 15u);
  }
  const uint4 pv = packed[v];
  const uint32_t words[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t a[4];
    if (zp)
      decode8_zp(words[j], c_lo, c_hi, a);
    else
      decode8(words[j], a);
#pragma unroll
    for (int reg = 0; reg < 4; ++reg) {
      const uint32_t h = hmul2_u32(a[reg], (reg & 1) ? s_row_g8 : s_row_g);
      const long long n = vc.nb * 16LL + g + 8 * (reg & 1);
      const long long k = vc.kb * 64LL + 16 * j + 4 * t + 2 * (reg >> 1);
      bhat[k * N + n] = static_cast<uint16_t>(h & 0xffffu);
      bhat[(k + 1) * N + n] = static_cast<uint16_t>(h >> 16);
    }
  }
}

inline unsigned grid_for(long long n, int block) { return static_cast<unsigned>((n + block - 1) / block); }

}  // namespace

cudaError_t launch_repack(const uint8_t* q, const uint16_t* s, int K, int N, int G, uint32_t* packed,
                          uint16_t* scales_p, cudaStream_t stream) {
  const unsigned tiles = static_cast<unsigned>(static_cast<long long>(N / 128) * (K / 64));
  repack_codes_kernel<<<tiles, kTileThreads, 0, stream>>>(q, K, N, reinterpret_cast<uint4*>(packed));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long ns = static_cast<long long>(K / G) * N;
  permute_scales_kernel<<<grid_for(ns, 256), 256, 0, stream>>>(s, scales_p, N, K / G, ns, 0);
  return cudaGetLastError();
}

cudaError_t launch_quantize_repack(const uint16_t* w, const uint16_t* s, const uint8_t* z, int K, int N, int G,
                                   uint32_t* packed, uint16_t* scales_p, cudaStream_t stream) {
  const unsigned tiles = static_cast<unsigned>(static_cast<long long>(N / 128) * (K / 64));
  quantize_codes_kernel<<<tiles, kTileThreads, 0, stream>>>(w, s, z, K, N, G, reinterpret_cast<uint4*>(packed));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long ns = static_cast<long long>(K / G) * N;
  permute_scales_kernel<<<grid_for(ns, 256), 256, 0, stream>>>(s, scales_p, N, K / G, ns, 0);
  return cudaGetLastError();
}

cudaError_t launch_minmax_scales(const uint16_t* w, int K, int N, int G, uint16_t* s, uint8_t* z,
                                 cudaStream_t stream) {
  const dim3 grid(grid_for(N / 2, 256), static_cast<unsigned>(K / G));
  minmax_scales_kernel<<<grid, 256, 0, stream>>>(w, N, G, s, z);
  return cudaGetLastError();
}

cudaError_t launch_permute_scales(const uint16_t* s, int K, int N, int G, uint16_t* scales_p, cudaStream_t stream) {
  const long long ns = static_cast<long long>(K / G) * N;
  permute_scales_kernel<<<grid_for(ns, 256), 256, 0, stream>>>(s, scales_p, N, K / G, ns, 0);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint32_t* packed, const uint16_t* scales_p, int K, int N, int G, uint8_t* q,
                          uint16_t* s, cudaStream_t stream) {
  const long long nvec = static_cast<long long>(K) * N / 32;
  unpack_codes_kernel<<<grid_for(nvec, 256), 256, 0, stream>>>(reinterpret_cast<const uint4*>(packed), K, N, q,
                                                                nvec);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long ns = static_cast<long long>(K / G) * N;
  permute_scales_kernel<<<grid_for(ns, 256), 256, 0, stream>>>(scales_p, s, N, K / G, ns, 1);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const uint32_t* packed, const uint16_t* scales_p, const uint8_t* zeros_p, int K, int N,
                           int G, uint16_t* bhat, cudaStream_t stream) {
  const long long nvec = static_cast<long long>(K) * N / 32;
  dequant_kernel<<<grid_for(nvec, 256), 256, 0, stream>>>(reinterpret_cast<const uint4*>(packed), scales_p, zeros_p,
                                                           K, N, G, bhat, nvec);
  return cudaGetLastError();
}

cudaError_t launch_repack_zeros(const uint8_t* z, int K, int N, int G, uint8_t* zeros_p, cudaStream_t stream) {
  const long long count = static_cast<long long>(K / G) * N;
  permute_zeros_kernel<<<grid_for(count, 256), 256, 0, stream>>>(z, zeros_p, N, K / G, count);
  return cudaGetLastError();
}

cudaError_t read_and_clear_repack_flag(unsigned int* flag, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(flag, g_repack_flag, sizeof(unsigned int), 0, cudaMemcpyDeviceToHost,
                                            stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  if (*flag) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_repack_flag, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
  }
  return e;
}

}  // namespace w4a16
