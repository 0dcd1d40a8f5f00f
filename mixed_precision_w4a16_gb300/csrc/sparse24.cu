// Offline steps of the 2:4-sparse W4A16 layer (the Sparse-Marlin analogue):
// dense 2:4 codes <-> the packed stream the streaming GEMM's SP24 variant reads.
//
// The MARLIN paper (Section 2.1.1, "Modern Tensor Core Units") describes the 2:4
// format: the sparse operand is cut into vectors of four along the reduction
// dimension, two values of each are kept, and metadata gives each kept value's
// position in its group.  The deep-dive article (section "Sparse-Marlin 再叠加
// 2:4 结构化稀疏") keeps the values as 4-bit codes with 2-bit positions.
//
// Packed stream, per 128-column strip and 64-row piece (768 words, 3 KB against
// 4 KB dense): codes [8 column blocks][32 lanes][2 words], then positions
// [8][32][1 word].  Code word m of lane (g, t) holds, in the decode's nibble
// slots (slot i: low half of register i, slot i + 4: its high half), the kept
// values of rows g + 8 (i & 1), groups t + 4 (i >> 1) of sparse MMA m (reduction
// rows 32m .. 32m + 31 of the piece): kept entry 0 in the low half, 1 in the high
// half.  Position word of lane (g, t): MMA t >> 1 (its sparsity selector), groups
// 4 (t & 1) .. + 3, nibbles 0..3 for row g and 4..7 for row g + 8, each nibble
// i0 | i1 << 2 with i0 < i1 -- the lane layout the tensor cores read, measured on
// a GB300 (see gemm_mma.cu).
#include <cuda_runtime.h>

#include "../../include/w4a16.h"
#include "sparse24.h"

namespace w4a16 {

// Error flag of the 2:4 repack / unpack (read and cleared by w4a16_get_status).
__device__ unsigned int g_sparse_flag;

namespace {

// Kept positions and codes of the group of four rows starting at row 4*grp of column n: the
// positions of the codes != 8 in increasing order, filled up with the lowest remaining
// positions.  More than two codes != 8 sets `bad`.
__device__ __forceinline__ void group_entry(const uint8_t* __restrict__ q, int N, int grp, int n, int& i0, int& i1,
                                            uint32_t& c0, uint32_t& c1, bool& bad) {
  uint32_t codes[4];
  uint32_t mask = 0;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    codes[r] = q[(4LL * grp + r) * N + n];
    if (codes[r] != 8u) mask |= 1u << r;
  }
  if (__popc(mask) > 2) bad = true;
  while (__popc(mask) < 2) mask |= ~mask & (mask + 1u);  // add the lowest free position
  i0 = __ffs(mask) - 1;
  i1 = 31 - __clz(mask);
  c0 = codes[i0] & 15u;
  c1 = codes[i1] & 15u;
}

// one thread per (strip, 64-row piece, column block, lane): two code words and one metadata word
__global__ void repack24_kernel(const uint8_t* __restrict__ q, int K, int N, uint32_t* __restrict__ packed24,
                                long long nthreads) {
  const long long v = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (v >= nthreads) return;
  const int lane = static_cast<int>(v & 31);
  const int nb = static_cast<int>((v >> 5) & 7);
  const long long rest = v >> 8;
  const int P = static_cast<int>(rest % (K / 64));
  const long long strip = rest / (K / 64);
  const int g = lane >> 2, t = lane & 3;
  const int n0 = static_cast<int>(strip * 128) + 16 * nb + g;
  bool bad = false;
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int i0, i1;
      uint32_t c0, c1;
      group_entry(q, N, 16 * P + 8 * m + t + 4 * (i >> 1), n0 + 8 * (i & 1), i0, i1, c0, c1, bad);
      w[m] |= (c0 << (4 * i)) | (c1 << (4 * (i + 4)));
    }
  const int m = t >> 1, r = t & 1;  // this lane's metadata: MMA m (selector m), groups 4r .. 4r + 3
  uint32_t meta = 0;
#pragma unroll
  for (int h = 0; h < 4; ++h)
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      int i0, i1;
      uint32_t c0, c1;
      group_entry(q, N, 16 * P + 8 * m + 4 * r + h, n0 + 8 * rr, i0, i1, c0, c1, bad);
      meta |= static_cast<uint32_t>(i0 | (i1 << 2)) << (4 * (h + 4 * rr));
    }
  const long long base = (strip * (K / 64) + P) * kPiece24Words;
  packed24[base + (nb * 32 + lane) * 2 + 0] = w[0];
  packed24[base + (nb * 32 + lane) * 2 + 1] = w[1];
  packed24[base + 512 + nb * 32 + lane] = meta;
  if (bad) atomicOr(&g_sparse_flag, kDevErrValue);
}

// inverse: the same thread grid; each thread writes the four rows of its own (row, group) pairs,
// taking the positions from the lane that holds them (a warp is one column block of one piece)
__global__ void unpack24_kernel(const uint32_t* __restrict__ packed24, int K, int N, uint8_t* __restrict__ q,
                                long long nthreads) {
  const long long v = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (v >= nthreads) return;  // nthreads is a multiple of 32: whole warps return together
  const int lane = static_cast<int>(v & 31);
  const int nb = static_cast<int>((v >> 5) & 7);
  const long long rest = v >> 8;
  const int P = static_cast<int>(rest % (K / 64));
  const long long strip = rest / (K / 64);
  const int g = lane >> 2, t = lane & 3;
  const int n0 = static_cast<int>(strip * 128) + 16 * nb + g;
  const long long base = (strip * (K / 64) + P) * kPiece24Words;
  const uint32_t w[2] = {packed24[base + (nb * 32 + lane) * 2], packed24[base + (nb * 32 + lane) * 2 + 1]};
  const uint32_t meta = packed24[base + 512 + nb * 32 + lane];
  bool bad = false;
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      // groups t + 4*half of MMA m: positions in lane (g, 2m + half), nibble t (row g) / 4 + t (row g + 8)
      const uint32_t mm = __shfl_sync(0xffffffffu, meta, g * 4 + 2 * m + half);
      const int grp = 16 * P + 8 * m + t + 4 * half;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int i = rr + 2 * half;  // register holding rows g + 8*rr, groups t + 4*half
        const uint32_t nib = (mm >> (4 * (t + 4 * rr))) & 15u;
        const int i0 = nib & 3, i1 = nib >> 2;
        if (i0 >= i1) bad = true;
        const uint32_t c0 = (w[m] >> (4 * i)) & 15u, c1 = (w[m] >> (4 * (i + 4))) & 15u;
        const int n = n0 + 8 * rr;
#pragma unroll
        for (int r = 0; r < 4; ++r)
          q[(4LL * grp + r) * N + n] = static_cast<uint8_t>(r == i0 ? c0 : (r == i1 ? c1 : 8u));
      }
    }
  if (bad) atomicOr(&g_sparse_flag, kDevErrValue);
}

inline unsigned grid_for(long long n, int block) { return static_cast<unsigned>((n + block - 1) / block); }

}  // namespace

cudaError_t launch_repack24(const uint8_t* q, int K, int N, uint32_t* packed24, cudaStream_t stream) {
  const long long n = static_cast<long long>(N / 128) * (K / 64) * 256;
  repack24_kernel<<<grid_for(n, 256), 256, 0, stream>>>(q, K, N, packed24, n);
  return cudaGetLastError();
}

cudaError_t launch_unpack24(const uint32_t* packed24, int K, int N, uint8_t* q, cudaStream_t stream) {
  const long long n = static_cast<long long>(N / 128) * (K / 64) * 256;
  unpack24_kernel<<<grid_for(n, 256), 256, 0, stream>>>(packed24, K, N, q, n);
  return cudaGetLastError();
}

cudaError_t read_and_clear_sparse_flag(unsigned int* flag, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(flag, g_sparse_flag, sizeof(unsigned int), 0, cudaMemcpyDeviceToHost,
                                            stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  if (*flag) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_sparse_flag, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
  }
  return e;
}

}  // namespace w4a16
