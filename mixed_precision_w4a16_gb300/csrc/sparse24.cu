// 2:4-sparse W4A16 GEMM for small batches (the Sparse-Marlin analogue).
//
// The MARLIN paper (Section 2.1.1, "Modern Tensor Core Units") describes the
// 2:4 format: the sparse operand is cut into vectors of four along the
// reduction dimension, two values of each are kept, and a metadata structure
// gives each kept value's position in its group; the sparse tensor cores use
// the metadata to pick the matching rows of the dense operand.  The deep-dive
// article (section "Sparse-Marlin 再叠加 2:4 结构化稀疏") adds that the kept
// weights stay 4-bit codes with 2-bit positions, and that the hardware wants
// the sparse matrix in a fixed operand slot, so the product is taken as
// (B^T A^T)^T.  Here the weights already sit on the 16-row (A) side of the
// streaming kernel's MMA, so mma.sp takes them as they are:
//
//  * mma.sp::ordered_metadata.m16n8k32 (f16 in, f32 accumulate): the 16 x 16
//    compressed weight fragment covers 32 reduction rows; a 64-row piece is
//    two such MMAs, the first with sparsity selector 0 and the second with 1;
//  * metadata lane layout, read off a GB300 by an in-bounds probe (one MMA per
//    metadata nibble flipped): with selector s the lanes t = 2s, 2s + 1 of each
//    quad supply it; lane (g, 2s + r) holds in nibbles 0..3 the position pairs
//    of row g for the MMA's groups 4r .. 4r + 3, in nibbles 4..7 those of row
//    g + 8.  So every lane supplies exactly one useful word per piece;
//  * packed stream, per 128-column strip and 64-row piece (768 words, 3 KB
//    against 4 KB dense): codes [8 column blocks][32 lanes][2 words], then
//    metadata [8][32][1 word].  Code word j of lane (g, t) holds, in the
//    decode's nibble slots (slot i: low half of register i, slot i + 4: its
//    high half), the kept values of rows g + 8 (i & 1), groups t + 4 (i >> 1)
//    of MMA j, kept entry 0 in the low half and 1 in the high half;
//  * the rest of the pipeline is the streaming kernel's: one producer lane
//    fills a stage with three copies (weights evict-first, activation tile,
//    scale rows), eight consumer warps (2 column halves x 4 K-split), split-
//    strip reduction in fixed CTA order.
#include <cuda_runtime.h>

#include <algorithm>

#include "../../include/w4a16.h"
#include "common.cuh"
#include "sparse24.h"

namespace w4a16 {

// Error flag of the 2:4 repack / unpack (read and cleared by w4a16_get_status).
__device__ unsigned int g_sparse_flag;

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kNbw = 4;                           // 16-column blocks per consumer warp
constexpr int kPieceBytes = kPiece24Words * 4;    // 3072
constexpr int kCodeBytes = 2048;                  // codes part of a piece
constexpr long long kDrainCycles = 2000000000LL;  // bound on the final drain wait

__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// D = A (2:4 compressed 16 x 16, f16) x B (32 x 8, f16) + C, metadata e with sparsity selector SEL.
template <int SEL>
__device__ __forceinline__ void mma_sp_16832(float d[4], const uint32_t a[4], const uint32_t b[4], uint32_t e,
                                             const float c[4]) {
  asm volatile(
      "mma.sp::ordered_metadata.sync.aligned.m16n8k32.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9, %10, %11}, {%12, %13, %14, %15}, %16, %17;"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]), "r"(b[2]), "r"(b[3]), "f"(c[0]),
        "f"(c[1]), "f"(c[2]), "f"(c[3]), "r"(e), "n"(SEL));
}

__device__ __forceinline__ uint16_t f32_to_f16_bits(float x) { return __half_as_ushort(__float2half_rn(x)); }

template <int MT>
__global__ void __launch_bounds__(kMmaThreads, 1)
    gemm24_kernel(const __grid_constant__ CUtensorMap tmA, const GemmParams p) {
  constexpr int MB = 8 * MT;
  constexpr int A_BOX = MB * 128;  // bytes of one 64-row activation piece
  constexpr int SLOT = 128 * MB;   // floats in one strip partial
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int S = p.stages;
  const int KQ = p.kq;
  const uint32_t bar_full = sbase + p.bar_off;
  const uint32_t bar_empty = bar_full + 8 * S;
  volatile int* flags = reinterpret_cast<volatile int*>(smem + p.flag_off);
  volatile int* abort_flag = flags + 0;
  volatile int* last_flag = flags + 1;
  volatile int* seg_abort = flags + 2;
  volatile int* zero_flag = flags + 3;
  float* red = reinterpret_cast<float*>(smem + p.red_off);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const int u_begin = cta * p.T;
  const int u_end = min(p.units, u_begin + p.T);
  const int nunits = max(0, u_end - u_begin);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kConsumerWarps);
    }
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = 0;
    flags[3] = 0;
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) prefetch_tensormap(&tmA);
    const uint64_t pol_w = (p.ablate & kAblateNoEvictFirst) ? policy_evict_normal() : policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    const int NG = p.K / p.G;
    const uint32_t w_bytes = static_cast<uint32_t>(KQ) * kPieceBytes;
    int issued = 0;
    int s = 0, round = 0;
    int j = nunits > 0 ? u_begin / p.KU : 0, kt = u_begin - j * p.KU;
    for (int it = 0; it < nunits; ++it) {
      if (it >= S) {
        bool ok = true;
        if (lane == 0) ok = mbar_wait_bounded(bar_empty + 8 * s, (round - 1) & 1, p.wait_limit, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          if (lane == 0 && !*abort_flag) {
            *abort_flag = 1;
            atomicOr(p.status, kDevErrTimeout);
          }
          break;
        }
      }
      if (!(p.debug_stall && it == 0)) {
        if (lane == 0) {
          const uint32_t st = sbase + s * p.stage_bytes;
          const uint32_t fb = bar_full + 8 * s;
          mbar_arrive_expect_tx(fb, p.tx_bytes);
          const uint32_t* wsrc =
              p.packed + (static_cast<long long>(j) * (p.K / 64) + static_cast<long long>(kt) * KQ) * kPiece24Words;
          bulk_g2s(st + p.w_off, wsrc, w_bytes, fb, pol_w);
          tma_load_3d(st, &tmA, 0, p.m0, kt * KQ, fb, pol_a);
          const int grp0 = (p.G == 128) ? kt * p.srows : 0;
          const uint16_t* ssrc = p.scales + (static_cast<long long>(j) * NG + grp0) * 128;
          bulk_g2s(st + p.s_off, ssrc, static_cast<uint32_t>(p.srows) * 256u, fb, pol_a);
        }
        __syncwarp();
        issued = it + 1;
      }
      if (++s == S) {
        s = 0;
        ++round;
      }
      if (++kt == p.KU) {
        kt = 0;
        ++j;
      }
    }
    named_bar_sync(3, kMmaThreads);
    if (*abort_flag && lane == 0) {
      const int first_filled = p.debug_stall ? 1 : 0;
      for (int it = max(first_filled, issued - S); it < issued; ++it)
        mbar_wait_bounded(bar_full + 8 * (it % S), (it / S) & 1, kDrainCycles, zero_flag);
    }
    return;
  }

  // -------------------------------------------------------------------- consumers
  const int ng = warp >> 2;  // column half: blocks 4*ng .. 4*ng + 3
  const int kq0 = warp & 3;  // first 64-row piece of each unit (then kq0 + 4, ...)
  const int g = lane >> 2, t = lane & 3;
  const int swz = (p.ablate & kAblateNoSwizzle) ? 0 : g;
  const int first_col = nunits > 0 ? u_begin / p.KU : 0;

  float acc[kNbw][MT][4];
#pragma unroll
  for (int i = 0; i < kNbw; ++i)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][mt][e] = 0.f;
  const float zero4[4] = {0.f, 0.f, 0.f, 0.f};

  int s = 0, round = 0;
  int j = first_col, kt = u_begin - first_col * p.KU;
  for (int it = 0; it < nunits; ++it) {
    const uint32_t st = sbase + s * p.stage_bytes;
    bool have = false;
    const bool go = __shfl_sync(0xffffffffu, *abort_flag == 0, 0);
    if (go) {
      have = mbar_wait_bounded(bar_full + 8 * s, round & 1, p.wait_limit, abort_flag);
      have = __all_sync(0xffffffffu, have);
      if (!have && lane == 0 && !*abort_flag) {
        *abort_flag = 1;
        atomicOr(p.status, kDevErrTimeout);
      }
    }
    if (have) {
#pragma unroll
      for (int pc = 0; pc < 4; ++pc) {
        const int kq = kq0 + 4 * pc;
        if (kq >= KQ) break;
        // activations: MMA m (reduction rows 32m .. 32m + 31 of the piece) wants in register q of lane
        // (g, t) the pair A[token][32m + 8q + 2t .. + 1]: one 4-byte load from 16-byte chunk 4m + q
        // (128-byte swizzle: chunk c of row r at c ^ (r & 7)).
        const uint32_t a_box = st + kq * A_BOX;
        uint32_t bf[2][MT][4];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int q = 0; q < 4; ++q)
              bf[m][mt][q] = lds32(a_box + (mt * 8 + g) * 128 + (((4 * m + q) ^ swz) << 4) + 4 * t);
        const int srow = (p.G == 128) ? (kq >> 1) : 0;
        const uint32_t wpiece = st + p.w_off + kq * kPieceBytes;
        uint2 cw[kNbw];
        uint32_t mw[kNbw], spv[kNbw];
#pragma unroll
        for (int i = 0; i < kNbw; ++i) {
          const int nb = ng * kNbw + i;
          cw[i] = lds64(wpiece + (nb * 32 + lane) * 8);
          mw[i] = lds32(wpiece + kCodeBytes + (nb * 32 + lane) * 4);
          spv[i] = lds32(st + p.s_off + (srow * 128 + nb * 16 + 2 * g) * 2);
        }
#pragma unroll
        for (int i = 0; i < kNbw; ++i) {
          float tmp[MT][4];
          uint32_t a[4];
          decode8(cw[i].x, a);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) mma_sp_16832<0>(tmp[mt], a, bf[0][mt], mw[i], zero4);
          decode8(cw[i].y, a);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) mma_sp_16832<1>(tmp[mt], a, bf[1][mt], mw[i], tmp[mt]);
          const float s_lo = __half2float(__ushort_as_half(static_cast<uint16_t>(spv[i] & 0xffffu)));
          const float s_hi = __half2float(__ushort_as_half(static_cast<uint16_t>(spv[i] >> 16)));
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            acc[i][mt][0] = fmaf(s_lo, tmp[mt][0], acc[i][mt][0]);
            acc[i][mt][1] = fmaf(s_lo, tmp[mt][1], acc[i][mt][1]);
            acc[i][mt][2] = fmaf(s_hi, tmp[mt][2], acc[i][mt][2]);
            acc[i][mt][3] = fmaf(s_hi, tmp[mt][3], acc[i][mt][3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }
    if (++s == S) {
      s = 0;
      ++round;
    }
    const bool seg_end = (kt == p.KU - 1) || (it == nunits - 1);
    if (++kt == p.KU) kt = 0;
    if (!seg_end) continue;

    // ---------------------------------------------------------- segment epilogue (strip j)
    if (kq0 != 0) {
#pragma unroll
      for (int i = 0; i < kNbw; ++i)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            red[(((((kq0 - 1) * 2 + ng) * kNbw + i) * MT + mt) * 4 + e) * 32 + lane] = acc[i][mt][e];
    }
    named_bar_sync(1, kConsumerWarps * 32);
    if (warp == 0 && lane == 0) *seg_abort = *abort_flag;
    if (kq0 == 0) {
#pragma unroll
      for (int i = 0; i < kNbw; ++i)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r0 = ((((0 * 2 + ng) * kNbw + i) * MT + mt) * 4 + e) * 32 + lane;
            const int stride = 2 * kNbw * MT * 4 * 32;
            acc[i][mt][e] = ((acc[i][mt][e] + red[r0]) + red[r0 + stride]) + red[r0 + 2 * stride];
          }
    }
    named_bar_sync(1, kConsumerWarps * 32);
    const bool skip = *seg_abort != 0;
    if (kq0 == 0 && !skip) {
      const int c_first = (j * p.KU) / p.T;
      const int c_last = min(((j + 1) * p.KU - 1) / p.T, p.grid - 1);
      const int sidx0 = ng * kNbw * MT * 4 * 32 + lane;
      bool write_now = true;
      if (c_first != c_last) {
        const int slot = (j == first_col) ? 2 * cta : 2 * cta + 1;
        float* dst = p.slots + static_cast<long long>(slot) * SLOT + sidx0;
#pragma unroll
        for (int i = 0; i < kNbw; ++i)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[((i * MT + mt) * 4 + e) * 32] = acc[i][mt][e];
        __threadfence();
        named_bar_sync(2, 2 * 32);
        if (warp == 0 && lane == 0) {
          const unsigned old = atomicAdd(p.counters + j, 1u);
          *last_flag = (old == static_cast<unsigned>(c_last - c_first)) ? 1 : 0;
        }
        named_bar_sync(2, 2 * 32);
        write_now = *last_flag != 0;
        if (write_now) {
          __threadfence();
#pragma unroll
          for (int i = 0; i < kNbw; ++i)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[i][mt][e] = 0.f;
          for (int c = c_first; c <= c_last; ++c) {
            const int cslot = (j == (c * p.T) / p.KU) ? 2 * c : 2 * c + 1;
            const float* src = p.slots + static_cast<long long>(cslot) * SLOT + sidx0;
#pragma unroll
            for (int i = 0; i < kNbw; ++i)
#pragma unroll
              for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[i][mt][e] += __ldcg(src + ((i * MT + mt) * 4 + e) * 32);
          }
          if (warp == 0 && lane == 0) p.counters[j] = 0u;
        }
      }
      if (write_now) {
#pragma unroll
        for (int i = 0; i < kNbw; ++i) {
          const int n_base = j * kStrip + (ng * kNbw + i) * 16 + g;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int token = p.m0 + mt * 8 + 2 * t + (e & 1);
              const int n = n_base + 8 * (e >> 1);
              if (token < p.M) p.C[static_cast<long long>(token) * p.N + n] = f32_to_f16_bits(acc[i][mt][e]);
            }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kNbw; ++i)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][mt][e] = 0.f;
    ++j;
  }
  named_bar_sync(3, kMmaThreads);
}

// ---------------------------------------------------------------------------
// Offline: dense 2:4 codes <-> packed stream
// ---------------------------------------------------------------------------

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

MmaLayout layout24(int m_tiles, int kq, int srows, int stages) {
  MmaLayout l{};
  const int MB = 8 * m_tiles;
  l.w_off = kq * MB * 128;                // activation pieces first (multiples of 1024 bytes)
  l.s_off = l.w_off + kq * kPieceBytes;  // then the packed 2:4 pieces, then the scale rows
  l.z_off = l.s_off + srows * 256;
  l.stage_bytes = (l.z_off + 1023) / 1024 * 1024;
  l.tx_bytes = kq * MB * 128 + kq * kPieceBytes + srows * 256;
  l.red_off = stages * l.stage_bytes;
  l.bar_off = l.red_off + 3 * 2 * kNbw * m_tiles * 4 * 32 * 4;
  l.flag_off = l.bar_off + 16 * stages;
  l.moe_off = l.flag_off + 64;
  l.smem_bytes = 1024 + l.moe_off;
  return l;
}

template <int MT>
cudaError_t launch24(const MmaConfig& cfg, const CUtensorMap& tmA, const GemmParams& p, cudaStream_t stream) {
  auto kern = gemm24_kernel<MT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, cfg.smem_bytes);
  if (e != cudaSuccess) return e;
  kern<<<p.grid, kMmaThreads, cfg.smem_bytes, stream>>>(tmA, p);
  return cudaGetLastError();
}

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

Plan24 make_plan24(int M, int K, int N, int G, int sms, int smem_optin, int ablate) {
  Plan24 pl{};
  const int mt = std::min(std::max(M, 1), 16) <= 8 ? 1 : 2;
  pl.strips = N / kStrip;
  // Unit depth KT = 64 * kq, chosen as for the dense streaming kernel with 3 KB of
  // weights per 64-row piece (~67 ns of copy-engine time each, plus ~80 ns per unit).
  int best_kq = 0;
  long long best_cost = 0;
  const int cands[5] = {16, 12, 8, 4, 2};
  for (int c = 0; c < 5; ++c) {
    const int kq = cands[c];
    if (K % (64 * kq) != 0) continue;
    const int srows = (G <= 64 * kq) ? (64 * kq) / G : 1;
    const MmaLayout l0 = layout24(mt, kq, srows, 0);
    const int stages = (smem_optin - l0.smem_bytes) / (l0.stage_bytes + 16);
    if (stages < 3 && kq != 2) continue;
    const long long units = static_cast<long long>(pl.strips) * (K / (64 * kq));
    const long long T = (units + sms - 1) / sms;
    const long long cost = T * (67LL * kq + 80);
    if (best_kq == 0 || cost < best_cost) {
      best_kq = kq;
      best_cost = cost;
    }
  }
  if (!best_kq) best_kq = 2;
  const int kq = best_kq;
  const int KT = 64 * kq;
  pl.srows = (G <= KT) ? KT / G : 1;
  const MmaLayout l0 = layout24(mt, kq, pl.srows, 0);
  int stages = (smem_optin - l0.smem_bytes) / (l0.stage_bytes + 16);
  stages = std::max(2, std::min(stages, 8));
  if (ablate & kAblateStages2) stages = 2;
  pl.lay = layout24(mt, kq, pl.srows, stages);
  pl.cfg.m_tiles = mt;
  pl.cfg.kq = kq;
  pl.cfg.stages = stages;
  pl.cfg.smem_bytes = pl.lay.smem_bytes;
  pl.cfg.threads = kMmaThreads;
  pl.m_chunk = 8 * mt;
  pl.KU = K / KT;
  pl.units = pl.strips * pl.KU;
  pl.T = (pl.units + sms - 1) / sms;
  pl.grid = (pl.units + pl.T - 1) / pl.T;
  pl.workspace = kStatusBytes + counter_bytes(pl.strips) +
                 2ull * pl.grid * (static_cast<size_t>(kStrip) * 8 * mt) * sizeof(float);
  return pl;
}

int run_gemm24(const Plan24& pl, const GemmCall& c) {
  uint8_t* ws = static_cast<uint8_t*>(c.workspace);
  CUtensorMap map;
  const int er = encode_a_map(&map, c.A, c.M, c.K, pl.m_chunk, pl.cfg.kq, !(c.ablate & kAblateNoSwizzle));
  if (er != W4A16_OK) return er;
  GemmParams p{};
  p.packed = c.packed;
  p.scales = c.scales;
  p.C = c.C;
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.counters = reinterpret_cast<uint32_t*>(ws + kStatusBytes);
  p.slots = reinterpret_cast<float*>(ws + kStatusBytes + counter_bytes(pl.strips));
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
  p.stage_bytes = pl.lay.stage_bytes;
  p.tx_bytes = pl.lay.tx_bytes;
  p.red_off = pl.lay.red_off;
  p.bar_off = pl.lay.bar_off;
  p.flag_off = pl.lay.flag_off;
  p.wait_limit = c.wait_limit;
  p.debug_stall = c.debug_stall;
  p.ablate = c.ablate;
  for (int m0 = 0; m0 < c.M; m0 += pl.m_chunk) {
    p.m0 = m0;
    const cudaError_t e = pl.cfg.m_tiles == 1 ? launch24<1>(pl.cfg, map, p, c.stream)
                                              : launch24<2>(pl.cfg, map, p, c.stream);
    if (e != cudaSuccess) return W4A16_ERR_CUDA;
  }
  return W4A16_OK;
}

}  // namespace w4a16
