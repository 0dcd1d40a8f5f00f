// Streaming W4A16 GEMM for small batches (up to 32 token rows per launch).
//
// The MARLIN paper (Section 3.4, "Bound By Weight Loading") makes the point
// that for small M the kernel should be bound by reading the 4-bit weights
// once.  This kernel is built around that stream on sm_103a:
//
//  * a work unit is one 128-column strip x KT = 64*KQ reduction rows; the
//    packed layout stores it as ONE contiguous chunk (KQ * 4 KB), so a single
//    producer lane fills a pipeline stage with three copy-engine (TMA)
//    operations: the weight chunk (1-D bulk copy, L2 evict-first), the
//    activation tile (3-D tensor copy, 128-byte swizzle, L2 evict-last) and
//    the unit's scale rows (1-D bulk copy); completion is tracked by an
//    mbarrier transaction count;
//  * eight consumer warps split each unit 2 ways along the columns (4 blocks
//    of 16 each) and 4 ways along K (64-row pieces kq0, kq0 + 4, ...; up to 16
//    pieces per unit); a warp
//    loads the activation fragments of its piece once (8-byte shared loads) and reuses
//    them for its 4 column blocks;
//  * each 32-bit word decodes to four FP16x2 operand registers (exact LOP3 +
//    packed-FP16 decode) feeding mma.sync.m16n8k16 with the weights on the
//    16-row side and the tokens on the 8-column side, so tiny M wastes only
//    the 8-wide slot;
//  * each 64-row piece's FP32 partial product is scaled by its group's FP32
//    scale with one FMA per accumulator;
//  * before waiting for the previous kernel of the stream (programmatic
//    dependent launch), thread 0 prefetches the first units' weights and scales
//    into L2;
//  * units are dealt to CTAs in contiguous stripes of T = ceil(units / CTAs)
//    running down a strip and wrapping into the next (the deep-dive article's
//    striped partitioning).  At a strip boundary the 4 K-split warps fold
//    their partials through shared memory in fixed order; strips split
//    between CTAs are reduced through FP32 slots with an arrival counter, the
//    last arriver summing the slots in CTA order (deterministic, no spin
//    waits);
//  * the grouped expert GEMM (MOE) runs the same pipeline over the rows of
//    all experts in one launch: a column of work units is one strip of one
//    row segment (up to 8*MT rows of one expert; MT = 1 or 2), so an expert's weights are
//    streamed once per segment and experts without rows cost nothing.  Each
//    CTA derives the segment table from the device-side expert offsets in
//    its prologue (a block-wide prefix sum), so the launch needs no host
//    synchronisation;
//  * the 2:4-sparse variant (SP24; the Sparse-Marlin analogue: the MARLIN
//    paper, Section 2.1.1 "Modern Tensor Core Units", keeps two of every four
//    weights along K with their positions as metadata) runs the same pipeline
//    on a stream of 3 KB per strip and 64-row piece and multiplies with
//    mma.sp::ordered_metadata.m16n8k32, two per piece (sparsity selectors 0
//    and 1).  Metadata lane layout, read off a GB300 by an in-bounds probe
//    that flips one nibble per MMA: with selector s the lanes t = 2s, 2s + 1
//    of each quad supply it; lane (g, 2s + r) holds in nibbles 0..3 the
//    position pairs of row g for the MMA's groups 4r .. 4r + 3, in nibbles
//    4..7 those of row g + 8.  So each lane loads one useful metadata word
//    per piece (the stream is laid out by w4a16_repack_24, sparse24.cu).
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace w4a16 {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kNbw = 4;                           // 16-column blocks per consumer warp
constexpr long long kDrainCycles = 2000000000LL;  // bound on the final drain wait

__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ uint16_t f32_to_f16_bits(float x) { return __half_as_ushort(__float2half_rn(x)); }

// 3-D tensor copy global -> shared (activations viewed as [K/64][M][64]).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}


__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// ZP: codes carry a zero point per group and column (p.zeros), else the constant 8.
// MOE: grouped expert GEMM over p.E experts (p.expert_off), else one GEMM on rows p.m0 ..
// SP24: p.packed is the 2:4-sparse stream (no zero points, no experts).
// FINAL8: the build whose last split-strip sum is shared by all eight consumer warps (dense
// layers with two token tiles, or one tile and at most two units per CTA); a separate build
// because with one token tile the larger epilogue costs the main loop up to ~1.7 % through code
// generation.
template <int MT, bool ZP, bool MOE, bool SP24, bool FINAL8>
__global__ void __launch_bounds__(kMmaThreads, 1)
    gemm_mma_kernel(const __grid_constant__ CUtensorMap tmA, const GemmParams p) {
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
  volatile int* abort_flag = flags + 0;  // set by any warp whose wait ran out
  volatile int* last_flag = flags + 1;   // "this CTA is the last arriver" broadcast
  volatile int* seg_abort = flags + 2;   // abort decision frozen for one epilogue
  volatile int* zero_flag = flags + 3;   // always 0 (for the drain wait)
  float* red = reinterpret_cast<float*>(smem + p.red_off);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  pdl_launch_dependents();
  if (MOE) pdl_wait();  // the expert offsets below may come from the previous kernel
  int units = p.units, T = p.T;
  const int* pref = nullptr;  // grouped GEMM: segment prefix per expert [E + 1]
  const int* offs = nullptr;  // grouped GEMM: expert row offsets [E + 1]
  if (MOE) {
    int* s_pref = reinterpret_cast<int*>(smem + p.moe_off);
    int* s_offs = s_pref + (p.E + 1);
    int* scan = s_offs + (p.E + 1);
    const int nseg = moe_segments<kMmaThreads>(p.expert_off, p.E, p.M, p.max_seg, MB, p.status, s_pref, s_offs,
                                               scan, warp, lane);
    if (nseg < 0) return;  // invalid offsets: every thread leaves here, before any copy
    pref = s_pref;
    offs = s_offs;
    units = nseg * p.strips * p.KU;
    T = (units + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
  }
  const int u_begin = cta * T;
  const int u_end = min(units, u_begin + T);
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
    if (!MOE) {
      // the weights and scales of the first units (as many as the stages hold) into L2 while the
      // previous kernel drains
      constexpr uint32_t kPieceWords = SP24 ? kPiece24Words : 1024u;
      const int NG = p.K / p.G;
      for (int it = 0, j = u_begin / p.KU, kt = u_begin % p.KU; it < min(S, nunits); ++it) {
        const int grp0 = (p.G == 128) ? kt * p.srows : 0;
        prefetch_l2(p.packed + (static_cast<long long>(j) * (p.K / 64) + static_cast<long long>(kt) * KQ) * kPieceWords,
                    static_cast<uint32_t>(KQ) * kPieceWords * 4u);
        prefetch_l2(p.scales + (static_cast<long long>(j) * NG + grp0) * 128, static_cast<uint32_t>(p.srows) * 256u);
        if (ZP)
          prefetch_l2(p.zeros + (static_cast<long long>(j) * NG + grp0) * 128, static_cast<uint32_t>(p.srows) * 128u);
        if (++kt == p.KU) {
          kt = 0;
          ++j;
        }
      }
    }
  }
  if (!MOE) pdl_wait();  // the previous kernel of the stream has completed: global memory is safe
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) prefetch_tensormap(&tmA);
    const uint64_t pol_w = (p.ablate & kAblateNoEvictFirst) ? policy_evict_normal() : policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    const int NG = p.K / p.G;
    constexpr uint32_t kPieceWords = SP24 ? kPiece24Words : 1024u;  // packed words per 64-row piece
    const uint32_t w_bytes = static_cast<uint32_t>(KQ) * kPieceWords * 4u;
    int issued = 0;
    // incremental counters: stage s / its fill round, strip j / unit kt within the strip
    int s = 0, round = 0;
    int j = nunits > 0 ? u_begin / p.KU : 0, kt = u_begin - j * p.KU;
    SegPos sp{0, 0, 0};
    if (MOE && nunits > 0) sp = seg_locate(pref, p.E, p.strips, j);
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
      if (!(p.debug_stall && it == 0)) {  // with debug_stall, stage 0 stays empty: nothing completes its barrier
        if (lane == 0) {
          const uint32_t st = sbase + s * p.stage_bytes;
          const uint32_t fb = bar_full + 8 * s;
          mbar_arrive_expect_tx(fb, p.tx_bytes);
          int strip = j, row0 = p.m0;
          const uint32_t* pk = p.packed;
          const uint16_t* sc = p.scales;
          if (MOE) {
            strip = sp.j;
            row0 = offs[sp.e] + MB * sp.ci;
            pk += sp.e * p.w_stride;
            sc += sp.e * p.s_stride;
          }
          const uint32_t* wsrc =
              pk + (static_cast<long long>(strip) * (p.K / 64) + static_cast<long long>(kt) * KQ) * kPieceWords;
          bulk_g2s(st + p.w_off, wsrc, w_bytes, fb, pol_w);
          tma_load_3d(st, &tmA, 0, row0, kt * KQ, fb, pol_a);
          const int grp0 = (p.G == 128) ? kt * p.srows : 0;  // G is 128 or K (K >= KT)
          const uint16_t* ssrc = sc + (static_cast<long long>(strip) * NG + grp0) * 128;
          bulk_g2s(st + p.s_off, ssrc, static_cast<uint32_t>(p.srows) * 256u, fb, pol_a);
          if (ZP)  // the zero codes of the same scale rows, permuted the same way
            bulk_g2s(st + p.z_off, p.zeros + (static_cast<long long>(j) * NG + grp0) * 128,
                     static_cast<uint32_t>(p.srows) * 128u, fb, pol_a);
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
        if (MOE && it + 1 < nunits) seg_next(sp, pref, p.E, p.strips);
      }
    }
    named_bar_sync(3, kMmaThreads);
    // After a timeout, make sure no copy is still landing in shared memory.
    if (*abort_flag && lane == 0) {
      const int first_filled = p.debug_stall ? 1 : 0;
      for (int it = max(first_filled, issued - S); it < issued; ++it)
        mbar_wait_bounded(bar_full + 8 * (it % S), (it / S) & 1, kDrainCycles, zero_flag);
    }
    return;
  }

  // -------------------------------------------------------------------- consumers
  const int ng = warp >> 2;  // column half of the strip: blocks 4*ng .. 4*ng + 3
  const int kq0 = warp & 3;  // first 64-row piece of each unit (then kq0 + 4, ...)
  const int g = lane >> 2, t = lane & 3;
  const int swz = (p.ablate & kAblateNoSwizzle) ? 0 : g;  // row-dependent XOR of the 16-byte chunks
  const int first_col = nunits > 0 ? u_begin / p.KU : 0;
  SegPos sp{0, 0, 0};
  if (MOE && nunits > 0) sp = seg_locate(pref, p.E, p.strips, first_col);

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
      // this warp's pieces kq0, kq0 + 4, ... of the unit (KQ <= 16), unrolled so the next piece's
      // loads and decode can overlap the first piece's multiply chain
#pragma unroll
      for (int pc = 0; pc < 4; ++pc) {
        const int kq = kq0 + 4 * pc;
        if (kq >= KQ) break;
if constexpr (SP24) {
          // activations: sparse MMA m (reduction rows 32m .. 32m + 31 of the piece) wants in register q
          // of lane (g, t) the pair A[token][32m + 8q + 2t .. + 1]: a 4-byte load from 16-byte chunk
          // 4m + q of the swizzled tile
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
          // the piece: 2048 bytes of code pairs [8 blocks][32 lanes][2 words], then 1024 bytes of
          // position words [8][32][1]
          const uint32_t wpiece = st + p.w_off + kq * (kPiece24Words * 4);
          uint2 cw[kNbw];
          uint32_t mw[kNbw], spv[kNbw];
#pragma unroll
          for (int i = 0; i < kNbw; ++i) {
            const int nb = ng * kNbw + i;
            cw[i] = lds64(wpiece + (nb * 32 + lane) * 8);
            mw[i] = lds32(wpiece + 2048 + (nb * 32 + lane) * 4);
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
        } else {
                // activation fragments of this 64-row piece: 4 k16 steps x MT token tiles.  The packed
        // weights hold k = 4t .. 4t+3 of each 16-row block where the m16n8k16 fragment expects
        // 2t, 2t+1, 2t+8, 2t+9, so the matching activation pair is one 8-byte load of
        // A[token][16 jj + 4t .. 4t+3] (128-byte swizzle: 16-byte chunk c of row r is at c ^ (r & 7);
        // without it, at c).
        const uint32_t a_box = st + kq * A_BOX;
        uint32_t bf[4][MT][2];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const int token = mt * 8 + g;
            const int chunk = 2 * jj + (t >> 1);
            const uint2 v = lds64(a_box + token * 128 + ((chunk ^ swz) << 4) + (t & 1) * 8);
            bf[jj][mt][0] = v.x;
            bf[jj][mt][1] = v.y;
          }
        const int srow = (p.G == 128) ? (kq >> 1) : 0;
        uint4 wv[kNbw];
        uint32_t spv[kNbw];
        uint32_t zpv[kNbw];
#pragma unroll
        for (int i = 0; i < kNbw; ++i) {
          const int nb = ng * kNbw + i;
          wv[i] = lds128(st + p.w_off + (kq * 8 + nb) * 512 + lane * 16);
          spv[i] = lds32(st + p.s_off + (srow * 128 + nb * 16 + 2 * g) * 2);
          zpv[i] = ZP ? lds_u16(st + p.z_off + srow * 128 + nb * 16 + 2 * g) : 0u;  // (z of row g, z of row g + 8)
        }
        // k16 step outermost: the kNbw x MT accumulator chains advance together, so consecutive
        // multiplies are independent (measured: M = 16 about 3 % faster than block by block)
        uint32_t c_lo[kNbw], c_hi[kNbw];
#pragma unroll
        for (int i = 0; i < kNbw; ++i) {
          c_lo[i] = ZP ? zp_const_lo(zpv[i] & 15u) : 0u;
          c_hi[i] = ZP ? zp_const_hi((zpv[i] >> 8) & 15u) : 0u;
        }
        float tmp[kNbw][MT][4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
          for (int i = 0; i < kNbw; ++i) {
            const uint32_t word = jj == 0 ? wv[i].x : jj == 1 ? wv[i].y : jj == 2 ? wv[i].z : wv[i].w;
            uint32_t a[4];
            if (ZP)
              decode8_zp(word, c_lo[i], c_hi[i], a);
            else
              decode8(word, a);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
              mma_16816(tmp[i][mt], a, bf[jj][mt][0], bf[jj][mt][1], jj == 0 ? zero4 : tmp[i][mt]);
          }
        }
#pragma unroll
        for (int i = 0; i < kNbw; ++i) {
          const float s_lo = __half2float(__ushort_as_half(static_cast<uint16_t>(spv[i] & 0xffffu)));
          const float s_hi = __half2float(__ushort_as_half(static_cast<uint16_t>(spv[i] >> 16)));
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            acc[i][mt][0] = fmaf(s_lo, tmp[i][mt][0], acc[i][mt][0]);
            acc[i][mt][1] = fmaf(s_lo, tmp[i][mt][1], acc[i][mt][1]);
            acc[i][mt][2] = fmaf(s_hi, tmp[i][mt][2], acc[i][mt][2]);
            acc[i][mt][3] = fmaf(s_hi, tmp[i][mt][3], acc[i][mt][3]);
          }
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
    // 1) fold the 4 K-split warps of each column half (kq0 = 1, 2, 3 -> kq0 = 0), fixed order
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
    if constexpr (FINAL8) {
      // small layers (at most two units per CTA): at a CTA's last segment all eight consumer
      // warps share the last arriver's sum of a split strip
      const bool skip = *seg_abort != 0;  // the same in every consumer warp
      const int c_first = (j * p.KU) / T;
      const int c_last = min(((j + 1) * p.KU - 1) / T, static_cast<int>(gridDim.x) - 1);
      int strip = j, row0 = p.m0, row_end = p.M;
      if (MOE) {
        strip = sp.j;
        row0 = offs[sp.e] + MB * sp.ci;
        row_end = min(row0 + MB, offs[sp.e + 1]);
      }
      // C for 16-column block i of this warp's column half (+ bias, FP32 -> FP16 RNE)
      auto store_block = [&](int i, const float (&v)[MT][4]) {
        const int n_base = strip * kStrip + (ng * kNbw + i) * 16 + g;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int token = row0 + mt * 8 + 2 * t + (e & 1);
            const int n = n_base + 8 * (e >> 1);
            float c = v[mt][e];
            if (p.bias) c += __half2float(__ushort_as_half(p.bias[n]));
            if (token < row_end) p.C[static_cast<long long>(token) * p.N + n] = f32_to_f16_bits(c);
          }
      };
      if (c_first == c_last) {
        // the strip lies inside this CTA: the folded sums are the result
        if (kq0 == 0 && !skip) {
#pragma unroll
          for (int i = 0; i < kNbw; ++i) store_block(i, acc[i]);
        }
      } else if (!skip) {
        // 2) this strip is split between CTAs: the folded warps publish the partial, one thread
        // counts the arrival.  Mid-range, only the two folded warps take part (the other six go on
        // decoding the next unit); at the CTA's last segment all eight share the last arriver's sum.
        const bool all8 = (it == nunits - 1);
        const bool part = all8 || kq0 == 0;
        auto sync = [&]() {
          if (all8)
            named_bar_sync(1, kConsumerWarps * 32);
          else if (kq0 == 0)
            named_bar_sync(2, 2 * 32);
        };
        if (kq0 == 0) {
          const int slot = (j == first_col) ? 2 * cta : 2 * cta + 1;
          float* dst = p.slots + static_cast<long long>(slot) * SLOT + ng * kNbw * MT * 4 * 32 + lane;
#pragma unroll
          for (int i = 0; i < kNbw; ++i)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
              for (int e = 0; e < 4; ++e) dst[((i * MT + mt) * 4 + e) * 32] = acc[i][mt][e];
          __threadfence();
        }
        sync();
        if (warp == 0 && lane == 0) {
          const unsigned old = atomicAdd(p.counters + j, 1u);
          *last_flag = (old == static_cast<unsigned>(c_last - c_first)) ? 1 : 0;
        }
        sync();
        if (part && *last_flag != 0) {
          // 3) last arriver: sum every CTA's slot in CTA order (deterministic)
          __threadfence();
          if (all8) {
            // each of the eight warps sums its block i = kq0; the loads of kU CTAs (16 floats a
            // thread) are in flight together
            constexpr int kU = 4 / MT;
            float sum[MT][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
              for (int e = 0; e < 4; ++e) sum[mt][e] = 0.f;
            const int sidx = (ng * kNbw + kq0) * MT * 4 * 32 + lane;
            for (int c0 = c_first; c0 <= c_last; c0 += kU) {
              float v[kU][MT][4];
#pragma unroll
              for (int u = 0; u < kU; ++u) {
                const int c = c0 + u;
                if (c <= c_last) {
                  const int cslot = (j == (c * T) / p.KU) ? 2 * c : 2 * c + 1;
                  const float* src = p.slots + static_cast<long long>(cslot) * SLOT + sidx;
#pragma unroll
                  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[u][mt][e] = __ldcg(src + (mt * 4 + e) * 32);
                }
              }
#pragma unroll
              for (int u = 0; u < kU; ++u)
                if (c0 + u <= c_last) {
#pragma unroll
                  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sum[mt][e] += v[u][mt][e];
                }
            }
            store_block(kq0, sum);
          } else {
            // the two folded warps sum all their blocks, one CTA's slot (all blocks' loads in
            // flight together) at a time
#pragma unroll
            for (int i = 0; i < kNbw; ++i)
#pragma unroll
              for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[i][mt][e] = 0.f;
            for (int c = c_first; c <= c_last; ++c) {
              const int cslot = (j == (c * T) / p.KU) ? 2 * c : 2 * c + 1;
              const float* src = p.slots + static_cast<long long>(cslot) * SLOT + ng * kNbw * MT * 4 * 32 + lane;
#pragma unroll
              for (int i = 0; i < kNbw; ++i)
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                  for (int e = 0; e < 4; ++e) acc[i][mt][e] += __ldcg(src + ((i * MT + mt) * 4 + e) * 32);
            }
#pragma unroll
            for (int i = 0; i < kNbw; ++i) store_block(i, acc[i]);
          }
          if (warp == 0 && lane == 0) p.counters[j] = 0u;
        }
      }
    } else {
      const bool skip = *seg_abort != 0;
      if (kq0 == 0 && !skip) {
        const int c_first = (j * p.KU) / T;
        const int c_last = min(((j + 1) * p.KU - 1) / T, static_cast<int>(gridDim.x) - 1);
        const int sidx0 = ng * kNbw * MT * 4 * 32 + lane;  // this warp's part of a strip partial
        bool write_now = true;
        if (c_first != c_last) {
          // 2) this strip is split between CTAs: publish the partial, count arrivals
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
            // 3) last arriver: sum every CTA's slot in CTA order (deterministic)
            __threadfence();
#pragma unroll
            for (int i = 0; i < kNbw; ++i)
#pragma unroll
              for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[i][mt][e] = 0.f;
            for (int c = c_first; c <= c_last; ++c) {
              const int cslot = (j == (c * T) / p.KU) ? 2 * c : 2 * c + 1;
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
          int strip = j, row0 = p.m0, row_end = p.M;
          if (MOE) {
            strip = sp.j;
            row0 = offs[sp.e] + MB * sp.ci;
            row_end = min(row0 + MB, offs[sp.e + 1]);
          }
#pragma unroll
          for (int i = 0; i < kNbw; ++i) {
            const int n_base = strip * kStrip + (ng * kNbw + i) * 16 + g;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int token = row0 + mt * 8 + 2 * t + (e & 1);
                const int n = n_base + 8 * (e >> 1);
                float c = acc[i][mt][e];
                if (p.bias) c += __half2float(__ushort_as_half(p.bias[n]));
                if (token < row_end) p.C[static_cast<long long>(token) * p.N + n] = f32_to_f16_bits(c);
              }
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
    if (MOE && it + 1 < nunits) seg_next(sp, pref, p.E, p.strips);
  }
  named_bar_sync(3, kMmaThreads);
}

template <int MT, bool ZP, bool MOE = false, bool SP24 = false, bool FINAL8 = false>
cudaError_t launch_one(const MmaConfig& cfg, const CUtensorMap& tmA, const GemmParams& p, cudaStream_t stream) {
  auto kern = gemm_mma_kernel<MT, ZP, MOE, SP24, FINAL8>;
  static int smem_cache[64];
  cudaError_t e = ensure_smem(kern, cfg.smem_bytes, smem_cache);
  if (e != cudaSuccess) return e;
  return launch_overlapped(kern, p.grid, kMmaThreads, cfg.smem_bytes, stream, tmA, p);
}

}  // namespace

MmaLayout mma_layout(int m_tiles, int kq, int srows, int stages, bool zp, int moe_E, int piece_bytes) {
  MmaLayout l{};
  const int MB = 8 * m_tiles;
  l.w_off = kq * MB * 128;        // activation pieces first (each a multiple of 1024 bytes)
  l.s_off = l.w_off + kq * piece_bytes;  // then the weight chunk, then the scale rows
  l.z_off = l.s_off + srows * 256;  // then, with zero points, their rows (128 bytes each)
  const int zbytes = zp ? srows * 128 : 0;
  l.stage_bytes = (l.z_off + zbytes + 1023) / 1024 * 1024;
  l.tx_bytes = kq * MB * 128 + kq * piece_bytes + srows * 256 + zbytes;
  l.red_off = stages * l.stage_bytes;
  l.bar_off = l.red_off + 3 * 2 * kNbw * m_tiles * 4 * 32 * 4;
  l.flag_off = l.bar_off + 16 * stages;
  l.moe_off = l.flag_off + 64;
  // grouped GEMM: segment prefix and offsets ([E + 1] ints each), then the scan's 1 + 9 ints
  const int moe_bytes = moe_E > 0 ? (2 * (moe_E + 1) + 1 + kMmaThreads / 32) * 4 : 0;
  l.smem_bytes = 1024 + l.moe_off + (moe_bytes + 15) / 16 * 16;
  return l;
}

cudaError_t launch_gemm_mma(const MmaConfig& cfg, const CUtensorMap& tmA, const GemmParams& p, cudaStream_t stream) {
  const bool zp = p.zeros != nullptr;
  if (cfg.final8) {
    switch (cfg.m_tiles) {
      case 1:
        return zp ? launch_one<1, true, false, false, true>(cfg, tmA, p, stream)
                  : launch_one<1, false, false, false, true>(cfg, tmA, p, stream);
      case 2:
        return zp ? launch_one<2, true, false, false, true>(cfg, tmA, p, stream)
                  : launch_one<2, false, false, false, true>(cfg, tmA, p, stream);
      default: break;
    }
  }
  switch (cfg.m_tiles) {
    case 1: return zp ? launch_one<1, true>(cfg, tmA, p, stream) : launch_one<1, false>(cfg, tmA, p, stream);
    case 2: return zp ? launch_one<2, true>(cfg, tmA, p, stream) : launch_one<2, false>(cfg, tmA, p, stream);
    case 4: return zp ? launch_one<4, true>(cfg, tmA, p, stream) : launch_one<4, false>(cfg, tmA, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_moe_mma(const MmaConfig& cfg, const CUtensorMap& tmA, const GemmParams& p, cudaStream_t stream) {
  switch (cfg.m_tiles) {
    case 1: return launch_one<1, false, true>(cfg, tmA, p, stream);
    case 2: return launch_one<2, false, true>(cfg, tmA, p, stream);  // segments are at most 16 rows
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm_sp24(const MmaConfig& cfg, const CUtensorMap& tmA, const GemmParams& p, cudaStream_t stream) {
  switch (cfg.m_tiles) {
    case 1: return launch_one<1, false, false, true>(cfg, tmA, p, stream);
    case 2: return launch_one<2, false, false, true>(cfg, tmA, p, stream);
    case 4: return launch_one<4, false, false, true>(cfg, tmA, p, stream);  // 32 token rows per launch
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace w4a16
