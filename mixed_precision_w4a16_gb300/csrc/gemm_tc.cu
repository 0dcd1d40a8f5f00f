// Tensor-memory W4A16 GEMM (tcgen05) for larger batches.
//
// Once M is large enough that the product is a real dense contraction (the
// MARLIN paper's roofline, Section 3.4: intensity ~4M FLOP/byte), the legacy
// mma.sync pipe is the limit.  This kernel feeds the sm_103a 5th-generation
// tensor cores instead.
//
//  * Work unit: a PAIR of 128-column strips x KT = 128*CH reduction rows (US = 2),
//    or, in the wide mode for more than 128 token rows (US = 1), one strip whose
//    decoded chunks feed multiplies of up to 256 tokens.  The unit's strips'
//    packed chunks (each contiguous along K) and their scale rows are
//    streamed into a ring of weight stages by one producer lane (bulk copies, L2
//    evict-first); the activation tile of each 128-row chunk ([2][MB][64] FP16,
//    128-byte swizzle) comes through a separate ring from a second producer lane
//    (3-D tensor copy, L2 evict-last) and serves the multiplies of both strips,
//    so activations are read from L2 once per 256 output columns (pair mode).
//  * Dequant: four warpgroups.  Warpgroup w serves strip w % US and the chunks
//    gs = w / US, w / US + 4 / US, ... of it; each of its warps decodes its 32-column
//    lane quarter of a whole 128-row chunk (16 packed words per thread: exact
//    q - 8, times the FP16 group scale with one RNE multiply -- the value
//    w4a16_dequant returns) and writes it with tcgen05.st.16x256b into that
//    strip's ring of A buffers in tensor memory (the packed word of lane (g, t)
//    is that store's fragment: rows g and g + 8, k = 4t .. 4t + 3).  In the wide
//    mode the four warpgroups take turns over four to seven A buffers.
//  * Multiply: one warp per strip (an elected lane) issues the chunk's eight
//    tcgen05.mma.kind::f16 (A = the chunk in tensor memory, 128 rows = the
//    strip's output columns; B = the activation stage through a shared-memory
//    descriptor; D = FP32 [128 x MB] in tensor memory, one accumulator per
//    strip, MB up to 128 in pair mode and 256 in the wide mode), then commits
//    the A buffer and the activation stage.  One issuer per strip completes its
//    chunks in order, which is what makes every parity wait of the ring protocol
//    name a unique phase.
//  * Epilogue, at the end of each unit-column segment, by all sixteen dequant
//    warps: tcgen05.ld of the accumulators (one output column per thread, 16
//    tokens per load), the per-column scale when G = K, the bias, and C -- or,
//    for pairs split between CTAs, FP32 slots reduced by the last arriver in CTA
//    order (deterministic, no spin waits).
//
// Before waiting for the previous kernel of the stream (programmatic dependent
// launch), thread 0 prefetches the first units' weights and scales into L2.
//
// Every wait is bounded; a timeout records W4A16_ERR_TIMEOUT, stops all roles,
// drains copies and multiplies in flight and always frees the tensor memory.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace w4a16 {

namespace {

// warps: 0 weight producer, 1 activation producer, 2..3 MMA issuers of strips 0 and 1 (warp 2
// owns the tensor memory), 4..19 dequant (warpgroup w = warps 4 + 4w .. 7 + 4w)
constexpr int kWeightWarp = 0;
constexpr int kActWarp = 1;
constexpr int kIssuerWarp0 = 2;
constexpr int kDequantWarp0 = 4;
constexpr int kDequantWarps = 16;
constexpr int kEpiThreads = 32 * kDequantWarps;
constexpr int kTmemCols = 512;
constexpr int kChunkCols = 64;  // 128 k of FP16 A = 64 32-bit columns
constexpr int kPairBytes = 8192;  // packed bytes of one strip's 128-row chunk
constexpr long long kDrainCycles = 2000000000LL;

// ---- tcgen05 wrappers -------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// The eight multiplies of one 128-row chunk: D[tmem] (+)= A[tmem] * B[smem], kind::f16,
// FP32 accumulate.  A: the chunk's 64 tensor-memory columns starting at `a`, 8 per
// k16 step.  B: descriptor {lo, hi} of the chunk's activation stage; k16 step kk
// starts (kk & 3) * 32 bytes into 64-row piece kk >> 2 (pieces `box16` * 16 bytes
// apart).  The first multiply overwrites D when `accumulate` is 0.
// Called by a whole warp with warp-uniform operands: one elected lane issues.  Kept
// uniform, the operands stay in the uniform datapath, and one warp issues a multiply
// every ~20 cycles (measured on GB300 at N = 32; at N >= 64 the tensor pipe is the
// limit) -- against ~50 when a single lane runs the issue loop on its own registers.
__device__ __forceinline__ void tc_mma_chunk(uint32_t d, uint32_t a, uint32_t lo, uint32_t hi, uint32_t box16,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 l, l4, t;\n\t.reg .b64 b;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "mov.b64 b, {%2, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b, %5, p;\n\t"
      "setp.eq.b32 p, %2, %2;\n\t"
      "add.u32 l, %2, 2;\n\tadd.u32 t, %1, 8;\n\tmov.b64 b, {l, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %5, p;\n\t"
      "add.u32 l, %2, 4;\n\tadd.u32 t, %1, 16;\n\tmov.b64 b, {l, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %5, p;\n\t"
      "add.u32 l, %2, 6;\n\tadd.u32 t, %1, 24;\n\tmov.b64 b, {l, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %5, p;\n\t"
      "add.u32 l4, %2, %4;\n\tadd.u32 t, %1, 32;\n\tmov.b64 b, {l4, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %5, p;\n\t"
      "add.u32 l, l4, 2;\n\tadd.u32 t, %1, 40;\n\tmov.b64 b, {l, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %5, p;\n\t"
      "add.u32 l, l4, 4;\n\tadd.u32 t, %1, 48;\n\tmov.b64 b, {l, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %5, p;\n\t"
      "add.u32 l, l4, 6;\n\tadd.u32 t, %1, 56;\n\tmov.b64 b, {l, %3};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %5, p;\n\t}" ::"r"(d),
      "r"(a), "r"(lo), "r"(hi), "r"(box16), "r"(idesc), "r"(accumulate)
      : "memory");
}
// tcgen05.commit by one elected lane of a converged warp: `bar` gets one arrival once
// every multiply this warp issued before has completed.
__device__ __forceinline__ void tc_commit_warp(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tmem_st_16x256b_x4(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes in 8-row (1024-byte) atoms.  Fields: start address >> 4 (bits
// 0..13), leading-dimension byte offset >> 4 (16..29, unused for swizzled
// K-major: 1), stride byte offset >> 4 (32..45: 1024 bytes between 8-row
// groups), descriptor version 1 (46..47), layout type 2 = 128-byte swizzle
// (61..63).  Returned as its low and high 32-bit words.
__device__ __forceinline__ uint32_t smem_desc_sw128_lo(uint32_t saddr) { return ((saddr & 0x3FFFFu) >> 4) | (1u << 16); }
__device__ __forceinline__ uint32_t smem_desc_sw128_hi() { return (1024u >> 4) | (1u << (46 - 32)) | (2u << (61 - 32)); }

__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ uint16_t f32_to_f16_bits(float x) { return __half_as_ushort(__float2half_rn(x)); }

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// position of output column r (0..127) of a strip inside its permuted scale row
__device__ __forceinline__ int scale_pos(int r) { return (r & ~15) + 2 * (r & 7) + ((r >> 3) & 1); }

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// Barrier block (8 bytes each, from p.bar_off): wfull[kTcMaxSW], wempty[kTcMaxSW],
// afull[kTcMaxNS], aempty[kTcMaxNS], cfull[2][kTcMaxNA], consumed[2][kTcMaxNA], dfull, dempty,
// drain[2].
constexpr int kBarWfull = 0;
constexpr int kBarWempty = kBarWfull + kTcMaxSW;
constexpr int kBarAfull = kBarWempty + kTcMaxSW;
constexpr int kBarAempty = kBarAfull + kTcMaxNS;
constexpr int kBarCfull = kBarAempty + kTcMaxNS;
constexpr int kBarConsumed = kBarCfull + 2 * kTcMaxNA;
constexpr int kBarDfull = kBarConsumed + 2 * kTcMaxNA;
constexpr int kBarDempty = kBarDfull + 1;
constexpr int kBarDrain = kBarDempty + 1;
constexpr int kBarCount = kBarDrain + 2;

// US: strips per work unit -- 2 (a strip pair, one issuer and two warpgroups per strip), or 1
// (wide mode: one issuer, four warpgroups taking turns over four to seven A buffers, CH = 4).
// ZP: codes carry a zero point per group and column (p.zeros), else the constant 8.
// BIAS: p.bias is added to C.
// MOE: grouped expert GEMM over p.E experts (p.expert_off, rows sorted by expert), pair mode: a
// unit column is (row segment of MB rows of one expert, strip pair), found from the offsets on the
// device; each segment multiplies its expert's weights.
// All four are compile-time, and every grouped-GEMM step sits under MOE, so the plain layer's
// build is unchanged.
template <int US, bool ZP, bool BIAS, bool MOE>
__global__ void __launch_bounds__(kTcThreads, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const TcParams p) {
  static_assert(US == 1 || US == 2, "one or two strips per unit");
  static_assert(!MOE || (US == 2 && !ZP && !BIAS), "the grouped GEMM runs in pair mode, symmetric, without bias");
  constexpr int RK = 4 / US;  // warpgroups per strip: each takes every RK-th chunk of it
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int SW = p.w_stages;
  const int NS = p.a_stages;
  const int NA = p.na;
  const int CH = p.ch;
  const int MB = p.mb;
  const uint32_t bars = sbase + p.bar_off;
  const uint32_t bar_wfull = bars + 8 * kBarWfull;
  const uint32_t bar_wempty = bars + 8 * kBarWempty;
  const uint32_t bar_afull = bars + 8 * kBarAfull;
  const uint32_t bar_aempty = bars + 8 * kBarAempty;
  const uint32_t bar_cfull = bars + 8 * kBarCfull;        // [strip][a]
  const uint32_t bar_consumed = bars + 8 * kBarConsumed;  // [strip][a]
  const uint32_t bar_dfull = bars + 8 * kBarDfull;
  const uint32_t bar_dempty = bars + 8 * kBarDempty;
  const uint32_t bar_drain = bars + 8 * kBarDrain;
  volatile int* flags = reinterpret_cast<volatile int*>(smem + p.flag_off);
  volatile int* abort_flag = flags + 0;
  volatile int* last_flag = flags + 1;
  volatile int* seg_abort = flags + 2;
  volatile int* zero_flag = flags + 3;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(flags + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  // the CTA's units; the grouped GEMM finds them after its prologue (only it reassigns these)
  int u_begin = cta * p.T;
  int u_end = min(p.units, u_begin + p.T);
  int nunits = u_end - u_begin;
  int first_pair = u_begin / p.KU;
  int kt0 = u_begin - first_pair * p.KU;
  int T_moe = 0, grid_moe = 0;   // grouped GEMM: units per CTA and CTAs
  const int* pref = nullptr;     // grouped GEMM: segment prefix per expert [E + 1]
  const int* offs = nullptr;     // grouped GEMM: expert row offsets [E + 1]
  const int pairs = (p.strips + 1) / 2;  // grouped GEMM: unit columns per row segment

  if (threadIdx.x == 0) {
    for (int s = 0; s < SW; ++s) {
      mbar_init(bar_wfull + 8 * s, 1);
      // the warpgroups with a chunk in the unit read the stage: all four, or (pair mode, units of
      // one chunk) one per strip
      mbar_init(bar_wempty + 8 * s, CH * US >= 4 ? kDequantWarps : 4 * CH * US);
    }
    for (int a = 0; a < NS; ++a) {
      mbar_init(bar_afull + 8 * a, 1);
      mbar_init(bar_aempty + 8 * a, US);  // every strip's multiplies read the stage
    }
    for (int i = 0; i < kTcStrips * kTcMaxNA; ++i) {
      mbar_init(bar_cfull + 8 * i, 4);      // the four warps of the writing warpgroup
      mbar_init(bar_consumed + 8 * i, 1);   // the strip's issuer
    }
    mbar_init(bar_dfull, US);
    mbar_init(bar_dempty, kDequantWarps);
    for (int i = 0; i < kTcStrips; ++i) mbar_init(bar_drain + 8 * i, 1);
    for (int i = 0; i < 4; ++i) flags[i] = 0;  // flags[4] receives the tensor-memory address
    mbar_fence_init();
    // the weights and scales of the first units (as many as the weight ring holds) into L2 while
    // the previous kernel drains (the grouped GEMM learns its units only from the offsets)
    const int NG = p.K / p.G;
    for (int it = 0, j = first_pair, kt = kt0; !MOE && it < min(SW, nunits); ++it) {
      const int nst = (US == 2 && 2 * j + 1 < p.strips) ? 2 : 1;
      const int grp0 = (p.G == 128) ? kt * p.srows : 0;
      for (int t = 0; t < nst; ++t) {
        const long long strip = US * j + t;
        prefetch_l2(p.packed + (strip * (p.K / 64) + static_cast<long long>(kt) * 2 * CH) * 1024,
                    static_cast<uint32_t>(CH) * kPairBytes);
        prefetch_l2(p.scales + (strip * NG + grp0) * 128, static_cast<uint32_t>(p.srows) * 256u);
        if (ZP) prefetch_l2(p.zeros + (strip * NG + grp0) * 128, static_cast<uint32_t>(p.srows) * 128u);
      }
      if (++kt == p.KU) {
        kt = 0;
        ++j;
      }
    }
  }
  if (warp == kIssuerWarp0) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
    tmem_relinquish();
  }
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel of the stream has completed: global memory is safe
  bool moe_bad = false;
  if constexpr (MOE) {
    int* s_pref = reinterpret_cast<int*>(smem + p.moe_off);
    int* s_offs = s_pref + (p.E + 1);
    int* scan = s_offs + (p.E + 1);
    const int nseg = moe_segments<kTcThreads>(p.expert_off, p.E, p.M, p.max_seg, MB, p.status, s_pref, s_offs,
                                              scan, warp, lane);
    moe_bad = nseg < 0;  // the same in every thread
    pref = s_pref;
    offs = s_offs;
    const int units = max(nseg, 0) * pairs * p.KU;
    grid_moe = static_cast<int>(gridDim.x);
    T_moe = max(1, (units + grid_moe - 1) / grid_moe);
    u_begin = cta * T_moe;
    u_end = min(units, u_begin + T_moe);
    nunits = max(0, u_end - u_begin);
    first_pair = nunits > 0 ? u_begin / p.KU : 0;
    kt0 = nunits > 0 ? u_begin - first_pair * p.KU : 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if constexpr (MOE) {
    if (moe_bad) {  // invalid offsets: nothing copied or written; free the tensor memory
      if (warp == kIssuerWarp0) tmem_dealloc(tmem, kTmemCols);
      return;
    }
  }

  auto raise_abort = [&]() {
    if (!*abort_flag) {
      *abort_flag = 1;
      atomicOr(p.status, kDevErrTimeout);
    }
  };

  if (warp == kWeightWarp) {
    // ------------------------------- producer: both strips' weights + scale rows, one stage per unit
    int issued = 0;
    if (lane == 0) {
      const uint64_t pol = (p.ablate & kAblateNoEvictFirst) ? policy_evict_normal() : policy_evict_first();
      const uint64_t pol_s = policy_evict_last();
      const int NG = p.K / p.G;
      const uint32_t w_bytes = static_cast<uint32_t>(CH) * kPairBytes;
      const uint32_t s_bytes = static_cast<uint32_t>(p.srows) * 256u;
      const uint32_t z_bytes = static_cast<uint32_t>(p.srows) * 128u;
      int s = 0, round = 0;
      int j = first_pair, kt = kt0;
      SegPos cp{0, 0, 0};  // grouped GEMM: the unit column's expert, row segment and strip pair
      if constexpr (MOE) {
        if (nunits > 0) cp = seg_locate(pref, p.E, pairs, first_pair);
      }
      for (int it = 0; it < nunits; ++it) {
        if (it >= SW && !mbar_wait_bounded_sleep(bar_wempty + 8 * s, (round - 1) & 1, p.wait_limit, abort_flag)) {
          raise_abort();
          break;
        }
        if (!(p.debug_stall && it == 0)) {  // with debug_stall, stage 0 stays empty: nothing completes its barrier
          const int pr = MOE ? cp.j : j;  // strip pair
          const int nst = (US == 2 && 2 * pr + 1 < p.strips) ? 2 : 1;
          const uint32_t fb = bar_wfull + 8 * s;
          const uint32_t* pk = MOE ? p.packed + cp.e * p.w_stride : p.packed;  // the column's expert
          const uint16_t* sk = MOE ? p.scales + cp.e * p.s_stride : p.scales;
          const uint32_t st = sbase + p.w_base + s * p.w_stage_bytes;
          mbar_arrive_expect_tx(fb, static_cast<uint32_t>(nst) * (w_bytes + s_bytes + (ZP ? z_bytes : 0u)));
          const int grp0 = (p.G == 128) ? kt * p.srows : 0;
          for (int t = 0; t < nst; ++t) {
            const long long strip = US * pr + t;
            bulk_g2s(st + t * w_bytes, pk + (strip * (p.K / 64) + static_cast<long long>(kt) * 2 * CH) * 1024,
                     w_bytes, fb, pol);
            bulk_g2s(st + p.s_off + t * s_bytes, sk + (strip * NG + grp0) * 128, s_bytes, fb, pol_s);
            if (ZP)  // the zero codes of the same scale rows, permuted the same way
              bulk_g2s(st + p.z_off + t * z_bytes, p.zeros + (strip * NG + grp0) * 128, z_bytes, fb, pol_s);
          }
          issued = it + 1;
        }
        if (++s == SW) {
          s = 0;
          ++round;
        }
        if (++kt == p.KU) {
          kt = 0;
          ++j;
          if constexpr (MOE) {
            if (it + 1 < nunits) seg_next(cp, pref, p.E, pairs);
          }
        }
      }
    }
    __syncwarp();
    named_bar_sync(3, kTcThreads);
    if (*abort_flag && lane == 0) {  // copies possibly in flight: the last SW issued
      const int first_filled = p.debug_stall ? 1 : 0;
      for (int it = max(first_filled, issued - SW); it < issued; ++it)
        mbar_wait_bounded(bar_wfull + 8 * (it % SW), (it / SW) & 1, kDrainCycles, zero_flag);
    }
    return;
  }

  if (warp == kActWarp) {
    // --------------------------- activation producer: chunk gs's tile into stage gs % NS, once the
    // stage's previous chunk has been multiplied for both strips
    int last = -1;  // last chunk whose copy was issued
    if (lane == 0) {
      prefetch_tensormap(&tmA);
      const uint64_t pol = policy_evict_last();
      const int nch = nunits * CH;
      const uint32_t a_bytes = static_cast<uint32_t>(MB) * 256u;
      int a = 0, c = 0, kt = kt0;
      uint32_t ph = 0;  // phase bit (gs / NS) & 1
      SegPos cp{0, 0, 0};  // grouped GEMM: the chunk's unit column
      if constexpr (MOE) {
        if (nunits > 0) cp = seg_locate(pref, p.E, pairs, first_pair);
      }
      for (int gs = 0; gs < nch; ++gs) {
        if (gs >= NS && !mbar_wait_bounded_sleep(bar_aempty + 8 * a, ph ^ 1u, p.wait_limit, abort_flag)) {
          raise_abort();
          break;
        }
        if (!(p.debug_stall && gs == 0)) {  // with debug_stall, stage 0 stays empty
          mbar_arrive_expect_tx(bar_afull + 8 * a, a_bytes);
          const int row0 = MOE ? offs[cp.e] + MB * cp.ci : p.m0;  // the launch's (segment's) first row
          tma_load_3d(sbase + a * p.a_stage_bytes, &tmA, 0, row0, (kt * CH + c) * 2, bar_afull + 8 * a, pol);
          last = gs;
        }
        if (++a == NS) {
          a = 0;
          ph ^= 1u;
        }
        if (++c == CH) {
          c = 0;
          if (++kt == p.KU) {
            kt = 0;
            if constexpr (MOE) {
              if (gs + 1 < nch) seg_next(cp, pref, p.E, pairs);
            }
          }
        }
      }
    }
    __syncwarp();
    named_bar_sync(3, kTcThreads);
    if (*abort_flag && lane == 0) {  // copies possibly in flight: the latest one on each stage
      const int first_filled = p.debug_stall ? 1 : 0;
      for (int gs = last; gs >= first_filled && gs > last - NS; --gs)
        mbar_wait_bounded(bar_afull + 8 * (gs % NS), (gs / NS) & 1, kDrainCycles, zero_flag);
    }
    return;
  }

  if (warp < kDequantWarp0) {
    // ------------------------------------------------------------- MMA issuers
    // Warp s multiplies every chunk of strip s of every unit, in order.  The whole warp runs
    // the loop with warp-uniform state; each multiply and commit is issued by one elected lane.
    const int s = warp - kIssuerWarp0;
    if (s >= US) {  // wide mode: one issuer
      __syncwarp();
      named_bar_sync(3, kTcThreads);
      return;
    }
    const uint32_t a_tmem = tmem + static_cast<uint32_t>(s * NA * kChunkCols);
    const uint32_t d_tmem = tmem + static_cast<uint32_t>(US * NA * kChunkCols + s * MB);
    const uint32_t lo0 = smem_desc_sw128_lo(sbase);  // activation stage 0 sits at the base
    const uint32_t hi = smem_desc_sw128_hi();
    const uint32_t stage16 = static_cast<uint32_t>(p.a_stage_bytes) >> 4;
    const uint32_t box16 = static_cast<uint32_t>(MB * 128) >> 4;
    const uint32_t cfull0 = bar_cfull + 8 * (s * kTcMaxNA), consumed0 = bar_consumed + 8 * (s * kTcMaxNA);
    int a = 0, st = 0, segs = 0, kt = kt0, j = first_pair;
    SegPos cp{0, 0, 0};  // grouped GEMM: the unit column
    if constexpr (MOE) {
      if (nunits > 0) cp = seg_locate(pref, p.E, pairs, first_pair);
    }
    uint32_t ph = 0, sph = 0;  // phase bits of A buffer a and activation stage st
    bool first = true;         // the next chunk starts the accumulator of a segment
    bool ok = true;
    for (int it = 0; it < nunits; ++it) {
      const bool seg_end = (kt == p.KU - 1) || (it == nunits - 1);
      const bool real = US * (MOE ? cp.j : j) + s < p.strips;  // the last pair of an odd strip count has one strip
      for (int c = 0; c < CH; ++c) {
        // The A chunk was written after the multiplies of chunk gs - NA completed (the dequant
        // waits for them), and this warp waited for chunk gs - NA's A chunk and activation stage
        // before; so both parity waits name a unique phase.  Both spin: a sleeping wait wakes
        // a few hundred cycles late, and this warp's chunk-to-chunk latency sets the pace.
        ok = mbar_wait_bounded(cfull0 + 8 * a, ph, p.wait_limit, abort_flag) &&
             mbar_wait_bounded(bar_afull + 8 * st, sph, p.wait_limit, abort_flag);
        // the previous segment's accumulator must have been read out
        if (ok && first && segs > 0) ok = mbar_wait_bounded(bar_dempty, (segs - 1) & 1, p.wait_limit, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        if (real)
          tc_mma_chunk(d_tmem, a_tmem + a * kChunkCols, lo0 + st * stage16, hi, box16, p.idesc, first ? 0u : 1u);
        tc_commit_warp(consumed0 + 8 * a);     // A buffer free once these multiplies complete
        tc_commit_warp(bar_aempty + 8 * st);   // activation stage: one of its strips done
        first = false;
        if (++a == NA) {
          a = 0;
          ph ^= 1u;
        }
        if (++st == NS) {
          st = 0;
          sph ^= 1u;
        }
      }
      if (!ok) {
        if (lane == 0) raise_abort();
        break;
      }
      if (seg_end) {
        tc_commit_warp(bar_dfull);
        ++segs;
        first = true;
      }
      if (++kt == p.KU) {
        kt = 0;
        ++j;
        if constexpr (MOE) {
          if (it + 1 < nunits) seg_next(cp, pref, p.E, pairs);
        }
      }
    }
    // wait for every multiply this warp issued before the memory is released
    tc_commit_warp(bar_drain + 8 * s);
    mbar_wait_bounded(bar_drain + 8 * s, 0, kDrainCycles, zero_flag);
    __syncwarp();
    named_bar_sync(3, kTcThreads);
    if (warp == kIssuerWarp0) {
      tc_fence_after();
      tmem_dealloc(tmem, kTmemCols);
    }
    return;
  }

  // ----------------------------------------------------------------- dequant
  const int dw = warp - kDequantWarp0;
  // loop-invariant launch parameters, kept in registers
  const int KU = p.KU, strips = p.strips, w_stage_bytes = p.w_stage_bytes;
  const long long wlim = p.wait_limit;
  const int wg = dw >> 2;
  const int s = wg % US;              // strip of the unit this warpgroup serves
  const int r = wg / US;              // it takes that strip's chunks gs with gs % RK == r
  const int q = warp & 3;             // tensor-memory lane quarter: rows 32q .. 32q + 31 (blocks 2q, 2q + 1)
  const int g = lane >> 2;
  const bool grouped = p.G == 128;
  const int NG = p.K / p.G;
  const uint32_t w_bytes = static_cast<uint32_t>(CH) * kPairBytes;
  // byte offsets inside a weight stage: this strip's packed piece (2c + h), block (2q + bi), and
  // its scale pair / zero pair of rows g, g + 8
  const uint32_t w_lane = static_cast<uint32_t>(s) * w_bytes + static_cast<uint32_t>((2 * q) * 512 + lane * 16);
  const uint32_t s_lane = static_cast<uint32_t>(p.s_off + s * p.srows * 256 + 2 * q * 32 + 4 * g);
  const uint32_t z_lane = static_cast<uint32_t>(p.z_off + s * p.srows * 128 + 2 * q * 16 + 2 * g);
  // tensor-memory address of this warp's lane quarter in this strip's A ring
  const uint32_t t_warp = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(s * NA * kChunkCols);
  const uint32_t cfull0 = bar_cfull + 8 * (s * kTcMaxNA), consumed0 = bar_consumed + 8 * (s * kTcMaxNA);
  // ring position of this warpgroup's next chunk gs (= r, r + RK, ...): A buffer a = gs % NA, phase
  // bit ph = (gs / NA) & 1
  int gs = r, a = r;
  uint32_t ph = 0;
  uint32_t stw = sbase + p.w_base;  // weight stage ws
  int ws = 0, wround = 0, segs = 0;
  int j = first_pair, kt = kt0;
  SegPos cp{0, 0, 0};  // grouped GEMM: the unit column
  if constexpr (MOE) {
    if (nunits > 0) cp = seg_locate(pref, p.E, pairs, first_pair);
  }
  for (int it = 0; it < nunits; ++it) {
    const bool seg_end = (kt == KU - 1) || (it == nunits - 1);
    // this warpgroup's first chunk of the unit (then every RK-th; the wide mode has CH = 4)
    const int c0 = (US == 2 && (CH & 1)) ? ((r ^ it) & 1) : r;
    const bool real = US * (MOE ? cp.j : j) + s < strips;
    if (c0 < CH) {
      bool have = false;
      if (!*abort_flag) {
        have = mbar_wait_bounded(bar_wfull + 8 * ws, wround & 1, wlim, abort_flag);
        if (!have && lane == 0) raise_abort();
      }
      have = __all_sync(0xffffffffu, have);
      if (have) {
        // This warp's words, scales and zero codes of one chunk at a time: the second chunk's are
        // read once the first chunk's stores are issued, and the stage is released after the last
        // read (it is refilled for a unit two units on, so holding it a chunk longer costs nothing).
        uint4 wv[2][2];  // [block bi][64-row piece h]
        uint32_t sc[2];
        uint32_t zc[2];
        auto load_chunk = [&](int c) {
          if (real) {
#pragma unroll
            for (int bi = 0; bi < 2; ++bi) {
#pragma unroll
              for (int h = 0; h < 2; ++h) wv[bi][h] = lds128(stw + w_lane + (2 * c + h) * 4096 + bi * 512);
              sc[bi] = grouped ? lds32(stw + s_lane + c * 256 + bi * 32) : 0x3c003c00u;
              zc[bi] = ZP ? lds_u16(stw + z_lane + (grouped ? c * 128 : 0) + bi * 16) : 0u;
            }
          }
        };
        load_chunk(c0);
        if (c0 + RK >= CH) {  // the warp's only chunk of the unit: release the stage now
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_wempty + 8 * ws);
        }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          if (c0 + RK * cc >= CH) break;
          if (gs >= NA) {  // A buffer a is free once the multiplies of chunk gs - NA have completed
            const bool ok = mbar_wait_bounded(consumed0 + 8 * a, ph ^ 1u, wlim, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
              if (lane == 0) raise_abort();
              have = false;
              break;
            }
          }
          tc_fence_after();
          if (real) {
#pragma unroll
            for (int bi = 0; bi < 2; ++bi) {
              const uint32_t s_g = __byte_perm(sc[bi], 0u, 0x1010u);   // scale of row g in both halves
              const uint32_t s_g8 = __byte_perm(sc[bi], 0u, 0x3232u);  // scale of row g + 8
              const uint32_t c_lo = ZP ? zp_const_lo(zc[bi] & 15u) : 0u;
              const uint32_t c_hi = ZP ? zp_const_hi((zc[bi] >> 8) & 15u) : 0u;
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const uint32_t words[4] = {wv[bi][h].x, wv[bi][h].y, wv[bi][h].z, wv[bi][h].w};
                uint32_t rr[16];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                  uint32_t v[4];
                  if (ZP)
                    decode8_zp(words[jj], c_lo, c_hi, v);
                  else
                    decode8(words[jj], v);
                  if (grouped) {
                    v[0] = hmul2_u32(v[0], s_g);
                    v[1] = hmul2_u32(v[1], s_g8);
                    v[2] = hmul2_u32(v[2], s_g);
                    v[3] = hmul2_u32(v[3], s_g8);
                  }
                  // .16x256b fragment order: (row g, col 2t), (row g, col 2t+1), (row g+8, col 2t), (row g+8, col 2t+1)
                  rr[4 * jj + 0] = v[0];
                  rr[4 * jj + 1] = v[2];
                  rr[4 * jj + 2] = v[1];
                  rr[4 * jj + 3] = v[3];
                }
                tmem_st_16x256b_x4(t_warp + (static_cast<uint32_t>(16 * bi) << 16) +
                                       static_cast<uint32_t>(a * kChunkCols + 32 * h), rr);
              }
            }
          }
          if (cc == 0 && c0 + RK < CH) {  // the second chunk's words, then release the stage
            load_chunk(c0 + RK);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_wempty + 8 * ws);
          }
          if (real) tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(cfull0 + 8 * a);
          gs += RK;
          a += RK;
          if (a >= NA) {
            a -= NA;
            ph ^= 1u;
          }
        }
      }
    }
    if (seg_end) {
      // ------------------------------------------------ epilogue (unit column j), all dequant warps
      named_bar_sync(1, kEpiThreads);
      if (dw == 0 && lane == 0) *seg_abort = *abort_flag;
      named_bar_sync(1, kEpiThreads);
      if (!*seg_abort) {
        bool ok = mbar_wait_bounded(bar_dfull, segs & 1, wlim, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && lane == 0) raise_abort();
        named_bar_sync(1, kEpiThreads);
        if (dw == 0 && lane == 0) *seg_abort = *abort_flag;
        named_bar_sync(1, kEpiThreads);
      }
      if (!*seg_abort) {
        tc_fence_after();
        const int row = 32 * q + lane;  // output column within its strip
        const int pr = MOE ? cp.j : j;  // strip pair (strip, wide mode)
        const int nst = (US == 2 && 2 * pr + 1 < strips) ? 2 : 1;
        const int ngrp = MB / 16;       // 16-token groups of the accumulator
        // rows of this column: the launch's, or (grouped GEMM) the segment's within its expert
        const int row0 = MOE ? offs[cp.e] + MB * cp.ci : p.m0;
        const int row_end = MOE ? min(offs[cp.e + 1], row0 + MB) : p.M;
        const int ntask = nst * ngrp;   // (strip, token group) read-outs, dealt to the warpgroups
        float scale[2], bias_n[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int strip = min(US * pr + t, strips - 1);
          const uint16_t* sk = MOE ? p.scales + cp.e * p.s_stride : p.scales;
          scale[t] = grouped ? 1.f : __half2float(__ushort_as_half(sk[static_cast<long long>(strip) * NG * 128 + scale_pos(row)]));
          bias_n[t] = BIAS ? __half2float(__ushort_as_half(p.bias[strip * kStrip + row])) : 0.f;
        }
        const uint32_t dbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(US * NA * kChunkCols);
        const int T = MOE ? T_moe : p.T;
        const int c_first = (j * KU) / T;
        const int c_last = min(((j + 1) * KU - 1) / T, (MOE ? grid_moe : p.grid) - 1);
        const int slot_floats = US * MB * 128;
        if (c_first == c_last) {
          for (int e = wg; e < ntask; e += 4) {
            const int t = e / ngrp, grp = e - t * ngrp;
            uint32_t v[16];
            tmem_ld_32x32b_x16(dbase + static_cast<uint32_t>(t * MB + grp * 16), v);
            tmem_ld_wait();
            const long long n = static_cast<long long>(US * pr + t) * kStrip + row;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int token = row0 + grp * 16 + i;
              if (token < row_end)
                p.C[static_cast<long long>(token) * p.N + n] = f32_to_f16_bits(__uint_as_float(v[i]) * scale[t] + bias_n[t]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_dempty);
        } else {
          // pair split between CTAs: FP32 partial [strip][token][column] into this CTA's slot
          const int slot = (j == first_pair) ? 2 * cta : 2 * cta + 1;
          float* dst = p.slots + static_cast<long long>(slot) * slot_floats;
          for (int e = wg; e < ntask; e += 4) {
            const int t = e / ngrp, grp = e - t * ngrp;
            uint32_t v[16];
            tmem_ld_32x32b_x16(dbase + static_cast<uint32_t>(t * MB + grp * 16), v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) dst[(t * MB + grp * 16 + i) * 128 + row] = __uint_as_float(v[i]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_dempty);
          __threadfence();
          named_bar_sync(2, kEpiThreads);
          if (dw == 0 && lane == 0) {
            const unsigned old = atomicAdd(p.counters + j, 1u);
            *last_flag = (old == static_cast<unsigned>(c_last - c_first)) ? 1 : 0;
          }
          named_bar_sync(2, kEpiThreads);
          if (*last_flag) {
            __threadfence();
            // sum the partials in CTA order, 8 tokens at a time: the 8 loads of one slot are
            // independent, so their latencies overlap
            for (int e = wg; e < ntask; e += 4) {
              const int t = e / ngrp, grp = e - t * ngrp;
              const long long n = static_cast<long long>(US * pr + t) * kStrip + row;
              for (int m = 0; m < 16 && row0 + grp * 16 + m < row_end; m += 8) {
                float acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = 0.f;
                for (int c = c_first; c <= c_last; ++c) {
                  const int cslot = (j == (c * T) / KU) ? 2 * c : 2 * c + 1;
                  const float* src =
                      p.slots + static_cast<long long>(cslot) * slot_floats + (t * MB + grp * 16 + m) * 128 + row;
                  float tv[8];
#pragma unroll
                  for (int i = 0; i < 8; ++i) tv[i] = __ldcg(src + i * 128);
#pragma unroll
                  for (int i = 0; i < 8; ++i) acc[i] += tv[i];
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const int token = row0 + grp * 16 + m + i;
                  if (token < row_end) p.C[static_cast<long long>(token) * p.N + n] = f32_to_f16_bits(acc[i] * scale[t] + bias_n[t]);
                }
              }
            }
            if (dw == 0 && lane == 0) p.counters[j] = 0u;
          }
        }
      }
      ++segs;
    }
    stw += w_stage_bytes;
    if (++ws == SW) {
      ws = 0;
      ++wround;
      stw = sbase + p.w_base;
    }
    if (++kt == KU) {
      kt = 0;
      ++j;
      if constexpr (MOE) {
        if (it + 1 < nunits) seg_next(cp, pref, p.E, pairs);
      }
    }
  }
  named_bar_sync(3, kTcThreads);
}

}  // namespace

TcLayout tc_layout(int us, int mb, int ch, int srows, int a_stages, int w_stages, bool zp, int moe_E) {
  TcLayout l{};
  l.a_stage_bytes = 2 * mb * 128;  // one 128-row chunk: a multiple of 1024 keeps the swizzle atoms aligned
  // weight stage: the unit's strips' packed chunks, their scale rows, then (with zero points) their zero rows
  l.s_off = us * ch * kPairBytes;
  l.z_off = l.s_off + us * srows * 256;
  l.w_stage_bytes = (l.z_off + (zp ? us * srows * 128 : 0) + 1023) / 1024 * 1024;
  l.w_base = a_stages * l.a_stage_bytes;
  l.bar_off = l.w_base + w_stages * l.w_stage_bytes;
  l.flag_off = l.bar_off + 8 * kBarCount;
  l.moe_off = l.flag_off + 64;
  // grouped GEMM: segment prefix and offsets ([E + 1] ints each), then the scan's 1 + 20 ints
  const int moe_bytes = moe_E > 0 ? (2 * (moe_E + 1) + 1 + kTcThreads / 32) * 4 : 0;
  l.smem_bytes = 1024 + l.moe_off + (moe_bytes + 15) / 16 * 16;
  return l;
}

// instruction descriptor, kind::f16: D = F32 (bits 4..5 = 1), A = B = F16 (bits 7..12 = 0),
// both K-major (bits 15, 16 = 0), N >> 3 in bits 17..22, M >> 4 in bits 24..28
uint32_t tc_idesc(int m, int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

cudaError_t launch_gemm_tc(int smem_bytes, const CUtensorMap& tmA, const TcParams& p, cudaStream_t stream) {
  // outside what the ring protocol and tensor memory allow: pair mode 2..3 A buffers per strip and
  // up to 128 token rows, an even weight ring for one-chunk units; wide mode four to seven A
  // buffers, units of four chunks and up to 256 token rows
  const bool pair_ok = p.us == 2 && p.na >= 2 && p.na <= 3 && p.mb <= 128 && !(p.ch == 1 && (p.w_stages & 1));
  const bool wide_ok = p.us == 1 && p.na >= 4 && p.na <= kTcMaxNA && p.ch == 4 && p.mb <= 256;
  if (!(pair_ok || wide_ok) || p.a_stages < 2 || p.a_stages > kTcMaxNS || p.w_stages < 2 ||
      p.w_stages > kTcMaxSW || p.mb < 16 || (p.mb & 15) || p.us * (p.na * kChunkCols + p.mb) > kTmemCols)
    return cudaErrorInvalidConfiguration;
  using Kern = void (*)(const CUtensorMap, const TcParams);
  static const Kern kerns[2][2][2] = {
      {{gemm_tc_kernel<1, false, false, false>, gemm_tc_kernel<1, false, true, false>},
       {gemm_tc_kernel<1, true, false, false>, gemm_tc_kernel<1, true, true, false>}},
      {{gemm_tc_kernel<2, false, false, false>, gemm_tc_kernel<2, false, true, false>},
       {gemm_tc_kernel<2, true, false, false>, gemm_tc_kernel<2, true, true, false>}}};
  const bool moe = p.expert_off != nullptr;
  if (moe && (p.us != 2 || p.zeros || p.bias || p.E < 1)) return cudaErrorInvalidConfiguration;
  const int zp = p.zeros ? 1 : 0, bias = p.bias ? 1 : 0;
  const Kern kern = moe ? gemm_tc_kernel<2, false, false, true> : kerns[p.us - 1][zp][bias];
  static int smem_cache[9][64];  // per kernel variant
  cudaError_t e = ensure_smem(kern, smem_bytes, smem_cache[moe ? 8 : (p.us - 1) * 4 + zp * 2 + bias]);
  if (e != cudaSuccess) return e;
  return launch_overlapped(kern, p.grid, kTcThreads, smem_bytes, stream, tmA, p);
}

}  // namespace w4a16
