// Tensor-memory W4A16 GEMM (tcgen05) for larger batches.
//
// Once M is large enough that the product is a real dense contraction (the
// MARLIN paper's roofline, Section 3.4: intensity ~4M FLOP/byte), the legacy
// mma.sync pipe is the limit.  This kernel feeds the sm_103a 5th-generation
// tensor cores instead:
//
//  * a CTA owns stripes of work units exactly like the streaming kernel: one
//    128-column strip x KT = 128*CH reduction rows per unit, loaded by one
//    producer lane with three copy-engine operations (weights, activations as a
//    swizzled [K/64][M][64] tile, scale rows) into a ring of shared-memory stages;
//  * two teams of dequant warps (two warpgroups each) take alternate 128-row
//    chunks; a warpgroup decodes one 64-row half of its team's chunk to FP16
//    (exact q - 8, times the FP16 group scale with one RNE multiply -- the same
//    value w4a16_dequant returns) and writes it with tcgen05.st.16x256b straight
//    into tensor memory, where it forms the A operand (128 rows = the strip's
//    output columns, K along the 32-bit columns).  The packed word of lane
//    (g, t) is that store's fragment: rows g and g + 8, k = 4t .. 4t + 3.  With
//    two teams, one team's hand-off latency (store drain, fences, barrier
//    waits) overlaps the other team's decode arithmetic;
//  * up to four threads, each in its own warp on its own SM sub-partition,
//    issue tcgen05.mma.kind::f16 (A from tensor memory, B = the activation tile
//    through a shared-memory descriptor, FP32 accumulators D[128 x MB] in
//    tensor memory, one per issuer).  The dequant warps keep the integer and
//    FP16 pipes busy, so an issuer gets few issue slots: its per-chunk path is
//    one wait per barrier, one asm block with the chunk's eight multiplies and a
//    single tcgen05.commit.  Activation stage a and tensor-memory A buffer a
//    belong to the same chunk, so that one commit frees both;
//  * at the end of each strip segment the first warpgroup reads D back with
//    tcgen05.ld (one output column per thread, the tokens along registers),
//    applies the per-column scale when G = K, and writes C -- or, for strips
//    split between CTAs, FP32 slots reduced by the last arriver in CTA order
//    (deterministic, no spin waits).
//
// Every wait is bounded; a timeout records W4A16_ERR_TIMEOUT, stops all roles,
// drains copies and MMAs in flight and always frees the tensor memory.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace w4a16 {

namespace {

// warps: 0 weight producer, 1..2 activation producers (even / odd chunks), 3..6 MMA
// issuers 0..3 (warp 3 owns the tensor memory), 7 idle (it completes the second
// warpgroup), 8..23 dequant (team 0: warps 8..15, team 1: warps 16..23)
constexpr int kActWarp0 = 1;
constexpr int kIssuerWarp0 = 3;
constexpr int kDequantWarp0 = 8;
// Register split (setmaxnreg): the two helper warpgroups drop to kHelperRegs per thread and
// the four dequant warpgroups rise to kDequantRegs.  The launch allocates numRegs * kTcThreads;
// the rise must be covered by what the drop releases, which launch_gemm_tc checks before it
// launches (an uncovered rise would wait forever).
constexpr int kHelperRegs = 40;
constexpr int kDequantRegs = 96;
constexpr int kHelperThreads = 32 * kDequantWarp0;
constexpr int kDequantThreads = kTcThreads - kHelperThreads;
constexpr int kDequantWarps = 16;  // both teams; every one releases each weight stage
constexpr int kTeamWarps = 8;      // one team: the writers of one A chunk
constexpr int kEpiThreads = 32 * kTeamWarps;  // team 0 runs the epilogue
constexpr int kTmemCols = 512;
constexpr int kChunkCols = 64;           // 128 k of FP16 A = 64 32-bit columns
constexpr int kMaxNA = 7;                // A chunks in flight in tensor memory (p.na <= 7)
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
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// The eight multiplies of one 128-row chunk: D[tmem] (+)= A[tmem] * B[smem], kind::f16,
// FP32 accumulate.  A: the chunk's 64 tensor-memory columns starting at `a`, 8 per
// k16 step.  B: descriptor {lo, hi} of the chunk's activation stage; k16 step kk
// starts (kk & 3) * 32 bytes into 64-row piece kk >> 2 (pieces `box16` * 16 bytes
// apart).  The first multiply overwrites D when `accumulate` is 0.
__device__ __forceinline__ void tc_mma_chunk(uint32_t d, uint32_t a, uint32_t lo, uint32_t hi, uint32_t box16,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b32 l, l4, t;\n\t.reg .b64 b;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "mov.b64 b, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b, %5, p;\n\t"
      "setp.eq.b32 p, %2, %2;\n\t"
      "add.u32 l, %2, 2;\n\tadd.u32 t, %1, 8;\n\tmov.b64 b, {l, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %5, p;\n\t"
      "add.u32 l, %2, 4;\n\tadd.u32 t, %1, 16;\n\tmov.b64 b, {l, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %5, p;\n\t"
      "add.u32 l, %2, 6;\n\tadd.u32 t, %1, 24;\n\tmov.b64 b, {l, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %5, p;\n\t"
      "add.u32 l4, %2, %4;\n\tadd.u32 t, %1, 32;\n\tmov.b64 b, {l4, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %5, p;\n\t"
      "add.u32 l, l4, 2;\n\tadd.u32 t, %1, 40;\n\tmov.b64 b, {l, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %5, p;\n\t"
      "add.u32 l, l4, 4;\n\tadd.u32 t, %1, 48;\n\tmov.b64 b, {l, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %5, p;\n\t"
      "add.u32 l, l4, 6;\n\tadd.u32 t, %1, 56;\n\tmov.b64 b, {l, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t], b, %5, p;\n\t}" ::"r"(d),
      "r"(a), "r"(lo), "r"(hi), "r"(box16), "r"(idesc), "r"(accumulate)
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

// ZP: codes carry a zero point per group and column (p.zeros), else the constant 8.
// BIAS: p.bias is added to C.  Both are compile-time so the plain layer's build is unchanged.
template <bool ZP, bool BIAS>
__global__ void __launch_bounds__(kTcThreads, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int SW = p.w_stages;         // weight + scale ring (released by the dequant warps)
  const int CH = p.ch;
  const int KQ = 2 * CH;
  const int MB = p.mb;
  const int A_BOX = MB * 128;
  // Chunk gc of the CTA uses activation stage and tensor-memory A buffer gc % NA;
  // the accumulators follow the A buffers in tensor memory.
  const int NA = p.na;
  const int NI = p.ni;               // MMA-issuing threads, each with its own accumulator region
  const int kDCol = NA * kChunkCols;
  const uint32_t bar_afull = sbase + p.bar_off;        // activation stage landed
  const uint32_t bar_wfull = bar_afull + 8 * kMaxNA;   // weight stage landed
  const uint32_t bar_wempty = bar_wfull + 8 * SW;      // weight stage read by the dequant warps
  const uint32_t bar_cfull = bar_wempty + 8 * SW;      // A chunk written to tensor memory
  const uint32_t bar_consumed = bar_cfull + 8 * kMaxNA;  // chunk's multiplies done: stage and A buffer free
  const uint32_t bar_dfull = bar_consumed + 8 * kMaxNA;
  const uint32_t bar_dempty = bar_dfull + 8;
  const uint32_t bar_drain = bar_dempty + 8;
  volatile int* flags = reinterpret_cast<volatile int*>(smem + p.flag_off);
  volatile int* abort_flag = flags + 0;
  volatile int* last_flag = flags + 1;
  volatile int* seg_abort = flags + 2;
  volatile int* zero_flag = flags + 3;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(flags + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const int u_begin = cta * p.T;
  const int u_end = min(p.units, u_begin + p.T);
  const int nunits = u_end - u_begin;
  const int first_col = u_begin / p.KU;
  const int kt0 = u_begin - first_col * p.KU;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SW; ++s) {
      mbar_init(bar_wfull + 8 * s, 1);
      mbar_init(bar_wempty + 8 * s, kDequantWarps);
    }
    for (int a = 0; a < NA; ++a) {
      mbar_init(bar_afull + 8 * a, 1);
      mbar_init(bar_cfull + 8 * a, kTeamWarps);
      mbar_init(bar_consumed + 8 * a, 1);
    }
    mbar_init(bar_dfull, NI);
    mbar_init(bar_dempty, kTeamWarps);
    for (int i = 0; i < 4; ++i) mbar_init(bar_drain + 8 * i, 1);
    for (int i = 0; i < 4; ++i) flags[i] = 0;  // flags[4] receives the tensor-memory address from warp 2
    mbar_fence_init();
  }
  if (warp == kIssuerWarp0) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // warpgroup-uniform: warps 0..7 are warpgroups 0 and 1, warps 8..23 warpgroups 2..5
  if (warp < kDequantWarp0)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kHelperRegs));
  else
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kDequantRegs));

  auto raise_abort = [&]() {
    if (!*abort_flag) {
      *abort_flag = 1;
      atomicOr(p.status, kDevErrTimeout);
    }
  };

  if (warp == 0) {
    // ------------------------------------------- producer: weights + scale rows, one stage per unit
    const uint64_t pol = (p.ablate & kAblateNoEvictFirst) ? policy_evict_normal() : policy_evict_first();
    const uint64_t pol_s = policy_evict_last();
    const int NG = p.K / p.G;
    const uint32_t w_bytes = static_cast<uint32_t>(KQ) * 4096u;
    int issued = 0;
    int s = 0, round = 0;
    int j = first_col, kt = kt0;
    for (int it = 0; it < nunits; ++it) {
      if (it >= SW) {
        bool ok = true;
        if (lane == 0) ok = mbar_wait_bounded_sleep(bar_wempty + 8 * s, (round - 1) & 1, p.wait_limit, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          if (lane == 0) raise_abort();
          break;
        }
      }
      if (!(p.debug_stall && it == 0)) {  // with debug_stall, stage 0 stays empty: nothing completes its barrier
        if (lane == 0) {
          const uint32_t fb = bar_wfull + 8 * s;
          const uint32_t st = sbase + p.w_base + s * p.w_stage_bytes;
          mbar_arrive_expect_tx(fb, w_bytes + static_cast<uint32_t>(p.srows) * (ZP ? 384u : 256u));
          const uint32_t* wsrc =
              p.packed + (static_cast<long long>(j) * (p.K / 64) + static_cast<long long>(kt) * KQ) * 1024;
          bulk_g2s(st, wsrc, w_bytes, fb, pol);
          const int grp0 = (p.G == 128) ? kt * p.srows : 0;
          const uint16_t* ssrc = p.scales + (static_cast<long long>(j) * NG + grp0) * 128;
          bulk_g2s(st + w_bytes, ssrc, static_cast<uint32_t>(p.srows) * 256u, fb, pol_s);
          if (ZP)  // the zero codes of the same scale rows, permuted the same way
            bulk_g2s(st + p.z_off, p.zeros + (static_cast<long long>(j) * NG + grp0) * 128,
                     static_cast<uint32_t>(p.srows) * 128u, fb, pol_s);
        }
        __syncwarp();
        issued = it + 1;
      }
      if (++s == SW) {
        s = 0;
        ++round;
      }
      if (++kt == p.KU) {
        kt = 0;
        ++j;
      }
    }
    named_bar_sync(3, kTcThreads);
    if (*abort_flag && lane == 0) {
      const int first_filled = p.debug_stall ? 1 : 0;
      for (int it = max(first_filled, issued - SW); it < issued; ++it)
        mbar_wait_bounded(bar_wfull + 8 * (it % SW), (it / SW) & 1, kDrainCycles, zero_flag);
    }
    return;
  }

  if (warp < kIssuerWarp0) {
    // ------------------------------- activation producers: chunk gc's tile into stage gc % NA, warp
    // kActWarp0 + (gc & 1) for chunk gc (NA is even, so each producer owns every other stage).  One
    // thread's loop is slow while the dequant warps hold the issue slots; two share the chunks.
    const int ap = warp - kActWarp0;
    int last = -1;  // last chunk whose copy this lane issued
    if (lane == 0) {
      prefetch_tensormap(&tmA);
      const uint64_t pol = policy_evict_last();
      const int nch = nunits * CH;
      int a = ap, c = ap, kt = kt0;
      uint32_t ph = 0;  // phase bit (gc / NA) & 1 of chunk gc's stage
      while (c >= CH) {
        c -= CH;
        if (++kt == p.KU) kt = 0;
      }
      for (int gc = ap; gc < nch; gc += 2) {
        if (gc >= NA &&
            !mbar_wait_bounded_sleep(bar_consumed + 8 * a, ph ^ 1u, p.wait_limit, abort_flag)) {
          raise_abort();
          break;
        }
        if (!(p.debug_stall && gc == 0)) {  // with debug_stall, stage 0 stays empty
          mbar_arrive_expect_tx(bar_afull + 8 * a, static_cast<uint32_t>(2 * A_BOX));
          tma_load_3d(sbase + a * p.a_stage_bytes, &tmA, 0, p.m0, kt * KQ + 2 * c, bar_afull + 8 * a, pol);
          last = gc;
        }
        a += 2;
        if (a >= NA) {
          a -= NA;
          ph ^= 1u;
        }
        c += 2;
        while (c >= CH) {
          c -= CH;
          if (++kt == p.KU) kt = 0;
        }
      }
    }
    __syncwarp();
    named_bar_sync(3, kTcThreads);
    if (*abort_flag && lane == 0) {
      // copies possibly in flight: this producer's latest one on each of its stages
      for (int gc = last; gc >= 0 && gc > last - NA; gc -= 2)
        mbar_wait_bounded(bar_afull + 8 * (gc % NA), (gc / NA) & 1, kDrainCycles, zero_flag);
    }
    return;
  }

  if (warp < kDequantWarp0) {
    // ------------------------------------------------------------- MMA issuers
    // A single thread can issue a tcgen05.mma only every ~90 cycles, far below the
    // tensor core's rate for small N; NI threads therefore issue in parallel, issuer i
    // taking the chunks gc = i mod NI into its own accumulator.  The loop visits only
    // those chunks: a starved thread pays for every instruction.
    const int issuer = warp - kIssuerWarp0;
    if (lane == 0 && issuer < NI) {
      const uint32_t d_tmem = tmem + kDCol + issuer * MB;
      const uint32_t lo0 = smem_desc_sw128_lo(sbase);  // activation stage 0 sits at the base
      const uint32_t hi = smem_desc_sw128_hi();
      const uint32_t stage16 = static_cast<uint32_t>(p.a_stage_bytes) >> 4;
      const uint32_t box16 = static_cast<uint32_t>(A_BOX) >> 4;
      int a = issuer, segs = 0, kt = kt0;  // a = gc % NA of this issuer's next chunk
      uint32_t ph = 0;                     // phase bit (gc / NA) & 1
      bool first = true;  // next chunk of this issuer starts its accumulator for the segment
      bool ok = true;
      for (int it = 0; it < nunits; ++it) {
        const bool seg_end = (kt == p.KU - 1) || (it == nunits - 1);
        const int c0 = (issuer - it * CH) & (NI - 1);  // first own chunk of the unit (NI is a power of two)
        for (int c = c0; c < CH; c += NI) {
          // The A chunk first.  Its arrival means that this team's chunk gc - NA was decoded
          // after the multiplies of chunk gc - NA completed, and those had waited for that chunk's
          // activation copy; only then does the parity wait on the activation stage (shared with
          // chunks of other issuers when NA is not a multiple of NI) name a unique phase.  Waited
          // the other way round, an activation copy still in flight for chunk gc - NA could be
          // taken for chunk gc's.
          ok = mbar_wait_bounded_sleep(bar_cfull + 8 * a, ph, p.wait_limit, abort_flag) &&
               mbar_wait_bounded_sleep(bar_afull + 8 * a, ph, p.wait_limit, abort_flag);
          // the previous segment's accumulators must have been read out
          if (ok && first && segs > 0) ok = mbar_wait_bounded(bar_dempty, (segs - 1) & 1, p.wait_limit, abort_flag);
          if (!ok) break;
          tc_fence_after();
          tc_mma_chunk(d_tmem, tmem + a * kChunkCols, lo0 + a * stage16, hi, box16, p.idesc, first ? 0u : 1u);
          tc_commit(bar_consumed + 8 * a);  // stage and A buffer free once these multiplies complete
          first = false;
          a += NI;
          if (a >= NA) {
            a -= NA;
            ph ^= 1u;
          }
        }
        if (!ok) {
          raise_abort();
          break;
        }
        if (seg_end) {
          // An issuer without a chunk in this segment (fewer chunks than issuers: a CTA's range
          // ending just past a strip boundary) has not waited for the previous segment's
          // read-out; without that wait its commit could complete the previous phase of
          // bar_dfull, ahead of another issuer's multiplies.
          if (first && segs > 0 && !mbar_wait_bounded(bar_dempty, (segs - 1) & 1, p.wait_limit, abort_flag)) {
            raise_abort();
            break;
          }
          tc_commit(bar_dfull);
          ++segs;
          first = true;
        }
        if (++kt == p.KU) kt = 0;
      }
      // wait for every multiply this thread issued before the memory is released
      tc_commit(bar_drain + 8 * issuer);
      mbar_wait_bounded(bar_drain + 8 * issuer, 0, kDrainCycles, zero_flag);
    }
    __syncwarp();
    named_bar_sync(3, kTcThreads);
    if (warp == kIssuerWarp0) {
      tc_fence_after();
      tmem_dealloc(tmem, kTmemCols);
    }
    return;
  }

  // ----------------------------------------------------------------- dequant
  // The decode shares the SM's half-rate integer / FP16 issue with every
  // integer instruction around it, so the loop keeps its bookkeeping small:
  // ring positions advance by counters, addresses by offsets fixed here.
  const int dw = warp - kDequantWarp0;
  const int team = dw >> 3;          // this team writes the chunks with gc % 2 == team
  const int wg = (dw >> 2) & 1;      // which 64-row half of each 128-row chunk
  const int q = warp & 3;            // tensor-memory lane quarter: rows 32q .. 32q + 31 (blocks 2q, 2q + 1)
  const int g = lane >> 2;
  const bool grouped = p.G == 128;
  const int NG = p.K / p.G;
  const bool epi_lead = warp == kDequantWarp0;  // first warp of team 0
  const bool epi_group = team == 0;  // team 0 reads the accumulators out, each warpgroup half of the tokens
  // byte offsets inside a weight stage: packed block (kq = 2c + wg, b = 2q + bi) and its scale pair
  const uint32_t w_lane = static_cast<uint32_t>((wg * 8 + 2 * q) * 512 + lane * 16);
  const uint32_t s_lane = static_cast<uint32_t>(KQ * 4096 + 2 * q * 32 + 4 * g);
  const uint32_t z_lane = static_cast<uint32_t>(p.z_off + 2 * q * 16 + 2 * g);  // zero pair of rows g, g + 8
  // tensor-memory address of this warp's first store: lanes 32q.., columns of half wg
  const uint32_t t_warp = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(wg * 32);
  // this team's chunks are gc = team, team + 2, ...: A buffer a = gc % NA, phase ph = (gc / NA) & 1
  int a = team, tcount = 0;
  uint32_t ph = 0;
  const int reuse_from = (NA - team + 1) >> 1;  // team chunks before this team's first gc >= NA
  uint32_t st = sbase + p.w_base;    // weight stage s
  int s = 0, round = 0, segs = 0, seg_units = 0;
  int j = first_col, kt = kt0;
  for (int it = 0; it < nunits; ++it) {
    ++seg_units;
    const bool seg_end = (kt == p.KU - 1) || (it == nunits - 1);
    const int c0 = (CH & 1) ? ((team ^ it) & 1) : team;  // this team's first chunk of the unit (then every second one)
    const bool go = __shfl_sync(0xffffffffu, *abort_flag == 0, 0);
    bool have = false;
    if (go) {
      have = mbar_wait_bounded(bar_wfull + 8 * s, round & 1, p.wait_limit, abort_flag);
      have = __all_sync(0xffffffffu, have);
      if (!have && lane == 0) raise_abort();
    }
    if (have) {
      // read this warp's share of the team's chunks and their scales, then release the stage
      uint4 wv[2][2];
      uint32_t sc[2][2];
      uint32_t zc[2][2];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = c0 + 2 * cc;
        if (c < CH) {
#pragma unroll
          for (int bi = 0; bi < 2; ++bi) {
            wv[cc][bi] = lds128(st + w_lane + c * 8192 + bi * 512);
            sc[cc][bi] = grouped ? lds32(st + s_lane + c * 256 + bi * 32) : 0x3c003c00u;
            zc[cc][bi] = ZP ? lds_u16(st + z_lane + (grouped ? c * 128 : 0) + bi * 16) : 0u;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_wempty + 8 * s);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        if (c0 + 2 * cc >= CH || !have) break;
        if (tcount >= reuse_from) {
          bool ok = mbar_wait_bounded(bar_consumed + 8 * a, ph ^ 1u, p.wait_limit, abort_flag);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) {
            if (lane == 0) raise_abort();
            have = false;
            break;
          }
        }
        tc_fence_after();
#pragma unroll
        for (int bi = 0; bi < 2; ++bi) {
          const uint32_t s_g = __byte_perm(sc[cc][bi], 0u, 0x1010u);   // scale of row g in both halves
          const uint32_t s_g8 = __byte_perm(sc[cc][bi], 0u, 0x3232u);  // scale of row g + 8
          const uint32_t words[4] = {wv[cc][bi].x, wv[cc][bi].y, wv[cc][bi].z, wv[cc][bi].w};
          const uint32_t c_lo = ZP ? zp_const_lo(zc[cc][bi] & 15u) : 0u;
          const uint32_t c_hi = ZP ? zp_const_hi((zc[cc][bi] >> 8) & 15u) : 0u;
          uint32_t r[16];
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
            r[4 * jj + 0] = v[0];
            r[4 * jj + 1] = v[2];
            r[4 * jj + 2] = v[1];
            r[4 * jj + 3] = v[3];
          }
          tmem_st_16x256b_x4(t_warp + (static_cast<uint32_t>(16 * bi) << 16) + a * kChunkCols, r);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_cfull + 8 * a);
        ++tcount;
        a += 2;
        if (a >= NA) {
          a -= NA;
          ph ^= 1u;
        }
      }
    }
    if (seg_end && epi_group) {
      // ------------------------------------------------------ epilogue (strip j)
      named_bar_sync(1, kEpiThreads);
      if (epi_lead && lane == 0) *seg_abort = *abort_flag;
      named_bar_sync(1, kEpiThreads);
      if (!*seg_abort) {
        bool ok = mbar_wait_bounded(bar_dfull, segs & 1, p.wait_limit, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && lane == 0) raise_abort();
        named_bar_sync(1, kEpiThreads);
        if (epi_lead && lane == 0) *seg_abort = *abort_flag;
        named_bar_sync(1, kEpiThreads);
      }
      if (!*seg_abort) {
        tc_fence_after();
        const int row = 32 * q + lane;
        const int n = j * kStrip + row;
        const float scale =
            grouped ? 1.f
                    : __half2float(__ushort_as_half(p.scales[static_cast<long long>(j) * NG * 128 + scale_pos(row)]));
        const float bias_n = BIAS ? __half2float(__ushort_as_half(p.bias[n])) : 0.f;
        const int c_first = (j * p.KU) / p.T;
        const int c_last = min(((j + 1) * p.KU - 1) / p.T, p.grid - 1);
        const int nchunks = MB / 16;
        const int half = (nchunks + 1) >> 1;       // 16-token groups of warpgroup 0; warpgroup 1 takes the rest
        const int ch_lo = wg * half, ch_hi = min(nchunks, ch_lo + half);
        // accumulator regions written in this segment: chunk gc went to issuer gc % NI,
        // summed in a fixed order starting at the segment's first chunk
        const int nseg = seg_units * CH;
        const int nact = min(NI, nseg);
        const int r_first = (nseg >= NI) ? 0 : (((it - seg_units + 1) * CH) & (NI - 1));
        const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + kDCol;
        // sum of the active accumulator regions for tokens ch*16 .. ch*16+15 (fixed order)
        auto load_sum = [&](int ch, float (&out)[16]) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(taddr + r_first * MB + ch * 16, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) out[i] = __uint_as_float(v[i]);
          for (int t = 1; t < nact; ++t) {
            tmem_ld_32x32b_x16(taddr + ((r_first + t) & (NI - 1)) * MB + ch * 16, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) out[i] += __uint_as_float(v[i]);
          }
        };
        if (c_first == c_last) {
          for (int ch = ch_lo; ch < ch_hi; ++ch) {
            float v[16];
            load_sum(ch, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int token = p.m0 + ch * 16 + i;
              if (token < p.M) p.C[static_cast<long long>(token) * p.N + n] = f32_to_f16_bits(BIAS ? v[i] * scale + bias_n : v[i] * scale);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_dempty);
        } else {
          // strip split between CTAs: FP32 partial [token][row] into this CTA's slot
          const int slot = (j == first_col) ? 2 * cta : 2 * cta + 1;
          float* dst = p.slots + static_cast<long long>(slot) * (128 * MB);
          for (int ch = ch_lo; ch < ch_hi; ++ch) {
            float v[16];
            load_sum(ch, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) dst[(ch * 16 + i) * 128 + row] = v[i];
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_dempty);
          __threadfence();
          named_bar_sync(2, kEpiThreads);
          if (epi_lead && lane == 0) {
            const unsigned old = atomicAdd(p.counters + j, 1u);
            *last_flag = (old == static_cast<unsigned>(c_last - c_first)) ? 1 : 0;
          }
          named_bar_sync(2, kEpiThreads);
          if (*last_flag) {
            __threadfence();
            // sum the partials in CTA order, 8 tokens at a time: the 8 loads of one
            // slot are independent, so their latencies overlap
            for (int m0 = 16 * ch_lo; m0 < 16 * ch_hi && p.m0 + m0 < p.M; m0 += 8) {
              float acc[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) acc[i] = 0.f;
              for (int c = c_first; c <= c_last; ++c) {
                const int cslot = (j == (c * p.T) / p.KU) ? 2 * c : 2 * c + 1;
                const float* src = p.slots + static_cast<long long>(cslot) * (128 * MB) + m0 * 128 + row;
                float t[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) t[i] = __ldcg(src + i * 128);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] += t[i];
              }
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int token = p.m0 + m0 + i;
                if (token < p.M)
                  p.C[static_cast<long long>(token) * p.N + n] = f32_to_f16_bits(BIAS ? acc[i] * scale + bias_n : acc[i] * scale);
              }
            }
            if (epi_lead && lane == 0) p.counters[j] = 0u;
          }
        }
      }
      ++segs;
    }
    if (seg_end) seg_units = 0;
    st += p.w_stage_bytes;
    if (++s == SW) {
      s = 0;
      ++round;
      st = sbase + p.w_base;
    }
    if (++kt == p.KU) {
      kt = 0;
      ++j;
    }
  }
  named_bar_sync(3, kTcThreads);
}

}  // namespace

TcLayout tc_layout(int mb, int ch, int srows, int a_stages, int w_stages, bool zp) {
  TcLayout l{};
  const int kq = 2 * ch;
  l.a_stage_bytes = 2 * mb * 128;  // one 128-row chunk; a multiple of 1024 keeps the swizzle atoms aligned
  l.z_off = kq * 4096 + srows * 256;  // weight stage: packed chunk, scale rows, then (with zero points) zero rows
  l.w_stage_bytes = (l.z_off + (zp ? srows * 128 : 0) + 1023) / 1024 * 1024;
  l.w_base = a_stages * l.a_stage_bytes;
  l.bar_off = l.w_base + w_stages * l.w_stage_bytes;
  l.flag_off = l.bar_off + 8 * (3 * kMaxNA + 2 * w_stages + 6);
  l.smem_bytes = 1024 + l.flag_off + 64;
  return l;
}

// instruction descriptor, kind::f16: D = F32 (bits 4..5 = 1), A = B = F16 (bits 7..12 = 0),
// both K-major (bits 15, 16 = 0), N >> 3 in bits 17..22, M >> 4 in bits 24..28
uint32_t tc_idesc(int m, int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

cudaError_t launch_gemm_tc(int smem_bytes, const CUtensorMap& tmA, const TcParams& p, cudaStream_t stream) {
  auto kern = p.zeros ? (p.bias ? gemm_tc_kernel<true, true> : gemm_tc_kernel<true, false>)
                      : (p.bias ? gemm_tc_kernel<false, true> : gemm_tc_kernel<false, false>);
  cudaFuncAttributes fa{};
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (static_cast<long long>(fa.numRegs) * kTcThreads <
      static_cast<long long>(kHelperRegs) * kHelperThreads + static_cast<long long>(kDequantRegs) * kDequantThreads)
    return cudaErrorInvalidConfiguration;  // the register split would not be covered
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  kern<<<p.grid, kTcThreads, smem_bytes, stream>>>(tmA, p);
  return cudaGetLastError();
}

}  // namespace w4a16
