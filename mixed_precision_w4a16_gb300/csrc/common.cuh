// Device-side building blocks shared by the W4A16 kernels (sm_103a).
//
// Inline PTX for: mbarrier waits with a time bound, 1-D bulk copies and 2-D
// tensor copies (TMA) into shared memory with L2 cache-policy hints, ldmatrix,
// the m16n8k16 FP16 tensor-core multiply, and the 4-bit -> FP16x2 decode.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace w4a16 {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for phase `parity` of `bar` to complete, for at most `limit` clock
// cycles.  Gives up early when `*abort` becomes non-zero (another warp timed
// out).  Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long limit,
                                                  const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > limit) return false;
  }
}

// try_wait with a suspend-time hint: the thread may sleep (up to `ns`) until
// the phase completes instead of re-polling, leaving issue slots to other warps.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return done != 0;
}

// Like mbar_wait_bounded, but the thread sleeps between polls, leaving issue
// slots to the warps that do the arithmetic.  For single-thread roles (copy
// issue, MMA issue) whose waits tolerate a little wake-up latency.
__device__ __forceinline__ bool mbar_wait_bounded_sleep(uint32_t bar, uint32_t parity, long long limit,
                                                        const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 2000u)) return true;
    if (*abort) return false;
    if (clock64() - t0 > limit) return false;
  }
}

// ---------------------------------------------------------------------------
// L2 cache policies and bulk / tensor copies into shared memory
// ---------------------------------------------------------------------------

// Warms L2 with `bytes` (a multiple of 16) from the 16-byte aligned global address `src`.  A
// prefetch cannot make a later read return stale data (device memory is kept coherent in L2), so
// a kernel may issue it before waiting for the previous kernel of the stream: the weights of its
// first work units then stream from HBM while that kernel drains.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 1-D bulk copy global -> shared, completing `bytes` on mbarrier `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// 2-D tiled tensor copy global -> shared (box given by the tensor map).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// Programmatic dependent launch.  A GEMM launched with the programmatic-serialization
// attribute may start while the previous kernel of its stream is still running: its CTAs
// set up barriers and tensor memory, then wait here until that kernel has completed and its
// writes are visible, before touching any global memory (so inputs just written by a repack or
// by the layer before stay safe).  The kernels allow their own dependents to launch at once:
// every GEMM grid is a single wave, so a dependent CTA only takes an SM that is free.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// shared-memory loads and the tensor-core multiply
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// D = A * B + C, m16n8k16, A row-major FP16, B column-major FP16, FP32 accumulate.
// A pure register operation: not volatile, so the compiler may interleave it
// with the decode arithmetic and the shared-memory loads of other blocks.
__device__ __forceinline__ void mma_16816(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1,
                                          const float c[4]) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %11, %12, %13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
        "f"(c[3]));
}

// D = A (2:4 compressed 16 x 16, f16) x B (32 x 8, f16) + C with metadata e and
// sparsity selector SEL (which pair of lanes in each quad supplies the metadata).
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

// ---------------------------------------------------------------------------
// 4-bit -> FP16x2 decode (the Marlin deep-dive article, section "INT4 只是存储
// 类型，不是这条路径的计算类型": the codes become FP16 values by placing their
// bits inside FP16 bit patterns, with no integer-to-float conversion).
//
// Construction, from the binary16 format (10 fraction bits; an exponent e
// gives the fraction's least significant bit the weight 2^(e - 10)):
//  * a code in bits 0..3 of a half: choose e = 10 (pattern 0x6400 = 1024.0,
//    lsb weight 1), so OR-ing the nibble in gives exactly 1024 + q;
//  * a code in bits 4..7 of a half: choose e = 6 (pattern 0x5400 = 64.0, lsb
//    weight 1/16), so the nibble's bit 4 weighs 16/16 = 1 and OR-ing it in gives
//    exactly 64 + q.
// One packed subtraction of the same pattern with the zero point added to the
// fraction (1024 + 8 = 0x6408, 64 + 8 = 0x5480) then leaves q - 8: both
// operands and the difference are exactly representable, so the result is
// exact.  A zero point z replaces the 8 in that constant (0x6400 | z,
// 0x5400 | z << 4).
//
// Word layout: nibble slot i (bits 4i..4i+3) for i < 4 is the low half and
// slot i + 4 the high half of operand register i.  Register i holds slots i
// and i + 4, i.e. nibble position (i & 1) of byte (i >> 1) in each half word:
// registers 0 and 2 take position 0 (bits 0..3 of the half after shifting the
// word right by 8 * (i >> 1)), registers 1 and 3 position 1 (bits 4..7).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  // truth table (a & b) | c with a = 0xF0, b = 0xCC, c = 0xAA
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}


__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Per nibble position p of a half word: the mask selecting it in both halves,
// the exponent pattern whose fraction lsb weighs 2^-4p, and how a zero point z
// sits in that pattern's fraction.
template <int P>
struct NibblePos {
  static constexpr uint32_t mask = 0x000f000fu << (4 * P);
  static constexpr uint32_t base = P == 0 ? 0x64006400u : 0x54005400u;  // 1024.0 / 64.0 in both halves
  __device__ static constexpr uint32_t offset(uint32_t z) { return ((base & 0xffffu) | (z << (4 * P))) * 0x10001u; }
};

// The codes of position P of `w` (in both halves), biased by the base: exactly
// base + q as FP16; subtracting base + z leaves q - z.
template <int P>
__device__ __forceinline__ uint32_t nibbles_minus(uint32_t w, uint32_t base_plus_z) {
  return hsub2_u32(lop3_and_or(w, NibblePos<P>::mask, NibblePos<P>::base), base_plus_z);
}

// Zero-point constants (base + z in both halves) of positions 0 and 1.
__device__ __forceinline__ uint32_t zp_const_lo(uint32_t z) { return NibblePos<0>::offset(z); }
__device__ __forceinline__ uint32_t zp_const_hi(uint32_t z) { return NibblePos<1>::offset(z); }

// One packed word -> four FP16x2 registers holding (q - z) exactly, the zero
// point given per register position by its constant (c_lo for the codes of
// rows g, registers 0 and 2; c_hi for rows g + 8, registers 1 and 3).
__device__ __forceinline__ void decode8_zp(uint32_t w, uint32_t c_lo, uint32_t c_hi, uint32_t a[4]) {
  const uint32_t w8 = w >> 8;  // byte 1 of each half moved to byte 0
  a[0] = nibbles_minus<0>(w, c_lo);
  a[1] = nibbles_minus<1>(w, c_hi);
  a[2] = nibbles_minus<0>(w8, c_lo);
  a[3] = nibbles_minus<1>(w8, c_hi);
}

// The symmetric format: zero point 8 everywhere.
__device__ __forceinline__ void decode8(uint32_t w, uint32_t a[4]) {
  decode8_zp(w, NibblePos<0>::offset(8u), NibblePos<1>::offset(8u), a);
}

// ---------------------------------------------------------------------------
// Grouped expert GEMM: the row segments of each expert
// ---------------------------------------------------------------------------

// Column of work units in a grouped expert GEMM: expert e, its row segment ci
// (rows off[e] + mb * ci ..), unit column j within the segment (a strip, or a
// strip pair).  pref[e] = row segments of the experts before e, pref[E] = all of them.
struct SegPos {
  int e, ci, j;
};

// Column jj (segment jj / cols, column jj % cols); jj < pref[E] * cols.
__device__ __forceinline__ SegPos seg_locate(const int* pref, int E, int cols, int jj) {
  const int seg = jj / cols;
  int lo = 0, hi = E;  // pref[lo] <= seg < pref[hi]; experts without rows have pref[e] == pref[e + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pref[mid] <= seg)
      lo = mid;
    else
      hi = mid;
  }
  return SegPos{lo, seg - pref[lo], jj - seg * cols};
}

// The next column (call only while one exists).
__device__ __forceinline__ void seg_next(SegPos& sp, const int* pref, int E, int cols) {
  if (++sp.j < cols) return;
  sp.j = 0;
  if (++sp.ci < pref[sp.e + 1] - pref[sp.e]) return;
  sp.ci = 0;
  do {
    ++sp.e;
  } while (sp.e < E && pref[sp.e + 1] == pref[sp.e]);
}

// Grouped-GEMM prologue, run by all NT threads of the CTA: copies the expert
// offsets to shared memory (offs[E + 1]), checks them (0 = off[0] <= ... <=
// off[E] = M) and writes the segment prefix (pref[E + 1], segments of mb rows)
// with a block-wide scan (scan[1 + NT / 32]).  Returns the number of segments, or
// -1 (kDevErrValue set in *status) when the offsets are invalid or need more
// segments than the workspace holds; the result is the same in every thread.
// The caller's next __syncthreads publishes pref.
template <int NT>
__device__ int moe_segments(const int* expert_off, int E, int M, int max_seg, int mb, uint32_t* status, int* pref,
                            int* offs, int* scan, int warp, int lane) {
  const int per = (E + NT - 1) / NT;
  const int e0 = threadIdx.x * per;
  bool bad = false;
  long long local = 0;
  for (int i = 0; i < per; ++i) {
    const int e = e0 + i;
    if (e < E) {
      const int lo = expert_off[e], hi = expert_off[e + 1];
      offs[e] = lo;
      const long long rows = static_cast<long long>(hi) - lo;
      bad |= rows < 0 || rows > M;
      if (rows > 0 && rows <= M) local += (rows + mb - 1) / mb;
    }
  }
  if (threadIdx.x == 0) {
    const int last = expert_off[E];
    offs[E] = last;
    bad |= expert_off[0] != 0 || last != M;
  }
  const int mine = static_cast<int>(min(local, static_cast<long long>(max_seg) + 1));  // no overflow below
  int incl = mine;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) scan[1 + warp] = incl;
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) {
    int run = 0;
    for (int w = 0; w < NT / 32; ++w) {
      const int v = scan[1 + w];
      scan[1 + w] = run;
      run += v;
    }
    scan[0] = run;
  }
  __syncthreads();
  const int total = scan[0];
  if (bad || total > max_seg) {
    if (threadIdx.x == 0) atomicOr(status, kDevErrValue);
    return -1;
  }
  int run = scan[1 + warp] + incl - mine;
  for (int i = 0; i < per; ++i) {
    const int e = e0 + i;
    if (e < E) {
      pref[e] = run;
      const int rows = offs[e + 1] - offs[e];
      if (rows > 0) run += (rows + mb - 1) / mb;
    }
  }
  if (threadIdx.x == 0) pref[E] = total;
  return total;
}

}  // namespace w4a16
