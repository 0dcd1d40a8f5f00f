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

#include <algorithm>

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

// Both tile walkers below are persistent: CTA c takes the tiles [c*T, (c+1)*T) of the packed
// stream's order (strip by strip, 64-row blocks down each strip), so its output is one
// contiguous range and consecutive tiles of a strip share their scale group.  A tile is 64 rows
// x 128 columns (one strip, one 64-row block); its 256 output vectors (16 bytes, one per
// thread: warp b = 16-column block, lane = fragment lane) are consecutive in the packed stream.
// Tiles are copied into a ring of three shared buffers (cp.async, 16 bytes per copy), two tiles
// ahead of the one being packed; one block barrier per tile both publishes the tile's copies and
// frees the buffer the next copy overwrites (the one packed in the previous iteration).
constexpr int kTileThreads = 256;
constexpr int kTileCtasPerSm = 4;
constexpr int kTileStages = 3;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most kTileStages - 2 committed groups (the tiles after this one) are in flight
__device__ __forceinline__ void cp_async_wait_tile() {
  asm volatile("cp.async.wait_group %0;" ::"n"(kTileStages - 2) : "memory");
}

struct TileRange {
  long long t0, t1;
};
__device__ __forceinline__ TileRange tile_range(int T, long long tiles) {
  const long long t0 = static_cast<long long>(blockIdx.x) * T;
  return {t0, t0 + T < tiles ? t0 + T : tiles};
}

// (strip, 64-row block) of a tile, stepped along the CTA's range without dividing per tile
struct TilePos {
  int strip;
  int kb;
  __device__ __forceinline__ TilePos next(int kTiles) const {
    return kb + 1 == kTiles ? TilePos{strip + 1, 0} : TilePos{strip, kb + 1};
  }
};

// The copy side of the ring: issue(pos, stage) copies one tile; every call commits exactly one
// group (empty past the range's end), so the group count per iteration stays uniform.
template <class Issue>
struct TileFeed {
  Issue issue;
  TilePos pos;      // next tile to copy
  long long left;   // tiles of the range not yet copied
  int kTiles;
  __device__ __forceinline__ void push(int stage) {
    if (left > 0) {
      issue(pos, stage);
      pos = pos.next(kTiles);
      --left;
    }
    cp_async_commit();
  }
};

// Codes: a tile is 64 rows of 128 bytes in shared memory.  In one load instruction the lanes of
// a warp read rows 4t + c (t = 0..3, c fixed) at the same 16-byte chunk b, so chunk b of row k is
// stored at chunk b ^ ((k >> 2) & 3): the four rows then sit in four different bank groups.
__device__ __forceinline__ int code_chunk(int k, int chunk) { return chunk ^ ((k >> 2) & 3); }

__global__ void __launch_bounds__(kTileThreads, kTileCtasPerSm)
    repack_codes_kernel(const uint8_t* __restrict__ q, int K, int N, int T, long long tiles,
                        uint4* __restrict__ packed) {
  __shared__ __align__(16) uint8_t buf[kTileStages][64][128];
  const TileRange tr = tile_range(T, tiles);
  if (tr.t0 >= tr.t1) return;
  const int kTiles = K / 64;
  const int tid = threadIdx.x;
  auto issue = [&](TilePos tp, int stage) {
    const uint8_t* src = q + tp.kb * 64LL * N + tp.strip * 128;
#pragma unroll
    for (int i = 0; i < 2; ++i) {  // 64 rows x 8 chunks
      const int c = tid + kTileThreads * i, r = c >> 3, ch = c & 7;
      cp_async16(smem_u32(&buf[stage][r][16 * code_chunk(r, ch)]), src + static_cast<long long>(r) * N + 16 * ch);
    }
  };
  TileFeed<decltype(issue)> feed{issue, {static_cast<int>(tr.t0 / kTiles), static_cast<int>(tr.t0 % kTiles)},
                                 tr.t1 - tr.t0, kTiles};
  for (int st = 0; st < kTileStages - 1; ++st) feed.push(st);
  const int b = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  uint32_t seen = 0;  // OR of every code read: a code above 15 sets a bit above the nibble
  int stage = 0;
  for (long long tile = tr.t0; tile < tr.t1; ++tile) {
    cp_async_wait_tile();
    __syncthreads();
    feed.push(stage == 0 ? kTileStages - 1 : stage - 1);
    uint32_t words[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // nibble slots 7 .. 0, most significant first; a code above 15 is masked to its nibble
      uint32_t w = 0;
#pragma unroll
      for (int slot_i = 7; slot_i >= 0; --slot_i) {
        int r, c;
        slot_rc(slot_i, g, t, r, c);
        const int k = 16 * j + c;
        const uint32_t code = buf[stage][k][16 * code_chunk(k, b) + r];
        seen |= code;
        w = (w << 4) | (code & 15u);
      }
      words[j] = w;
    }
    packed[tile * kTileThreads + tid] = make_uint4(words[0], words[1], words[2], words[3]);
    stage = stage + 1 == kTileStages ? 0 : stage + 1;
  }
  if (seen > 15u) atomicOr(&g_repack_flag, kDevErrCodeRange);
}

// FP16 weights: a tile is 64 rows of 128 halves, each shared row padded to 136 halves (272
// bytes, 17 16-byte chunks).  The packing reads it with transposed 8x8 matrix loads: matrix m of
// 16-row block j holds rows 16j + 4i' + 2(m >> 1) + {0, 1} (i' = 0..3) of columns 16b + 8(m & 1)
// + 0..7, which hands lane (g, t) exactly its register m (reduction rows 4t + 2(m >> 1) + {0, 1}
// of column g + 8(m & 1)).  Rows k and k + 8 would share a bank group, so rows with bit 3 set swap
// row pairs (k ^ 2): the eight rows of one matrix then fall into eight different groups.
constexpr int kHalfRow = 136;
// one stage: the tile, then the 128 scales and 128 zero codes of its group row
constexpr int kQuantTileBytes = 64 * kHalfRow * 2;
constexpr int kQuantStageBytes = kQuantTileBytes + 128 * 2 + 128;
constexpr int kQuantSmem = kTileStages * kQuantStageBytes;
__device__ __forceinline__ int half_row(int k) { return k ^ (((k >> 3) & 1) << 1); }

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t d[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
               : "r"(addr));
}

// Per column (and scale group) constants of the quantiser's fast path.
struct QuantCol {
  float s;       // the scale
  float lo;      // -offset: the smallest rint(w / s) that still stores as code 0 or above
  float hi;      // 15 - offset
  float off;     // the offset: 8, or the zero code
  uint64_t y2;   // RN(1 / s), twice (a float pair)
  uint64_t ns2;  // -s, twice
  bool bad;      // s is zero, infinite or NaN: the fast path does not apply to the column
};
__device__ __forceinline__ uint64_t f32_pair(float x) {
  return (static_cast<uint64_t>(__float_as_uint(x)) << 32) | __float_as_uint(x);
}
__device__ __forceinline__ QuantCol quant_col(uint16_t s_bits, float off) {
  QuantCol c;
  c.s = __half2float(__ushort_as_half(s_bits));
  c.off = off;
  c.lo = -c.off;
  c.hi = 15.0f - c.off;
  c.y2 = f32_pair(__frcp_rn(c.s));
  c.ns2 = f32_pair(-c.s);
  c.bad = (c.s == 0.0f) || !isfinite(c.s);
  return c;
}

// Both FP16 halves of a fragment register (the same column, reduction rows k and k + 1): their
// float32 quotients by the column's scale (packed pairs: q0 = RN(w y), r = fma(q0, -s, w),
// q1 = fma(r, y, q0)), clamped to [lo, hi], plus 1.5 * 2^23 (packed); returns the two sums' bits.
// nan_acc = fma(halves, 0, nan_acc) stays zero unless a half is infinite or NaN.
__device__ __forceinline__ void quant_pair(uint32_t d, const QuantCol& c, uint32_t& v_lo, uint32_t& v_hi,
                                           uint32_t& nan_acc) {
  asm("{\n"
      "  .reg .b16 h0, h1;\n"
      "  .reg .f32 w0, w1, a0, a1;\n"
      "  .reg .b64 w2, q0, r2, q1, m2;\n"
      "  .reg .b32 zero;\n"
      "  mov.b32 zero, 0;\n"
      "  mov.b32 {h0, h1}, %3;\n"
      "  cvt.f32.f16 w0, h0;\n"
      "  cvt.f32.f16 w1, h1;\n"
      "  fma.rn.f16x2 %2, %3, zero, %2;\n"
      "  mov.b64 w2, {w0, w1};\n"
      "  mul.rn.f32x2 q0, w2, %4;\n"
      "  fma.rn.f32x2 r2, q0, %5, w2;\n"
      "  fma.rn.f32x2 q1, r2, %4, q0;\n"
      "  mov.b64 {a0, a1}, q1;\n"
      "  max.f32 a0, a0, %6;\n"
      "  max.f32 a1, a1, %6;\n"
      "  min.f32 a0, a0, %7;\n"
      "  min.f32 a1, a1, %7;\n"
      "  mov.b64 q1, {a0, a1};\n"
      "  add.rn.f32x2 m2, q1, %8;\n"
      "  mov.b64 {%0, %1}, m2;\n"
      "}\n"
      : "=r"(v_lo), "=r"(v_hi), "+r"(nan_acc)
      : "r"(d), "l"(c.y2), "l"(c.ns2), "f"(c.lo), "f"(c.hi), "l"(0x4B4000004B400000ull));
}

// The reference rule for one weight: the IEEE float32 quotient, rounded half to even, plus the
// offset, clamped; a non-finite quotient gives code 8 and flags the call.
__device__ __forceinline__ uint32_t quant_exact(float wf, const QuantCol& c, bool& bad) {
  const float quot = __fdiv_rn(wf, c.s);
  if (!isfinite(quot)) {
    bad = true;
    return 8u;
  }
  return static_cast<uint32_t>(fminf(fmaxf(rintf(quot) + c.off, 0.0f), 15.0f));
}

__device__ __forceinline__ float half_of(const uint32_t d[4], int si) {
  const int m = si & 3;
  return __half2float(__ushort_as_half(static_cast<uint16_t>(si >= 4 ? d[m] >> 16 : d[m] & 0xffffu)));
}

// Quantise FP16 weights with their FP16 scales straight into the packed layout (the original
// Layer.pack step, deep-dive article section "可复现的调用链"): q = clamp(rint(w / s) + 8, 0, 15)
// (or + z), the quotient an IEEE float32 division, rint rounding half to even.
//
// The quotient is formed without a division: with y = RN(1/s), q0 = RN(w y), the residual
// r = fma(-q0, s, w) (exact) and q1 = fma(r, y, q0).  For FP16 operands q1 equals the correctly
// rounded float32 quotient RN(w/s): this one-step correction (Markstein's) holds whenever no
// intermediate under- or overflows, true for every FP16 pair (|w/s| lies in [2^-40, 2^40]), and
// an exhaustive check over all pairs of FP16 significands at several exponent offsets found no
// exception.  Clamping q1 to [-offset, 15 - offset] commutes with rounding to an integer (the
// bounds are integers), and adding 1.5 * 2^23 rounds it half to even into the low mantissa bits;
// the eight slots are summed into the word with their offsets added back.  Both halves of a
// fragment register share their column, so the quotient and the rounding run on float pairs.
// An infinite or NaN weight is caught by fma(w, 0, acc) accumulated over the thread's tile; its
// words, and the columns whose scale is zero, infinite or NaN, are recomputed with the
// reference rule slot by slot.
// z: zero codes uint8[K/G][N] row-major, or null for the symmetric offset 8.
__global__ void __launch_bounds__(kTileThreads, kTileCtasPerSm)
    quantize_codes_kernel(const uint16_t* __restrict__ w, const uint16_t* __restrict__ s,
                          const uint8_t* __restrict__ z, int K, int N, int G, int T, long long tiles,
                          uint4* __restrict__ packed) {
  extern __shared__ __align__(16) uint8_t qbuf[];  // kTileStages x (tile, scales, zero codes)
  const TileRange tr = tile_range(T, tiles);
  if (tr.t0 >= tr.t1) return;
  const int kTiles = K / 64;
  const int tid = threadIdx.x;
  const uint32_t qbase = smem_u32(qbuf);
  auto row_addr = [&](int stage, int row) {
    return qbase + static_cast<uint32_t>(stage * kQuantStageBytes + row * kHalfRow * 2);
  };
  auto issue = [&](TilePos tp, int stage) {
    const uint16_t* src = w + tp.kb * 64LL * N + tp.strip * 128LL;
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // 64 rows x 16 chunks
      const int c = tid + kTileThreads * i, r = c >> 4, ch = c & 15;
      cp_async16(row_addr(stage, half_row(r)) + 16 * ch, src + static_cast<long long>(r) * N + 8 * ch);
    }
    // the group row's 128 scales (16 chunks) and zero codes (8 chunks)
    const long long gi = static_cast<long long>(G == 128 ? tp.kb >> 1 : 0) * N + tp.strip * 128LL;
    const uint32_t sdst = qbase + static_cast<uint32_t>(stage * kQuantStageBytes + kQuantTileBytes);
    if (tid < 16)
      cp_async16(sdst + 16 * tid, s + gi + 8 * tid);
    else if (z && tid < 24)
      cp_async16(sdst + 256 + 16 * (tid - 16), z + gi + 16 * (tid - 16));
  };
  TilePos pos{static_cast<int>(tr.t0 / kTiles), static_cast<int>(tr.t0 % kTiles)};
  TileFeed<decltype(issue)> feed{issue, pos, tr.t1 - tr.t0, kTiles};
  for (int st = 0; st < kTileStages - 1; ++st) feed.push(st);
  const int b = tid >> 5, lane = tid & 31;
  const int g = lane >> 2;
  // this lane's row and column in the transposed matrix loads
  const int mi = lane >> 3, ri = lane & 7;
  const int ld_row = 4 * (ri >> 1) + 2 * (mi >> 1) + (ri & 1);
  const int ld_col = 16 * b + 8 * (mi & 1);
  constexpr uint32_t kMagicBits = 0x4B400000u;              // bits of 1.5 * 2^23
  constexpr uint32_t kMagicSum = kMagicBits * 0x11111111u;  // its sum over the eight nibble slots
  bool bad = false;
  QuantCol col[2];
  uint32_t word_add = 0;  // per word: the offsets of the eight slots minus the magic constants
  int kb = pos.kb;
  bool first = true;
  int stage = 0;
  for (long long tile = tr.t0; tile < tr.t1; ++tile) {
    cp_async_wait_tile();
    __syncthreads();
    feed.push(stage == 0 ? kTileStages - 1 : stage - 1);
    // a new scale group starts at every strip's first tile and, for G = 128, every even block
    if (first || (G == 128 ? (kb & 1) == 0 : kb == 0)) {  // uniform over the CTA
      first = false;
      const uint8_t* sg = qbuf + stage * kQuantStageBytes + kQuantTileBytes;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int n = 16 * b + 8 * h + g;
        col[h] = quant_col(reinterpret_cast<const uint16_t*>(sg)[n], z ? static_cast<float>(sg[256 + n]) : 8.0f);
      }
      // even slots belong to column g, odd slots to column g + 8
      word_add = static_cast<uint32_t>(col[0].off) * 0x01010101u + static_cast<uint32_t>(col[1].off) * 0x10101010u -
                 kMagicSum;
    }
    kb = kb + 1 == kTiles ? 0 : kb + 1;
    uint32_t words[4];
    uint32_t need = (col[0].bad || col[1].bad) ? 15u : 0u;  // bit j: word j takes the reference rule
    uint32_t nan_acc = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t d[4];
      ldmatrix_x4_trans(row_addr(stage, half_row(16 * j + ld_row)) + 2 * ld_col, d);
      // slot m + 4e holds half e of register m (column half m & 1): slots 0-3 in the low and
      // slots 4-7 in the high half of the word
      uint32_t acc_lo = 0, acc_hi = 0;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        uint32_t v_lo, v_hi;
        quant_pair(d[m], col[m & 1], v_lo, v_hi, nan_acc);
        acc_lo += v_lo << (4 * m);
        acc_hi += v_hi << (4 * m);
      }
      words[j] = acc_lo + (acc_hi << 16) + word_add;
    }
    if (nan_acc & 0x7fff7fffu) need = 15u;  // an infinite or NaN weight in this thread's tile
    if (__any_sync(0xffffffffu, need != 0)) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (__any_sync(0xffffffffu, (need >> j) & 1u)) {  // warp-uniform: the matrix load is collective
          uint32_t d[4];
          ldmatrix_x4_trans(row_addr(stage, half_row(16 * j + ld_row)) + 2 * ld_col, d);
          if ((need >> j) & 1u) {
            uint32_t word = 0;
#pragma unroll
            for (int si = 7; si >= 0; --si) word = (word << 4) | quant_exact(half_of(d, si), col[si & 1], bad);
            words[j] = word;
          }
        }
      }
    }
    packed[tile * kTileThreads + tid] = make_uint4(words[0], words[1], words[2], words[3]);
    stage = stage + 1 == kTileStages ? 0 : stage + 1;
  }
  if (bad) atomicOr(&g_repack_flag, kDevErrValue);
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

// One thread per 16-column block of one scale row: permuted position p of the block holds natural
// column perm_row(p), i.e. positions 2k and 2k + 1 hold columns k and k + 8, so the 16 permuted
// scales are the two natural 8-column halves interleaved.  Both sides are 32 contiguous bytes
// (two 16-byte loads and stores).  Forward (inverse = 0): s natural -> sp permuted; inverse = 1:
// s permuted -> sp natural.
__global__ void permute_scales_kernel(const uint16_t* __restrict__ s, uint16_t* __restrict__ sp, int N, int NG,
                                      long long nblocks, int inverse) {
  const long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (i >= nblocks) return;
  const int per_strip = NG * 8;
  const long long strip = i / per_strip;
  const int r = static_cast<int>(i - strip * per_strip);
  const int g = r >> 3, blk = r & 7;
  const long long nat = static_cast<long long>(g) * N + strip * 128 + blk * 16;  // natural: row g, 16 columns
  const long long per = (strip * NG + g) * 128 + blk * 16;                      // permuted: 16 positions
  const uint4* src = reinterpret_cast<const uint4*>(s + (inverse ? per : nat));
  uint4* dst = reinterpret_cast<uint4*>(sp + (inverse ? nat : per));
  const uint4 x0 = src[0], x1 = src[1];
  const uint32_t a[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
  uint32_t o[8];
  if (!inverse) {
    // permuted word m = (column m, column m + 8): low or high halves of natural words m/2, 4 + m/2
#pragma unroll
    for (int m = 0; m < 8; ++m) o[m] = __byte_perm(a[m >> 1], a[4 + (m >> 1)], (m & 1) ? 0x7632 : 0x5410);
  } else {
    // natural word k of the first half = low halves of permuted words 2k, 2k + 1; of the second
    // half, their high halves
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      o[k] = __byte_perm(a[2 * k], a[2 * k + 1], 0x5410);
      o[4 + k] = __byte_perm(a[2 * k], a[2 * k + 1], 0x7632);
    }
  }
  dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
  dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
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

// Zero codes uint8[K/G][N] -> the scales' permuted order (uint8[N/128][K/G][128]), one thread per
// 16-column block of one row: permuted bytes 2k and 2k + 1 hold columns k and k + 8 (one 16-byte
// load and store, byte permutes for the interleave).  Codes above 15 are masked to 4 bits and flag.
__global__ void permute_zeros_kernel(const uint8_t* __restrict__ z, uint8_t* __restrict__ zp, int N, int NG,
                                     long long nblocks) {
  const long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (i >= nblocks) return;
  const int per_strip = NG * 8;
  const long long strip = i / per_strip;
  const int r = static_cast<int>(i - strip * per_strip);
  const int g = r >> 3, blk = r & 7;
  const uint4 x = *reinterpret_cast<const uint4*>(z + static_cast<long long>(g) * N + strip * 128 + blk * 16);
  if ((x.x | x.y | x.z | x.w) & 0xF0F0F0F0u) atomicOr(&g_repack_flag, kDevErrCodeRange);
  const uint32_t w0 = x.x & 0x0F0F0F0Fu, w1 = x.y & 0x0F0F0F0Fu, w2 = x.z & 0x0F0F0F0Fu, w3 = x.w & 0x0F0F0F0Fu;
  *reinterpret_cast<uint4*>(zp + (strip * NG + g) * 128 + blk * 16) =
      make_uint4(__byte_perm(w0, w2, 0x5140), __byte_perm(w0, w2, 0x7362), __byte_perm(w1, w3, 0x5140),
                 __byte_perm(w1, w3, 0x7362));
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

// T tiles per CTA, for kTileCtasPerSm CTAs on every SM
inline int tiles_per_cta(long long tiles, int sms) {
  const long long ctas = static_cast<long long>(std::max(sms, 1)) * kTileCtasPerSm;
  return static_cast<int>((tiles + ctas - 1) / ctas);
}

cudaError_t launch_repack(const uint8_t* q, const uint16_t* s, int K, int N, int G, uint32_t* packed,
                          uint16_t* scales_p, int sms, cudaStream_t stream) {
  const long long tiles = static_cast<long long>(N / 128) * (K / 64);
  const int T = tiles_per_cta(tiles, sms);
  repack_codes_kernel<<<grid_for(tiles, T), kTileThreads, 0, stream>>>(q, K, N, T, tiles,
                                                                       reinterpret_cast<uint4*>(packed));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long ns = static_cast<long long>(K / G) * N;
  permute_scales_kernel<<<grid_for(ns / 16, 256), 256, 0, stream>>>(s, scales_p, N, K / G, ns / 16, 0);
  return cudaGetLastError();
}

cudaError_t launch_quantize_repack(const uint16_t* w, const uint16_t* s, const uint8_t* z, int K, int N, int G,
                                   uint32_t* packed, uint16_t* scales_p, int sms, cudaStream_t stream) {
  const long long tiles = static_cast<long long>(N / 128) * (K / 64);
  const int T = tiles_per_cta(tiles, sms);
  cudaError_t e = cudaFuncSetAttribute(quantize_codes_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQuantSmem);
  if (e != cudaSuccess) return e;
  quantize_codes_kernel<<<grid_for(tiles, T), kTileThreads, kQuantSmem, stream>>>(
      w, s, z, K, N, G, T, tiles, reinterpret_cast<uint4*>(packed));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long ns = static_cast<long long>(K / G) * N;
  permute_scales_kernel<<<grid_for(ns / 16, 256), 256, 0, stream>>>(s, scales_p, N, K / G, ns / 16, 0);
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
  permute_scales_kernel<<<grid_for(ns / 16, 256), 256, 0, stream>>>(s, scales_p, N, K / G, ns / 16, 0);
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
  permute_scales_kernel<<<grid_for(ns / 16, 256), 256, 0, stream>>>(scales_p, s, N, K / G, ns / 16, 1);
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
  const long long nblocks = static_cast<long long>(K / G) * N / 16;
  permute_zeros_kernel<<<grid_for(nblocks, 256), 256, 0, stream>>>(z, zeros_p, N, K / G, nblocks);
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
