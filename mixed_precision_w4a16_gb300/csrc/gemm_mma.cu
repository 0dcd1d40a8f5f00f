// Streaming W4A16 GEMM for small batches (M <= 64 rows per launch).
//
// The MARLIN paper (Section 3.4, "Bound By Weight Loading") makes the point
// that for small M the kernel should be bound by reading the 4-bit weights
// once.  This kernel is built around that stream on sm_103a:
//
//  * one producer warp issues 1-D bulk copies (TMA engine) of the packed
//    weights (L2 evict-first) and 2-D tensor copies of the activation tile
//    (L2 evict-last, 128-byte swizzle) into a ring of shared-memory stages,
//    signalled by mbarriers with transaction counts;
//  * eight consumer warps decode each 32-bit word into four FP16x2 operand
//    registers (exact LOP3 + packed-FP16 decode) and feed
//    mma.sync.m16n8k16 with the weights on the 16-row side and the tokens on
//    the 8-column side (so tiny M wastes only the 8-wide slot);
//  * each group's FP32 partial product is scaled by its FP32 scale (one FMA
//    per accumulator instead of one FP16 multiply per weight);
//  * work units (n_tile output columns x 128 reduction rows) are dealt to
//    CTAs in contiguous stripes of T = ceil(units / CTAs) units running down
//    a column tile and wrapping into the next (the deep-dive article's
//    striped partitioning); column tiles split between CTAs are reduced
//    through FP32 slots with an arrival counter, the last arriver summing
//    the slots in CTA order (fixed order: deterministic, no spin waits).
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace w4a16 {

namespace {

constexpr int kConsumerWarps = 8;
constexpr long long kDrainCycles = 2000000000LL;  // bound on the final drain wait

template <int MT, int NBW>
struct Layout {
  static constexpr int MB = 8 * MT;                 // token rows per launch
  static constexpr int NT = 64 * NBW;               // output columns per unit
  static constexpr int A_BOX = MB * 128;            // one 64-column activation box (bytes)
  static constexpr int A_OFF = 0;                   // two boxes, 1024-aligned
  static constexpr int W_OFF = 2 * A_BOX;           // NT/16 runs of 1024 bytes
  static constexpr int S_OFF = W_OFF + NT * 64;     // NT fp16 scales
  static constexpr int STAGE = ((S_OFF + NT * 2) + 1023) / 1024 * 1024;
  static constexpr int TX = 2 * A_BOX + NT * 64 + NT * 2;
  static constexpr int RED = 4 * NBW * MT * 4 * 32 * 4;  // kh = 1 partials
  static constexpr int red_off(int stages) { return stages * STAGE; }
  static constexpr int bar_off(int stages) { return red_off(stages) + RED; }
  static constexpr int flag_off(int stages) { return bar_off(stages) + 16 * stages; }
  static constexpr int total(int stages) { return 1024 + flag_off(stages) + 64; }
};

__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ uint16_t f32_to_f16_bits(float x) { return __half_as_ushort(__float2half_rn(x)); }

template <int MT, int NBW>
__global__ void __launch_bounds__(kMmaThreads, 1)
    gemm_mma_kernel(const __grid_constant__ CUtensorMap tmA, const GemmParams p) {
  using L = Layout<MT, NBW>;
  constexpr int NT = L::NT;
  constexpr int MB = L::MB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int S = p.stages;
  const uint32_t bar_full = sbase + L::bar_off(S);
  const uint32_t bar_empty = bar_full + 8 * S;
  volatile int* flags = reinterpret_cast<volatile int*>(smem + L::flag_off(S));
  volatile int* abort_flag = flags + 0;  // set by any warp whose wait ran out
  volatile int* last_flag = flags + 1;   // "this CTA is the last arriver" broadcast
  volatile int* seg_abort = flags + 2;   // abort decision frozen for one epilogue
  volatile int* zero_flag = flags + 3;   // always 0 (for the drain wait)
  float* red = reinterpret_cast<float*>(smem + L::red_off(S));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const int u_begin = cta * p.T;
  const int u_end = min(p.units, u_begin + p.T);
  const int nunits = u_end - u_begin;

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
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    const int ktiles64 = p.K / 64;
    int issued = 0;
    for (int it = 0; it < nunits; ++it) {
      const int s = it % S;
      if (it >= S) {
        bool ok = true;
        if (lane == 0) ok = mbar_wait_bounded(bar_empty + 8 * s, ((it / S) - 1) & 1, p.wait_limit, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          if (lane == 0 && !*abort_flag) {
            *abort_flag = 1;
            atomicOr(p.status, kDevErrTimeout);
          }
          break;
        }
      }
      const int u = u_begin + it;
      const int j = u / p.KU;
      const int kt = u - j * p.KU;
      const uint32_t st = sbase + s * L::STAGE;
      const uint32_t fb = bar_full + 8 * s;
      if (p.debug_stall && it == 0) continue;  // leave stage 0 empty: nothing will complete its barrier
      if (lane == 0) mbar_arrive_expect_tx(fb, L::TX);
      __syncwarp();
      if (lane < NT / 16) {
        const long long nbg = static_cast<long long>(j) * (NT / 16) + lane;
        const uint32_t* src = p.packed + (nbg * ktiles64 + 2LL * kt) * 128;
        bulk_g2s(st + L::W_OFF + lane * 1024, src, 1024, fb, pol_w);
      }
      if (lane == 31) {
        tma_load_2d(st + L::A_OFF, &tmA, kt * 128, p.m0, fb, pol_a);
        tma_load_2d(st + L::A_OFF + L::A_BOX, &tmA, kt * 128 + 64, p.m0, fb, pol_a);
      }
      if (lane == 30) {
        const int grp = (kt * 128) / p.G;
        const uint16_t* src = p.scales + static_cast<long long>(grp) * p.N + static_cast<long long>(j) * NT;
        bulk_g2s(st + L::S_OFF, src, NT * 2, fb, pol_a);
      }
      issued = it + 1;
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
  const int kh = warp & 1;   // which 64-row half of the 128-row unit
  const int ng = warp >> 1;  // which group of NBW 16-column blocks
  const int g = lane >> 2, t = lane & 3;
  const int first_col = u_begin / p.KU;

  float acc[NBW][MT][4];
#pragma unroll
  for (int i = 0; i < NBW; ++i)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][mt][e] = 0.f;
  const float zero4[4] = {0.f, 0.f, 0.f, 0.f};

  for (int it = 0; it < nunits; ++it) {
    const int s = it % S;
    const int u = u_begin + it;
    const uint32_t st = sbase + s * L::STAGE;
    bool have = false;
    const bool go = __shfl_sync(0xffffffffu, *abort_flag == 0, 0);
    if (go) {
      have = mbar_wait_bounded(bar_full + 8 * s, (it / S) & 1, p.wait_limit, abort_flag);
      have = __all_sync(0xffffffffu, have);
      if (!have && lane == 0 && !*abort_flag) {
        *abort_flag = 1;
        atomicOr(p.status, kDevErrTimeout);
      }
    }
    if (have) {
      // activation fragments of this warp's 64-row half: 4 k16 steps x MT token tiles
      const uint32_t a_box = st + L::A_OFF + kh * L::A_BOX;
      uint32_t bf[4][MT][2];
      const int mi = lane >> 3, rr = lane & 7;
      if constexpr (MT == 1) {
#pragma unroll
        for (int jj = 0; jj < 4; jj += 2) {
          const int chunk = 2 * jj + mi;
          ldmatrix_x4(a_box + rr * 128 + ((chunk ^ rr) << 4), bf[jj][0][0], bf[jj][0][1], bf[jj + 1][0][0],
                      bf[jj + 1][0][1]);
        }
      } else {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
          for (int mp = 0; mp < MT / 2; ++mp) {
            const int token = (2 * mp + (mi >> 1)) * 8 + rr;
            const int chunk = 2 * jj + (mi & 1);
            ldmatrix_x4(a_box + token * 128 + ((chunk ^ rr) << 4), bf[jj][2 * mp][0], bf[jj][2 * mp][1],
                        bf[jj][2 * mp + 1][0], bf[jj][2 * mp + 1][1]);
          }
      }
#pragma unroll
      for (int i = 0; i < NBW; ++i) {
        const int lnb = ng * NBW + i;
        const uint4 wv = lds128(st + L::W_OFF + lnb * 1024 + kh * 512 + lane * 16);
        const uint32_t sp = lds32(st + L::S_OFF + (lnb * 16 + 2 * g) * 2);
        const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
        float tmp[MT][4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          uint32_t a[4];
          decode8(words[jj], a);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) mma_16816(tmp[mt], a, bf[jj][mt][0], bf[jj][mt][1], jj == 0 ? zero4 : tmp[mt]);
        }
        const float s_lo = __half2float(__ushort_as_half(static_cast<uint16_t>(sp & 0xffffu)));
        const float s_hi = __half2float(__ushort_as_half(static_cast<uint16_t>(sp >> 16)));
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          acc[i][mt][0] = fmaf(s_lo, tmp[mt][0], acc[i][mt][0]);
          acc[i][mt][1] = fmaf(s_lo, tmp[mt][1], acc[i][mt][1]);
          acc[i][mt][2] = fmaf(s_hi, tmp[mt][2], acc[i][mt][2]);
          acc[i][mt][3] = fmaf(s_hi, tmp[mt][3], acc[i][mt][3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }

    // ---------------------------------------------------------- segment epilogue
    const bool seg_end = ((u + 1) % p.KU == 0) || (it == nunits - 1);
    if (!seg_end) continue;
    const int j = u / p.KU;
    // 1) fold the two 64-row halves together (kh = 1 -> shared memory -> kh = 0)
    if (kh == 1) {
#pragma unroll
      for (int i = 0; i < NBW; ++i)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) red[(((ng * NBW + i) * MT + mt) * 4 + e) * 32 + lane] = acc[i][mt][e];
    }
    named_bar_sync(1, kConsumerWarps * 32);
    if (warp == 0 && lane == 0) *seg_abort = *abort_flag;
    if (kh == 0) {
#pragma unroll
      for (int i = 0; i < NBW; ++i)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[i][mt][e] += red[(((ng * NBW + i) * MT + mt) * 4 + e) * 32 + lane];
    }
    named_bar_sync(1, kConsumerWarps * 32);
    const bool skip = *seg_abort != 0;
    if (kh == 0 && !skip) {
      const int c_first = (j * p.KU) / p.T;
      const int c_last = min(((j + 1) * p.KU - 1) / p.T, p.grid - 1);
      bool write_now = true;
      if (c_first != c_last) {
        // 2) this column tile is split between CTAs: publish the partial, count arrivals
        const int slot = (j == first_col) ? 2 * cta : 2 * cta + 1;
        float* dst = p.slots + static_cast<long long>(slot) * (NT * MB);
#pragma unroll
        for (int i = 0; i < NBW; ++i)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[(((ng * NBW + i) * MT + mt) * 4 + e) * 32 + lane] = acc[i][mt][e];
        __threadfence();
        named_bar_sync(2, 4 * 32);
        if (warp == 0 && lane == 0) {
          const unsigned old = atomicAdd(p.counters + j, 1u);
          *last_flag = (old == static_cast<unsigned>(c_last - c_first)) ? 1 : 0;
        }
        named_bar_sync(2, 4 * 32);
        write_now = *last_flag != 0;
        if (write_now) {
          // 3) last arriver: sum every CTA's slot in CTA order (deterministic)
          __threadfence();
#pragma unroll
          for (int i = 0; i < NBW; ++i)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[i][mt][e] = 0.f;
          for (int c = c_first; c <= c_last; ++c) {
            const int cslot = (j == (c * p.T) / p.KU) ? 2 * c : 2 * c + 1;
            const float* src = p.slots + static_cast<long long>(cslot) * (NT * MB);
#pragma unroll
            for (int i = 0; i < NBW; ++i)
#pragma unroll
              for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  acc[i][mt][e] += __ldcg(src + (((ng * NBW + i) * MT + mt) * 4 + e) * 32 + lane);
          }
          if (warp == 0 && lane == 0) p.counters[j] = 0u;
        }
      }
      if (write_now) {
#pragma unroll
        for (int i = 0; i < NBW; ++i) {
          const int n_base = j * NT + (ng * NBW + i) * 16 + g;
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
    for (int i = 0; i < NBW; ++i)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][mt][e] = 0.f;
  }
  named_bar_sync(3, kMmaThreads);
}

template <int MT, int NBW>
cudaError_t launch_one(const MmaConfig& cfg, const CUtensorMap& tmA, const GemmParams& p, cudaStream_t stream) {
  auto kern = gemm_mma_kernel<MT, NBW>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, cfg.smem_bytes);
  if (e != cudaSuccess) return e;
  kern<<<p.grid, kMmaThreads, cfg.smem_bytes, stream>>>(tmA, p);
  return cudaGetLastError();
}

// Instantiated configurations (registers: 9 warps leave at most 168 per thread,
// so wider token tiles get fewer column blocks per warp).
template <int MT>
cudaError_t launch_mt(const MmaConfig& cfg, const CUtensorMap& tmA, const GemmParams& p, cudaStream_t stream) {
  switch (cfg.nbw) {
    case 1: return launch_one<MT, 1>(cfg, tmA, p, stream);
    case 2:
      if constexpr (MT <= 4) return launch_one<MT, 2>(cfg, tmA, p, stream);
      return cudaErrorInvalidValue;
    case 4:
      if constexpr (MT <= 2) return launch_one<MT, 4>(cfg, tmA, p, stream);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

template <int MT, int NBW>
constexpr int stage_bytes_of() { return Layout<MT, NBW>::STAGE; }

}  // namespace

int mma_stage_bytes(int m_tiles, int nbw) {
  const int MB = 8 * m_tiles, NT = 64 * nbw;
  const int s_off = 2 * MB * 128 + NT * 64;
  return (s_off + NT * 2 + 1023) / 1024 * 1024;
}

int mma_smem_bytes(int m_tiles, int nbw, int stages) {
  const int red = 4 * nbw * m_tiles * 4 * 32 * 4;
  return 1024 + stages * mma_stage_bytes(m_tiles, nbw) + red + 16 * stages + 64;
}

static_assert(stage_bytes_of<2, 4>() == 21504, "stage layout");

cudaError_t launch_gemm_mma(const MmaConfig& cfg, const CUtensorMap& tmA, const GemmParams& p, cudaStream_t stream) {
  switch (cfg.m_tiles) {
    case 1: return launch_mt<1>(cfg, tmA, p, stream);
    case 2: return launch_mt<2>(cfg, tmA, p, stream);
    case 4: return launch_mt<4>(cfg, tmA, p, stream);
    case 8: return launch_mt<8>(cfg, tmA, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace w4a16
