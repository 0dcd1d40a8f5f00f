/*
 * w4a16.h -- C ABI of the GB300 (sm_103a) W4A16 linear-layer library.
 *
 * The operation ("MARLIN: Mixed-Precision Auto-Regressive Parallel Inference
 * on Large Language Models", Section 3.4 "Kernel Design"; the Marlin
 * deep-dive article "Marlin 完全拆解", section "Marlin 要解决的精确问题"):
 *
 *     C[M x N] = A[M x K] * B^[K x N],   B^[k, n] = s[floor(k / G), n] * (q[k, n] - 8)
 *
 * A and C are IEEE binary16 (FP16), q are 4-bit codes 0..15 (symmetric, zero
 * point 8), s are FP16 scales, one per G consecutive rows of each column
 * (G = 128) or one per column (G = K, also spelt -1).
 *
 * Conventions shared by every entry point:
 *  - FP16 data are passed as uint16_t bit patterns.
 *  - All buffers are caller-owned; the library never allocates device memory.
 *    Device pointers must be 16-byte aligned.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Kernel launches are asynchronous on that stream; only the size
 *    queries, w4a16_plan and w4a16_get_status are synchronous.
 *  - Every call validates its arguments on the host first and returns a
 *    w4a16_status; nothing is launched when validation fails.  The device
 *    never traps: errors found on the device (a code above 15, a pipeline
 *    wait that ran out of time) are recorded in a status word and returned
 *    by w4a16_get_status.
 *  - The library is built for sm_103a only and returns W4A16_ERR_ARCH on any
 *    other device.  There is no CPU fallback.
 *
 * Shapes: K % 128 == 0, N % 128 == 0, groupsize in {128, K, -1}, M >= 0.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define W4A16_API __attribute__((visibility("default")))
#else
#define W4A16_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  W4A16_OK = 0,
  W4A16_ERR_NULL = 1,        /* a required pointer is NULL */
  W4A16_ERR_SHAPE = 2,       /* K, N or M outside the supported shapes */
  W4A16_ERR_GROUP = 3,       /* groupsize not in {128, K, -1} */
  W4A16_ERR_CODE_RANGE = 4,  /* repack saw a code above 15 (device-detected) */
  W4A16_ERR_WORKSPACE = 5,   /* workspace missing or smaller than w4a16_workspace_bytes */
  W4A16_ERR_CUDA = 6,        /* a CUDA runtime call or launch failed */
  W4A16_ERR_TIMEOUT = 7,     /* a pipeline wait ran out of time (device-detected) */
  W4A16_ERR_ARCH = 8,        /* current device is not compute capability 10.3 */
  W4A16_ERR_ALIGN = 9,       /* a device pointer is not 16-byte aligned */
  W4A16_ERR_VALUE = 10       /* quantisation saw a non-finite w / s (zero, NaN or infinite input; device-detected) */
} w4a16_status;

/* Human-readable name of a status code (static string, never NULL). */
W4A16_API const char* w4a16_status_string(int status);

/* Version of this ABI (incremented on any incompatible change). */
W4A16_API int w4a16_abi_version(void);

/* ---------------------------------------------------------------------------
 * Size queries (host only, pure functions; 0 on invalid shapes).
 * ------------------------------------------------------------------------- */

/* Bytes of the packed weight stream: K * N / 2 (4 bits per weight). */
W4A16_API size_t w4a16_packed_bytes(int K, int N);

/* Number of FP16 scales: (K / G) * N, G = K for groupsize K or -1. */
W4A16_API size_t w4a16_scales_count(int K, int N, int groupsize);

/* Bytes of workspace w4a16_gemm needs for this shape on the current device.
 * Layout: a status word, one arrival counter per output column tile, and
 * FP32 partial-sum slots for column tiles whose K range is split between
 * CTAs.  The caller zeroes it once (cudaMemsetAsync) before first use; every
 * successful call leaves the counters at zero, so it can be reused on the
 * same stream without re-zeroing.  After a call reports W4A16_ERR_TIMEOUT the
 * caller must zero it again.  One workspace per concurrently running stream. */
W4A16_API size_t w4a16_workspace_bytes(int M, int K, int N, int groupsize);

/* ---------------------------------------------------------------------------
 * Offline repack (the pages: MARLIN paper Section 3.4 "Maximizing Loading
 * Bandwidth" -- 16x64 tiles stored contiguously, one 16-byte vector per thread
 * carrying the codes of four 16x16 tensor-core blocks; deep-dive article
 * sections "直接生成 MMA 所需的寄存器 fragment" and "全局内存布局").
 *
 *   q        device, uint8[K][N] row-major, codes 0..15
 *   s        device, fp16[K/G][N] row-major scales
 *   packed   device, uint32[K*N/8] output, layout below
 *   scales_p device, fp16[(K/G)*N] output, layout below
 *
 * Packed layout (this library's own ABI): uint32[N/128][K/64][8][32][4].
 * Output columns are cut into 128-column strips, each stored contiguously
 * along K, so a kernel work unit (a strip x a run of 64-row blocks) is one
 * contiguous copy.  Code q[k][n] sits in word
 *   (((n/128 * K/64 + k/64) * 8 + (n%128)/16) * 32 + lane) * 4 + (k%64)/16
 * at bits [4*slot, 4*slot+4), with r = n%16, c = k%16,
 *   lane = 4*(r%8) + c/4,   slot = r/8 + 2*((c%4)/2) + 4*(c%2),
 * i.e. register i of lane L = 4g + t (slot i low half, slot i + 4 high half)
 * holds row g + 8*(i%2) at k = 4t + 2*(i/2) + {0, 1}: each lane owns four
 * consecutive k of rows g and g + 8 of a 16x16 block whose 16 rows are output
 * columns (the per-thread fragment of a tcgen05.st.16x256b store; the
 * mma.m16n8k16 kernel reads the activations in the same k order).
 * Permuted scales fp16[N/128][K/G][128]:
 * s[g][n] is stored at ((n/128) * K/G + g) * 128 + 16*((n%128)/16) + 2*(r%8) + r/8.
 * Codes above 15 are masked to 4 bits and flag W4A16_ERR_CODE_RANGE for
 * w4a16_get_status(NULL, stream).
 * ------------------------------------------------------------------------- */
W4A16_API int w4a16_repack(const uint8_t* q, const uint16_t* s, int K, int N, int groupsize,
                 uint32_t* packed, uint16_t* scales_p, void* stream);

/* ---------------------------------------------------------------------------
 * Fused quantise + repack from FP16 weights and given FP16 scales (the
 * original Layer.pack step, deep-dive article section "可复现的调用链": the
 * weights are divided by the scale, rounded, offset by 8 and clamped to
 * [0, 15], then laid out like w4a16_repack).
 *
 *   w         device, fp16[K][N] row-major: the weights to quantise
 *   s         device, fp16[K/G][N] row-major: their scales (any sign)
 *   packed    device, uint32[K*N/8], written: same layout as w4a16_repack
 *   scales_p  device, fp16[K/G*N], written: s permuted as by w4a16_repack
 *
 * Per weight: q = clamp(rint(w / s) + 8, 0, 15), where w / s is the IEEE
 * float32 quotient of the two FP16 values (correctly rounded) and rint
 * rounds half to even.  A quotient that is NaN or infinite (s = 0, or a
 * NaN / infinite input) stores code 8 and flags W4A16_ERR_VALUE for
 * w4a16_get_status(NULL, stream).  Inputs and outputs must not overlap.
 * ------------------------------------------------------------------------- */
W4A16_API int w4a16_quantize_repack(const uint16_t* w, const uint16_t* s, int K, int N, int groupsize,
                          uint32_t* packed, uint16_t* scales_p, void* stream);

/* w4a16_quantize_repack with a zero code per group and column (the
 * asymmetric format of w4a16_gemm_zp): q = clamp(rint(w / s) + z, 0, 15),
 * same quotient, rounding and errors.  z: device, uint8[K/G][N] row-major
 * codes 0..15 (NULL: the offset 8, i.e. w4a16_quantize_repack).  The zero
 * codes themselves go through w4a16_repack_zeros for the GEMM. */
W4A16_API int w4a16_quantize_repack_zp(const uint16_t* w, const uint16_t* s, const uint8_t* z, int K, int N,
                                       int groupsize, uint32_t* packed, uint16_t* scales_p, void* stream);

/* ---------------------------------------------------------------------------
 * Scales (and zero codes) of FP16 weights by the min-max rule (MARLIN paper,
 * Section 2.2 "Mixed-Precision Inference on LLMs", paragraph "Weight
 * Quantization": the step is (max - min) / (2^b - 1), the minimum maps to
 * code 0), per group of G consecutive rows of one column.
 *
 *   w   device, fp16[K][N] row-major: the weights
 *   s   device, fp16[K/G][N] row-major, written: the scales
 *   z   device, uint8[K/G][N] row-major, written: zero codes -- or NULL
 *
 * z = NULL: symmetric rule for the offset-8 format, s = RNE_fp16(f32(2 a) / 15)
 * with a = max |w| over the group.  z given: asymmetric rule with the range
 * widened to contain 0 (lo = min(min w, 0), hi = max(max w, 0)):
 * s = RNE_fp16(f32(hi - lo) / 15), z = clamp(rint(f32(-lo / s)), 0, 15).
 * Every step is one IEEE float32 rounding (f32), rint ties to even.  A scale
 * that rounds to 0 (all-zero group) is written as 1.  A NaN or infinite
 * weight writes s = 1 (z = 0) for its group and flags W4A16_ERR_VALUE for
 * w4a16_get_status(NULL, stream).  Feed s (and z) to
 * w4a16_quantize_repack(_zp).  Inputs and outputs must not overlap.
 * ------------------------------------------------------------------------- */
W4A16_API int w4a16_minmax_scales(const uint16_t* w, int K, int N, int groupsize, uint16_t* s, uint8_t* z,
                                  void* stream);

/* Inverse of w4a16_repack (diagnostic; the pages' layout check "repack then
 * unpack recovers the same codes and scales", deep-dive article section
 * "适用边界与工程陷阱").  Outputs q uint8[K][N] and s fp16[K/G][N]. */
W4A16_API int w4a16_unpack(const uint32_t* packed, const uint16_t* scales_p, int K, int N, int groupsize,
                 uint8_t* q, uint16_t* s, void* stream);

/* Dequantised weights B^ as FP16, fp16[K][N] row-major (diagnostic):
 * Bhat[k][n] = round_to_nearest_even(s[k/G][n] * (q[k][n] - 8)), decoded from
 * the packed stream with the same in-register decode the GEMM uses
 * (deep-dive article section "INT4 只是存储类型，不是这条路径的计算类型"). */
W4A16_API int w4a16_dequant(const uint32_t* packed, const uint16_t* scales_p, int K, int N, int groupsize,
                  uint16_t* Bhat, void* stream);

/* ---------------------------------------------------------------------------
 * The fused W4A16 GEMM (MARLIN paper Section 3.4; deep-dive article sections
 * "软件流水线", "并行划分" and "Split-K 与全局归约").
 *
 *   A         device, fp16[M][K] row-major (lda = K)
 *   packed    device, output of w4a16_repack
 *   scales_p  device, output of w4a16_repack
 *   C         device, fp16[M][N] row-major (ldc = N), written, never read
 *   workspace device, >= w4a16_workspace_bytes(M, K, N, groupsize) bytes,
 *             zeroed by the caller before first use (see above)
 *
 * Accumulation is FP32.  Up to 16 token rows, each group's partial product is
 * scaled by its FP32 scale; from 17 rows on, the weights are dequantised to
 * FP16 (RNE(s * (q - 8)), the value w4a16_dequant returns) before the
 * tensor-core multiply.  Split-K partials are summed in a fixed order, so
 * repeated calls give bitwise-identical C.  M == 0 returns W4A16_OK without a
 * launch.
 * ------------------------------------------------------------------------- */
W4A16_API int w4a16_gemm(const uint16_t* A, const uint32_t* packed, const uint16_t* scales_p, uint16_t* C,
               int M, int K, int N, int groupsize, void* workspace, size_t workspace_bytes,
               void* stream);

/* ---------------------------------------------------------------------------
 * Zero points and bias (the affine form of the deep-dive article, section
 * "Marlin 要解决的精确问题": B^[k, n] = s[g, n] * (q[k, n] - z[g, n]); the
 * production variant with a zero point per group and a bias, section
 * "Marlin 已从一个 Kernel 变成一族实现").
 *
 * w4a16_repack_zeros: zero codes z uint8[K/G][N] row-major (values 0..15, one
 * per byte, G as for the scales) -> zeros_p uint8[(K/G)*N] in the permuted
 * order of the scales (z[g][n] at the index w4a16_repack gives s[g][n]).
 * Codes above 15 are masked to 4 bits and flag W4A16_ERR_CODE_RANGE for
 * w4a16_get_status(NULL, stream).
 *
 * w4a16_gemm_zp: w4a16_gemm with optional zero points and bias:
 *   C[m][n] = RNE( sum_k A[m][k] * s[k/G][n] * (q[k][n] - z[k/G][n]) + bias[n] )
 * accumulated in FP32.  zeros_p = NULL means z = 8 (the symmetric codes of
 * w4a16_gemm); bias (fp16[N]) = NULL means no bias.  Same operands, workspace
 * (w4a16_workspace_bytes covers both forms), determinism and errors as
 * w4a16_gemm; zeros_p and bias, when given, are 16-byte aligned device
 * pointers.
 *
 * w4a16_dequant_zp: Bhat[k][n] = RNE(s[k/G][n] * (q[k][n] - z[k/G][n]))
 * (diagnostic, like w4a16_dequant).
 * ------------------------------------------------------------------------- */
W4A16_API int w4a16_repack_zeros(const uint8_t* z, int K, int N, int groupsize, uint8_t* zeros_p, void* stream);

W4A16_API int w4a16_gemm_zp(const uint16_t* A, const uint32_t* packed, const uint16_t* scales_p,
                            const uint8_t* zeros_p, const uint16_t* bias, uint16_t* C, int M, int K, int N,
                            int groupsize, void* workspace, size_t workspace_bytes, void* stream);

W4A16_API int w4a16_dequant_zp(const uint32_t* packed, const uint16_t* scales_p, const uint8_t* zeros_p, int K,
                               int N, int groupsize, uint16_t* Bhat, void* stream);

/* ---------------------------------------------------------------------------
 * 2:4-sparse W4A16 (the Sparse-Marlin analogue).  The MARLIN paper, Section
 * 2.1.1 "Modern Tensor Core Units", describes the 2:4 format: in every vector
 * of four along the reduction dimension two values are kept, with metadata
 * giving their positions; the deep-dive article, section "Sparse-Marlin 再叠加
 * 2:4 结构化稀疏", keeps them as 4-bit codes with 2-bit positions.  Here a
 * pruned weight is the code 8 (B^ = 0), and a layer is 2:4 sparse when every
 * group of four consecutive rows k = 4i .. 4i + 3 of every column holds at
 * most two codes != 8.  Its product is the dense one of those codes:
 * C = A * B^ exactly as for w4a16_gemm.  Shapes and groups as for w4a16_gemm.
 *
 * w4a16_packed24_bytes: bytes of the packed 2:4 stream, 3 K N / 8 (3 bits per
 * weight: two 4-bit codes and two 2-bit positions per group of four).
 *
 * w4a16_repack_24: dense codes q uint8[K][N] (2:4 as above) and scales
 * s fp16[K/G][N] -> packed24 (uint32[3 K N / 32], this library's layout:
 * per 128-column strip and 64-row piece, 2048 bytes of codes then 1024 bytes
 * of positions in the lane order of the sparse tensor-core instruction) and
 * scales_p (permuted exactly as by w4a16_repack).  The kept positions of a
 * group are those of its codes != 8, filled up with its lowest other
 * positions.  A group with three or more codes != 8 flags W4A16_ERR_VALUE for
 * w4a16_get_status(NULL, stream) (its stored entries are then unspecified).
 *
 * w4a16_unpack_24: packed24 -> dense codes q uint8[K][N] (8 at pruned
 * positions); positions that are not a rising pair flag W4A16_ERR_VALUE.
 * It checks a stream of unknown origin before w4a16_gemm_24 reads it.
 *
 * w4a16_gemm_24: C fp16[M][N] = A fp16[M][K] * B^ from packed24 and
 * scales_p, computed with the sparse tensor-core MMA; any M >= 0 (16 token
 * rows per launch).  packed24 must come from w4a16_repack_24 (or have passed
 * w4a16_unpack_24 without an error): its positions feed the tensor cores'
 * metadata operand, which requires rising pairs.  The workspace (size from
 * w4a16_workspace_bytes_24) follows the rules of w4a16_gemm's.
 * ------------------------------------------------------------------------- */
W4A16_API size_t w4a16_packed24_bytes(int K, int N);

W4A16_API int w4a16_repack_24(const uint8_t* q, const uint16_t* s, int K, int N, int groupsize, uint32_t* packed24,
                              uint16_t* scales_p, void* stream);

W4A16_API int w4a16_unpack_24(const uint32_t* packed24, int K, int N, uint8_t* q, void* stream);

W4A16_API size_t w4a16_workspace_bytes_24(int M, int K, int N, int groupsize);

W4A16_API int w4a16_gemm_24(const uint16_t* A, const uint32_t* packed24, const uint16_t* scales_p, uint16_t* C,
                            int M, int K, int N, int groupsize, void* workspace, size_t workspace_bytes,
                            void* stream);

/* ---------------------------------------------------------------------------
 * Grouped expert GEMM (MoE).  The deep-dive article, section "适用边界与工程
 * 陷阱" (items 1 and 4), notes that an MoE layer regroups the tokens by
 * expert, so every expert's GEMM has its own small M, and that the grouped
 * GEMM schedules differently from a dense layer.  One call runs all experts:
 *
 *   C[m][n] = sum_k A[m][k] * Bhat_e[k][n]   for the expert e that owns row m
 *
 *   A               device, fp16[M][K] row-major, rows sorted by expert
 *   packed          device, E layers of w4a16_repack output back to back
 *                   (expert e at word e * K * N / 8)
 *   scales_p        device, E permuted scale arrays back to back (expert e at
 *                   element e * (K/G) * N)
 *   expert_offsets  device, int32[E + 1]: expert e owns rows
 *                   expert_offsets[e] .. expert_offsets[e+1] - 1; they must
 *                   rise from 0 to M (an expert may own no rows)
 *   C               device, fp16[M][N] row-major, written
 *   max_rows        a bound on the rows of any one expert (<= 0: M).  It picks
 *                   the kernel and the row-segment height: up to 16, the
 *                   streaming mma.sync kernel with segments of 8 rows (when
 *                   max_rows <= 8) or 16; from 17, the tensor-memory (tcgen05)
 *                   kernel with segments of max_rows rounded up to 16, at most
 *                   128.  An expert with more rows than a segment is split into
 *                   segments, each of which streams that expert's weights once.
 *                   A bound that is too low only costs speed.
 *
 * Symmetric codes (z = 8), no bias; 1 <= E <= 2048, M <= 2^24, K, N, G as for
 * w4a16_gemm.  The offsets are read on the device only, so the call needs no
 * host synchronisation (CUDA-graph capturable).  Offsets that do not rise from
 * 0 to M leave C unwritten and record W4A16_ERR_VALUE for
 * w4a16_get_status(workspace, stream).  The workspace (size from
 * w4a16_moe_workspace_bytes) follows the rules of w4a16_gemm's workspace.
 * ------------------------------------------------------------------------- */
W4A16_API size_t w4a16_moe_workspace_bytes(int E, int M, int max_rows, int K, int N, int groupsize);

W4A16_API int w4a16_moe_gemm(const uint16_t* A, const uint32_t* packed, const uint16_t* scales_p,
                             const int32_t* expert_offsets, uint16_t* C, int E, int M, int max_rows, int K, int N,
                             int groupsize, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Allocation-free GEMM.  The paper has no counterpart: this entry point is a
 * convenience of this library for callers that cannot allocate device memory.
 *
 * Some callers cannot call cudaMalloc: code that runs while its stream is being
 * captured into a CUDA graph (an allocation is not a stream operation and the
 * default capture mode forbids it), serving loops that must never allocate or
 * synchronise the device on their hot path, and plugin hosts that own all
 * device memory and hand a kernel nothing but its inputs and outputs.  Such a
 * caller passes A, packed, scales_p and C exactly as for w4a16_gemm (same
 * meaning, layout and alignment) and no workspace.
 *
 * The scratch this call needs lives in the library itself: a file-scope device
 * array of W4A16_NOALLOC_SCRATCH_BYTES that every GPU which loads the library
 * holds until the process exits.  The first call on each device looks up the
 * array's device address with that device current; make that first call
 * before any stream capture begins.  Each call then clears the array's
 * arrival counters (cudaMemsetAsync on `stream`) and runs the same kernel as
 * w4a16_gemm, so its result is bitwise identical to w4a16_gemm's.  It calls
 * no cudaMalloc, no cudaFree and no allocating library routine.
 *
 * All calls share the one array and it keeps the previous call's contents, so
 * two calls that may execute at the same time on the GPU (for example on two
 * streams with no ordering between them) race and corrupt each other's output:
 * order them.  Shapes whose w4a16_workspace_bytes exceed the array are rejected
 * with W4A16_ERR_WORKSPACE before anything is launched.  A pipeline timeout
 * inside this call is recorded in the status word at the head of the
 * library's array; later calls leave that word alone, and
 * w4a16_get_status(NULL, stream) reports it (W4A16_ERR_TIMEOUT) and clears it.
 * ------------------------------------------------------------------------- */
#define W4A16_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

W4A16_API int w4a16_gemm_noalloc(const uint16_t* A, const uint32_t* packed, const uint16_t* scales_p, uint16_t* C,
                                 int M, int K, int N, int groupsize, void* stream);

/* Synchronises `stream`, then returns (and clears) the first error recorded on
 * the device: the repack code-range flag and, when `workspace` is non-NULL,
 * the GEMM status word in that workspace.  With `workspace` NULL, the status
 * word of w4a16_gemm_noalloc's array takes its place once a call of that entry
 * point has set the array up on the current device.  W4A16_OK when none. */
W4A16_API int w4a16_get_status(void* workspace, void* stream);

/* ---------------------------------------------------------------------------
 * Work plan (host only; deep-dive article section "为什么规则二维网格会浪费最后
 * 一波 SM": T = ceil(#tiles / #SMs) consecutive K-tiles per SM, wrapping into
 * the next column).  Describes how w4a16_gemm would split a shape over
 * `num_sms` SMs (num_sms <= 0: the current device's count).
 * ------------------------------------------------------------------------- */
typedef struct {
  int path;          /* 1 = mma.sync streaming kernel, 2 = tensor-memory (tcgen05) kernel */
  int m_tiles;       /* m_chunk / 8 */
  int m_chunk;       /* token rows per launch (8, 16 or 32 on path 1; a multiple of 16 up to
                        256 on path 2); launches = ceil(M / m_chunk) */
  int n_tile;        /* output columns per work unit: 128 (path 1, and path 2 in its wide
                        mode) or 256 (path 2, a strip pair) */
  int k_tile;        /* reduction rows per work unit (path 1: 128 to 1024; path 2: 128, 256
                        or 512) */
  int units;         /* work units per launch: ceil(N / n_tile) * (K / k_tile) */
  int units_per_cta; /* T */
  int grid;          /* CTAs per launch */
  int stages;        /* shared-memory pipeline depth */
  int smem_bytes;    /* dynamic shared memory per CTA */
  int threads;       /* threads per CTA */
  int final_sum_warps; /* warps that sum a split strip's FP32 slots at a CTA's last segment:
                          path 1: 8 with two token tiles, or one tile and at most two units per
                          CTA (measured faster there), else 2; path 2: the 16 dequant warps */
} w4a16_plan_t;

W4A16_API int w4a16_plan(int M, int K, int N, int groupsize, int num_sms, w4a16_plan_t* out);

/* Debug knob (not thread-safe): bound, in GPU clock cycles, on every pipeline
 * wait of later w4a16_gemm launches.  0 restores the default (about one
 * second).  A wait that runs out records W4A16_ERR_TIMEOUT and the kernel
 * winds down without trapping. */
W4A16_API void w4a16_debug_set_wait_cycles(long long cycles);

/* Failure-injection knob (not thread-safe): while enabled, w4a16_gemm launches
 * leave the first pipeline stage of every CTA unfilled, so the consumers' first
 * wait can only end by running out of its cycle bound.  The kernel then records
 * W4A16_ERR_TIMEOUT, skips all output and returns; the CUDA context stays
 * usable.  Used by the failure-detection tests; 0 disables it. */
W4A16_API void w4a16_debug_inject_stall(int enable);

/* Kernel-selection knob (not thread-safe), for tests and measurements: 1 runs
 * every later w4a16_gemm on the streaming mma.sync kernel; 2 on the
 * tensor-memory (tcgen05) kernel, in strip pairs up to 128 token rows and in
 * its wide mode (one strip per unit, up to 256 token rows per launch) above;
 * 3 on the tensor-memory kernel in strip pairs only; 4 on the tensor-memory
 * kernel in its wide mode wherever K is a multiple of 512 (strip pairs
 * otherwise); 0 restores the default (the mma.sync kernel up to 16 token rows,
 * then as 2).  w4a16_workspace_bytes and w4a16_plan follow the same choice. */
W4A16_API void w4a16_debug_force_path(int path);

/* Ablation switches: the MARLIN paper's Figure 12 ablations (discussed in the
 * deep-dive article, section "性能结果应该怎样读"), re-run on this library's
 * kernels.  `flags` is a bit mask, applied to every later GEMM call of the
 * process (0 restores the full design):
 *   1  the weight stream loses its L2 evict-first hint (evict-normal instead);
 *   2  the weight pipeline is 2 stages deep (streaming kernel: stages; tensor-
 *      memory kernel: weight ring);
 *   4  the activation tile is stored without the 128-byte XOR swizzle
 *      (streaming kernel and grouped GEMM only; the tensor-memory kernel's
 *      operand descriptors require the swizzled layout).
 * The results stay bitwise identical: none of the switches changes the order
 * of the arithmetic.  Diagnostic: not for concurrent use with GEMM calls. */
W4A16_API void w4a16_debug_ablate(int flags);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
