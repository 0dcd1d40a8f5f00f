"""Plain float64 CPU statement of the W4A16 layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
import this module.  It is independent of the CUDA library and imports nothing
from it.

Sources (page title, section):
  [P1] "MARLIN: Mixed-Precision Auto-Regressive Parallel Inference on Large
       Language Models" (arXiv HTML), Section 3.4 "Kernel Design" (problem
       statement: FP16 A, K x N INT4 B, symmetric quantisation with one FP16
       scale per column or per G consecutive weights of a column) and its
       paragraph "Bound By Weight Loading" (memory/FLOP counts); Section 2.2
       "Mixed-Precision Inference on LLMs", paragraph "Weight Quantization"
       (the min-max rule for the step and the zero); Section 2.1.1 "Modern
       Tensor Core Units" (the 2:4 sparse format: values plus positions).
  [P2] "Marlin 完全拆解：4-bit 权重如何喂满 GPU Tensor Core" (the Marlin
       deep-dive article), section "Marlin 要解决的精确问题" (the affine
       dequantisation B^[k,n] = s[g,n] (q[k,n] - z[g,n]), q in {0..15}),
       section "scale 为什么有时在内环乘，有时在末尾乘" (grouped sum
       C = sum_g s[g,n] sum_{k in g} A[m,k](q[k,n]-8) and the per-column form
       AB = (AQ) diag(s)), and section "量化数据如何进入 Tensor Core" (the
       symmetric zero point 8 folded into the decode), and section
       "适用边界与工程陷阱" (MoE layers: one GEMM per expert on the rows
       routed to it), and section "Sparse-Marlin 再叠加 2:4 结构化稀疏"
       (2:4 sparse weights: 4-bit kept values plus 2-bit positions).

Readings taken where the pages are silent (each also listed in the design notes):
  * zero point: the symmetric main path uses the constant z = 8; no zero tensor;
  * group index: g = floor(k / G), K a multiple of G; G = K (or -1) is the
    one-scale-per-column mode;
  * q arrives as uint8[K][N] row-major (one code per byte), s as fp16[K/G][N];
  * the reference result is the exact dense product, accumulated in float64 in
    plain k order (numpy matmul as the summation primitive);
  * parity bound (per element): |C - C_ref| <= 4e-3 * sum_k |A[m,k] B^[k,n]| + 1e-4;
  * the packed weight / permuted scale layout is this library's own ABI (the
    pages describe its purpose -- one 16-byte load per thread carrying the
    codes of four 16x16 tensor-core blocks, 16x64 tiles stored contiguously --
    but print no permutation table); it is defined here by a closed index
    formula, ``packed_position`` and ``scale_position``: 128-column strips,
    each stored contiguously along K, so that one work unit of the kernel is
    one large contiguous copy.  It needs K % 64 == 0 and N % 128 == 0.
"""
from __future__ import annotations

import numpy as np

#: symmetric INT4 zero point ([P2] "量化数据如何进入 Tensor Core": the zero 8 is folded into the decode)
Z_POINT = 8
#: per-element tolerance of the GEMM parity check
TOL_REL = 4e-3
TOL_ABS = 1e-4


# ---------------------------------------------------------------------------
# IEEE-754 binary16, written from the format definition (1 sign bit, 5
# exponent bits with bias 15, 10 fraction bits; subnormals at 2^-24 steps).
# ---------------------------------------------------------------------------

def fp16_bits_to_f64(bits) -> np.ndarray:
    """Decode binary16 bit patterns (uint16) to float64 exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where(b >> 15, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    f = (b & 0x3FF).astype(np.float64)
    normal = sign * np.ldexp(1.0 + f / 1024.0, (e - 15).astype(np.int64))
    sub = sign * np.ldexp(f, -24)
    out = np.where(e == 0, sub, normal)
    out = np.where((e == 31) & (f == 0), sign * np.inf, out)
    out = np.where((e == 31) & (f != 0), np.nan, out)
    return out


def f64_to_fp16_bits(x) -> np.ndarray:
    """Round float64 values to binary16 with round-to-nearest, ties-to-even.

    Scaling by powers of two is exact in float64, so ``np.rint`` (which rounds
    half to even) on the scaled magnitude performs exactly one RNE rounding.
    """
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x).astype(np.uint16) << 15
    a = np.abs(x)
    out = np.zeros(x.shape, dtype=np.uint16)
    # subnormal range |x| < 2^-14: integer multiples of 2^-24
    sub = a < 2.0 ** -14
    m_sub = np.rint(np.ldexp(a, 24)).astype(np.int64)  # 1024 -> smallest normal, which is bit pattern 0x0400
    # normal range
    with np.errstate(divide="ignore"):
        _, E = np.frexp(a)  # a = f * 2^E, f in [0.5, 1)
    e = E.astype(np.int64) - 1  # a in [2^e, 2^(e+1))
    m = np.rint(np.ldexp(a, (10 - e))).astype(np.int64)  # in [1024, 2048]
    carry = m == 2048
    e = np.where(carry, e + 1, e)
    m = np.where(carry, 1024, m)
    normal_bits = ((e + 15) << 10) | (m - 1024)
    normal_bits = np.where(e + 15 >= 31, 0x7C00, normal_bits)  # overflow -> infinity
    bits = np.where(sub, m_sub, normal_bits)
    bits = np.where(np.isinf(a), 0x7C00, bits)
    bits = np.where(np.isnan(a), 0x7E00, bits)
    out[...] = bits.astype(np.uint16)
    return out | sign


def _as_f64(h) -> np.ndarray:
    """float16 array (or its uint16 bit patterns) -> float64, exactly."""
    h = np.asarray(h)
    if h.dtype == np.float16:
        h = h.view(np.uint16)
    return fp16_bits_to_f64(h)


# ---------------------------------------------------------------------------
# Dequantisation and the dense product ([P1] Section 3.4; [P2] sections cited above)
# ---------------------------------------------------------------------------

def _group(K: int, G: int) -> int:
    G = K if G in (-1, K) else int(G)
    if G <= 0 or K % G:
        raise ValueError(f"K={K} is not a multiple of the group size {G}")
    return G


def dequant_exact(q, s, G: int) -> np.ndarray:
    """B^[k, n] = s[floor(k/G), n] * (q[k, n] - 8) in float64.

    An FP16 scale times an integer in [-8, 7] needs at most 11 + 4 significant
    bits, so the float64 product is exact.
    """
    q = np.asarray(q)
    K = q.shape[0]
    G = _group(K, G)
    if q.min(initial=0) < 0 or q.max(initial=0) > 15:
        raise ValueError("4-bit codes must lie in 0..15")
    s64 = _as_f64(s)
    if s64.shape != (K // G, q.shape[1]):
        raise ValueError("scales must have shape [K/G][N]")
    g_of_k = np.arange(K) // G
    return s64[g_of_k, :] * (q.astype(np.float64) - Z_POINT)


def dequant_fp16_bits(q, s, G: int) -> np.ndarray:
    """The FP16 dequantised weight: one RNE rounding of the exact B^ (uint16 bits)."""
    return f64_to_fp16_bits(dequant_exact(q, s, G))


def gemm_ref(A, q, s, G: int):
    """C_ref[m, n] = sum_k A[m, k] B^[k, n] and Bound[m, n] = sum_k |A[m, k] B^[k, n]|.

    Both in float64; numpy's matmul is the summation primitive.  Returns
    (C_ref, Bound), each float64[M][N].
    """
    A64 = _as_f64(A)
    B64 = dequant_exact(q, s, G)
    if A64.shape[1] != B64.shape[0]:
        raise ValueError("A is M x K and B is K x N")
    C = A64 @ B64
    bound = np.abs(A64) @ np.abs(B64)
    return C, bound


# ---------------------------------------------------------------------------
# Zero points and bias ([P2] section "Marlin 要解决的精确问题": the affine form
# B^[k,n] = s[g,n] (q[k,n] - z[g,n]); section "Marlin 已从一个 Kernel 变成一族实现":
# the production variants with a zero point per group and a bias)
# ---------------------------------------------------------------------------

def dequant_exact_zp(q, s, z, G: int) -> np.ndarray:
    """B^[k, n] = s[floor(k/G), n] * (q[k, n] - z[floor(k/G), n]) in float64 (exact:
    an FP16 scale times an integer in [-15, 15]).  Readings taken: z are 4-bit
    codes 0..15 (an integer zero point per group and column), shaped like s."""
    q = np.asarray(q)
    K, N = q.shape
    G = _group(K, G)
    z = np.asarray(z)
    if z.shape != (K // G, N):
        raise ValueError("zero points must have shape [K/G][N]")
    if q.min(initial=0) < 0 or q.max(initial=0) > 15 or z.min(initial=0) < 0 or z.max(initial=0) > 15:
        raise ValueError("codes and zero points must lie in 0..15")
    s64 = _as_f64(s)
    if s64.shape != (K // G, N):
        raise ValueError("scales must have shape [K/G][N]")
    g_of_k = np.arange(K) // G
    return s64[g_of_k, :] * (q.astype(np.float64) - z.astype(np.float64)[g_of_k, :])


def dequant_fp16_bits_zp(q, s, z, G: int) -> np.ndarray:
    """RNE(s (q - z)) as FP16 bit patterns."""
    return f64_to_fp16_bits(dequant_exact_zp(q, s, z, G))


def gemm_ref_zp(A, q, s, z, bias, G: int):
    """C_ref[m, n] = sum_k A[m, k] B^[k, n] + bias[n] and Bound[m, n] = sum_k |A[m, k] B^[k, n]| + |bias[n]|,
    B^ with zero points (z None: the symmetric z = 8; bias None: no bias).  Reading taken: the bias joins
    the absolute sum of the parity bound, so the FP16 rounding of a result dominated by the bias is covered."""
    if z is None:
        z = np.full(np.asarray(s).shape, Z_POINT, dtype=np.uint8)
    Bh = dequant_exact_zp(q, s, z, G)
    A64 = _as_f64(A)
    C = A64 @ Bh
    bound = np.abs(A64) @ np.abs(Bh)
    if bias is not None:
        b64 = _as_f64(bias).reshape(1, -1)
        C = C + b64
        bound = bound + np.abs(b64)
    return C, bound


def repack_zeros(z, G: int, K: int):
    """Zero codes uint8[K/G][N] -> uint8[(K/G)*N] in the permuted order of the scales (``scale_position``)."""
    z = np.asarray(z)
    G = _group(K, G)
    NG, N = z.shape
    if NG != K // G or z.dtype != np.uint8 or z.max(initial=0) > 15:
        raise ValueError("zero points must be uint8 codes 0..15 of shape [K/G][N]")
    gg, nn = np.meshgrid(np.arange(NG), np.arange(N), indexing="ij")
    zp = np.empty(NG * N, dtype=np.uint8)
    zp[scale_position(gg, nn, NG).ravel()] = z.ravel()
    return zp


def error_excess(C_gpu, C_ref, bound) -> np.ndarray:
    """|C_gpu - C_ref| - (4e-3 * Bound + 1e-4): an element passes iff <= 0."""
    c = _as_f64(C_gpu) if np.asarray(C_gpu).dtype in (np.float16, np.uint16) else np.asarray(C_gpu, np.float64)
    return np.abs(c - C_ref) - (TOL_REL * bound + TOL_ABS)


def error_ok(C_gpu, C_ref, bound) -> bool:
    """True iff every element lies within the parity bound (NaN fails)."""
    ex = error_excess(C_gpu, C_ref, bound)
    return bool(np.all(ex <= 0.0))


# ---------------------------------------------------------------------------
# Packed layout (this library's own ABI; purpose from [P1] Section 3.4
# "Maximizing Loading Bandwidth" and [P2] section "直接生成 MMA 所需的寄存器 fragment")
# ---------------------------------------------------------------------------

def packed_position(k, n, K: int):
    """Word index and bit offset of code q[k, n] in the packed uint32 stream.

    The stream is uint32[N/128][K/64][8][32][4]: output columns are cut into
    strips of 128, and each strip is stored contiguously along K, one
    16 x 64 tile (512 bytes) per (64-row block kb, 16-column block b) with the
    8 column blocks of a 64-row block side by side.  Inside a tile, lane L's
    four consecutive words (one 16-byte vector) are its operand fragments of
    the four 16 x 16 tensor-core blocks j = 0..3 (rows 16j .. 16j+15 of the
    tile).  Inside a 16x16 block, with r = n mod 16 (the fragment row) and
    c = k mod 16 (the reduction index inside the block):
        lane   = 4 * (r mod 8) + floor(c / 4)
        slot   = floor(r / 8) + 2 * floor((c mod 4) / 2) + 4 * (c mod 2)
        bits   = [4 * slot, 4 * slot + 4)
    Slot i < 4 is the low half and slot i + 4 the high half of the lane's
    i-th 32-bit register: register i holds row g + 8*(i mod 2) (g = lane/4)
    and reduction indices 4t + 2*floor(i/2) + {0, 1} (t = lane mod 4).  Each
    lane thus holds four consecutive k of rows g and g + 8 -- the per-thread
    fragment of a 16-row x 256-bit tensor-memory store -- and, read as an
    m16n8k16 A operand, the k order inside the block is the fixed permutation
    2t + e -> 4t + e, 2t + 8 + e -> 4t + 2 + e (the activation operand is
    loaded in the same order).
    """
    k = np.asarray(k, dtype=np.int64)
    n = np.asarray(n, dtype=np.int64)
    strip, b = n // 128, (n % 128) // 16
    r = n % 16
    kb, kk = k // 64, k % 64
    j, c = kk // 16, kk % 16
    lane = 4 * (r % 8) + c // 4
    slot = r // 8 + 2 * ((c % 4) // 2) + 4 * (c % 2)
    word = (((strip * (K // 64) + kb) * 8 + b) * 32 + lane) * 4 + j
    return word, 4 * slot


def scale_position(g, n, NG: int):
    """Index of scale s[g, n] in the permuted scale array (NG = K/G rows of scales).

    Layout fp16[N/128][NG][128]: each 128-column strip keeps its NG scale rows
    together; inside a row, every block of 16 columns puts fragment rows r and
    r + 8 (r < 8) side by side, so one 32-bit read gives a lane both of its
    rows' scales:
        index = (floor(n/128) * NG + g) * 128 + 16 * floor((n mod 128)/16) + 2 * (r mod 8) + floor(r / 8),
    with r = n mod 16.
    """
    g = np.asarray(g, dtype=np.int64)
    n = np.asarray(n, dtype=np.int64)
    r = n % 16
    return ((n // 128) * NG + g) * 128 + ((n % 128) // 16) * 16 + 2 * (r % 8) + r // 8


def _check_layout_shape(K: int, N: int):
    if K % 64 or N % 128 or K <= 0 or N <= 0:
        raise ValueError("the packed layout needs K % 64 == 0 and N % 128 == 0")


def quantize(w, s, G: int) -> np.ndarray:
    """4-bit codes of FP16 weights w[K][N] with FP16 scales s[K/G][N], the step
    before the repack ([P2] section "可复现的调用链": the original Layer.pack
    divides the weights by the scale, rounds, adds the offset 8 and clamps to
    [0, 15]):

        q[k, n] = clamp(rint(w[k, n] / s[floor(k/G), n]) + 8, 0, 15).

    Readings taken (the page prints no code): the quotient is the IEEE float32
    division of the two FP16 values (both are exact in float32, the division
    rounds once, to nearest); "round" is to nearest with ties to even.  A NaN
    or infinite quotient (a zero, NaN or infinite input) is an error.
    """
    w64 = _as_f64(w)
    if w64.ndim != 2:
        raise ValueError("weights must have shape [K][N]")
    K, N = w64.shape
    G = _group(K, G)
    s64 = _as_f64(s)
    if s64.shape != (K // G, N):
        raise ValueError("scales must have shape [K/G][N]")
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        quot = w64.astype(np.float32) / s64[np.arange(K) // G, :].astype(np.float32)
    if not np.all(np.isfinite(quot)):
        raise ValueError("w / s is NaN or infinite (zero, NaN or infinite input)")
    q = np.clip(np.rint(quot).astype(np.float64) + Z_POINT, 0, 15)
    return q.astype(np.uint8)


# ---------------------------------------------------------------------------
# 2:4 structured sparsity ([P1] Section 2.1.1 "Modern Tensor Core Units": the
# 2:4 format splits the sparse operand into vectors of four along the reduction
# dimension, keeps two values of each and stores them with a metadata
# structure giving each kept value's position inside its group of four;
# [P2] section "Sparse-Marlin 再叠加 2:4 结构化稀疏": the kept weights stay
# 4-bit codes, the positions are 2-bit metadata)
# ---------------------------------------------------------------------------

def sparse24_compress(q):
    """Dense codes uint8[K][N] with at most two codes != 8 (the zero weight) in
    every group of four consecutive rows of a column -> (qc uint8[K/2][N],
    idx uint8[K/2][N]): kept entry j (0, 1) of group i of column n is row
    2i + j, holding the code qc and its position idx in 0..3 inside the group.

    Readings taken: a pruned weight is the code 8 (B^ = 0); the kept positions
    are those of the codes != 8 in increasing order, and a group with fewer
    than two such codes is filled up with its lowest remaining positions, then
    the two positions are sorted (so idx0 < idx1 always).
    """
    q = np.asarray(q)
    if q.ndim != 2 or q.shape[0] % 4:
        raise ValueError("codes must be uint8[K][N] with K a multiple of 4")
    K, N = q.shape
    if q.min(initial=0) < 0 or q.max(initial=0) > 15:
        raise ValueError("codes must lie in 0..15")
    qc = np.empty((K // 2, N), dtype=np.uint8)
    idx = np.empty((K // 2, N), dtype=np.uint8)
    for i in range(K // 4):
        grp = q[4 * i:4 * i + 4, :]
        for n in range(N):
            nz = [p for p in range(4) if grp[p, n] != Z_POINT]
            if len(nz) > 2:
                raise ValueError(f"group {i} of column {n} has {len(nz)} non-zero weights (2:4 allows 2)")
            for p in range(4):
                if len(nz) == 2:
                    break
                if p not in nz:
                    nz.append(p)
            nz.sort()
            for j in range(2):
                qc[2 * i + j, n] = grp[nz[j], n]
                idx[2 * i + j, n] = nz[j]
    return qc, idx


def sparse24_expand(qc, idx):
    """Inverse of ``sparse24_compress``: dense codes with 8 at every pruned position."""
    qc = np.asarray(qc)
    idx = np.asarray(idx)
    K2, N = qc.shape
    if idx.shape != (K2, N) or K2 % 2:
        raise ValueError("qc and idx must both be uint8[K/2][N]")
    if np.any(idx[0::2] >= idx[1::2]) or idx.max(initial=0) > 3:
        raise ValueError("the two positions of a group must rise inside 0..3")
    q = np.full((2 * K2, N), Z_POINT, dtype=np.uint8)
    cols = np.arange(N)
    for j in range(K2):
        q[4 * (j // 2) + idx[j].astype(np.int64), cols] = qc[j]
    return q


def gemm24_ref(A, qc, idx, s, G: int):
    """The 2:4-sparse layer's product: the dense product ``gemm_ref`` of the expanded codes
    (pruned weights are exact zeros)."""
    return gemm_ref(A, sparse24_expand(qc, idx), s, G)


# ---------------------------------------------------------------------------
# Grouped expert GEMM ([P2] section "适用边界与工程陷阱", items 1 and 4: an MoE
# layer regroups the tokens by expert, so every expert's GEMM has its own,
# usually small, M, and the grouped GEMM schedules differently from a dense one)
# ---------------------------------------------------------------------------

def check_expert_offsets(offsets, M: int) -> np.ndarray:
    """offsets int[E+1]: 0 = offsets[0] <= offsets[1] <= ... <= offsets[E] = M."""
    off = np.asarray(offsets, dtype=np.int64)
    if off.ndim != 1 or off.size < 2 or off[0] != 0 or off[-1] != M or np.any(np.diff(off) < 0):
        raise ValueError("expert offsets must rise from 0 to M")
    return off


def moe_gemm_ref(A, offsets, q, s, G: int):
    """C_ref[m, n] = sum_k A[m, k] B^_e[k, n], e the expert that owns row m, and the
    matching Bound, each float64[M][N].

    Readings taken: the rows of A are already sorted by expert; expert e owns
    rows offsets[e] .. offsets[e+1] - 1 (an expert may own none); every expert
    has its own codes q[e] uint8[K][N] and scales s[e] fp16[K/G][N] with the
    same K, N and G; the symmetric zero point 8, no bias.  Each expert's block
    of rows is the plain product ``gemm_ref`` of that expert's weights.
    """
    A = np.asarray(A)
    if A.ndim != 2:
        raise ValueError("A must be fp16[M][K]")
    M = A.shape[0]
    off = check_expert_offsets(offsets, M)
    E = off.size - 1
    q = np.asarray(q)
    if q.ndim != 3 or q.shape[0] != E:
        raise ValueError("q must be uint8[E][K][N]")
    N = q.shape[2]
    C = np.zeros((M, N))
    bound = np.zeros((M, N))
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi > lo:
            C[lo:hi], bound[lo:hi] = gemm_ref(A[lo:hi], q[e], s[e], G)
    return C, bound


def minmax_scales(w, G: int, symmetric: bool = True):
    """Scales (and zero codes) of FP16 weights w[K][N] by the min-max rule of
    [P1] Section 2.2, paragraph "Weight Quantization": uniform quantisation of
    a vector v to b bits maps min(v) to code 0 and max(v) to code 2^b - 1, so
    the step is s = (max(v) - min(v)) / (2^b - 1); here b = 4 and v is one
    group (G consecutive rows of one column).

    Readings taken, so that the result fits the kernels' formats:
      * asymmetric (``symmetric=False``): the kernels store the zero point as
        a 4-bit code z with B^ = s (q - z), so the range is widened to contain
        0: lo = min(min v, 0), hi = max(max v, 0), s = (hi - lo) / 15 and
        z = clamp(rint(-lo / s), 0, 15);
      * symmetric (z = 8): the range is [-a, a] with a = max |v|, so
        s = 2a / 15;
      * arithmetic: hi - lo (or 2a) and the division by 15 in IEEE float32,
        one round-to-nearest each, then the scale rounded to FP16 (RNE);
        the zero code's quotient -lo / s in float32 with that FP16 s;
      * a group whose FP16 scale comes out 0 (all weights 0, or a range below
        FP16's reach) takes s = 1, so its codes reproduce 0;
      * a NaN or infinite weight is an error.

    Returns (s fp16[K/G][N], z uint8[K/G][N] or None when symmetric).
    """
    w64 = _as_f64(w)
    if w64.ndim != 2:
        raise ValueError("weights must have shape [K][N]")
    K, N = w64.shape
    G = _group(K, G)
    if not np.all(np.isfinite(w64)):
        raise ValueError("weights must be finite")
    grp = w64.reshape(K // G, G, N)
    lo = grp.min(axis=1)
    hi = grp.max(axis=1)
    if symmetric:
        a = np.maximum(np.abs(lo), np.abs(hi))
        span = np.float32(2.0) * a.astype(np.float32)            # exact: a doubling
    else:
        lo = np.minimum(lo, 0.0)
        hi = np.maximum(hi, 0.0)
        span = hi.astype(np.float32) - lo.astype(np.float32)     # one float32 rounding
    s32 = span / np.float32(15.0)                                 # one float32 rounding
    s16 = s32.astype(np.float16)                                  # RNE to FP16
    s16[s16 == 0] = np.float16(1.0)
    if symmetric:
        return s16, None
    zq = (-lo).astype(np.float32) / s16.astype(np.float32)
    z = np.clip(np.rint(zq), 0, 15).astype(np.uint8)
    return s16, z


def quantize_zp(w, s, z, G: int) -> np.ndarray:
    """4-bit codes with a zero code per group and column: the step before the
    repack for the asymmetric format,

        q[k, n] = clamp(rint(w[k, n] / s[floor(k/G), n]) + z[floor(k/G), n], 0, 15),

    so that s (q - z) is the nearest point of the grid to w inside the code
    range.  The quotient, rounding and errors are those of ``quantize``
    (float32 division, ties to even; a NaN or infinite quotient is an error).
    """
    w64 = _as_f64(w)
    if w64.ndim != 2:
        raise ValueError("weights must have shape [K][N]")
    K, N = w64.shape
    G = _group(K, G)
    s64 = _as_f64(s)
    z = np.asarray(z)
    if s64.shape != (K // G, N) or z.shape != (K // G, N):
        raise ValueError("scales and zero codes must have shape [K/G][N]")
    if z.min(initial=0) < 0 or z.max(initial=0) > 15:
        raise ValueError("zero codes must lie in 0..15")
    rows = np.arange(K) // G
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        quot = w64.astype(np.float32) / s64[rows, :].astype(np.float32)
    if not np.all(np.isfinite(quot)):
        raise ValueError("w / s is NaN or infinite (zero, NaN or infinite input)")
    q = np.clip(np.rint(quot).astype(np.float64) + z.astype(np.float64)[rows, :], 0, 15)
    return q.astype(np.uint8)


def repack(q, s, G: int):
    """Codes uint8[K][N] and scales fp16[K/G][N] -> (packed uint32[K*N/8], permuted fp16[(K/G)*N])."""
    q = np.asarray(q)
    K, N = q.shape
    _check_layout_shape(K, N)
    G = _group(K, G)
    if q.dtype != np.uint8 or q.max(initial=0) > 15:
        raise ValueError("4-bit codes must be uint8 values in 0..15")
    kk, nn = np.meshgrid(np.arange(K), np.arange(N), indexing="ij")
    word, shift = packed_position(kk, nn, K)
    nibbles = np.zeros((K * N // 8, 8), dtype=np.uint32)
    nibbles[word.ravel(), (shift // 4).ravel()] = q.ravel()
    packed = np.zeros(K * N // 8, dtype=np.uint32)
    for slot in range(8):
        packed |= nibbles[:, slot] << np.uint32(4 * slot)
    s = np.asarray(s)
    NG = K // G
    if s.shape != (NG, N):
        raise ValueError("scales must have shape [K/G][N]")
    gg, nn = np.meshgrid(np.arange(NG), np.arange(N), indexing="ij")
    sp = np.empty(NG * N, dtype=s.dtype)
    sp[scale_position(gg, nn, NG).ravel()] = s.ravel()
    return packed, sp


def unpack(packed, sp, K: int, N: int, G: int):
    """Inverse of ``repack``: (packed, permuted scales) -> (q uint8[K][N], s fp16[K/G][N])."""
    _check_layout_shape(K, N)
    G = _group(K, G)
    packed = np.asarray(packed, dtype=np.uint32)
    if packed.size != K * N // 8:
        raise ValueError("packed stream has the wrong length")
    kk, nn = np.meshgrid(np.arange(K), np.arange(N), indexing="ij")
    word, shift = packed_position(kk, nn, K)
    q = ((packed[word] >> shift.astype(np.uint32)) & np.uint32(15)).astype(np.uint8)
    NG = K // G
    sp = np.asarray(sp).ravel()
    gg, nn = np.meshgrid(np.arange(NG), np.arange(N), indexing="ij")
    s = sp[scale_position(gg, nn, NG)]
    return q, s
