"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each pin is chosen so that a plausible slip in the oracle -- a wrong zero
point, a group index taken modulo instead of by division, a transposed
operand, a mis-rounded FP16 conversion, a layout that is not a bijection --
fails at least one test here.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import w4a16_oracle as ow
from mixed_precision_w4a16_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# binary16 encoder / decoder
# --------------------------------------------------------------------------

def _golden_fp16():
    rows = []
    with open(os.path.join(GOLDEN, "fp16_binary16.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            v, b = line.split()[:2]
            rows.append((float.fromhex(v), int(b, 16)))
    return rows


def test_fp16_golden_encode():
    for v, b in _golden_fp16():
        got = int(oracle.f64_to_fp16_bits(np.array([v]))[0])
        assert got == b, (v, hex(got), hex(b))


def test_fp16_golden_decode():
    for v, b in _golden_fp16():
        back = float(oracle.fp16_bits_to_f64(np.array([b], np.uint16))[0])
        if b == 0x7C00:
            assert back == float("inf")
        elif abs(v) == 0.0 or float(np.float16(v)) == v:
            # exactly representable inputs decode to themselves (sign of zero included)
            assert back == v and np.signbit(back) == np.signbit(v)


def test_fp16_encoder_matches_numpy_cast():
    # numpy's float64 -> float16 cast is an independent implementation of the same rounding.
    rng = np.random.default_rng(123)
    mags = np.ldexp(rng.uniform(1, 2, 200000), rng.integers(-30, 17, 200000))
    x = mags * rng.choice([-1.0, 1.0], 200000)
    # add exact ties at several binades
    m = rng.integers(1024, 2048, 5000)
    e = rng.integers(-14, 15, 5000)
    ties = np.ldexp(m + 0.5, e - 10)
    x = np.concatenate([x, ties, -ties])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = oracle.f64_to_fp16_bits(x)
    assert np.array_equal(got, ref)


def test_fp16_decoder_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.fp16_bits_to_f64(bits)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


# --------------------------------------------------------------------------
# the dense product against exact integer brute force
# --------------------------------------------------------------------------

def _exact_fp16(x) -> int:
    """FP16 value as an integer multiple of 2^-24 (exact; uses Python's Fraction)."""
    f = Fraction(float(x)) * (1 << 24)
    assert f.denominator == 1
    return int(f)


def _brute_force(A, q, s, G):
    """Exact C * 2^48 and Bound * 2^48 as Python integers."""
    M, K = A.shape
    N = q.shape[1]
    a = [[_exact_fp16(A[m, k]) for k in range(K)] for m in range(M)]
    sc = [[_exact_fp16(s[g, n]) for n in range(N)] for g in range(s.shape[0])]
    C = [[0] * N for _ in range(M)]
    B = [[0] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = 0
            bnd = 0
            for k in range(K):
                # the zero point, written out: codes 0..15 stand for -8..7
                w = sc[k // G][n] * (int(q[k, n]) - 8)
                acc += a[m][k] * w
                bnd += abs(a[m][k] * w)
            C[m][n] = acc
            B[m][n] = bnd
    return C, B


@pytest.mark.parametrize("M,K,N,G", [(1, 128, 16, 128), (3, 256, 32, 128), (4, 256, 16, 256), (2, 192, 16, 64)])
def test_gemm_matches_exact_brute_force(M, K, N, G):
    q, s = synth.make_weights(K, N, G, seed=7 + K + N)
    A = synth.make_activations(M, K, seed=11 + M)
    C, bound = oracle.gemm_ref(A, q, s, G)
    Ce, Be = _brute_force(A, q, s, G)
    scale = 2.0 ** -48
    for m in range(M):
        for n in range(N):
            exact = Ce[m][n] * scale
            ebound = Be[m][n] * scale
            assert abs(C[m, n] - exact) <= K * 2.0 ** -52 * ebound + 1e-300, (m, n)
            assert abs(bound[m, n] - ebound) <= K * 2.0 ** -52 * ebound + 1e-300, (m, n)


def test_planted_zero_point_mistake_is_caught(monkeypatch):
    # A wrong zero point planted in the oracle must fail the brute-force pin.
    M, K, N, G = 2, 128, 16, 128
    q, s = synth.make_weights(K, N, G, seed=5)
    A = synth.make_activations(M, K, seed=6)
    monkeypatch.setattr(ow, "Z_POINT", 7)
    C, _ = oracle.gemm_ref(A, q, s, G)
    Ce, Be = _brute_force(A, q, s, G)
    worst = max(abs(C[m, n] - Ce[m][n] * 2.0 ** -48) / (Be[m][n] * 2.0 ** -48)
                for m in range(M) for n in range(N))
    assert worst > 1e-3


# --------------------------------------------------------------------------
# closed forms and special cases
# --------------------------------------------------------------------------

def test_zero_codes_give_exact_zero():
    K, N, G = 256, 32, 128
    _, s = synth.make_weights(K, N, G, seed=1)
    q = np.full((K, N), 8, np.uint8)
    A = synth.make_activations(5, K, seed=2)
    C, bound = oracle.gemm_ref(A, q, s, G)
    assert np.all(C == 0.0) and np.all(bound == 0.0)


def test_identity_rows_return_dequantised_rows():
    K, N, G = 256, 48, 128
    q, s = synth.make_weights(K, N, G, seed=3)
    rows = [0, 5, 127, 128, 200, 255]
    A = np.zeros((len(rows), K), np.float16)
    for m, k in enumerate(rows):
        A[m, k] = 1.0
    C, _ = oracle.gemm_ref(A, q, s, G)
    Bh = oracle.dequant_exact(q, s, G)
    assert np.array_equal(C, Bh[rows, :])
    # the FP16 dequantised weight is one RNE rounding of the exact value
    assert np.array_equal(oracle.f64_to_fp16_bits(C), oracle.dequant_fp16_bits(q, s, G)[rows, :])


def test_groups_are_consecutive_rows():
    # "one scale per G consecutive weights in each column": codes 9 (value +1) in the first
    # group only and zero elsewhere give C = G * s[0, n] for an all-ones activation row;
    # codes 9 everywhere give G * sum_g s[g, n].
    K, N, G = 512, 32, 128
    _, s = synth.make_weights(K, N, G, seed=4)
    s64 = s.astype(np.float64)
    A = np.ones((1, K), np.float16)
    q = np.full((K, N), 8, np.uint8)
    q[:G, :] = 9
    C, _ = oracle.gemm_ref(A, q, s, G)
    assert np.array_equal(C[0], G * s64[0])
    q[:, :] = 9
    C, _ = oracle.gemm_ref(A, q, s, G)
    assert np.allclose(C[0], G * s64.sum(axis=0), rtol=1e-15, atol=0)
    q[:, :] = 0  # value -8
    C, _ = oracle.gemm_ref(A, q, s, G)
    assert np.allclose(C[0], -8 * G * s64.sum(axis=0), rtol=1e-15, atol=0)


def test_per_column_mode_is_diag_scaling():
    # group = K: AB = (A Q) diag(s), Q = q - 8 (integer matrix)
    M, K, N = 3, 256, 32
    q, s = synth.make_weights(K, N, -1, seed=8)
    A = synth.make_activations(M, K, seed=9)
    C, _ = oracle.gemm_ref(A, q, s, -1)
    AQ = A.astype(np.float64) @ (q.astype(np.float64) - 8.0)
    assert np.allclose(C, AQ * s.astype(np.float64)[0], rtol=1e-13, atol=1e-13)


def test_integer_gemm_textbook():
    # s = 1 and small integer activations: C is an integer GEMM, computed here in int64.
    rng = np.random.default_rng(10)
    M, K, N, G = 4, 256, 64, 128
    Ai = rng.integers(-4, 5, (M, K))
    q = rng.integers(0, 16, (K, N)).astype(np.uint8)
    s = np.ones((K // G, N), np.float16)
    C, _ = oracle.gemm_ref(Ai.astype(np.float16), q, s, G)
    ref = Ai.astype(np.int64) @ (q.astype(np.int64) - 8)
    assert np.array_equal(C, ref.astype(np.float64))


def test_error_bound_semantics():
    C_ref = np.array([[1.0, -2.0]])
    bound = np.array([[10.0, 0.0]])
    ok = np.array([[1.0 + 4e-2, -2.0 + 1e-4]])
    bad = np.array([[1.0 + 4.1e-2, -2.0]])
    assert oracle.error_ok(ok, C_ref, bound)
    assert not oracle.error_ok(bad, C_ref, bound)
    assert not oracle.error_ok(np.array([[np.nan, -2.0]]), C_ref, bound)


def test_code_range_rejected():
    q = np.full((128, 128), 16, np.uint8)
    s = np.ones((1, 128), np.float16)
    with pytest.raises(ValueError):
        oracle.dequant_exact(q, s, 128)
    with pytest.raises(ValueError):
        oracle.repack(q, s, 128)


# --------------------------------------------------------------------------
# packed layout
# --------------------------------------------------------------------------

# PTX ISA, "Matrix Fragments for mma.m16n8k16 with floating point type": the A operand
# (16 x 16, .f16) is four .f16x2 registers per lane; with groupID = lane / 4 and
# tig = lane % 4 the eight elements a0..a7 sit at (row, col):
ISA_A_FRAGMENT = {
    0: (0, 0), 1: (0, 1),      # a0, a1: (groupID,     2*tig + {0,1})
    2: (8, 0), 3: (8, 1),      # a2, a3: (groupID + 8, 2*tig + {0,1})
    4: (0, 8), 5: (0, 9),      # a4, a5: (groupID,     2*tig + 8 + {0,1})
    6: (8, 8), 7: (8, 9),      # a6, a7: (groupID + 8, 2*tig + 8 + {0,1})
}
# The layout stores, in the lane/register the ISA assigns to fragment column 2*tig + e
# (resp. 2*tig + 8 + e), the weight of reduction index 4*tig + e (resp. 4*tig + 2 + e).
def PERM_K(tig, col_offset):
    return 4 * tig + (2 if col_offset >= 8 else 0) + (col_offset % 2)

# PTX ISA, tcgen05 "Matrix fragments for .16x256b": four 32-bit registers per thread,
# (lane groupID, column 2*tig), (lane groupID, column 2*tig + 1), (lane groupID + 8,
# column 2*tig), (lane groupID + 8, column 2*tig + 1); a 32-bit column holds two FP16 k.
TMEM_16x256b = [(0, 0), (0, 1), (8, 0), (8, 1)]


def test_packed_layout_is_the_permuted_isa_fragment():
    K = 64
    for lane in range(32):
        g, t = lane // 4, lane % 4
        for p, (dr, dc) in ISA_A_FRAGMENT.items():
            for j in range(4):
                for nb in range(8):
                    n = nb * 16 + g + dr
                    k = 16 * j + PERM_K(t, dc)
                    word, shift = oracle.packed_position(k, n, K)
                    reg, half = p // 2, p % 2
                    # register `reg` = (low half, high half) = (a_{2reg}, a_{2reg+1}); slot = reg + 4*half
                    assert int(word) == (nb * 32 + lane) * 4 + j
                    assert int(shift) == 4 * (reg + 4 * half)


def test_packed_words_are_tensor_memory_store_fragments():
    # register order (r0, r2, r1, r3) of a word is the .16x256b fragment: row g / g+8, columns 2t / 2t+1,
    # column c holding k = 2c, 2c + 1 of the 16x16 block
    K = 64
    for lane in range(32):
        g, t = lane // 4, lane % 4
        for frag_reg, (dr, dcol) in enumerate(TMEM_16x256b):
            reg = [0, 2, 1, 3][frag_reg]
            for e in range(2):
                n = g + dr
                k = 2 * (2 * t + dcol) + e
                word, shift = oracle.packed_position(k, n, K)
                assert int(word) == lane * 4 and int(shift) == 4 * (reg + 4 * e)


def test_packed_layout_is_a_bijection():
    K, N = 256, 384
    kk, nn = np.meshgrid(np.arange(K), np.arange(N), indexing="ij")
    word, shift = oracle.packed_position(kk, nn, K)
    code = word * 8 + shift // 4
    assert np.array_equal(np.sort(code.ravel()), np.arange(K * N))


def test_16x64_tiles_are_contiguous_and_vectors_span_four_blocks():
    # 16 x 64 tiles are stored contiguously (512 bytes); each lane's 16-byte vector
    # carries codes from four distinct 16 x 16 blocks.
    K, N = 256, 256
    kk, nn = np.meshgrid(np.arange(K), np.arange(N), indexing="ij")
    word, _ = oracle.packed_position(kk, nn, K)
    tile = ((nn // 128) * (K // 64) + kk // 64) * 8 + (nn % 128) // 16
    for t in np.unique(tile):
        w = np.unique(word[tile == t])
        assert w.size == 128 and w[-1] - w[0] == 127 and w[0] == t * 128
    vec = word // 4
    blk = (kk // 16) * 1000 + nn // 16
    for v in np.unique(vec)[:64]:
        assert np.unique(blk[vec == v]).size == 4


def test_strips_are_contiguous_along_k():
    # a 128-column strip x any run of 64-row blocks is one contiguous range of the stream
    K, N = 512, 384
    for strip in range(N // 128):
        for kb0, kb1 in [(0, 8), (2, 6), (4, 8)]:
            kk, nn = np.meshgrid(np.arange(64 * kb0, 64 * kb1), np.arange(128 * strip, 128 * strip + 128), indexing="ij")
            w, _ = oracle.packed_position(kk, nn, K)
            lo, hi = int(w.min()), int(w.max())
            assert hi - lo + 1 == (kb1 - kb0) * 8 * 128 and np.unique(w).size == hi - lo + 1
            assert lo == (strip * (K // 64) + kb0) * 1024


def test_scale_position_pairs_rows_r_and_r_plus_8():
    NG, N = 3, 256
    gg, nn = np.meshgrid(np.arange(NG), np.arange(N), indexing="ij")
    p = oracle.scale_position(gg, nn, NG)
    assert np.array_equal(np.sort(p.ravel()), np.arange(NG * N))
    for g in range(NG):
        for r in range(8):
            assert p[g, r + 8] == p[g, r] + 1 and p[g, r] % 2 == 0
    # a strip's NG scale rows are one contiguous block of NG * 128 entries
    for strip in range(N // 128):
        blk = p[:, strip * 128:(strip + 1) * 128]
        assert blk.min() == strip * NG * 128 and blk.max() == (strip + 1) * NG * 128 - 1


@pytest.mark.parametrize("K,N,G", [(128, 128, 128), (256, 256, 128), (512, 384, -1), (1024, 128, 128)])
def test_repack_unpack_round_trip(K, N, G):
    q, s = synth.make_weights(K, N, G, seed=K + N)
    packed, sp = oracle.repack(q, s, G)
    assert packed.dtype == np.uint32 and packed.size == K * N // 8
    q2, s2 = oracle.unpack(packed, sp, K, N, G)
    assert np.array_equal(q2, q)
    assert np.array_equal(np.asarray(s2).view(np.uint16), s.view(np.uint16))


def test_repack_word_decodes_to_fragment_values():
    # Decoding one word by its nibble slots must give the lane's eight A-fragment codes.
    K, N, G = 64, 128, 64
    q, s = synth.make_weights(K, N, G, seed=21)
    packed, _ = oracle.repack(q, s, G)
    for lane in range(32):
        g, t = lane // 4, lane % 4
        for j in range(4):
            w = int(packed[lane * 4 + j])
            for p, (dr, dc) in ISA_A_FRAGMENT.items():
                slot = p // 2 + 4 * (p % 2)
                assert (w >> (4 * slot)) & 15 == q[16 * j + PERM_K(t, dc), g + dr]


# ---------------------------------------------------------------------------
# quantise (the Layer.pack step: divide by the scale, round, add 8, clamp)
# ---------------------------------------------------------------------------

def _f32_round_exact(fr: Fraction) -> Fraction:
    """The float32 nearest to an exact rational (ties to even), found by exact
    comparison with the neighbouring float32 values -- independent of any
    floating-point division."""
    x = np.float32(float(fr))  # within one float32 ulp of the answer
    cands = {np.nextafter(x, np.float32(-np.inf)), x, np.nextafter(x, np.float32(np.inf))}
    best = None
    for c in sorted(cands, key=float):
        d = abs(Fraction(float(c)) - fr)
        if best is None or d < best[0] or (d == best[0] and (int(np.float32(c).view(np.uint32)) & 1) == 0):
            best = (d, c)
    return Fraction(float(best[1]))


def _round_half_even(fr: Fraction) -> int:
    f = fr.numerator // fr.denominator
    rem = fr - f
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and f % 2 == 1):
        return f + 1
    return f


def _h(values):
    return np.asarray(values, dtype=np.float16)


def test_quantize_matches_exact_rational_arithmetic():
    """Every code equals clamp(round_half_even(f32(w / s)) + 8), computed with exact
    rationals and an independent float32 rounding (pins the division precision,
    the rounding, the offset and the clamp)."""
    rng = np.random.default_rng(31)
    K, N, G = 256, 16, 128
    s = _h(rng.uniform(0.002, 0.05, (K // G, N)) * rng.choice([-1, 1], (K // G, N)))
    w = _h(rng.normal(0, 0.15, (K, N)))
    q = oracle.quantize(w, s, G)
    for k in range(K):
        for n in range(N):
            fr = Fraction(float(w[k, n])) / Fraction(float(s[k // G, n]))
            want = min(max(_round_half_even(_f32_round_exact(fr)) + 8, 0), 15)
            assert q[k, n] == want, (k, n, float(w[k, n]), float(s[k // G, n]))


@pytest.mark.parametrize("G", [128, -1])
def test_quantize_inverts_dequantisation(G):
    """quantise(RNE(s (q - 8)), s) == q for every code, positive and negative scales."""
    rng = np.random.default_rng(32)
    K, N = 256, 64
    NG = 2 if G == 128 else 1
    q = np.tile(np.arange(16, dtype=np.uint8), K * N // 16).reshape(K, N)
    rng.shuffle(q.ravel())
    s = _h(rng.uniform(0.001, 3.0, (NG, N)) * rng.choice([-1, 1], (NG, N)))
    w = oracle.dequant_fp16_bits(q, s, G).view(np.float16)
    assert np.array_equal(oracle.quantize(w, s, G), q)


def test_quantize_ties_round_to_even_and_clamp():
    w = _h([[0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, -3.5, 7.5, -8.5, 8.0, -9.0, 7.0, -8.0, 1000.0, -1000.0]])
    s = _h(np.ones((1, 16)))
    want = [8, 10, 10, 12, 8, 6, 6, 4, 15, 0, 15, 0, 15, 0, 15, 0]
    assert oracle.quantize(w, s, 1).ravel().tolist() == want
    # the same ties with a scale of 0.25 and the weights scaled by it (all exact)
    assert oracle.quantize(_h(w.astype(np.float64) * 0.25), _h(np.full((1, 16), 0.25)), 1).ravel().tolist() == want


def test_quantize_rejects_non_finite_quotients():
    w = _h(np.ones((128, 1)))
    with pytest.raises(ValueError):
        oracle.quantize(w, _h(np.zeros((1, 1))), 128)
    with pytest.raises(ValueError):
        oracle.quantize(_h(np.full((128, 1), np.inf)), _h(np.ones((1, 1))), 128)


# ---------------------------------------------------------------------------
# zero points and bias
# ---------------------------------------------------------------------------

def _brute_force_zp(A, q, s, z, bias, G):
    """Exact (C - bias) * 2^48 and Bound * 2^48 as Python integers, zero points written out."""
    M, K = A.shape
    N = q.shape[1]
    a = [[_exact_fp16(A[m, k]) for k in range(K)] for m in range(M)]
    sc = [[_exact_fp16(s[g, n]) for n in range(N)] for g in range(s.shape[0])]
    C = [[0] * N for _ in range(M)]
    B = [[0] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = bnd = 0
            for k in range(K):
                wv = sc[k // G][n] * (int(q[k, n]) - int(z[k // G, n]))
                acc += a[m][k] * wv
                bnd += abs(a[m][k] * wv)
            C[m][n] = acc
            B[m][n] = bnd
    return C, B


def _zp_inputs(K, N, G, seed):
    rng = np.random.default_rng(seed)
    q, s = synth.make_weights(K, N, G, seed=seed)
    z = rng.integers(0, 16, (K // synth.effective_group(K, G), N)).astype(np.uint8)
    bias = rng.normal(0, 1.0, N).astype(np.float16)
    return q, s, z, bias


@pytest.mark.parametrize("M,K,N,G", [(1, 128, 16, 128), (3, 256, 16, 128), (2, 256, 16, 256)])
def test_gemm_zp_matches_exact_brute_force(M, K, N, G):
    q, s, z, bias = _zp_inputs(K, N, G, 40 + K)
    A = synth.make_activations(M, K, seed=41 + M)
    C, bound = oracle.gemm_ref_zp(A, q, s, z, bias, G)
    Ce, Be = _brute_force_zp(A, q, s, z, bias, G)
    for m in range(M):
        for n in range(N):
            exact = Ce[m][n] * 2.0 ** -48 + float(bias[n])
            ebound = Be[m][n] * 2.0 ** -48 + abs(float(bias[n]))
            assert abs(C[m, n] - exact) <= K * 2.0 ** -52 * ebound + 1e-300, (m, n)
            assert abs(bound[m, n] - ebound) <= K * 2.0 ** -52 * ebound + 1e-300, (m, n)


def test_planted_zero_point_row_mistake_is_caught(monkeypatch):
    # using the zero point of the next group (a wrong group index for z) must fail the brute force
    M, K, N, G = 2, 256, 16, 128
    q, s, z, bias = _zp_inputs(K, N, G, 50)
    A = synth.make_activations(M, K, seed=51)
    real = ow.dequant_exact_zp
    monkeypatch.setattr(ow, "dequant_exact_zp", lambda q_, s_, z_, G_: real(q_, s_, np.roll(z_, 1, axis=0), G_))
    C, _ = oracle.gemm_ref_zp(A, q, s, z, None, G)
    Ce, Be = _brute_force_zp(A, q, s, z, None, G)
    worst = max(abs(C[m, n] - Ce[m][n] * 2.0 ** -48) / (Be[m][n] * 2.0 ** -48 + 1e-30)
                for m in range(M) for n in range(N))
    assert worst > 1e-3


def test_zero_point_eight_is_the_symmetric_layer():
    K, N, G = 256, 32, 128
    q, s = synth.make_weights(K, N, G, seed=60)
    A = synth.make_activations(3, K, seed=61)
    z8 = np.full((K // G, N), 8, np.uint8)
    C0, B0 = oracle.gemm_ref(A, q, s, G)
    C1, B1 = oracle.gemm_ref_zp(A, q, s, z8, None, G)
    assert np.array_equal(C0, C1) and np.array_equal(B0, B1)


def test_codes_equal_to_zero_points_give_the_bias():
    K, N, G = 256, 32, 128
    _, s, z, bias = _zp_inputs(K, N, G, 62)
    q = np.repeat(z, G, axis=0)
    A = synth.make_activations(4, K, seed=63)
    C, bound = oracle.gemm_ref_zp(A, q, s, z, bias, G)
    assert np.array_equal(C, np.tile(bias.astype(np.float64), (4, 1)))
    assert np.array_equal(bound, np.tile(np.abs(bias.astype(np.float64)), (4, 1)))


def test_identity_rows_with_zero_points():
    K, N, G = 256, 48, 128
    q, s, z, _ = _zp_inputs(K, N, G, 64)
    rows = [0, 127, 128, 255]
    A = np.zeros((len(rows), K), np.float16)
    for m, k in enumerate(rows):
        A[m, k] = 1.0
    C, _ = oracle.gemm_ref_zp(A, q, s, z, None, G)
    # the rows of s (q - z), written out per element
    for m, k in enumerate(rows):
        want = np.array([float(s[k // G, n]) * (int(q[k, n]) - int(z[k // G, n])) for n in range(N)])
        assert np.array_equal(C[m], want)


def test_integer_gemm_with_zero_points_textbook():
    rng = np.random.default_rng(65)
    M, K, N, G = 3, 256, 32, 128
    Ai = rng.integers(-4, 5, (M, K))
    q = rng.integers(0, 16, (K, N)).astype(np.uint8)
    z = rng.integers(0, 16, (K // G, N)).astype(np.uint8)
    s = np.ones((K // G, N), np.float16)
    C, _ = oracle.gemm_ref_zp(Ai.astype(np.float16), q, s, z, None, G)
    ref = Ai.astype(np.int64) @ (q.astype(np.int64) - np.repeat(z.astype(np.int64), G, axis=0))
    assert np.array_equal(C, ref.astype(np.float64))


def test_repack_zeros_follows_the_scale_permutation():
    K, N, G = 512, 256, 128
    _, s, z, _ = _zp_inputs(K, N, G, 66)
    _, sp = oracle.repack(np.zeros((K, N), np.uint8), s, G)
    zp = oracle.repack_zeros(z, G, K)
    # wherever the scale of (g, n) went, its zero point went too
    for g in range(K // G):
        for n in (0, 7, 8, 15, 16, 127, 128, 255):
            i = int(oracle.scale_position(g, n, K // G))
            assert sp[i] == s[g, n] and zp[i] == z[g, n]


# ---------------------------------------------------------------------------
# min-max scale rule (MARLIN paper, Section 2.2, "Weight Quantization")
# ---------------------------------------------------------------------------

def _fp16_is_nearest(h: np.float16, x: Fraction) -> bool:
    """h is an FP16 value nearest to x (its FP16 neighbours are not closer)."""
    d = abs(Fraction(float(h)) - x)
    for nb in (np.nextafter(h, np.float16(-np.inf)), np.nextafter(h, np.float16(np.inf))):
        if np.isfinite(nb) and abs(Fraction(float(nb)) - x) < d:
            return False
    return True


def _minmax_groups(rng, G, N):
    """Weights [2G][N]: groups of mixed sign, all positive, all negative, tiny and wide ranges."""
    w = rng.normal(0, 0.05, (2 * G, N))
    w[:, 1] = np.abs(w[:, 1]) + 0.01          # all positive
    w[:, 2] = -np.abs(w[:, 2]) - 0.02         # all negative
    w[:, 3] *= 1e-4                           # small range (subnormal FP16 scale)
    w[:, 4] *= 300.0                          # wide range
    w[:G, 5] = 0.0                            # one all-zero group
    return _h(w)


@pytest.mark.parametrize("symmetric", [True, False])
def test_minmax_scales_match_exact_rational_arithmetic(symmetric):
    """Each scale is the FP16 nearest to f32(f32(span) / 15), span = hi - lo (or 2 max|v|), and each zero
    code is clamp(round_half_even(f32(-lo / s)), 0, 15), all computed with exact rationals (pins the
    divisor 2^4 - 1, the widened range, the symmetric range and the zero code's rounding)."""
    rng = np.random.default_rng(71)
    G, N = 128, 12
    w = _minmax_groups(rng, G, N)
    s, z = oracle.minmax_scales(w, G, symmetric=symmetric)
    assert s.dtype == np.float16 and s.shape == (2, N)
    assert (z is None) == symmetric
    for g in range(2):
        for n in range(N):
            v = [Fraction(float(x)) for x in w[g * G:(g + 1) * G, n]]
            if symmetric:
                span = 2 * max(abs(min(v)), abs(max(v)))
            else:
                lo, hi = min(min(v), Fraction(0)), max(max(v), Fraction(0))
                span = _f32_round_exact(hi - lo)
            s32 = _f32_round_exact(span / 15)
            if s32 <= Fraction(1, 2 ** 25):               # rounds to FP16 zero: s = 1
                assert float(s[g, n]) == 1.0, (g, n)
            else:
                assert _fp16_is_nearest(s[g, n], s32), (g, n, float(s[g, n]), float(s32))
            if not symmetric:
                zq = _f32_round_exact(-lo / Fraction(float(s[g, n])))
                assert z[g, n] == min(max(_round_half_even(zq), 0), 15), (g, n)


def test_minmax_zero_range_group_takes_unit_scale():
    w = _h(np.zeros((256, 2)))
    w[128:, 1] = 0.25
    s, z = oracle.minmax_scales(w, 128, symmetric=False)
    assert float(s[0, 0]) == 1.0 and z[0, 0] == 0
    assert np.all(oracle.dequant_exact_zp(oracle.quantize_zp(w, s, z, 128), s, z, 128)[:128] == 0.0)
    s, _ = oracle.minmax_scales(w, 128, symmetric=True)
    assert float(s[0, 0]) == 1.0 and np.all(oracle.quantize(w, s, 128)[:128] == 8)


def test_minmax_exact_grid_is_reproduced():
    """Weights on the grid c*k: asymmetric k in -7..8 gives s = c, z = 7; symmetric k in -7..7 with
    one weight 7.5c gives s = c (both exact), and every grid weight comes back exactly."""
    c = 2.0 ** -6
    ks = np.array(list(range(-7, 9)) * 8, dtype=np.float64)        # 128 rows, each k 8 times
    w = _h((c * ks).reshape(128, 1))
    s, z = oracle.minmax_scales(w, 128, symmetric=False)
    assert float(s[0, 0]) == c and z[0, 0] == 7
    q = oracle.quantize_zp(w, s, z, 128)
    assert np.array_equal(q.ravel(), (ks + 7).astype(np.uint8))
    assert np.array_equal(oracle.dequant_exact_zp(q, s, z, 128), w.astype(np.float64))
    ks2 = np.array((list(range(-7, 8)) * 9)[:127] + [7.5])
    w2 = _h((c * ks2).reshape(128, 1))
    s2, _ = oracle.minmax_scales(w2, 128, symmetric=True)
    assert float(s2[0, 0]) == c
    q2 = oracle.quantize(w2, s2, 128)
    assert np.array_equal(q2.ravel()[:127], (ks2[:127] + 8).astype(np.uint8))
    assert q2[127, 0] == 15                          # 7.5 rounds to 8 (even), clamped: error c/2


@pytest.mark.parametrize("symmetric", [True, False])
def test_minmax_reconstruction_error_bound(symmetric):
    """The point of the rule: every weight is reproduced within half a step where its code is not
    clamped (exactly, by the tie argument), and within a step anywhere; the group minimum gets code 0
    (asymmetric, lo < 0) and the maximum a code >= 14."""
    rng = np.random.default_rng(72)
    G, N = 128, 64
    w = _minmax_groups(rng, G, N)
    w64 = w.astype(np.float64)
    s, z = oracle.minmax_scales(w, G, symmetric=symmetric)
    if symmetric:
        q = oracle.quantize(w, s, G)
        Bh = oracle.dequant_exact(q, s, G)
        zz = np.full(s.shape, 8)
    else:
        q = oracle.quantize_zp(w, s, z, G)
        Bh = oracle.dequant_exact_zp(q, s, z, G)
        zz = z.astype(np.int64)
    step = np.repeat(s.astype(np.float64), G, axis=0)
    err = np.abs(Bh - w64)
    inner = (q > 0) & (q < 15)
    assert np.all(err[inner] <= step[inner] / 2)
    lim = (0.5 * (1 + 14 * 2.0 ** -10)) if symmetric else 1.0
    assert np.all(err <= lim * step * (1 + 2.0 ** -10) + 2.0 ** -24)
    if not symmetric:
        for g in range(2):
            blk, zq = w64[g * G:(g + 1) * G], zz[g]
            for n in range(N):
                col = blk[:, n]
                if col.min() < 0 and zq[n] < 15:
                    assert q[g * G + int(np.argmin(col)), n] == 0, (g, n)
                if col.max() > 0:
                    assert q[g * G + int(np.argmax(col)), n] >= 14, (g, n)


def test_minmax_rejects_non_finite_weights():
    w = _h(np.ones((128, 2)))
    w[5, 1] = np.inf
    for sym in (True, False):
        with pytest.raises(ValueError):
            oracle.minmax_scales(w, 128, symmetric=sym)


def test_quantize_zp_matches_exact_rational_arithmetic():
    rng = np.random.default_rng(73)
    K, N, G = 256, 8, 128
    s = _h(rng.uniform(0.002, 0.05, (K // G, N)))
    z = rng.integers(0, 16, (K // G, N)).astype(np.uint8)
    w = _h(rng.normal(0, 0.15, (K, N)))
    q = oracle.quantize_zp(w, s, z, G)
    for k in range(K):
        for n in range(N):
            fr = Fraction(float(w[k, n])) / Fraction(float(s[k // G, n]))
            want = min(max(_round_half_even(_f32_round_exact(fr)) + int(z[k // G, n]), 0), 15)
            assert q[k, n] == want, (k, n)
    # z = 8 everywhere is the symmetric quantiser
    z8 = np.full((K // G, N), 8, np.uint8)
    assert np.array_equal(oracle.quantize_zp(w, s, z8, G), oracle.quantize(w, s, G))


# ---------------------------------------------------------------------------
# grouped expert GEMM
# ---------------------------------------------------------------------------

def test_moe_gemm_integer_brute_force():
    """Integer activations and unit scales: every row is its own expert's integer product, the owner found
    by a binary search of the offsets (independent of the oracle's slicing); pins the row ownership at
    every boundary, empty experts and the per-expert weights."""
    rng = np.random.default_rng(81)
    K, N, G = 256, 16, 128
    off = np.array([0, 3, 3, 4, 9, 9, 12])            # experts 1 and 4 own no rows
    E, M = off.size - 1, int(off[-1])
    A = rng.integers(-3, 4, (M, K))
    q = rng.integers(0, 16, (E, K, N)).astype(np.uint8)
    s = np.ones((E, K // G, N), np.float16)
    C, bound = oracle.moe_gemm_ref(A.astype(np.float16), off, q, s, G)
    for m in range(M):
        e = int(np.searchsorted(off, m, side="right")) - 1
        want = A[m].astype(np.int64) @ (q[e].astype(np.int64) - 8)
        assert np.array_equal(C[m], want.astype(np.float64)), m
        assert np.array_equal(bound[m], (np.abs(A[m]).astype(np.int64) @ np.abs(q[e].astype(np.int64) - 8)))


def test_moe_gemm_with_one_shared_weight_is_the_dense_product():
    rng = np.random.default_rng(82)
    K, N, G, E = 256, 32, 128, 5
    q1, s1 = synth.make_weights(K, N, G, seed=83)
    A = synth.make_activations(20, K, seed=84)
    off = np.array([0, 2, 2, 11, 19, 20])
    C, bound = oracle.moe_gemm_ref(A, off, np.stack([q1] * E), np.stack([s1] * E), G)
    C_d, bound_d = oracle.gemm_ref(A, q1, s1, G)
    assert np.array_equal(C, C_d) and np.array_equal(bound, bound_d)


def test_moe_gemm_rejects_bad_offsets():
    K, N, G = 128, 8, 128
    q = np.zeros((2, K, N), np.uint8)
    s = np.ones((2, 1, N), np.float16)
    A = np.zeros((4, K), np.float16)
    for off in ([1, 2, 4], [0, 3, 2], [0, 2, 5], [0, 4]):
        with pytest.raises(ValueError):
            oracle.moe_gemm_ref(A, off, q, s, G)


# ---------------------------------------------------------------------------
# 2:4 structured sparsity
# ---------------------------------------------------------------------------

def test_sparse24_compress_keeps_the_nonzero_positions_in_order():
    q = np.full((8, 3), 8, np.uint8)
    q[0:4, 0] = [3, 8, 8, 12]       # positions 0 and 3
    q[4:8, 0] = [8, 5, 8, 8]        # one non-zero at 1: filled up with 0 -> (0, 1)
    q[0:4, 1] = [8, 8, 8, 8]        # none: (0, 1)
    q[4:8, 1] = [8, 8, 9, 1]        # (2, 3)
    q[0:4, 2] = [8, 8, 0, 8]        # one at 2: filled with 0 -> (0, 2)
    q[4:8, 2] = [15, 8, 8, 8]       # one at 0: filled with 1 -> (0, 1)
    qc, idx = oracle.sparse24_compress(q)
    assert idx[:, 0].tolist() == [0, 3, 0, 1] and qc[:, 0].tolist() == [3, 12, 8, 5]
    assert idx[:, 1].tolist() == [0, 1, 2, 3] and qc[:, 1].tolist() == [8, 8, 9, 1]
    assert idx[:, 2].tolist() == [0, 2, 0, 1] and qc[:, 2].tolist() == [8, 0, 15, 8]


def test_sparse24_round_trip_and_structure():
    q, _ = synth.make_weights_24(256, 64, 128, seed=41)
    # the generator's structure: at most two codes != 8 in every group of four
    assert np.all((q.reshape(64, 4, 64) != 8).sum(axis=1) <= 2)
    qc, idx = oracle.sparse24_compress(q)
    assert np.all(idx[0::2] < idx[1::2]) and idx.max() <= 3
    assert np.array_equal(oracle.sparse24_expand(qc, idx), q)


def test_sparse24_rejects_three_nonzeros_and_bad_positions():
    q = np.full((4, 1), 8, np.uint8)
    q[:3, 0] = [1, 2, 3]
    with pytest.raises(ValueError):
        oracle.sparse24_compress(q)
    with pytest.raises(ValueError):
        oracle.sparse24_expand(np.zeros((2, 1), np.uint8), np.array([[2], [1]], np.uint8))


def test_gemm24_integer_brute_force_over_kept_entries():
    """C = sum over groups and kept entries of A[m, 4i + idx] (qc - 8): the sparse sum written out,
    against the oracle's dense product of the expanded codes (pins the position arithmetic)."""
    rng = np.random.default_rng(42)
    M, K, N, G = 3, 128, 8, 128
    q, _ = synth.make_weights_24(K, N, G, seed=43)
    qc, idx = oracle.sparse24_compress(q)
    Ai = rng.integers(-4, 5, (M, K))
    C, _ = oracle.gemm24_ref(Ai.astype(np.float16), qc, idx, np.ones((1, N), np.float16), G)
    for m in range(M):
        for n in range(N):
            want = sum(int(Ai[m, 4 * (j // 2) + int(idx[j, n])]) * (int(qc[j, n]) - 8) for j in range(K // 2))
            assert C[m, n] == want, (m, n)
