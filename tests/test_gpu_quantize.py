"""The offline quantiser on the GPU against the CPU oracle (byte exact): fused
quantise + repack from FP16 weights, q = clamp(rint(w / s) + 8, 0, 15) (or + z)
in the packed layout, and the min-max scales and zero codes in front of it."""
import numpy as np
import pytest

import oracle
from mixed_precision_w4a16_gb300 import synth
import w4a16_testlib as tl

pytestmark = pytest.mark.gpu

SHAPES = [(128, 128, 128), (256, 384, 128), (1024, 1024, 128), (512, 384, -1), (4096, 512, 128),
          (11008, 256, 128), (1024, 640, 1024)]


@pytest.fixture(scope="module")
def w():
    return tl.lib()


def _quantize_on_device(w, wt, s, G):
    torch = tl.torch_mod()
    packed, sp = w.quantize_repack(tl.to_dev(wt), tl.to_dev(s), G)
    torch.cuda.synchronize()
    return packed.cpu().numpy().view(np.uint32), sp.cpu().numpy().view(np.uint16).ravel()


@pytest.mark.parametrize("K,N,G", SHAPES)
@pytest.mark.parametrize("signed", [False, True])
def test_quantize_repack_matches_oracle_bytes(w, K, N, G, signed):
    wt, s = synth.make_fp16_weights(K, N, G, seed=K + 5 * N, signed_scales=signed)
    got_packed, got_sp = _quantize_on_device(w, wt, s, G)
    ref_packed, ref_sp = oracle.repack(oracle.quantize(wt, s, G), s, G)
    assert np.array_equal(got_packed, ref_packed)
    assert np.array_equal(got_sp, ref_sp.view(np.uint16))
    assert w.w4a16_get_status() == 0


def test_quantize_ties_and_clamps(w):
    """Exact half-integer quotients round to even; out-of-range quotients clamp."""
    K, N = 128, 128
    vals = np.array([0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, -3.5, 7.5, -8.5, 8.0, -9.0, 7.0, -8.0, 1000.0, -1000.0])
    wt = np.tile(vals, K * N // 16).reshape(K, N)
    for scale in (1.0, 0.25):
        wts = (wt * scale).astype(np.float16)
        s = np.full((1, N), scale, dtype=np.float16)
        got_packed, _ = _quantize_on_device(w, wts, s, -1)
        want = np.tile(np.array([8, 10, 10, 12, 8, 6, 6, 4, 15, 0, 15, 0, 15, 0, 15, 0], np.uint8), K * N // 16)
        assert np.array_equal(got_packed, oracle.repack(want.reshape(K, N), s, -1)[0])


@pytest.mark.parametrize("K,N,G", [(1024, 512, 128), (512, 384, -1)])
def test_quantize_of_dequantised_weights_recovers_packed_stream(w, K, N, G):
    """quantise_repack(dequant(packed)) == packed: the device round trip through FP16 weights."""
    q, s = synth.make_weights(K, N, G, seed=77 + K)
    _, s_d, packed, sp = tl.device_layer(w, q, s, G)
    bhat = w.dequant(packed, sp, K, N, G)
    packed2, sp2 = w.quantize_repack(bhat, s_d, G)
    tl.torch_mod().cuda.synchronize()
    assert np.array_equal(packed2.cpu().numpy(), packed.cpu().numpy())
    assert np.array_equal(sp2.cpu().numpy(), sp.cpu().numpy())


def test_zero_scale_is_reported_and_cleared(w):
    K, N, G = 256, 128, 128
    wt, s = synth.make_fp16_weights(K, N, G, seed=5)
    s[1, 7] = 0.0
    got_packed, _ = _quantize_on_device(w, wt, s, G)
    assert w.w4a16_get_status() == 10  # W4A16_ERR_VALUE
    assert w.w4a16_get_status() == 0   # read and cleared
    # every other code is still the oracle's; the column with the zero scale stores code 8 there
    s_ok = s.copy()
    s_ok[1, 7] = 1.0
    ref_q = oracle.quantize(wt, s_ok, G)
    ref_q[128:256, 7] = 8
    assert np.array_equal(got_packed, oracle.repack(ref_q, s, G)[0])


def test_non_finite_weights_are_reported_and_stored_as_8(w):
    """Infinite and NaN weights make the quotient non-finite: the call flags W4A16_ERR_VALUE and
    stores code 8 there; every other code (including the rest of those words) is the oracle's."""
    K, N, G = 256, 256, 128
    wt, s = synth.make_fp16_weights(K, N, G, seed=6)
    bad_at = [(3, 5), (70, 130), (130, 255), (255, 0), (17, 17)]
    for (r, c), v in zip(bad_at, [np.inf, -np.inf, np.nan, np.inf, np.nan]):
        wt[r, c] = np.float16(v)
    got_packed, _ = _quantize_on_device(w, wt, s, G)
    assert w.w4a16_get_status() == 10  # W4A16_ERR_VALUE
    assert w.w4a16_get_status() == 0
    ok = wt.copy()
    for r, c in bad_at:
        ok[r, c] = 0
    ref_q = oracle.quantize(ok, s, G)
    for r, c in bad_at:
        ref_q[r, c] = 8
    assert np.array_equal(got_packed, oracle.repack(ref_q, s, G)[0])


def test_quantize_full_k_sampled_strips(w):
    """K = 18432 (the big layer's depth), N = 8192; four 128-column strips checked byte for byte."""
    K, N, G = 18432, 8192, 128
    wt, s = synth.make_fp16_weights(K, N, G, seed=2)
    got_packed, got_sp = _quantize_on_device(w, wt, s, G)
    words_per_strip = K * 128 // 8
    for j in (0, 17, 40, N // 128 - 1):
        cols = slice(128 * j, 128 * (j + 1))
        ref_packed, ref_sp = oracle.repack(oracle.quantize(wt[:, cols], s[:, cols], G), s[:, cols], G)
        assert np.array_equal(got_packed[j * words_per_strip:(j + 1) * words_per_strip], ref_packed)
        sps = (K // G) * 128
        assert np.array_equal(got_sp[j * sps:(j + 1) * sps], ref_sp.view(np.uint16))


# ---------------------------------------------------------------------------
# min-max scales (MARLIN paper, Section 2.2, "Weight Quantization")
# ---------------------------------------------------------------------------

MINMAX_SHAPES = [(128, 128, 128), (256, 384, 128), (1024, 512, -1), (4096, 256, 128), (1024, 640, 1024)]


def _minmax_on_device(w, wt, G, symmetric):
    torch = tl.torch_mod()
    s, z = w.minmax_scales(tl.to_dev(wt), G, symmetric=symmetric)
    torch.cuda.synchronize()
    return s.cpu().numpy(), (None if z is None else z.cpu().numpy())


@pytest.mark.parametrize("K,N,G", MINMAX_SHAPES)
@pytest.mark.parametrize("symmetric", [True, False])
def test_minmax_scales_match_oracle_bits(w, K, N, G, symmetric):
    wt = synth.make_raw_weights(K, N, seed=K + 3 * N)
    s, z = _minmax_on_device(w, wt, G, symmetric)
    s_ref, z_ref = oracle.minmax_scales(wt, G, symmetric=symmetric)
    assert np.array_equal(s.view(np.uint16), s_ref.view(np.uint16))
    if symmetric:
        assert z is None and z_ref is None
    else:
        assert np.array_equal(z, z_ref)
    assert w.w4a16_get_status() == 0


@pytest.mark.parametrize("symmetric", [True, False])
def test_minmax_then_quantize_repack_matches_oracle(w, symmetric):
    """The whole offline step on the device (scales, codes, packed layout, permuted zeros) against
    the oracle, byte for byte."""
    torch = tl.torch_mod()
    K, N, G = 2048, 384, 128
    wt = synth.make_raw_weights(K, N, seed=91)
    wd = tl.to_dev(wt)
    s, z = w.minmax_scales(wd, G, symmetric=symmetric)
    packed, sp = w.quantize_repack(wd, s, G, z=z)
    zp = None if z is None else w.repack_zeros(z, K, G)
    torch.cuda.synchronize()
    s_ref, z_ref = oracle.minmax_scales(wt, G, symmetric=symmetric)
    q_ref = oracle.quantize(wt, s_ref, G) if symmetric else oracle.quantize_zp(wt, s_ref, z_ref, G)
    ref_packed, ref_sp = oracle.repack(q_ref, s_ref, G)
    assert np.array_equal(packed.cpu().numpy().view(np.uint32), ref_packed)
    assert np.array_equal(sp.cpu().numpy().view(np.uint16).ravel(), ref_sp.view(np.uint16))
    if not symmetric:
        assert np.array_equal(zp.cpu().numpy(), oracle.repack_zeros(z_ref, G, K))
    assert w.w4a16_get_status() == 0


@pytest.mark.parametrize("M", [5, 40])
def test_gemm_on_minmax_quantised_weights(w, M):
    """Quantise with the asymmetric min-max rule on the device, then run the zero-point GEMM: within
    the parity bound of the oracle's product of the oracle's codes."""
    torch = tl.torch_mod()
    K, N, G = 1024, 512, 128
    wt = synth.make_raw_weights(K, N, seed=92)
    A = synth.make_activations(M, K, seed=93)
    wd = tl.to_dev(wt)
    s, z = w.minmax_scales(wd, G, symmetric=False)
    packed, sp = w.quantize_repack(wd, s, G, z=z)
    zp = w.repack_zeros(z, K, G)
    C = w.gemm_zp(tl.to_dev(A), packed, sp, zp, None, N, G)
    torch.cuda.synchronize()
    s_ref, z_ref = oracle.minmax_scales(wt, G, symmetric=False)
    C_ref, bound = oracle.gemm_ref_zp(A, oracle.quantize_zp(wt, s_ref, z_ref, G), s_ref, z_ref, None, G)
    assert oracle.error_ok(C.cpu().numpy(), C_ref, bound)


def test_minmax_non_finite_weight_is_reported(w):
    K, N, G = 256, 128, 128
    wt = synth.make_raw_weights(K, N, seed=94)
    wt[130, 9] = np.float16(np.inf)
    for symmetric in (True, False):
        s, z = _minmax_on_device(w, wt, G, symmetric)
        assert w.w4a16_get_status() == 10   # W4A16_ERR_VALUE
        assert w.w4a16_get_status() == 0
        assert float(s[1, 9]) == 1.0 and (z is None or z[1, 9] == 0)
        # every other group is the oracle's
        ok = wt.copy()
        ok[130, 9] = 0
        s_ref, z_ref = oracle.minmax_scales(ok, G, symmetric=symmetric)
        mask = np.ones(s.shape, bool)
        mask[1, 9] = False
        assert np.array_equal(s.view(np.uint16)[mask], s_ref.view(np.uint16)[mask])
        if z is not None:
            assert np.array_equal(z[mask], z_ref[mask])


@pytest.mark.parametrize("G", [128, -1])
def test_minmax_full_k_sampled_columns(w, G):
    """K = 18432 (the big layer's depth), N = 8192: sampled columns against the oracle."""
    K, N = 18432, 8192
    wt = synth.make_raw_weights(K, N, seed=95)
    for symmetric in (True, False):
        s, z = _minmax_on_device(w, wt, G, symmetric)
        cols = np.array([0, 1, 2, 3, 4, 5, 777, 4096, N - 2, N - 1])
        s_ref, z_ref = oracle.minmax_scales(wt[:, cols], G, symmetric=symmetric)
        assert np.array_equal(s[:, cols].view(np.uint16), s_ref.view(np.uint16))
        if not symmetric:
            assert np.array_equal(z[:, cols], z_ref)


def test_quantize_quotients_near_half_integers_match_oracle(w):
    """Weights placed at (x + 1/2 + delta) * s for random FP16 scales (inexact reciprocals) and tiny
    delta of either sign: the quotients sit next to the rounding boundaries, where the kernel must
    fall back to the correctly rounded division; codes byte for byte against the oracle."""
    rng = np.random.default_rng(97)
    K, N, G = 512, 512, 128
    s = rng.uniform(0.003, 0.05, size=(K // G, N)).astype(np.float16)
    x = rng.integers(-9, 8, size=(K, N)).astype(np.float64)
    delta = rng.choice([-1.0, 1.0], size=(K, N)) * 10.0 ** rng.uniform(-7, -2, size=(K, N))
    delta[rng.random((K, N)) < 0.2] = 0.0
    wt = ((x + 0.5 + delta) * np.repeat(s.astype(np.float64), G, axis=0)).astype(np.float16)
    got_packed, got_sp = _quantize_on_device(w, wt, s, G)
    ref_packed, _ = oracle.repack(oracle.quantize(wt, s, G), s, G)
    assert np.array_equal(got_packed, ref_packed)
    assert w.w4a16_get_status() == 0
