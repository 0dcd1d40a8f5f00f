"""Zero points and bias on the GPU against the CPU oracle: repacked zero codes
and dequantised weights bit-exact, GEMM outputs within the parity bound on both
kernels, special cases exact."""
import numpy as np
import pytest

import oracle
from mixed_precision_w4a16_gb300 import synth
import w4a16_testlib as tl

pytestmark = pytest.mark.gpu

PATHS = {"mma_sync": 1, "tcgen05": 2, "tcgen05_wide": 4}


@pytest.fixture(scope="module")
def w():
    return tl.lib()


@pytest.fixture(params=sorted(PATHS))
def path(request, w):
    w.w4a16_debug_force_path(PATHS[request.param])
    yield request.param
    w.w4a16_debug_force_path(0)


def zp_layer(K, N, G, seed):
    q, s = synth.make_weights(K, N, G, seed)
    rng = np.random.default_rng(seed + 1)
    z = rng.integers(0, 16, (K // synth.effective_group(K, G), N)).astype(np.uint8)
    bias = rng.normal(0, 1.0, N).astype(np.float16)
    return q, s, z, bias


def device_zp_layer(w, q, s, z, G):
    K = q.shape[0]
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    zp = w.repack_zeros(tl.to_dev(z), K, G)
    return packed, sp, zp


def run_zp(w, A, packed, sp, zp, bias_d, N, G, ws=None):
    torch = tl.torch_mod()
    C = w.gemm_zp(tl.to_dev(A), packed, sp, zp, bias_d, N, G, workspace=ws)
    torch.cuda.synchronize()
    return tl.c_numpy(C)


@pytest.mark.parametrize("K,N,G", [(256, 128, 128), (1024, 384, 128), (512, 256, -1)])
def test_repack_zeros_and_dequant_zp_bit_exact(w, K, N, G):
    q, s, z, _ = zp_layer(K, N, G, K + N)
    packed, sp, zp = device_zp_layer(w, q, s, z, G)
    assert np.array_equal(zp.cpu().numpy(), oracle.repack_zeros(z, G, K))
    bhat = w.dequant_zp(packed, sp, zp, K, N, G)
    tl.torch_mod().cuda.synchronize()
    assert np.array_equal(bhat.cpu().numpy().view(np.uint16), oracle.dequant_fp16_bits_zp(q, s, z, G))
    assert w.w4a16_get_status() == 0


SHAPES = [(1, 256, 128, 128), (7, 1024, 256, 128), (16, 1024, 384, 128), (17, 512, 256, 128), (32, 2048, 512, 128),
          (64, 1024, 256, -1), (100, 768, 384, 128), (8, 4096, 640, 128)]


@pytest.mark.parametrize("M,K,N,G", SHAPES)
@pytest.mark.parametrize("with_bias", [False, True])
def test_gemm_zp_parity(w, path, M, K, N, G, with_bias):
    q, s, z, bias = zp_layer(K, N, G, 3 * M + K)
    A = synth.make_activations(M, K, seed=M + 5)
    packed, sp, zp = device_zp_layer(w, q, s, z, G)
    C = run_zp(w, A, packed, sp, zp, tl.to_dev(bias) if with_bias else None, N, G)
    C_ref, bound = oracle.gemm_ref_zp(A, q, s, z, bias if with_bias else None, G)
    tl.assert_within_bound(C, C_ref, bound, f"{path} M={M} K={K} N={N} G={G} bias={with_bias}")
    assert w.w4a16_get_status() == 0


@pytest.mark.parametrize("M,K,N,G", [(16, 1024, 256, 128), (48, 1024, 256, 128)])
def test_bias_only_parity(w, path, M, K, N, G):
    q, s, _, bias = zp_layer(K, N, G, 9)
    A = synth.make_activations(M, K, seed=10)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    C = run_zp(w, A, packed, sp, None, tl.to_dev(bias), N, G)
    C_ref, bound = oracle.gemm_ref_zp(A, q, s, None, bias, G)
    tl.assert_within_bound(C, C_ref, bound, f"{path} bias only")


def test_identity_rows_with_zero_points_bit_exact(w, path):
    K, N, G = 512, 256, 128
    q, s, z, _ = zp_layer(K, N, G, 21)
    rows = [0, 1, 127, 128, 300, 511]
    A = np.zeros((len(rows), K), np.float16)
    for m, k in enumerate(rows):
        A[m, k] = 1.0
    packed, sp, zp = device_zp_layer(w, q, s, z, G)
    C = run_zp(w, A, packed, sp, zp, None, N, G)
    assert np.array_equal(C.view(np.uint16), oracle.dequant_fp16_bits_zp(q, s, z, G)[rows, :])


def test_codes_at_their_zero_points_give_the_bias_exactly(w, path):
    K, N, G = 1024, 256, 128
    _, s, z, bias = zp_layer(K, N, G, 22)
    q = np.repeat(z, G, axis=0)
    A = synth.make_activations(20, K, seed=23)
    packed, sp, zp = device_zp_layer(w, q, s, z, G)
    C = run_zp(w, A, packed, sp, zp, tl.to_dev(bias), N, G)
    assert np.array_equal(C.view(np.uint16), np.tile(bias.view(np.uint16), (20, 1)))


@pytest.mark.parametrize("M", [8, 40])
def test_zero_point_eight_matches_the_symmetric_gemm_bitwise(w, path, M):
    K, N, G = 1024, 384, 128
    q, s = synth.make_weights(K, N, G, seed=24)
    A = synth.make_activations(M, K, seed=25)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    zp = w.repack_zeros(tl.to_dev(np.full((K // G, N), 8, np.uint8)), K, G)
    C_zp = run_zp(w, A, packed, sp, zp, None, N, G)
    C_sym = tl.c_numpy(tl.run_gemm(w, A, packed, sp, N, G))
    assert np.array_equal(C_zp.view(np.uint16), C_sym.view(np.uint16))


def test_zp_gemm_is_deterministic(w, path):
    K, N, G = 2048, 512, 128
    q, s, z, bias = zp_layer(K, N, G, 26)
    A = synth.make_activations(33, K, seed=27)
    packed, sp, zp = device_zp_layer(w, q, s, z, G)
    b = tl.to_dev(bias)
    C1 = run_zp(w, A, packed, sp, zp, b, N, G)
    C2 = run_zp(w, A, packed, sp, zp, b, N, G)
    assert np.array_equal(C1.view(np.uint16), C2.view(np.uint16))


def test_zero_code_range_flag(w):
    K, N, G = 256, 128, 128
    z = np.full((K // G, N), 3, np.uint8)
    z[1, 5] = 16
    zp = w.repack_zeros(tl.to_dev(z), K, G)
    assert w.w4a16_get_status() == 4  # W4A16_ERR_CODE_RANGE
    assert w.w4a16_get_status() == 0


def test_big_layer_zero_points_sampled_columns(w):
    """K = 18432, N = 73728, zero points and bias, the bench's launch configuration (M = 1, 16, 64, 128)."""
    K, N, G = 18432, 73728, 128
    q, s, z, bias = zp_layer(K, N, G, 500)
    packed, sp, zp = device_zp_layer(w, q, s, z, G)
    rng = np.random.default_rng(501)
    cols = np.unique(np.concatenate([np.arange(128), np.arange(N - 128, N), rng.choice(N, 1024, False)]))
    qc, sc, zc = np.ascontiguousarray(q[:, cols]), np.ascontiguousarray(s[:, cols]), np.ascontiguousarray(z[:, cols])
    del q
    b = tl.to_dev(bias)
    for M in (1, 16, 64, 128):
        A = synth.make_activations(M, K, seed=502 + M)
        C = run_zp(w, A, packed, sp, zp, b, N, G)
        C_ref, bound = oracle.gemm_ref_zp(A, qc, sc, zc, bias[cols], G)
        tl.assert_within_bound(C[:, cols], C_ref, bound, f"big layer zp M={M}")
    assert w.w4a16_get_status() == 0
