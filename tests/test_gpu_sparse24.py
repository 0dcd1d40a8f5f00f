"""2:4-sparse W4A16 on the GPU against the CPU oracle: the packed stream round
trip (byte exact), the sparse GEMM within the parity bound of the dense
product of the same codes, identity rows exact, the 2:4 violation check, and
the ablation switches bitwise neutral."""
import numpy as np
import pytest

import oracle
from mixed_precision_w4a16_gb300 import synth
import w4a16_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w():
    return tl.lib()


def _device24(w, q, s, G):
    packed, sp = w.repack_24(tl.to_dev(q), tl.to_dev(s), G)
    tl.torch_mod().cuda.synchronize()
    return packed, sp


def _gemm24(w, A, packed, sp, N, G):
    torch = tl.torch_mod()
    C = w.gemm_24(tl.to_dev(A), packed, sp, N, G)
    torch.cuda.synchronize()
    return C.cpu().numpy()


@pytest.mark.parametrize("K,N,G", [(128, 128, 128), (1024, 384, 128), (512, 256, -1), (4096, 256, 128)])
def test_repack_unpack_round_trip(w, K, N, G):
    q, s = synth.make_weights_24(K, N, G, seed=K + N)
    packed, sp = _device24(w, q, s, G)
    assert packed.numel() * 4 == w.w4a16_packed24_bytes(K, N) == 3 * K * N // 8
    q2 = w.unpack_24(packed, K, N)
    tl.torch_mod().cuda.synchronize()
    qc, idx = oracle.sparse24_compress(q)
    assert np.array_equal(q2.cpu().numpy(), oracle.sparse24_expand(qc, idx))
    assert np.array_equal(sp.cpu().numpy().view(np.uint16), oracle.repack(q, s, G)[1].view(np.uint16))
    assert w.w4a16_get_status() == 0


@pytest.mark.parametrize("M", [1, 5, 8, 13, 16, 17, 32, 33, 64, 70])
@pytest.mark.parametrize("K,N,G", [(1024, 512, 128), (2048, 384, -1), (768, 1280, 128)])
def test_gemm24_matches_oracle(w, M, K, N, G):
    q, s = synth.make_weights_24(K, N, G, seed=3 * M + K)
    A = synth.make_activations(M, K, seed=M + N)
    packed, sp = _device24(w, q, s, G)
    C = _gemm24(w, A, packed, sp, N, G)
    qc, idx = oracle.sparse24_compress(q)
    C_ref, bound = oracle.gemm24_ref(A, qc, idx, s, G)
    tl.assert_within_bound(C, C_ref, bound, f"2:4 M={M} K={K} N={N} G={G}")
    assert w.w4a16_get_status() == 0


def test_gemm24_identity_rows_are_exact(w):
    """Row m = e_k returns the FP16 dequantised row k of the sparse weights exactly (kept values at their
    positions, zeros elsewhere): pins the code/position pairing and the fragment layout."""
    K, N, G = 512, 256, 128
    q, s = synth.make_weights_24(K, N, G, seed=7)
    ks = list(range(0, 16)) + [37, 64, 127, 128, 255, 300, 509, 510, 511]
    A = np.zeros((len(ks), K), np.float16)
    for m, k in enumerate(ks):
        A[m, k] = 1.0
    packed, sp = _device24(w, q, s, G)
    C = np.concatenate([_gemm24(w, A[i:i + 16], packed, sp, N, G) for i in range(0, len(ks), 16)])
    want = oracle.dequant_fp16_bits(q, s, G)
    for m, k in enumerate(ks):
        assert np.array_equal(C[m].view(np.uint16), want[k]), k


def test_gemm24_integer_product_is_exact(w):
    rng = np.random.default_rng(11)
    K, N, G = 1024, 256, 128
    q, _ = synth.make_weights_24(K, N, G, seed=12)
    s = np.ones((K // G, N), np.float16)
    A = rng.integers(-2, 3, (9, K)).astype(np.float16)
    packed, sp = _device24(w, q, s, G)
    C = _gemm24(w, A, packed, sp, N, G)
    ref = A.astype(np.int64) @ (q.astype(np.int64) - 8)
    assert np.array_equal(C.astype(np.float64), ref.astype(np.float64))


def test_dense_and_sparse_kernels_agree(w):
    """The same codes through the dense GEMM and the sparse one: both within the bound of the oracle."""
    K, N, G, M = 2048, 512, 128, 12
    q, s = synth.make_weights_24(K, N, G, seed=21)
    A = synth.make_activations(M, K, seed=22)
    packed, sp = _device24(w, q, s, G)
    C24 = _gemm24(w, A, packed, sp, N, G)
    _, _, pk, spd = tl.device_layer(w, q, s, G)
    Cd = tl.c_numpy(tl.run_gemm(w, A, pk, spd, N, G))
    C_ref, bound = oracle.gemm_ref(A, q, s, G)
    tl.assert_within_bound(C24, C_ref, bound, "sparse")
    tl.assert_within_bound(Cd, C_ref, bound, "dense")


def test_three_nonzeros_in_a_group_are_reported(w):
    K, N, G = 256, 128, 128
    q, s = synth.make_weights_24(K, N, G, seed=31)
    q[40:44, 77] = [1, 2, 3, 8]
    _device24(w, q, s, G)
    assert w.w4a16_get_status() == 10   # W4A16_ERR_VALUE
    assert w.w4a16_get_status() == 0


def test_ablations_leave_the_sparse_result_bitwise_unchanged(w):
    K, N, G, M = 1024, 384, 128, 7
    q, s = synth.make_weights_24(K, N, G, seed=41)
    A = synth.make_activations(M, K, seed=42)
    packed, sp = _device24(w, q, s, G)
    base = _gemm24(w, A, packed, sp, N, G)
    try:
        for f in (1, 2, 4, 7):
            w.w4a16_debug_ablate(f)
            assert np.array_equal(_gemm24(w, A, packed, sp, N, G).view(np.uint16), base.view(np.uint16)), f
    finally:
        w.w4a16_debug_ablate(0)


@pytest.mark.parametrize("M", [16, 32, 64])
def test_gemm24_big_layer_sampled_strips(w, M):
    """K = 18432 (the big layer's depth), N = 8192: four 128-column strips against the oracle."""
    K, N, G = 18432, 8192, 128
    q, s = synth.make_weights_24(K, N, G, seed=51)
    A = synth.make_activations(M, K, seed=52)
    packed, sp = _device24(w, q, s, G)
    C = _gemm24(w, A, packed, sp, N, G)
    for j in (0, 17, 40, N // 128 - 1):
        cols = slice(128 * j, 128 * (j + 1))
        C_ref, bound = oracle.gemm_ref(A, q[:, cols], s[:, cols], G)
        tl.assert_within_bound(C[:, cols], C_ref, bound, f"strip {j}")


def test_gemm24_timeout_is_reported_and_context_survives(w):
    """Failure injection on the host side of the wait: the first stage of every CTA is never filled,
    so the consumers' first wait runs out of its short bound; W4A16_ERR_TIMEOUT, nothing written,
    and the next call on a re-zeroed workspace is correct."""
    torch = tl.torch_mod()
    M, K, N, G = 8, 4096, 2048, 128
    q, s = synth.make_weights_24(K, N, G, seed=61)
    A = synth.make_activations(M, K, seed=62)
    packed, sp = _device24(w, q, s, G)
    A_d = tl.to_dev(A)
    ws = torch.zeros(w.w4a16_workspace_bytes_24(M, K, N, G), dtype=torch.uint8, device="cuda")
    C = torch.full((M, N), 7.0, dtype=torch.float16, device="cuda")
    try:
        w.w4a16_debug_set_wait_cycles(2_000_000)  # about a millisecond
        w.w4a16_debug_inject_stall(True)
        w.w4a16_gemm_24(A_d, packed, sp, C, M, K, N, G, ws)
    finally:
        w.w4a16_debug_inject_stall(False)
        w.w4a16_debug_set_wait_cycles(0)
    assert w.w4a16_get_status(ws) == 7
    assert torch.all(C == 7.0)
    ws.zero_()
    C2 = w.gemm_24(A_d, packed, sp, N, G, workspace=ws)
    torch.cuda.synchronize()
    qc, idx = oracle.sparse24_compress(q)
    C_ref, bound = oracle.gemm24_ref(A, qc, idx, s, G)
    tl.assert_within_bound(C2.cpu().numpy(), C_ref, bound, "after timeout")
    assert w.w4a16_get_status(ws) == 0
