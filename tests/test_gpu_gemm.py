"""The fused W4A16 GEMM on the GPU against the CPU oracle.

Bar: every element within |C - C_ref| <= 4e-3 * sum_k |A B^| + 1e-4; special
cases that are exact in FP32/FP16 must match bit for bit; repeated calls must
be bitwise identical (deterministic split-K reduction).
"""
import numpy as np
import pytest

import oracle
from mixed_precision_w4a16_gb300 import synth
import w4a16_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w():
    return tl.lib()


@pytest.fixture(params=[1, 2, 4], ids=["mma_sync", "tcgen05", "tcgen05_wide"])
def path(request, w):
    """Run the test on the streaming mma.sync kernel, on the tensor-memory kernel (strip pairs up to
    128 token rows, its wide mode above), and on the tensor-memory kernel in its wide mode at every M
    (where K is a multiple of 512; other K fall back to strip pairs)."""
    w.w4a16_debug_force_path(request.param)
    yield request.param
    w.w4a16_debug_force_path(0)


# token counts around every 8-row tile edge, the launch chunks (128 rows in strip pairs, up to 256
# rows dealt evenly in the wide mode)
M_EDGES = [1, 2, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65, 100, 128, 129, 200, 256, 257, 400]


@pytest.mark.parametrize("M", M_EDGES)
@pytest.mark.parametrize("G", [128, -1])
def test_gemm_parity_small_layer(w, path, M, G):
    K, N = 1024, 1024
    A, q, s = tl.layer(M, K, N, G, seed=100 + M)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    C = tl.c_numpy(tl.run_gemm(w, A, packed, sp, N, G))
    C_ref, bound = oracle.gemm_ref(A, q, s, G)
    tl.assert_within_bound(C, C_ref, bound, f"M={M} G={G}")


@pytest.mark.parametrize("M,K,N,G", [
    (5, 128, 128, 128),         # one unit, one CTA
    (16, 256, 384, 128),        # three strips
    (16, 384, 640, -1),         # K/128 odd (128-row units), per-column scales
    (3, 11008, 256, 128),       # long K: stripes split every strip
    (24, 2048, 8192, 128),      # many strips
    (40, 4096, 640, -1),
    (9, 1536, 1280, 128),       # K/256 odd: 256-row units
])
def test_gemm_parity_shapes(w, path, M, K, N, G):
    A, q, s = tl.layer(M, K, N, G, seed=M + K + N)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    C = tl.c_numpy(tl.run_gemm(w, A, packed, sp, N, G))
    C_ref, bound = oracle.gemm_ref(A, q, s, G)
    tl.assert_within_bound(C, C_ref, bound, f"{(M, K, N, G)}")


@pytest.mark.parametrize("G", [128, -1])
def test_identity_rows_return_dequantised_weights_exactly(w, path, G):
    K, N = 2048, 512
    q, s = synth.make_weights(K, N, G, seed=31)
    rows = [0, 1, 63, 64, 127, 128, 1000, 2047, 5, 77, 1500, 640, 641, 1919, 300, 301, 999]
    A = np.zeros((len(rows), K), np.float16)
    for m, k in enumerate(rows):
        A[m, k] = 1.0
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    C = tl.c_numpy(tl.run_gemm(w, A, packed, sp, N, G))
    ref = oracle.dequant_fp16_bits(q, s, G)[rows, :]
    assert np.array_equal(C.view(np.uint16), ref)


def test_integer_gemm_is_exact(w, path):
    # s = 1, small integer activations: every partial sum is an exact FP32 integer below 2048
    rng = np.random.default_rng(12)
    M, K, N, G = 16, 256, 256, 128
    A = rng.integers(-1, 2, (M, K)).astype(np.float16)
    q = rng.integers(5, 12, (K, N)).astype(np.uint8)
    s = np.ones((K // G, N), np.float16)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    C = tl.c_numpy(tl.run_gemm(w, A, packed, sp, N, G))
    ref = A.astype(np.int64) @ (q.astype(np.int64) - 8)
    assert np.abs(ref).max() < 2048
    assert np.array_equal(C.astype(np.float64), ref.astype(np.float64))


@pytest.mark.parametrize("K", [1024, 18432])
def test_zero_codes_stay_within_the_absolute_bound(w, path, K):
    # q == 8 everywhere: B^ = 0, so Bound = 0 and every output must satisfy |C| <= 1e-4.
    # The decode yields q - 8 exactly, so C must come out zero however long K is (a decode that
    # offset the codes and removed the offset afterwards would fail here on long K).
    M, N, G = 9, 512, 128
    A, _, s = tl.layer(M, K, N, G, seed=3)
    q = np.full((K, N), 8, np.uint8)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    C = tl.c_numpy(tl.run_gemm(w, A, packed, sp, N, G))
    C_ref, bound = oracle.gemm_ref(A, q, s, G)
    assert np.all(bound == 0.0)
    tl.assert_within_bound(C, C_ref, bound, f"zero codes K={K}")


@pytest.mark.parametrize("M", [1, 16, 33])
def test_repeated_calls_are_bitwise_identical(w, path, M):
    torch = tl.torch_mod()
    K, N, G = 4096, 2048, 128
    A, q, s = tl.layer(M, K, N, G, seed=77)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    A_d = tl.to_dev(A)
    ws = w.workspace_for(M, K, N, G)
    outs = [tl.run_gemm(w, A_d, packed, sp, N, G, workspace=ws).clone() for _ in range(4)]
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    assert w.w4a16_get_status(ws) == 0


def test_column_block_permutation_permutes_output(w, path):
    # Permuting the 16-column blocks of (q, s) permutes C's columns bit for bit.  (A column's
    # place inside its block picks its decode bias, 256 or 16, so only block moves are exact;
    # any column permutation still agrees within the parity bound, as every parity test shows.)
    M, K, N, G = 16, 2048, 512, 128
    A, q, s = tl.layer(M, K, N, G, seed=8)
    blocks = np.random.default_rng(1).permutation(N // 16)
    perm = (blocks[:, None] * 16 + np.arange(16)[None, :]).ravel()
    _, _, p1, s1 = tl.device_layer(w, q, s, G)
    _, _, p2, s2 = tl.device_layer(w, np.ascontiguousarray(q[:, perm]), np.ascontiguousarray(s[:, perm]), G)
    C1 = tl.c_numpy(tl.run_gemm(w, A, p1, s1, N, G))
    C2 = tl.c_numpy(tl.run_gemm(w, A, p2, s2, N, G))
    assert np.array_equal(C1[:, perm].view(np.uint16), C2.view(np.uint16))


def _linearity_excess(C1, C2, C12, b1, b2, b12):
    """How far C(A1 + A2) - C(A1) - C(A2) exceeds the sum of the three GEMMs' error bounds
    (each |C - C_ref| <= 4e-3 * Bound + 1e-4, and the reference is linear in A)."""
    C1, C2, C12 = (np.asarray(c, dtype=np.float64) for c in (C1, C2, C12))
    return np.abs(C12 - C1 - C2) - (4e-3 * (b1 + b2 + b12) + 3e-4)


def test_linearity_in_activations(w, path):
    # A1, A2 and A1 + A2 are all exact in FP16 (multiples of 1/16 up to 2 in magnitude)
    M, K, N, G = 24, 2048, 1024, 128
    rng = np.random.default_rng(79)
    A1 = (rng.integers(-16, 17, (M, K)) / 16).astype(np.float16)
    A2 = (rng.integers(-16, 17, (M, K)) / 16).astype(np.float16)
    A12 = (A1.astype(np.float64) + A2.astype(np.float64)).astype(np.float16)
    assert np.array_equal(A12.astype(np.float64), A1.astype(np.float64) + A2.astype(np.float64))
    q, s = synth.make_weights(K, N, G, 80)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    C1, C2, C12 = (tl.c_numpy(tl.run_gemm(w, A, packed, sp, N, G)) for A in (A1, A2, A12))
    b1, b2, b12 = (oracle.gemm_ref(A, q, s, G)[1] for A in (A1, A2, A12))
    ex = _linearity_excess(C1, C2, C12, b1, b2, b12)
    assert np.all(ex <= 0), f"{int(np.sum(ex > 0))} elements break linearity beyond the bounds"


def test_group_invariance(w, path):
    # a scale constant over the groups of each column: group 128 and per-column agree within the bound
    M, K, N = 16, 2048, 512
    A, q, s1 = tl.layer(M, K, N, -1, seed=15)
    s128 = np.repeat(s1, K // 128, axis=0)
    _, _, pa, sa = tl.device_layer(w, q, s128, 128)
    _, _, pb, sb = tl.device_layer(w, q, s1, -1)
    Ca = tl.c_numpy(tl.run_gemm(w, A, pa, sa, N, 128))
    Cb = tl.c_numpy(tl.run_gemm(w, A, pb, sb, N, -1))
    C_ref, bound = oracle.gemm_ref(A, q, s1, -1)
    tl.assert_within_bound(Ca, C_ref, bound, "G=128")
    tl.assert_within_bound(Cb, C_ref, bound, "G=K")


def test_workspace_reuse_across_shapes(w, path):
    # counters are left at zero, so one zeroed workspace serves a sequence of calls
    torch = tl.torch_mod()
    big = max(w.w4a16_workspace_bytes(M, 4096, 4096, 128) for M in (1, 16, 32, 64))
    ws = torch.zeros(big, dtype=torch.uint8, device="cuda")
    for M, K, N in [(1, 4096, 4096), (16, 1024, 4096), (32, 4096, 1024), (64, 2048, 2048), (1, 4096, 4096)]:
        A, q, s = tl.layer(M, K, N, 128, seed=M * 3 + K)
        _, _, packed, sp = tl.device_layer(w, q, s, 128)
        C = tl.c_numpy(tl.run_gemm(w, A, packed, sp, N, 128, workspace=ws))
        C_ref, bound = oracle.gemm_ref(A, q, s, 128)
        tl.assert_within_bound(C, C_ref, bound, f"{(M, K, N)}")
    assert w.w4a16_get_status(ws) == 0


def test_gemm_error_codes(w):
    torch = tl.torch_mod()
    M, K, N, G = 4, 1024, 512, 128
    A, q, s = tl.layer(M, K, N, G, seed=2)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    A_d = tl.to_dev(A)
    C = torch.empty((M, N), dtype=torch.float16, device="cuda")
    need = w.w4a16_workspace_bytes(M, K, N, G)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(w.W4A16Error) as e:
        w.w4a16_gemm(A_d, packed, sp, C, M, K, N, G, ws, need - 1)
    assert e.value.status == 5
    with pytest.raises(w.W4A16Error) as e:
        w.w4a16_gemm(A_d.data_ptr() + 2, packed, sp, C, M, K, N, G, ws)
    assert e.value.status == 9
    with pytest.raises(w.W4A16Error) as e:
        w.w4a16_gemm(A_d, packed, sp, C, M, K, N, 256, ws)
    assert e.value.status == 3
    with pytest.raises(w.W4A16Error) as e:
        w.w4a16_gemm(A_d, packed, sp, C, M, K, 448, G, ws)
    assert e.value.status == 2
    w.w4a16_gemm(A_d, packed, sp, C, 0, K, N, G, ws)  # M == 0: no-op


def test_timeout_is_reported_and_context_survives(w, path):
    # Failure injection on the host side of the wait: the first stage of every CTA is never
    # filled, so the consumers' first wait can only end by running out of its (short) bound.
    # The kernel records W4A16_ERR_TIMEOUT, writes nothing and returns; the context stays usable.
    torch = tl.torch_mod()
    M, K, N, G = 16, 4096, 4096, 128
    A, q, s = tl.layer(M, K, N, G, seed=4)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    A_d = tl.to_dev(A)
    ws = w.workspace_for(M, K, N, G)
    C = torch.full((M, N), 7.0, dtype=torch.float16, device="cuda")
    try:
        w.w4a16_debug_set_wait_cycles(2_000_000)  # about a millisecond
        w.w4a16_debug_inject_stall(True)
        w.w4a16_gemm(A_d, packed, sp, C, M, K, N, G, ws)
    finally:
        w.w4a16_debug_inject_stall(False)
        w.w4a16_debug_set_wait_cycles(0)
    assert w.w4a16_get_status(ws) == 7
    assert torch.all(C == 7.0)  # nothing written after the abort
    ws.zero_()
    C = tl.c_numpy(tl.run_gemm(w, A_d, packed, sp, N, G, workspace=ws))
    C_ref, bound = oracle.gemm_ref(A, q, s, G)
    tl.assert_within_bound(C, C_ref, bound, "after timeout")
    assert w.w4a16_get_status(ws) == 0
