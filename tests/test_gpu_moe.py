"""Grouped expert (MoE) GEMM on the GPU against the CPU oracle: every row of C
is its own expert's product, within the parity bound, for routed batches of
several shapes (uniform, skewed with hot experts split into row segments, many
empty experts), plus exact identity rows, bitwise agreement with the dense GEMM
for one expert, and the device-side check of the expert offsets."""
import numpy as np
import pytest

import oracle
from mixed_precision_w4a16_gb300 import synth
import w4a16_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w():
    return tl.lib()


def _device_experts(w, q, s, G):
    """Repack every expert on the device and concatenate (expert e at word e*K*N/8)."""
    torch = tl.torch_mod()
    packed, sps = [], []
    for e in range(q.shape[0]):
        pk, sp = w.repack(tl.to_dev(q[e]), tl.to_dev(s[e]), G)
        packed.append(pk)
        sps.append(sp)
    return torch.cat(packed), torch.cat(sps)


def _run(w, lay, N, max_rows, packed=None, sp=None, workspace=None):
    torch = tl.torch_mod()
    if packed is None:
        packed, sp = _device_experts(w, lay["q"], lay["s"], lay["G"])
    C = w.moe_gemm(tl.to_dev(lay["A"]), packed, sp, tl.to_dev(lay["offsets"]), N, lay["G"], max_rows=max_rows,
                   workspace=workspace)
    torch.cuda.synchronize()
    return C.cpu().numpy()


CASES = [
    # tokens, topk, E, K, N, G, skew, max_rows
    (16, 2, 8, 1024, 512, 128, 0.0, 8),
    (16, 2, 8, 1024, 512, 128, 0.0, 0),
    (64, 4, 16, 512, 384, 128, 1.2, 16),
    (5, 1, 32, 768, 256, -1, 0.0, 8),
    (40, 2, 4, 2048, 256, 128, 2.0, 32),
    (3, 3, 3, 256, 128, 128, 0.0, 1),
]


@pytest.mark.parametrize("tokens,topk,E,K,N,G,skew,max_rows", CASES)
def test_moe_gemm_matches_oracle(w, tokens, topk, E, K, N, G, skew, max_rows):
    lay = synth.make_moe_layer(tokens, topk, E, K, N, G, seed=tokens * 7 + E, skew=skew)
    C = _run(w, lay, N, max_rows)
    C_ref, bound = oracle.moe_gemm_ref(lay["A"], lay["offsets"], lay["q"], lay["s"], G)
    tl.assert_within_bound(C, C_ref, bound, f"moe E={E} rows={np.diff(lay['offsets']).tolist()}")
    assert w.w4a16_get_status() == 0


@pytest.mark.parametrize("counts", [[0, 0, 37, 0], [37, 0, 0, 0], [0, 0, 0, 37], [1, 0, 1, 0, 1, 0, 1, 0, 1],
                                    [9, 8, 17, 16, 15]])
def test_moe_gemm_row_distributions(w, counts):
    """Hot, cold and empty experts at the first and last positions; segments of 8 rows with ragged tails."""
    K, N, G = 512, 256, 128
    lay = synth.make_moe_layer(0, 0, len(counts), K, N, G, seed=sum(counts) + len(counts), counts=counts)
    C = _run(w, lay, N, 8)
    C_ref, bound = oracle.moe_gemm_ref(lay["A"], lay["offsets"], lay["q"], lay["s"], G)
    tl.assert_within_bound(C, C_ref, bound, f"counts={counts}")


def test_moe_identity_rows_return_each_experts_dequantised_rows(w):
    """Row m = e_k gives the owning expert's FP16 dequantised row k exactly (ownership and weights per row)."""
    K, N, G = 512, 256, 128
    counts = [3, 0, 5, 2]
    lay = synth.make_moe_layer(0, 0, len(counts), K, N, G, seed=5, counts=counts)
    M = sum(counts)
    ks = [(37 * m + 11) % K for m in range(M)]
    A = np.zeros((M, K), np.float16)
    for m, k in enumerate(ks):
        A[m, k] = 1.0
    lay["A"] = A
    C = _run(w, lay, N, 8)
    off = lay["offsets"]
    for m, k in enumerate(ks):
        e = int(np.searchsorted(off, m, side="right")) - 1
        want = oracle.dequant_fp16_bits(lay["q"][e], lay["s"][e], G)[k]
        assert np.array_equal(C[m].view(np.uint16), want), (m, e, k)


@pytest.mark.parametrize("M", [1, 8, 13, 16])
def test_one_expert_is_bitwise_the_dense_gemm(w, M):
    """E = 1 with all M rows in one segment (<= 16): the same units, split and summation order as
    w4a16_gemm on the streaming kernel."""
    torch = tl.torch_mod()
    K, N, G = 2048, 768, 128
    lay = synth.make_moe_layer(0, 0, 1, K, N, G, seed=60 + M, counts=[M])
    packed, sp = _device_experts(w, lay["q"], lay["s"], G)
    C = _run(w, lay, N, M, packed, sp)
    w.w4a16_debug_force_path(1)
    try:
        Cd = tl.run_gemm(w, lay["A"], packed, sp, N, G).cpu().numpy()
    finally:
        w.w4a16_debug_force_path(0)
    assert np.array_equal(C.view(np.uint16), Cd.view(np.uint16))
    torch.cuda.synchronize()


def test_moe_repeated_calls_and_workspace_reuse_are_bitwise_identical(w):
    torch = tl.torch_mod()
    K, N, G = 1024, 384, 128
    lay = synth.make_moe_layer(24, 2, 8, K, N, G, seed=71, skew=1.0)
    packed, sp = _device_experts(w, lay["q"], lay["s"], G)
    M = int(lay["offsets"][-1])
    ws = w.moe_workspace_for(8, M, 8, K, N, G)
    C1 = _run(w, lay, N, 8, packed, sp, ws)
    C2 = _run(w, lay, N, 8, packed, sp, ws)
    assert np.array_equal(C1.view(np.uint16), C2.view(np.uint16))
    assert w.w4a16_get_status(ws) == 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("bad", [[1, 5, 12], [0, 7, 5], [0, 5, 11], [0, 5, 13], [-1, 5, 12]])
def test_invalid_offsets_are_reported_and_c_is_untouched(w, bad):
    torch = tl.torch_mod()
    K, N, G = 256, 128, 128
    lay = synth.make_moe_layer(0, 0, 2, K, N, G, seed=72, counts=[5, 7])
    packed, sp = _device_experts(w, lay["q"], lay["s"], G)
    M = 12
    ws = w.moe_workspace_for(2, M, 8, K, N, G)
    C = torch.full((M, N), 7.0, dtype=torch.float16, device="cuda")
    off = tl.to_dev(np.array(bad, np.int32))
    w.moe_gemm(tl.to_dev(lay["A"]), packed, sp, off, N, G, max_rows=8, workspace=ws, out=C)
    assert w.w4a16_get_status(ws) == 10   # W4A16_ERR_VALUE
    assert bool((C == 7.0).all())
    # the workspace is still usable: a valid call afterwards is correct
    C2 = w.moe_gemm(tl.to_dev(lay["A"]), packed, sp, tl.to_dev(lay["offsets"]), N, G, max_rows=8, workspace=ws)
    torch.cuda.synchronize()
    C_ref, bound = oracle.moe_gemm_ref(lay["A"], lay["offsets"], lay["q"], lay["s"], G)
    tl.assert_within_bound(C2.cpu().numpy(), C_ref, bound, "after invalid offsets")


def test_moe_host_checks(w):
    import mixed_precision_w4a16_gb300 as m
    assert m.w4a16_moe_workspace_bytes(0, 8, 8, 256, 128, 128) == 0        # no experts
    assert m.w4a16_moe_workspace_bytes(4097, 8, 8, 256, 128, 128) == 0     # too many experts
    assert m.w4a16_moe_workspace_bytes(4, 8, 8, 200, 128, 128) == 0        # K not a multiple of 128
    assert m.w4a16_moe_workspace_bytes(4, 0, 8, 256, 128, 128) > 0         # M = 0 is a no-op call
    with pytest.raises(m.W4A16Error):
        torch = tl.torch_mod()
        A = torch.zeros((4, 256), dtype=torch.float16, device="cuda")
        C = torch.zeros((4, 128), dtype=torch.float16, device="cuda")
        off = torch.tensor([0, 4], dtype=torch.int32, device="cuda")
        packed = torch.zeros(256 * 128 // 8, dtype=torch.int32, device="cuda")
        sp = torch.zeros(2 * 128, dtype=torch.float16, device="cuda")
        m.w4a16_moe_gemm(A, packed, sp, off, C, 1, 4, 4, 256, 128, 128, None, 0)   # no workspace


def test_moe_large_layer_sampled_experts(w):
    """64 experts of K = 2048, N = 1408 (an MoE FFN's shape), 32 tokens routed top-4 with skew: the rows of
    the hottest, a cold and the first and last non-empty experts against the oracle."""
    K, N, G, E = 2048, 1408, 128, 64
    counts = synth.make_expert_rows(32, 4, E, seed=73, skew=1.0)
    lay = synth.make_moe_layer(0, 0, E, K, N, G, seed=74, counts=counts)
    C = _run(w, lay, N, 8)
    off = lay["offsets"]
    nz = [e for e in range(E) if counts[e] > 0]
    pick = sorted({int(np.argmax(counts)), nz[0], nz[-1], nz[len(nz) // 2]})
    for e in pick:
        lo, hi = int(off[e]), int(off[e + 1])
        C_ref, bound = oracle.gemm_ref(lay["A"][lo:hi], lay["q"][e], lay["s"][e], G)
        tl.assert_within_bound(C[lo:hi], C_ref, bound, f"expert {e} rows {lo}..{hi}")


@pytest.mark.parametrize("E", [289, 1000, 2048])
def test_moe_many_experts_exercise_the_multi_expert_scan(w, E):
    """E > 288 experts: each thread of the prologue's scan owns several experts (up to 8 at the
    2048 maximum); most own no rows, the rows sit at the first, last and scattered experts."""
    K, N, G = 256, 128, 128
    counts = np.zeros(E, dtype=np.int64)
    for e, c in ((0, 3), (1, 0), (287, 9), (288, 2), (E // 2, 17), (E - 2, 1), (E - 1, 5)):
        counts[e] = c
    lay = synth.make_moe_layer(0, 0, E, K, N, G, seed=E, counts=counts)
    C = _run(w, lay, N, 0)
    C_ref, bound = oracle.moe_gemm_ref(lay["A"], lay["offsets"], lay["q"], lay["s"], G)
    tl.assert_within_bound(C, C_ref, bound, f"E={E}")
    assert w.w4a16_get_status() == 0


def test_moe_timeout_is_reported_and_context_survives(w):
    torch = tl.torch_mod()
    K, N, G = 2048, 1024, 128
    lay = synth.make_moe_layer(16, 2, 8, K, N, G, seed=75)
    packed, sp = _device_experts(w, lay["q"], lay["s"], G)
    M = int(lay["offsets"][-1])
    ws = w.moe_workspace_for(8, M, 8, K, N, G)
    C = torch.full((M, N), 7.0, dtype=torch.float16, device="cuda")
    A_d, off_d = tl.to_dev(lay["A"]), tl.to_dev(lay["offsets"])
    try:
        w.w4a16_debug_set_wait_cycles(2_000_000)  # about a millisecond
        w.w4a16_debug_inject_stall(True)
        w.moe_gemm(A_d, packed, sp, off_d, N, G, max_rows=8, workspace=ws, out=C)
    finally:
        w.w4a16_debug_inject_stall(False)
        w.w4a16_debug_set_wait_cycles(0)
    assert w.w4a16_get_status(ws) == 7
    assert bool((C == 7.0).all())
    ws.zero_()
    C2 = _run(w, lay, N, 8, packed, sp, ws)
    C_ref, bound = oracle.moe_gemm_ref(lay["A"], lay["offsets"], lay["q"], lay["s"], G)
    tl.assert_within_bound(C2, C_ref, bound, "after timeout")


# ---------------------------------------------------------------------------
# From 17 rows per expert the grouped GEMM runs on the tensor-memory kernel (pair mode, row
# segments of max_rows rounded up to 16, at most 128 rows): the same checks on that path.
# ---------------------------------------------------------------------------

TC_CASES = [
    # counts per expert, K, N, G, max_rows
    ([21, 3, 0, 17, 8, 19, 0, 12], 1024, 512, 128, 32),     # Mixtral-like: 2 of 8 experts per token
    ([40, 64, 1, 0], 4096, 1024, 128, 64),                  # 64-row segments
    ([200, 3, 0, 50], 2048, 768, 128, 200),                 # 200 rows: two 128-row segments of one expert
    ([33, 31, 32, 1], 768, 384, 128, 48),                   # K / 128 = 6 (256-row units), three strips
    ([20, 0, 19], 640, 256, -1, 32),                        # K / 128 = 5 (128-row units), per-column scales
    ([0, 0, 0, 90], 512, 1280, 128, 96),                    # only the last expert owns rows
]


@pytest.mark.parametrize("counts,K,N,G,max_rows", TC_CASES)
def test_moe_tensor_memory_path_matches_oracle(w, counts, K, N, G, max_rows):
    assert max_rows >= 17
    lay = synth.make_moe_layer(0, 0, len(counts), K, N, G, seed=sum(counts) + K, counts=counts)
    C = _run(w, lay, N, max_rows)
    C_ref, bound = oracle.moe_gemm_ref(lay["A"], lay["offsets"], lay["q"], lay["s"], G)
    tl.assert_within_bound(C, C_ref, bound, f"tcgen05 moe counts={counts} K={K} N={N} G={G}")
    assert w.w4a16_get_status() == 0


def test_moe_tensor_memory_identity_rows_are_exact(w):
    K, N, G = 1024, 512, 128
    counts = [18, 0, 23, 5]
    lay = synth.make_moe_layer(0, 0, len(counts), K, N, G, seed=81, counts=counts)
    M = sum(counts)
    ks = [(53 * m + 7) % K for m in range(M)]
    A = np.zeros((M, K), np.float16)
    for m, k in enumerate(ks):
        A[m, k] = 1.0
    lay["A"] = A
    C = _run(w, lay, N, 32)
    off = lay["offsets"]
    for m, k in enumerate(ks):
        e = int(np.searchsorted(off, m, side="right")) - 1
        want = oracle.dequant_fp16_bits(lay["q"][e], lay["s"][e], G)[k]
        assert np.array_equal(C[m].view(np.uint16), want), (m, e, k)


def test_moe_forced_tensor_memory_path_with_small_segments(w):
    """The tensor-memory path forced onto 8-row experts (16-row segments)."""
    K, N, G = 1024, 384, 128
    lay = synth.make_moe_layer(24, 2, 8, K, N, G, seed=82, skew=1.0)
    w.w4a16_debug_force_path(2)
    try:
        C = _run(w, lay, N, 8)
    finally:
        w.w4a16_debug_force_path(0)
    C_ref, bound = oracle.moe_gemm_ref(lay["A"], lay["offsets"], lay["q"], lay["s"], G)
    tl.assert_within_bound(C, C_ref, bound, "forced tcgen05 moe")


def test_moe_tensor_memory_repeats_are_bitwise_identical(w):
    torch = tl.torch_mod()
    K, N, G = 2048, 1024, 128
    counts = [30, 12, 0, 27, 31, 1, 19, 8]
    lay = synth.make_moe_layer(0, 0, len(counts), K, N, G, seed=83, counts=counts)
    packed, sp = _device_experts(w, lay["q"], lay["s"], G)
    M = sum(counts)
    ws = w.moe_workspace_for(len(counts), M, 32, K, N, G)
    first = _run(w, lay, N, 32, packed, sp, ws)
    for _ in range(12):
        again = _run(w, lay, N, 32, packed, sp, ws)
        assert np.array_equal(first.view(np.uint16), again.view(np.uint16))
    assert w.w4a16_get_status(ws) == 0
    C_ref, bound = oracle.moe_gemm_ref(lay["A"], lay["offsets"], lay["q"], lay["s"], G)
    tl.assert_within_bound(first, C_ref, bound, "tcgen05 moe repeats")
    torch.cuda.synchronize()


@pytest.mark.parametrize("bad", [[1, 20, 40], [0, 25, 20], [0, 20, 41]])
def test_moe_tensor_memory_invalid_offsets(w, bad):
    torch = tl.torch_mod()
    K, N, G = 512, 256, 128
    lay = synth.make_moe_layer(0, 0, 2, K, N, G, seed=84, counts=[20, 20])
    packed, sp = _device_experts(w, lay["q"], lay["s"], G)
    M = 40
    ws = w.moe_workspace_for(2, M, 32, K, N, G)
    C = torch.full((M, N), 7.0, dtype=torch.float16, device="cuda")
    w.moe_gemm(tl.to_dev(lay["A"]), packed, sp, tl.to_dev(np.array(bad, np.int32)), N, G, max_rows=32, workspace=ws,
               out=C)
    assert w.w4a16_get_status(ws) == 10   # W4A16_ERR_VALUE
    assert bool((C == 7.0).all())
    C2 = w.moe_gemm(tl.to_dev(lay["A"]), packed, sp, tl.to_dev(lay["offsets"]), N, G, max_rows=32, workspace=ws)
    torch.cuda.synchronize()
    C_ref, bound = oracle.moe_gemm_ref(lay["A"], lay["offsets"], lay["q"], lay["s"], G)
    tl.assert_within_bound(C2.cpu().numpy(), C_ref, bound, "tcgen05 moe after invalid offsets")


def test_moe_tensor_memory_timeout_is_reported_and_context_survives(w):
    torch = tl.torch_mod()
    K, N, G = 2048, 1024, 128
    counts = [20, 30, 0, 18]
    lay = synth.make_moe_layer(0, 0, len(counts), K, N, G, seed=85, counts=counts)
    packed, sp = _device_experts(w, lay["q"], lay["s"], G)
    M = sum(counts)
    ws = w.moe_workspace_for(len(counts), M, 32, K, N, G)
    C = torch.full((M, N), 7.0, dtype=torch.float16, device="cuda")
    A_d, off_d = tl.to_dev(lay["A"]), tl.to_dev(lay["offsets"])
    try:
        w.w4a16_debug_set_wait_cycles(2_000_000)  # about a millisecond
        w.w4a16_debug_inject_stall(True)
        w.moe_gemm(A_d, packed, sp, off_d, N, G, max_rows=32, workspace=ws, out=C)
    finally:
        w.w4a16_debug_inject_stall(False)
        w.w4a16_debug_set_wait_cycles(0)
    assert w.w4a16_get_status(ws) == 7
    assert bool((C == 7.0).all())
    ws.zero_()
    C2 = _run(w, lay, N, 32, packed, sp, ws)
    C_ref, bound = oracle.moe_gemm_ref(lay["A"], lay["offsets"], lay["q"], lay["s"], G)
    tl.assert_within_bound(C2, C_ref, bound, "tcgen05 moe after timeout")
