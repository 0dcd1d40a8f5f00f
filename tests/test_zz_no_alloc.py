"""The allocation-free GEMM entry point, checked against the workspace entry point.

Callers that cannot allocate device memory -- code recording a CUDA graph,
serving loops that must not allocate or synchronise on the hot path, plugin
hosts that hand a kernel only its inputs and outputs -- call
w4a16_gemm_noalloc, which runs on a scratch array compiled into the library
instead of a caller-provided workspace.  These tests call it twice in a row
through the C ABI (the second call reuses the scratch left by the first).
Both entry points run the same plan on the same kernel with a fixed-order
reduction, so each result must equal w4a16_gemm's bit for bit; each is also
held to the oracle within the parity tolerance used everywhere else,
|C - C_ref| <= 4e-3 * sum_k |A B^| + 1e-4.

This file is named so that pytest collects it last; it passes alone in a
fresh process (the first call on the device performs the scratch set-up) and
after the other tests.
"""
import numpy as np
import pytest

import oracle
import w4a16_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K,N,G", [(16, 4096, 4096, 128), (33, 2048, 1024, -1), (1, 18432, 2048, 128),
                                     (32, 2048, 2048, 128)])
def test_noalloc_matches_workspace_entry_point_on_two_calls(M, K, N, G):
    w = tl.lib()
    torch = tl.torch_mod()
    A, q, s = tl.layer(M, K, N, G, seed=900 + M)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    A_d = tl.to_dev(A)
    with_workspace = tl.c_numpy(tl.run_gemm(w, A_d, packed, sp, N, G))
    C_ref, bound = oracle.gemm_ref(A, q, s, G)
    for call in range(2):
        C = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        w.w4a16_gemm_noalloc(A_d, packed, sp, C, M, K, N, G)
        torch.cuda.synchronize()
        got = C.cpu().numpy()
        what = f"no-alloc call {call + 1}, {(M, K, N, G)}"
        assert np.array_equal(got.view(np.uint16), with_workspace.view(np.uint16)), what + ": not bitwise equal"
        tl.assert_within_bound(got, C_ref, bound, what)
    assert w.w4a16_get_status(None) == 0


def test_noalloc_rejects_plans_larger_than_its_array():
    w = tl.lib()
    torch = tl.torch_mod()
    M, K, N, G = 128, 4096, 16384, 128
    assert w.w4a16_workspace_bytes(M, K, N, G) > w.W4A16_NOALLOC_SCRATCH_BYTES
    A_d = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    packed = torch.zeros(K * N // 8, dtype=torch.int32, device="cuda")
    sp = torch.zeros((K // 128) * N, dtype=torch.float16, device="cuda")
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    with pytest.raises(w.W4A16Error) as e:
        w.w4a16_gemm_noalloc(A_d, packed, sp, C, M, K, N, G)
    assert e.value.status == 5  # W4A16_ERR_WORKSPACE, before any launch
    torch.cuda.synchronize()
    assert torch.isnan(C).all()


def test_noalloc_timeout_is_reported_until_read():
    """A pipeline wait that runs out inside the allocation-free call (stage never
    filled, short bound) is recorded in the library's array; later calls do not
    clear it, w4a16_get_status(NULL) reports and clears it, and the next call is
    correct."""
    w = tl.lib()
    torch = tl.torch_mod()
    M, K, N, G = 16, 4096, 4096, 128
    A, q, s = tl.layer(M, K, N, G, seed=931)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    A_d = tl.to_dev(A)
    C = torch.full((M, N), 7.0, dtype=torch.float16, device="cuda")
    try:
        w.w4a16_debug_set_wait_cycles(2_000_000)  # about a millisecond
        w.w4a16_debug_inject_stall(True)
        w.w4a16_gemm_noalloc(A_d, packed, sp, C, M, K, N, G)
    finally:
        w.w4a16_debug_inject_stall(False)
        w.w4a16_debug_set_wait_cycles(0)
    torch.cuda.synchronize()
    assert torch.all(C == 7.0)  # nothing written after the abort
    # a good call in between must neither hide the timeout nor be disturbed by it
    w.w4a16_gemm_noalloc(A_d, packed, sp, C, M, K, N, G)
    assert w.w4a16_get_status(None) == 7
    assert w.w4a16_get_status(None) == 0
    C_ref, bound = oracle.gemm_ref(A, q, s, G)
    tl.assert_within_bound(tl.c_numpy(C), C_ref, bound, "no-alloc after timeout")
    C2 = torch.empty_like(C)
    w.w4a16_gemm_noalloc(A_d, packed, sp, C2, M, K, N, G)
    torch.cuda.synchronize()
    assert torch.equal(C, C2)
