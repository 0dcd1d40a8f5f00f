"""The allocation-free GEMM entry point, checked against the workspace entry point.

Callers that cannot allocate device memory -- code recording a CUDA graph,
serving loops that must not allocate or synchronise on the hot path, plugin
hosts that hand a kernel only its inputs and outputs -- call
w4a16_gemm_noalloc, which runs on a scratch array compiled into the library
instead of a caller-provided workspace.  These tests call it twice in a row
through the C ABI (the second call reuses the scratch left by the first) and
compare each result with w4a16_gemm's, within the parity tolerance used
everywhere else: |C - C_ref| <= 4e-3 * sum_k |A B^| + 1e-4.

This file is named so that pytest collects it last; it passes alone in a
fresh process (the first call on the device performs the scratch set-up) and
after the other tests.
"""
import numpy as np
import pytest

import oracle
import w4a16_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K,N,G", [(16, 4096, 4096, 128), (33, 2048, 1024, -1), (1, 18432, 2048, 128)])
def test_noalloc_matches_workspace_entry_point_on_two_calls(M, K, N, G):
    w = tl.lib()
    torch = tl.torch_mod()
    A, q, s = tl.layer(M, K, N, G, seed=900 + M)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    A_d = tl.to_dev(A)
    with_workspace = tl.c_numpy(tl.run_gemm(w, A_d, packed, sp, N, G)).astype(np.float64)
    _, bound = oracle.gemm_ref(A, q, s, G)
    for call in range(2):
        C = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        w.w4a16_gemm_noalloc(A_d, packed, sp, C, M, K, N, G)
        torch.cuda.synchronize()
        tl.assert_within_bound(C.cpu().numpy(), with_workspace, bound, f"no-alloc call {call + 1}, {(M, K, N, G)}")
