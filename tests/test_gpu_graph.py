"""The GEMM entry points inside CUDA graphs: each call is captured once and
replayed with new inputs written into the captured buffers (new activations;
for the grouped GEMM also a new routing, since its expert offsets are read on
the device), and every replay is checked against the oracle."""
import numpy as np
import pytest

import oracle
from mixed_precision_w4a16_gb300 import synth
import w4a16_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w():
    return tl.lib()


def _capture(torch, fn):
    fn()  # first call outside the capture: per-device set-up, kernel attributes
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("M", [8, 40])
def test_gemm_replays_with_new_activations(w, M):
    torch = tl.torch_mod()
    K, N, G = 2048, 1024, 128
    _, q, s = tl.layer(M, K, N, G, seed=501)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    A_d = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    C = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    ws = w.workspace_for(M, K, N, G)
    g = _capture(torch, lambda: w.w4a16_gemm(A_d, packed, sp, C, M, K, N, G, ws))
    for r in range(3):
        A = synth.make_activations(M, K, seed=600 + r)
        A_d.copy_(torch.from_numpy(A))
        g.replay()
        torch.cuda.synchronize()
        C_ref, bound = oracle.gemm_ref(A, q, s, G)
        tl.assert_within_bound(C.cpu().numpy(), C_ref, bound, f"replay {r}, M={M}")
    assert w.w4a16_get_status(ws) == 0


def test_noalloc_gemm_replays(w):
    torch = tl.torch_mod()
    M, K, N, G = 16, 1024, 768, 128
    _, q, s = tl.layer(M, K, N, G, seed=502)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    A_d = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    C = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    g = _capture(torch, lambda: w.w4a16_gemm_noalloc(A_d, packed, sp, C, M, K, N, G))
    for r in range(3):
        A = synth.make_activations(M, K, seed=610 + r)
        A_d.copy_(torch.from_numpy(A))
        g.replay()
        torch.cuda.synchronize()
        C_ref, bound = oracle.gemm_ref(A, q, s, G)
        tl.assert_within_bound(C.cpu().numpy(), C_ref, bound, f"no-alloc replay {r}")


def test_moe_gemm_replays_with_a_new_routing(w):
    """Same number of rows, different rows per expert at every replay: the captured launch finds the
    new segments from the offsets in device memory."""
    torch = tl.torch_mod()
    E, K, N, G, M = 8, 1024, 512, 128, 32
    routings = [[4, 4, 4, 4, 4, 4, 4, 4], [0, 20, 0, 0, 3, 0, 9, 0], [32, 0, 0, 0, 0, 0, 0, 0],
                [1, 2, 3, 4, 5, 6, 7, 4]]
    lay0 = synth.make_moe_layer(0, 0, E, K, N, G, seed=503, counts=routings[0])
    packed, sps = [], []
    for e in range(E):
        pk, sp = w.repack(tl.to_dev(lay0["q"][e]), tl.to_dev(lay0["s"][e]), G)
        packed.append(pk)
        sps.append(sp)
    packed, sp = torch.cat(packed), torch.cat(sps)
    A_d = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    off_d = torch.from_numpy(lay0["offsets"]).cuda()
    C = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    ws = w.moe_workspace_for(E, M, 16, K, N, G)
    g = _capture(torch, lambda: w.w4a16_moe_gemm(A_d, packed, sp, off_d, C, E, M, 16, K, N, G, ws))
    for r, counts in enumerate(routings):
        offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        A = synth.make_activations(M, K, seed=620 + r)
        A_d.copy_(torch.from_numpy(A))
        off_d.copy_(torch.from_numpy(offsets))
        g.replay()
        torch.cuda.synchronize()
        C_ref, bound = oracle.moe_gemm_ref(A, offsets, lay0["q"], lay0["s"], G)
        tl.assert_within_bound(C.cpu().numpy(), C_ref, bound, f"routing {counts}")
    assert w.w4a16_get_status(ws) == 0
