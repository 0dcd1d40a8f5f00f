"""The Figure 12 ablation switches on the GPU: every switch and their
combination leaves the result bitwise identical to the full design (none of
them changes the order of the arithmetic) on both GEMM kernels and the grouped
expert GEMM, and within the parity bound of the oracle."""
import numpy as np
import pytest

import oracle
from mixed_precision_w4a16_gb300 import synth
import w4a16_testlib as tl

pytestmark = pytest.mark.gpu

FLAGS = [1, 2, 4, 7]


@pytest.fixture(scope="module")
def w():
    return tl.lib()


@pytest.mark.parametrize("M", [3, 16, 40, 128])
@pytest.mark.parametrize("G", [128, -1])
def test_ablations_are_bitwise_identical_and_within_bound(w, M, G):
    K, N = 2048, 512
    A, q, s = tl.layer(M, K, N, G, seed=M + 3)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    base = tl.c_numpy(tl.run_gemm(w, A, packed, sp, N, G))
    C_ref, bound = oracle.gemm_ref(A, q, s, G)
    tl.assert_within_bound(base, C_ref, bound, f"full design M={M}")
    try:
        for f in FLAGS:
            w.w4a16_debug_ablate(f)
            C = tl.c_numpy(tl.run_gemm(w, A, packed, sp, N, G))
            assert np.array_equal(C.view(np.uint16), base.view(np.uint16)), f"flags {f}"
    finally:
        w.w4a16_debug_ablate(0)
    assert w.w4a16_get_status() == 0


def test_ablations_on_the_grouped_gemm(w):
    torch = tl.torch_mod()
    K, N, G = 1024, 384, 128
    lay = synth.make_moe_layer(24, 2, 8, K, N, G, seed=9, skew=1.0)
    packed, sps = [], []
    for e in range(8):
        pk, sp = w.repack(tl.to_dev(lay["q"][e]), tl.to_dev(lay["s"][e]), G)
        packed.append(pk)
        sps.append(sp)
    packed, sp = torch.cat(packed), torch.cat(sps)
    A_d, off_d = tl.to_dev(lay["A"]), tl.to_dev(lay["offsets"])

    def run():
        C = w.moe_gemm(A_d, packed, sp, off_d, N, G, max_rows=16)
        torch.cuda.synchronize()
        return C.cpu().numpy()

    base = run()
    C_ref, bound = oracle.moe_gemm_ref(lay["A"], lay["offsets"], lay["q"], lay["s"], G)
    tl.assert_within_bound(base, C_ref, bound, "grouped, full design")
    try:
        for f in FLAGS:
            w.w4a16_debug_ablate(f)
            assert np.array_equal(run().view(np.uint16), base.view(np.uint16)), f"flags {f}"
    finally:
        w.w4a16_debug_ablate(0)
