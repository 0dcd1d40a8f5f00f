"""Parity at the benchmarked sizes, in the launch configuration bench.py times.

The 7B- and 70B-style layers are compared with the oracle on every output
element (the oracle runs over blocks of columns to bound its memory).  The big
layer and the prefill layer are compared on a sample of output columns (all M
rows x the first and last 256 columns and 2048 seeded random ones); columns are
independent, so this is an element-by-element check of those outputs."""
import numpy as np
import pytest

import oracle
from mixed_precision_w4a16_gb300 import synth
import w4a16_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w():
    return tl.lib()


def sample_cols(N, seed=0):
    rng = np.random.default_rng(seed)
    cols = np.concatenate([np.arange(min(256, N)), np.arange(max(0, N - 256), N), rng.choice(N, min(2048, N), False)])
    return np.unique(cols)


def check_layer(w, K, N, G, Ms, seed, every_column=False):
    q, s = synth.make_weights(K, N, G, seed)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    if every_column:
        blocks = [np.arange(c0, min(N, c0 + 2048)) for c0 in range(0, N, 2048)]
    else:
        blocks = [sample_cols(N, seed)]
    ws = w.workspace_for(max(Ms), K, N, G)
    for M in Ms:
        ws_need = w.w4a16_workspace_bytes(M, K, N, G)
        assert ws_need <= ws.numel()
        A = synth.make_activations(M, K, seed * 1000 + M)
        C = tl.c_numpy(tl.run_gemm(w, A, packed, sp, N, G, workspace=ws))
        for cols in blocks:
            C_ref, bound = oracle.gemm_ref(A, np.ascontiguousarray(q[:, cols]), np.ascontiguousarray(s[:, cols]), G)
            tl.assert_within_bound(C[:, cols], C_ref, bound, f"K={K} N={N} G={G} M={M} columns {cols[0]}..{cols[-1]}")
    assert w.w4a16_get_status(ws) == 0


def test_big_layer_sweep(w):
    check_layer(w, 18432, 73728, 128, [1, 2, 4, 8, 16, 32, 64, 128], seed=200)


@pytest.mark.parametrize("K,N", [(4096, 12288), (4096, 4096), (4096, 22016), (11008, 4096)])
def test_7b_decode_layers(w, K, N):
    check_layer(w, K, N, 128, [1, 16], seed=100 + K % 97, every_column=True)


@pytest.mark.parametrize("K,N", [(8192, 10240), (8192, 8192), (8192, 57344), (28672, 8192)])
@pytest.mark.parametrize("G", [128, -1])
def test_70b_layers(w, K, N, G):
    check_layer(w, K, N, G, [32], seed=300 + N % 89, every_column=True)


def test_prefill_layer(w):
    # the tensor-memory kernel's wide mode: 256 token rows per launch (300 = two launches of 160)
    check_layer(w, 8192, 28672, 128, [256, 300, 512, 1024], seed=400)


def test_big_layer_wide_mode(w):
    check_layer(w, 18432, 73728, 128, [200], seed=210)


# K not a multiple of 512: the tensor-memory path runs 256-row units, and some CTAs' ranges end
# one unit past a strip boundary, so that their last segment has fewer chunks than MMA issuers
# (the host tests check that these plans contain such segments).  Every column is checked.
@pytest.mark.parametrize("M,K,N", [(32, 11008, 4096), (64, 11008, 4096), (32, 2816, 4096)])
def test_segments_with_idle_issuers(w, M, K, N):
    G = 128
    q, s = synth.make_weights(K, N, G, 600 + M)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    A = synth.make_activations(M, K, 700 + M)
    ws = w.workspace_for(M, K, N, G)
    C_ref, bound = oracle.gemm_ref(A, q, s, G)
    for _ in range(3):  # the hazard was timing-dependent: repeat on the same buffers
        C = tl.c_numpy(tl.run_gemm(w, A, packed, sp, N, G, workspace=ws))
        tl.assert_within_bound(C, C_ref, bound, f"K={K} N={N} M={M}")
    assert w.w4a16_get_status(ws) == 0


# Standing guard for the tensor-memory kernel's hand-off protocol.  Two races were found in it
# by reading (an issuer's parity wait naming the wrong phase of an activation stage; an idle
# issuer committing a segment early); both showed only under particular timings, one of them in
# about 1 of 6 runs of the 70B-style down-projection below.  The reduction order is fixed, so
# every repetition on the same buffers must equal the first bit for bit; the first is held to
# the oracle on sampled columns (all columns for the small shapes).
# The wide mode (one strip per unit, four A buffers) is guarded the same way, at its own sizes and
# forced onto a small token count.
@pytest.mark.parametrize("M,K,N,G,reps,force", [
    (32, 8192, 57344, -1, 24, 0), (32, 11008, 4096, 128, 24, 0), (64, 11008, 4096, 128, 24, 0),
    (32, 2816, 4096, 128, 24, 0), (256, 8192, 28672, 128, 24, 0), (1000, 8192, 4096, -1, 24, 0),
    (32, 8192, 57344, -1, 24, 4)])
def test_tensor_memory_protocol_repeats(w, M, K, N, G, reps, force):
    w.w4a16_debug_force_path(force)
    try:
        _protocol_repeats(w, M, K, N, G, reps)
    finally:
        w.w4a16_debug_force_path(0)


def _protocol_repeats(w, M, K, N, G, reps):
    torch = tl.torch_mod()
    q, s = synth.make_weights(K, N, G, 800 + M + K % 7)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    A = synth.make_activations(M, K, 900 + M)
    A_d = tl.to_dev(A)
    ws = w.workspace_for(M, K, N, G)
    assert w.w4a16_plan(M, K, N, G, 0)["path"] == 2
    C = w.gemm(A_d, packed, sp, N, G, workspace=ws)
    first = tl.c_numpy(C).copy()
    cols = sample_cols(N, 5) if N > 8192 else np.arange(N)
    C_ref, bound = oracle.gemm_ref(A, np.ascontiguousarray(q[:, cols]), np.ascontiguousarray(s[:, cols]), G)
    tl.assert_within_bound(first[:, cols], C_ref, bound, f"K={K} N={N} G={G} M={M}")
    first_d = C.clone()
    mismatched = []
    for r in range(reps - 1):
        C = w.gemm(A_d, packed, sp, N, G, workspace=ws)
        if not torch.equal(C.view(torch.int16), first_d.view(torch.int16)):
            mismatched.append(r + 2)
    torch.cuda.synchronize()
    assert not mismatched, f"repetitions {mismatched} differ from the first"
    assert w.w4a16_get_status(ws) == 0
