"""Seeded random shapes through every kernel and mode, against the oracle element by element.

Each case draws K (a multiple of 128 up to 4608, so K/128 odd, K/256 odd and K % 512 == 0 all
occur), N (a multiple of 128 up to 2304, odd strip counts included), M (1 to 300, across the
16-, 128- and 256-row launch chunks), the group size (128 or per column) and the kernel choice
(automatic, streaming, tensor memory by M, strip pairs only, wide mode forced).  The draws are
fixed by the seed, so a failure names a reproducible case."""
import numpy as np
import pytest

import oracle
import w4a16_testlib as tl

pytestmark = pytest.mark.gpu

PATHS = (0, 1, 2, 3, 4)


def _cases(n, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        K = 128 * int(rng.integers(1, 37))
        N = 128 * int(rng.integers(1, 19))
        M = int(rng.choice([int(rng.integers(1, 17)), int(rng.integers(17, 129)), int(rng.integers(129, 301))]))
        G = 128 if rng.random() < 0.75 else -1
        path = PATHS[i % len(PATHS)]
        out.append((M, K, N, G, path))
    return out


CASES = _cases(100)


@pytest.fixture(scope="module")
def w():
    return tl.lib()


@pytest.mark.parametrize("M,K,N,G,path", CASES, ids=[f"M{m}-K{k}-N{n}-G{g}-p{p}" for m, k, n, g, p in CASES])
def test_random_shape_matches_oracle(w, M, K, N, G, path):
    A, q, s = tl.layer(M, K, N, G, seed=M * 7 + K + N)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    w.w4a16_debug_force_path(path)
    try:
        C = tl.c_numpy(tl.run_gemm(w, A, packed, sp, N, G))
    finally:
        w.w4a16_debug_force_path(0)
    C_ref, bound = oracle.gemm_ref(A, q, s, G)
    tl.assert_within_bound(C, C_ref, bound, f"M={M} K={K} N={N} G={G} path={path}")


def _moe_cases(n, seed=2027):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        E = int(rng.integers(1, 13))
        hot = int(rng.choice([8, 16, 40, 150]))  # the largest expert: streaming or tensor-memory path
        counts = rng.integers(0, hot + 1, E)
        counts[int(rng.integers(0, E))] = hot
        K = 128 * int(rng.integers(1, 25))
        N = 128 * int(rng.integers(1, 13))
        G = 128 if rng.random() < 0.75 else -1
        out.append(([int(c) for c in counts], K, N, G))
    return out


MOE_CASES = _moe_cases(30)


@pytest.mark.parametrize("counts,K,N,G", MOE_CASES, ids=[f"E{len(c)}-max{max(c)}-K{k}-N{n}-G{g}" for c, k, n, g in MOE_CASES])
def test_random_grouped_gemm_matches_oracle(w, counts, K, N, G):
    from mixed_precision_w4a16_gb300 import synth
    torch = tl.torch_mod()
    lay = synth.make_moe_layer(0, 0, len(counts), K, N, G, seed=sum(counts) + K + N, counts=counts)
    packed, sps = [], []
    for e in range(len(counts)):
        pk, sp = w.repack(tl.to_dev(lay["q"][e]), tl.to_dev(lay["s"][e]), G)
        packed.append(pk)
        sps.append(sp)
    C = w.moe_gemm(tl.to_dev(lay["A"]), torch.cat(packed), torch.cat(sps), tl.to_dev(lay["offsets"]), N, G,
                   max_rows=max(counts))
    torch.cuda.synchronize()
    C_ref, bound = oracle.moe_gemm_ref(lay["A"], lay["offsets"], lay["q"], lay["s"], G)
    tl.assert_within_bound(C.cpu().numpy(), C_ref, bound, f"counts={counts} K={K} N={N} G={G}")
    assert w.w4a16_get_status() == 0
