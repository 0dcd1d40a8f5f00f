"""Shared helpers of the GPU parity tests: seeded inputs -> device, library
calls through the C ABI binding, comparison against the CPU oracle."""
import numpy as np

import oracle
from mixed_precision_w4a16_gb300 import synth


def torch_mod():
    import torch
    return torch


def lib():
    from mixed_precision_w4a16_gb300 import build
    build.build()
    import mixed_precision_w4a16_gb300 as w
    return w


def to_dev(x):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def device_layer(w, q, s, G):
    """Repack on the device; returns (q_d, s_d, packed_d, sp_d)."""
    q_d, s_d = to_dev(q), to_dev(s)
    packed, sp = w.repack(q_d, s_d, G)
    return q_d, s_d, packed, sp


def run_gemm(w, A, packed, sp, N, G, workspace=None):
    torch = torch_mod()
    A_d = A if isinstance(A, torch.Tensor) else to_dev(A)
    M, K = A_d.shape
    C = w.gemm(A_d, packed, sp, N, G, workspace=workspace)
    torch.cuda.synchronize()
    return C


def c_numpy(C):
    return C.cpu().numpy()


def assert_within_bound(C_gpu, C_ref, bound, what=""):
    ex = oracle.error_excess(C_gpu.astype(np.float16), C_ref, bound)
    bad = np.argwhere(~(ex <= 0))
    if bad.size:
        m, n = bad[0]
        raise AssertionError(
            f"{what}: {bad.shape[0]} elements outside |C - C_ref| <= 4e-3*Bound + 1e-4; first at (m={m}, n={n}): "
            f"gpu={float(C_gpu[m, n])!r} ref={C_ref[m, n]!r} bound={bound[m, n]!r}")


def layer(M, K, N, G, seed):
    q, s = synth.make_weights(K, N, G, seed)
    A = synth.make_activations(M, K, seed)
    return A, q, s
