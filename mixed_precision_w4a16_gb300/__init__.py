"""GB300 (sm_103a) W4A16 linear layer: thin Python binding of ``libw4a16.so``.

Every function below marshals arguments (torch tensors or raw integer device
pointers) into the C ABI declared in ``include/w4a16.h`` and checks the
returned status; all of the work happens in the library's CUDA kernels.
PyTorch only provides device memory and streams.

There is no CPU fallback: the first call into the library fails loudly when it
has not been built (``python -m mixed_precision_w4a16_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "W4A16Error", "lib", "Plan",
    "w4a16_packed_bytes", "w4a16_scales_count", "w4a16_workspace_bytes", "w4a16_plan",
    "w4a16_repack", "w4a16_quantize_repack", "w4a16_unpack", "w4a16_dequant", "w4a16_gemm", "w4a16_gemm_noalloc",
    "w4a16_get_status", "w4a16_repack_zeros", "w4a16_gemm_zp", "w4a16_dequant_zp", "w4a16_quantize_repack_zp",
    "w4a16_minmax_scales", "w4a16_moe_workspace_bytes", "w4a16_moe_gemm", "w4a16_debug_ablate",
    "ABLATE_NO_EVICT_FIRST", "ABLATE_STAGES_2", "ABLATE_NO_SWIZZLE",
    "w4a16_packed24_bytes", "w4a16_repack_24", "w4a16_unpack_24", "w4a16_workspace_bytes_24", "w4a16_gemm_24",
    "w4a16_debug_set_wait_cycles", "w4a16_debug_inject_stall", "w4a16_debug_force_path", "w4a16_status_string",
    "EXPORTED_SYMBOLS",
    "repack", "quantize_repack", "unpack", "dequant", "gemm", "workspace_for", "repack_zeros", "gemm_zp",
    "dequant_zp", "minmax_scales", "moe_gemm", "moe_workspace_for", "repack_24", "unpack_24", "gemm_24",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libw4a16.so")

EXPORTED_SYMBOLS = (
    "w4a16_status_string", "w4a16_abi_version", "w4a16_packed_bytes", "w4a16_scales_count",
    "w4a16_workspace_bytes", "w4a16_repack", "w4a16_unpack", "w4a16_dequant", "w4a16_gemm",
    "w4a16_get_status", "w4a16_plan", "w4a16_debug_set_wait_cycles", "w4a16_debug_inject_stall",
    "w4a16_gemm_noalloc", "w4a16_debug_force_path", "w4a16_quantize_repack", "w4a16_repack_zeros",
    "w4a16_gemm_zp", "w4a16_dequant_zp", "w4a16_quantize_repack_zp", "w4a16_minmax_scales",
    "w4a16_moe_workspace_bytes", "w4a16_moe_gemm", "w4a16_debug_ablate",
    "w4a16_packed24_bytes", "w4a16_repack_24", "w4a16_unpack_24", "w4a16_workspace_bytes_24", "w4a16_gemm_24",
)


class W4A16Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {w4a16_status_string(status)} ({status})")


class Plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "path", "m_tiles", "m_chunk", "n_tile", "k_tile", "units", "units_per_cta", "grid",
        "stages", "smem_bytes", "threads", "final_sum_warps")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m mixed_precision_w4a16_gb300.build` "
            "(the W4A16 path has no CPU fallback)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "w4a16_status_string": (ctypes.c_char_p, [i]),
        "w4a16_abi_version": (i, []),
        "w4a16_packed_bytes": (sz, [i, i]),
        "w4a16_scales_count": (sz, [i, i, i]),
        "w4a16_workspace_bytes": (sz, [i, i, i, i]),
        "w4a16_repack": (i, [vp, vp, i, i, i, vp, vp, vp]),
        "w4a16_unpack": (i, [vp, vp, i, i, i, vp, vp, vp]),
        "w4a16_dequant": (i, [vp, vp, i, i, i, vp, vp]),
        "w4a16_gemm": (i, [vp, vp, vp, vp, i, i, i, i, vp, sz, vp]),
        "w4a16_get_status": (i, [vp, vp]),
        "w4a16_plan": (i, [i, i, i, i, i, ctypes.POINTER(Plan)]),
        "w4a16_debug_set_wait_cycles": (None, [ctypes.c_longlong]),
        "w4a16_debug_inject_stall": (None, [i]),
        "w4a16_gemm_noalloc": (i, [vp, vp, vp, vp, i, i, i, i, vp]),
        "w4a16_debug_force_path": (None, [i]),
        "w4a16_debug_ablate": (None, [i]),
        "w4a16_packed24_bytes": (sz, [i, i]),
        "w4a16_repack_24": (i, [vp, vp, i, i, i, vp, vp, vp]),
        "w4a16_unpack_24": (i, [vp, i, i, vp, vp]),
        "w4a16_workspace_bytes_24": (sz, [i, i, i, i]),
        "w4a16_gemm_24": (i, [vp, vp, vp, vp, i, i, i, i, vp, sz, vp]),
        "w4a16_quantize_repack": (i, [vp, vp, i, i, i, vp, vp, vp]),
        "w4a16_repack_zeros": (i, [vp, i, i, i, vp, vp]),
        "w4a16_gemm_zp": (i, [vp, vp, vp, vp, vp, vp, i, i, i, i, vp, sz, vp]),
        "w4a16_dequant_zp": (i, [vp, vp, vp, i, i, i, vp, vp]),
        "w4a16_quantize_repack_zp": (i, [vp, vp, vp, i, i, i, vp, vp, vp]),
        "w4a16_minmax_scales": (i, [vp, i, i, i, vp, vp, vp]),
        "w4a16_moe_workspace_bytes": (sz, [i, i, i, i, i, i]),
        "w4a16_moe_gemm": (i, [vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, sz, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


_LIB = None


def _lib():
    """The loaded library (loaded on first use; raises ImportError when it was never built)."""
    global _LIB
    if _LIB is None:
        _LIB = _load()
    return _LIB


def __getattr__(name):
    if name == "lib":
        return _lib()
    raise AttributeError(name)


# ---------------------------------------------------------------------------
# argument marshalling
# ---------------------------------------------------------------------------

def _ptr(x):
    """Device pointer of a torch tensor (must be contiguous), an int, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if hasattr(x, "is_contiguous") and not x.is_contiguous():
            raise ValueError("W4A16 buffers must be contiguous")
        return x.data_ptr()
    raise TypeError(f"expected a tensor or an integer pointer, got {type(x)!r}")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != 0:
        raise W4A16Error(status, where)


# ---------------------------------------------------------------------------
# the C ABI, one Python function per entry point
# ---------------------------------------------------------------------------

def w4a16_status_string(status: int) -> str:
    return _lib().w4a16_status_string(int(status)).decode()


def w4a16_packed_bytes(K: int, N: int) -> int:
    return int(_lib().w4a16_packed_bytes(K, N))


def w4a16_scales_count(K: int, N: int, groupsize: int) -> int:
    return int(_lib().w4a16_scales_count(K, N, groupsize))


def w4a16_workspace_bytes(M: int, K: int, N: int, groupsize: int) -> int:
    return int(_lib().w4a16_workspace_bytes(M, K, N, groupsize))


def w4a16_abi_version() -> int:
    return int(_lib().w4a16_abi_version())


def w4a16_plan(M: int, K: int, N: int, groupsize: int, num_sms: int = 0) -> dict:
    p = Plan()
    _check(_lib().w4a16_plan(M, K, N, groupsize, num_sms, ctypes.byref(p)), "w4a16_plan")
    return p.as_dict()


def w4a16_repack(q, s, K, N, groupsize, packed, scales_p, stream=None):
    _check(_lib().w4a16_repack(_ptr(q), _ptr(s), K, N, groupsize, _ptr(packed), _ptr(scales_p), _stream(stream)),
           "w4a16_repack")


def w4a16_quantize_repack(w, s, K, N, groupsize, packed, scales_p, stream=None):
    _check(_lib().w4a16_quantize_repack(_ptr(w), _ptr(s), K, N, groupsize, _ptr(packed), _ptr(scales_p),
                                        _stream(stream)), "w4a16_quantize_repack")


def w4a16_quantize_repack_zp(w, s, z, K, N, groupsize, packed, scales_p, stream=None):
    _check(_lib().w4a16_quantize_repack_zp(_ptr(w), _ptr(s), _ptr(z), K, N, groupsize, _ptr(packed),
                                           _ptr(scales_p), _stream(stream)), "w4a16_quantize_repack_zp")


def w4a16_minmax_scales(w, K, N, groupsize, s, z, stream=None):
    _check(_lib().w4a16_minmax_scales(_ptr(w), K, N, groupsize, _ptr(s), _ptr(z), _stream(stream)),
           "w4a16_minmax_scales")


def w4a16_moe_workspace_bytes(E, M, max_rows, K, N, groupsize) -> int:
    return int(_lib().w4a16_moe_workspace_bytes(E, M, max_rows, K, N, groupsize))


def w4a16_moe_gemm(A, packed, scales_p, expert_offsets, C, E, M, max_rows, K, N, groupsize, workspace,
                   workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(_lib().w4a16_moe_gemm(_ptr(A), _ptr(packed), _ptr(scales_p), _ptr(expert_offsets), _ptr(C), E, M,
                                 max_rows, K, N, groupsize, _ptr(workspace), int(workspace_bytes),
                                 _stream(stream)), "w4a16_moe_gemm")


def w4a16_packed24_bytes(K, N) -> int:
    return int(_lib().w4a16_packed24_bytes(K, N))


def w4a16_repack_24(q, s, K, N, groupsize, packed24, scales_p, stream=None):
    _check(_lib().w4a16_repack_24(_ptr(q), _ptr(s), K, N, groupsize, _ptr(packed24), _ptr(scales_p),
                                  _stream(stream)), "w4a16_repack_24")


def w4a16_unpack_24(packed24, K, N, q, stream=None):
    _check(_lib().w4a16_unpack_24(_ptr(packed24), K, N, _ptr(q), _stream(stream)), "w4a16_unpack_24")


def w4a16_workspace_bytes_24(M, K, N, groupsize) -> int:
    return int(_lib().w4a16_workspace_bytes_24(M, K, N, groupsize))


def w4a16_gemm_24(A, packed24, scales_p, C, M, K, N, groupsize, workspace, workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(_lib().w4a16_gemm_24(_ptr(A), _ptr(packed24), _ptr(scales_p), _ptr(C), M, K, N, groupsize,
                                _ptr(workspace), int(workspace_bytes), _stream(stream)), "w4a16_gemm_24")


def w4a16_unpack(packed, scales_p, K, N, groupsize, q, s, stream=None):
    _check(_lib().w4a16_unpack(_ptr(packed), _ptr(scales_p), K, N, groupsize, _ptr(q), _ptr(s), _stream(stream)),
           "w4a16_unpack")


def w4a16_dequant(packed, scales_p, K, N, groupsize, bhat, stream=None):
    _check(_lib().w4a16_dequant(_ptr(packed), _ptr(scales_p), K, N, groupsize, _ptr(bhat), _stream(stream)),
           "w4a16_dequant")


def w4a16_gemm(A, packed, scales_p, C, M, K, N, groupsize, workspace, workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(_lib().w4a16_gemm(_ptr(A), _ptr(packed), _ptr(scales_p), _ptr(C), M, K, N, groupsize, _ptr(workspace),
                          int(workspace_bytes), _stream(stream)), "w4a16_gemm")


def w4a16_repack_zeros(z, K, N, groupsize, zeros_p, stream=None):
    _check(_lib().w4a16_repack_zeros(_ptr(z), K, N, groupsize, _ptr(zeros_p), _stream(stream)), "w4a16_repack_zeros")


def w4a16_gemm_zp(A, packed, scales_p, zeros_p, bias, C, M, K, N, groupsize, workspace, workspace_bytes=None,
                  stream=None):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(_lib().w4a16_gemm_zp(_ptr(A), _ptr(packed), _ptr(scales_p), _ptr(zeros_p), _ptr(bias), _ptr(C), M, K, N,
                                groupsize, _ptr(workspace), int(workspace_bytes), _stream(stream)), "w4a16_gemm_zp")


def w4a16_dequant_zp(packed, scales_p, zeros_p, K, N, groupsize, bhat, stream=None):
    _check(_lib().w4a16_dequant_zp(_ptr(packed), _ptr(scales_p), _ptr(zeros_p), K, N, groupsize, _ptr(bhat),
                                   _stream(stream)), "w4a16_dequant_zp")


# Size of the library's scratch array used by w4a16_gemm_noalloc (W4A16_NOALLOC_SCRATCH_BYTES).
W4A16_NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024


def w4a16_gemm_noalloc(A, packed, scales_p, C, M, K, N, groupsize, stream=None):
    """The allocation-free GEMM: same operands as w4a16_gemm, no workspace (the library's
    own scratch array is used; calls must not overlap on the GPU)."""
    _check(_lib().w4a16_gemm_noalloc(_ptr(A), _ptr(packed), _ptr(scales_p), _ptr(C), M, K, N, groupsize,
                                     _stream(stream)), "w4a16_gemm_noalloc")


def w4a16_get_status(workspace=None, stream=None) -> int:
    return int(_lib().w4a16_get_status(_ptr(workspace), _stream(stream)))


def w4a16_debug_set_wait_cycles(cycles: int) -> None:
    _lib().w4a16_debug_set_wait_cycles(int(cycles))


def w4a16_debug_inject_stall(enable: bool) -> None:
    _lib().w4a16_debug_inject_stall(1 if enable else 0)


def w4a16_debug_force_path(path: int) -> None:
    """0 = automatic kernel choice, 1 = streaming mma.sync kernel, 2 = tensor-memory kernel (mode by M),
    3 = tensor-memory kernel in strip pairs only, 4 = tensor-memory kernel in its wide mode where K allows."""
    _lib().w4a16_debug_force_path(int(path))


#: ablation switches of w4a16_debug_ablate (the MARLIN paper's Figure 12), combinable
ABLATE_NO_EVICT_FIRST = 1
ABLATE_STAGES_2 = 2
ABLATE_NO_SWIZZLE = 4


def w4a16_debug_ablate(flags: int) -> None:
    """Remove design choices for every later GEMM call: ABLATE_* bits, 0 = the full design."""
    _lib().w4a16_debug_ablate(int(flags))


# ---------------------------------------------------------------------------
# conveniences: allocate outputs with torch, then call the entry points
# ---------------------------------------------------------------------------

def _group_rows(K: int, groupsize: int) -> int:
    return 1 if groupsize in (-1, K) else K // groupsize


def workspace_for(M: int, K: int, N: int, groupsize: int, device=None):
    """A zeroed workspace tensor of w4a16_workspace_bytes(M, K, N, groupsize) bytes."""
    import torch
    nbytes = w4a16_workspace_bytes(M, K, N, groupsize)
    if nbytes == 0:
        raise W4A16Error(2, "w4a16_workspace_bytes")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


def repack(q, s, groupsize: int, stream=None):
    """q uint8[K][N], s fp16[K/G][N] (CUDA tensors) -> (packed int32[K*N/8], permuted fp16[K/G][N])."""
    import torch
    K, N = q.shape
    packed = torch.empty(K * N // 8, dtype=torch.int32, device=q.device)
    sp = torch.empty(s.numel(), dtype=torch.float16, device=q.device)  # permuted: fp16[N/128][K/G][128]
    w4a16_repack(q, s, K, N, groupsize, packed, sp, stream)
    return packed, sp


def quantize_repack(w, s, groupsize: int, z=None, stream=None):
    """w fp16[K][N], s fp16[K/G][N] (CUDA tensors) -> (packed int32[K*N/8], permuted fp16[K/G][N])
    with q = clamp(rint(w / s) + 8, 0, 15), or + z (uint8[K/G][N] zero codes) when z is given."""
    import torch
    K, N = w.shape
    packed = torch.empty(K * N // 8, dtype=torch.int32, device=w.device)
    sp = torch.empty(s.numel(), dtype=torch.float16, device=w.device)
    if z is None:
        w4a16_quantize_repack(w, s, K, N, groupsize, packed, sp, stream)
    else:
        w4a16_quantize_repack_zp(w, s, z, K, N, groupsize, packed, sp, stream)
    return packed, sp


def minmax_scales(w, groupsize: int, symmetric: bool = True, stream=None):
    """w fp16[K][N] (CUDA tensor) -> (s fp16[K/G][N], z uint8[K/G][N] or None) by the min-max rule:
    symmetric for the offset-8 format, else with zero codes."""
    import torch
    K, N = w.shape
    s = torch.empty((_group_rows(K, groupsize), N), dtype=torch.float16, device=w.device)
    z = None if symmetric else torch.empty((_group_rows(K, groupsize), N), dtype=torch.uint8, device=w.device)
    w4a16_minmax_scales(w, K, N, groupsize, s, z, stream)
    return s, z


def unpack(packed, scales_p, K: int, N: int, groupsize: int, stream=None):
    import torch
    q = torch.empty((K, N), dtype=torch.uint8, device=packed.device)
    s = torch.empty((_group_rows(K, groupsize), N), dtype=torch.float16, device=packed.device)
    w4a16_unpack(packed, scales_p, K, N, groupsize, q, s, stream)
    return q, s


def dequant(packed, scales_p, K: int, N: int, groupsize: int, stream=None):
    import torch
    bhat = torch.empty((K, N), dtype=torch.float16, device=packed.device)
    w4a16_dequant(packed, scales_p, K, N, groupsize, bhat, stream)
    return bhat


def repack_zeros(z, K: int, groupsize: int, stream=None):
    """z uint8[K/G][N] zero codes (CUDA tensor) -> zeros_p uint8[(K/G)*N], permuted like the scales."""
    import torch
    N = z.shape[1]
    zp = torch.empty(z.numel(), dtype=torch.uint8, device=z.device)
    w4a16_repack_zeros(z, K, N, groupsize, zp, stream)
    return zp


def dequant_zp(packed, scales_p, zeros_p, K: int, N: int, groupsize: int, stream=None):
    import torch
    bhat = torch.empty((K, N), dtype=torch.float16, device=packed.device)
    w4a16_dequant_zp(packed, scales_p, zeros_p, K, N, groupsize, bhat, stream)
    return bhat


def gemm_zp(A, packed, scales_p, zeros_p, bias, N: int, groupsize: int, workspace=None, out=None, stream=None):
    """C fp16[M][N] = A * (s (q - z)) + bias; zeros_p / bias may be None."""
    import torch
    M, K = A.shape
    if workspace is None:
        workspace = workspace_for(M, K, N, groupsize, A.device)
    C = out if out is not None else torch.empty((M, N), dtype=torch.float16, device=A.device)
    w4a16_gemm_zp(A, packed, scales_p, zeros_p, bias, C, M, K, N, groupsize, workspace, None, stream)
    return C


def gemm(A, packed, scales_p, N: int, groupsize: int, workspace=None, out=None, stream=None):
    """C fp16[M][N] = A fp16[M][K] * dequant(packed, scales_p)."""
    import torch
    M, K = A.shape
    if workspace is None:
        workspace = workspace_for(M, K, N, groupsize, A.device)
    C = out if out is not None else torch.empty((M, N), dtype=torch.float16, device=A.device)
    w4a16_gemm(A, packed, scales_p, C, M, K, N, groupsize, workspace, None, stream)
    return C


def moe_workspace_for(E: int, M: int, max_rows: int, K: int, N: int, groupsize: int, device=None):
    """A zeroed workspace tensor for w4a16_moe_gemm."""
    import torch
    nbytes = w4a16_moe_workspace_bytes(E, M, max_rows, K, N, groupsize)
    if nbytes == 0:
        raise W4A16Error(2, "w4a16_moe_workspace_bytes")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


def moe_gemm(A, packed, scales_p, expert_offsets, N: int, groupsize: int, max_rows: int = 0, workspace=None,
             out=None, stream=None):
    """Grouped expert GEMM: A fp16[M][K] (rows sorted by expert), packed / scales_p the E experts'
    repacked layers concatenated, expert_offsets int32[E+1] on the device -> C fp16[M][N]."""
    import torch
    M, K = A.shape
    E = expert_offsets.numel() - 1
    if workspace is None:
        workspace = moe_workspace_for(E, M, max_rows, K, N, groupsize, A.device)
    C = out if out is not None else torch.empty((M, N), dtype=torch.float16, device=A.device)
    w4a16_moe_gemm(A, packed, scales_p, expert_offsets, C, E, M, max_rows, K, N, groupsize, workspace, None,
                   stream)
    return C


def repack_24(q, s, groupsize: int, stream=None):
    """2:4-sparse dense codes q uint8[K][N], s fp16[K/G][N] (CUDA tensors) -> (packed24 int32[3*K*N/32],
    permuted scales fp16[K/G*N])."""
    import torch
    K, N = q.shape
    packed = torch.empty(3 * K * N // 32, dtype=torch.int32, device=q.device)
    sp = torch.empty(s.numel(), dtype=torch.float16, device=q.device)
    w4a16_repack_24(q, s, K, N, groupsize, packed, sp, stream)
    return packed, sp


def unpack_24(packed24, K: int, N: int, stream=None):
    import torch
    q = torch.empty((K, N), dtype=torch.uint8, device=packed24.device)
    w4a16_unpack_24(packed24, K, N, q, stream)
    return q


def gemm_24(A, packed24, scales_p, N: int, groupsize: int, workspace=None, out=None, stream=None):
    """C fp16[M][N] = A fp16[M][K] * dequant of the 2:4-sparse packed24."""
    import torch
    M, K = A.shape
    if workspace is None:
        nbytes = w4a16_workspace_bytes_24(M, K, N, groupsize)
        if nbytes == 0:
            raise W4A16Error(2, "w4a16_workspace_bytes_24")
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=A.device)
    C = out if out is not None else torch.empty((M, N), dtype=torch.float16, device=A.device)
    w4a16_gemm_24(A, packed24, scales_p, C, M, K, N, groupsize, workspace, None, stream)
    return C
