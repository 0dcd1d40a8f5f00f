"""CPU oracle for the W4A16 (MARLIN-style) linear layer -- TEST INFRASTRUCTURE.

This package is the plain, slow, obviously correct statement of what the
product computes.  It is written in numpy, in float64, from the pages that
describe the method, and it shares no code with the CUDA library (no kernels,
headers, helpers, tables or constant generators).

Only the test suite (``tests/``), ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product path (``mixed_precision_w4a16_gb300``) never imports it and fails
loudly when its CUDA library is missing.

Every function here is pinned by ``tests/test_oracle.py`` to something other
than itself (IEEE-754 binary16 golden values, exact integer brute force,
closed forms, the PTX ISA fragment table, round trips); none is "parity
unpinned".
"""
from .w4a16_oracle import (  # noqa: F401
    Z_POINT,
    fp16_bits_to_f64,
    f64_to_fp16_bits,
    dequant_exact,
    dequant_fp16_bits,
    gemm_ref,
    error_ok,
    error_excess,
    packed_position,
    scale_position,
    quantize,
    quantize_zp,
    minmax_scales,
    moe_gemm_ref,
    sparse24_compress,
    sparse24_expand,
    gemm24_ref,
    check_expert_offsets,
    dequant_exact_zp,
    dequant_fp16_bits_zp,
    gemm_ref_zp,
    repack_zeros,
    repack,
    unpack,
    TOL_REL,
    TOL_ABS,
)
