"""Host-side checks of the C ABI (no GPU): the library builds, loads, exports
every entry point the header declares, and its pure host logic (sizes, work
plan, argument validation) behaves as documented."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


@pytest.fixture(scope="module")
def w():
    from mixed_precision_w4a16_gb300 import build
    build.build()
    import mixed_precision_w4a16_gb300 as w
    return w


def _declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"W4A16_API\s+[\w\s\*]+?\b(w4a16_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    syms = _declared_symbols()
    for name in ("w4a16_repack", "w4a16_gemm", "w4a16_workspace_bytes", "w4a16_get_status"):
        assert name in syms


def test_library_exports_every_declared_symbol(w):
    lib = ctypes.CDLL(w.LIB_PATH)
    for name in _declared_symbols():
        assert hasattr(lib, name), name
    assert set(_declared_symbols()) <= set(w.EXPORTED_SYMBOLS) | {"w4a16_abi_version"}


def test_binding_has_every_entry_point_under_its_c_name(w):
    missing = [name for name in _declared_symbols() if not callable(getattr(w, name, None))]
    assert not missing, missing
    assert w.w4a16_abi_version() == 1


def test_library_exports_nothing_else(w):
    # -fvisibility=hidden: only the declared C entry points are dynamic symbols
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", w.LIB_PATH], capture_output=True, text=True).stdout
    ours = sorted(l.split()[-1] for l in out.splitlines() if " T " in l and "w4a16" in l)
    assert ours == _declared_symbols()


def test_sizes(w):
    assert w.w4a16_packed_bytes(4096, 12288) == 4096 * 12288 // 2
    assert w.w4a16_scales_count(4096, 12288, 128) == 32 * 12288
    assert w.w4a16_scales_count(4096, 12288, -1) == 12288
    assert w.w4a16_scales_count(4096, 12288, 4096) == 12288
    assert w.w4a16_packed_bytes(100, 64) == 0
    assert w.w4a16_scales_count(1024, 96, 128) == 0      # N % 128
    assert w.w4a16_scales_count(1024, 192, 128) == 0
    assert w.w4a16_scales_count(1024, 128, 64) == 0      # unsupported group size


def test_status_strings(w):
    assert w.w4a16_status_string(0) == "W4A16_OK"
    assert w.w4a16_status_string(7) == "W4A16_ERR_TIMEOUT"
    assert w.w4a16_status_string(99) == "W4A16_ERR_UNKNOWN"


SHAPES = [(1, 1024, 1024), (16, 1024, 1024), (16, 4096, 12288), (1, 11008, 4096), (32, 8192, 57344),
          (64, 18432, 73728), (16, 18432, 73728), (100, 4096, 4096), (3, 128, 128), (40, 256, 384), (8, 11008, 4096)]


@pytest.mark.parametrize("M,K,N", SHAPES)
def test_plan_stripes_cover_every_unit_once(w, M, K, N):
    for sms in (152, 148, 7):
        p = w.w4a16_plan(M, K, N, 128, sms)
        # streaming kernel: 2..16 pieces of 64 rows, one strip; tensor-memory kernel: 1, 2 or 4 chunks of
        # 128 rows, a strip pair (the last pair has one strip when N / 128 is odd), or in its wide mode
        # (from 129 token rows, K a multiple of 512) 4 chunks of one strip
        allowed = (128, 256, 512, 768, 1024) if p["path"] == 1 else (128, 256, 512)
        wide = p["path"] == 2 and M >= 129 and K % 512 == 0
        assert p["k_tile"] in allowed and K % p["k_tile"] == 0
        assert p["n_tile"] == (128 if p["path"] == 1 or wide else 256)
        KU = K // p["k_tile"]
        assert p["units"] == -(-N // p["n_tile"]) * KU
        T, grid, U = p["units_per_cta"], p["grid"], p["units"]
        assert grid <= sms and grid * T >= U and (grid - 1) * T < U
        assert p["m_chunk"] == 8 * p["m_tiles"] and p["m_chunk"] >= min(M, 32 if p["path"] == 1 else 128)
        assert p["smem_bytes"] <= 232448 and p["stages"] >= 2
        # every unit belongs to exactly one CTA; every CTA has work
        owner = [u // T for u in range(U)]
        assert owner[-1] == grid - 1
        # split column tiles: the partial-sum slot (cta, first-or-later) is unique
        slots = set()
        for j in range(U // KU):
            c_first, c_last = (j * KU) // T, min(((j + 1) * KU - 1) // T, grid - 1)
            assert c_first == owner[j * KU] and c_last == owner[(j + 1) * KU - 1]
            if c_first == c_last:
                continue
            for c in range(c_first, c_last + 1):
                slot = 2 * c if j == (c * T) // KU else 2 * c + 1
                assert slot not in slots
                slots.add(slot)
        assert all(s < 2 * grid for s in slots)


def test_plan_token_tiles_and_kernel_choice(w):
    ms = (1, 8, 9, 16, 17, 32, 33, 64, 128, 129, 250, 300, 1000)
    plans = [w.w4a16_plan(m, 1024, 1024, 128, 152) for m in ms]
    # up to 16 rows: streaming mma.sync kernel, 8-row token tiles
    assert [p["path"] for p in plans] == [1] * 4 + [2] * 9
    assert [p["m_chunk"] for p in plans[:4]] == [8, 8, 16, 16]
    # from 17 rows: tensor-memory kernel, tokens padded to 16 (the MMA's N), strip pairs and at most
    # 128 rows per launch; from 129 rows its wide mode, one strip per unit and the rows dealt evenly
    # to launches of at most 256
    assert [p["m_chunk"] for p in plans[4:]] == [32, 32, 48, 64, 128, 144, 256, 160, 256]
    assert [p["n_tile"] for p in plans[4:]] == [256] * 5 + [128] * 4
    assert all(p["threads"] == 640 for p in plans[4:]) and all(p["threads"] == 288 for p in plans[:4])
    # the wide mode needs units of four 128-row chunks: K = 768 stays in strip pairs
    p = w.w4a16_plan(300, 768, 1024, 128, 152)
    assert (p["n_tile"], p["m_chunk"], p["k_tile"]) == (256, 128, 256)


def test_force_path_knob(w):
    try:
        w.w4a16_debug_force_path(2)
        assert w.w4a16_plan(1, 1024, 1024, 128, 152)["path"] == 2
        w.w4a16_debug_force_path(1)
        assert w.w4a16_plan(200, 1024, 1024, 128, 152)["path"] == 1
        w.w4a16_debug_force_path(3)  # tensor memory, strip pairs only
        p = w.w4a16_plan(1000, 1024, 1024, 128, 152)
        assert (p["path"], p["n_tile"], p["m_chunk"]) == (2, 256, 128)
        w.w4a16_debug_force_path(4)  # tensor memory, wide mode wherever K allows
        p = w.w4a16_plan(32, 1024, 1024, 128, 152)
        assert (p["path"], p["n_tile"], p["m_chunk"]) == (2, 128, 32)
        assert w.w4a16_plan(32, 768, 1024, 128, 152)["n_tile"] == 256
    finally:
        w.w4a16_debug_force_path(0)
    assert w.w4a16_plan(200, 1024, 1024, 128, 152)["path"] == 2


# a streaming-kernel case and a tensor-memory case (two-chunk units: K a multiple of 256, not 512)
# whose full-design plans are deeper than 2 stages
ABLATION_CASES = ((4, 4096, 1024), (64, 4352, 4096))


def _plans(w):
    return [w.w4a16_plan(m, k, n, 128, 152) for m, k, n in ABLATION_CASES]


def test_ablation_switch_sets_two_stages(w):
    full = _plans(w)
    assert [p["path"] for p in full] == [1, 2]
    assert all(p["stages"] > 2 for p in full)
    try:
        w.w4a16_debug_ablate(w.ABLATE_STAGES_2)
        abl = _plans(w)
        assert [p["stages"] for p in abl] == [2, 2]
        # nothing else of the plan changes: same kernel, tiles and split
        for a, f in zip(abl, full):
            assert {k: v for k, v in a.items() if k not in ("stages", "smem_bytes")} == \
                {k: v for k, v in f.items() if k not in ("stages", "smem_bytes")}
        w.w4a16_debug_ablate(w.ABLATE_NO_EVICT_FIRST | w.ABLATE_NO_SWIZZLE)
        assert _plans(w) == full
    finally:
        w.w4a16_debug_ablate(0)
    assert _plans(w) == full


def test_moe_gemm_validates_before_touching_the_device(w):
    L = w.lib
    # E out of range, bad K, null pointers, M == 0
    assert L.w4a16_moe_gemm(16, 16, 16, 16, 16, 0, 8, 8, 1024, 1024, 128, 16, 1 << 20, None) == 2
    assert L.w4a16_moe_gemm(16, 16, 16, 16, 16, 4097, 8, 8, 1024, 1024, 128, 16, 1 << 20, None) == 2
    assert L.w4a16_moe_gemm(16, 16, 16, 16, 16, 4, 8, 8, 1000, 1024, 128, 16, 1 << 20, None) == 2
    assert L.w4a16_moe_gemm(16, 16, 16, 16, 16, 4, -1, 8, 1024, 1024, 128, 16, 1 << 20, None) == 2


def test_plan_rejects_bad_shapes(w):
    with pytest.raises(w.W4A16Error):
        w.w4a16_plan(16, 1000, 1024, 128, 152)
    with pytest.raises(w.W4A16Error):
        w.w4a16_plan(16, 1024, 1000, 128, 152)
    with pytest.raises(w.W4A16Error):
        w.w4a16_plan(16, 1024, 1024, 32, 152)


def test_gemm_validates_before_touching_the_device(w):
    L = w.lib
    # bad shapes, bad group, null pointers: rejected on the host with the documented codes
    assert L.w4a16_gemm(16, 16, 16, 16, 4, 1000, 1024, 128, 16, 1 << 20, None) == 2
    assert L.w4a16_gemm(16, 16, 16, 16, 4, 1024, 1024, 96, 16, 1 << 20, None) == 3
    assert L.w4a16_gemm(None, 16, 16, 16, 4, 1024, 1024, 128, 16, 1 << 20, None) == 1
    assert L.w4a16_gemm(16, 16, 16, 16, 4, 1024, 1024, 128, None, 1 << 20, None) == 5
    assert L.w4a16_gemm(16, 16, 16, 16, -1, 1024, 1024, 128, 16, 1 << 20, None) == 2
    # M == 0 is a no-op
    assert L.w4a16_gemm(None, None, None, None, 0, 1024, 1024, 128, None, 0, None) == 0
    assert L.w4a16_repack(None, 16, 1024, 1024, 128, 16, 16, None) == 1
    assert L.w4a16_repack(16, 16, 1024, 1024, 100, 16, 16, None) == 3


def test_entry_points_report_missing_gpu(w):
    # On a machine without a GPU the device query fails: an error code, not a crash.
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    L = w.lib
    assert L.w4a16_gemm(16, 16, 16, 16, 4, 1024, 1024, 128, 16, 1 << 20, None) == 6
    assert L.w4a16_workspace_bytes(16, 1024, 1024, 128) == 0


def test_sparse_and_quantiser_entry_points_validate_on_the_host(w):
    L = w.lib
    # 2:4: sizes, bad shapes, null pointers, M == 0
    assert L.w4a16_packed24_bytes(1024, 1024) == 1024 * 1024 * 3 // 8
    assert L.w4a16_packed24_bytes(1000, 1024) == 0
    assert L.w4a16_gemm_24(16, 16, 16, 16, 4, 1000, 1024, 128, 16, 1 << 20, None) == 2
    assert L.w4a16_gemm_24(None, 16, 16, 16, 4, 1024, 1024, 128, 16, 1 << 20, None) == 1
    assert L.w4a16_gemm_24(16, 16, 16, 16, 4, 1024, 1024, 128, None, 1 << 20, None) == 5
    assert L.w4a16_gemm_24(None, None, None, None, 0, 1024, 1024, 128, None, 0, None) == 0
    assert L.w4a16_repack_24(None, 16, 1024, 1024, 128, 16, 16, None) == 1
    assert L.w4a16_repack_24(16, 16, 1024, 1024, 96, 16, 16, None) == 3
    assert L.w4a16_unpack_24(16, 1000, 1024, 16, None) == 2
    # quantiser: bad group, null scales, misaligned weights
    assert L.w4a16_minmax_scales(16, 1024, 1024, 96, 16, None, None) == 3
    assert L.w4a16_minmax_scales(16, 1024, 1024, 128, None, None, None) == 1
    assert L.w4a16_minmax_scales(17, 1024, 1024, 128, 16, None, None) == 9   # W4A16_ERR_ALIGN
    assert L.w4a16_quantize_repack_zp(16, 16, 17, 1024, 1024, 128, 16, 16, None) == 9


def test_big_layer_plans_are_the_measured_ones(w):
    """The plans the benchmark numbers were measured with (K = 18432, N = 73728, G = 128, 152 SMs):
    streaming kernel with 16-piece (1024-row) units in 2 stages up to M = 16, tensor-memory kernel
    with units of a strip pair x 512 rows above."""
    for M in (1, 8, 16):
        p = w.w4a16_plan(M, 18432, 73728, 128, 152)
        assert (p["path"], p["k_tile"], p["stages"], p["m_chunk"]) == (1, 1024, 2, 8 if M <= 8 else 16)
    for M in (32, 64, 128):
        p = w.w4a16_plan(M, 18432, 73728, 128, 152)
        assert (p["path"], p["k_tile"], p["n_tile"], p["m_chunk"]) == (2, 512, 256, M)


# (K, N) -> unit depth (rows) of the streaming kernel at M <= 16 on 152 SMs, as measured inside a
# CUDA graph: the deeper unit was faster where it is chosen and the shallower one where it is not
# (8192 x 10240: 512-row units 14.9 us against 15.4; 5120 x 5120: 9.0 against 9.5)
MEASURED_UNIT_ROWS = [((4096, 4096), 1024), ((4096, 22016), 1024), ((8192, 8192), 1024), ((8192, 10240), 512),
                      ((2048, 7168), 1024), ((7168, 2048), 1024), ((1024, 12288), 1024), ((18432, 4096), 768),
                      ((5120, 5120), 512), ((7168, 4096), 512), ((18432, 73728), 1024)]


@pytest.mark.parametrize("shape,rows", MEASURED_UNIT_ROWS, ids=[f"{k}x{n}" for (k, n), _ in MEASURED_UNIT_ROWS])
def test_streaming_unit_depth_is_the_measured_best(w, shape, rows):
    K, N = shape
    for M in (1, 8, 16):
        p = w.w4a16_plan(M, K, N, 128, 152)
        assert p["path"] == 1 and p["k_tile"] == rows, (M, p["k_tile"])


# (K, N, M) -> warps that sum a split strip at a CTA's last segment on 152 SMs, as chosen from
# same-box measurements of both streaming builds: eight with two token tiles at every layer size,
# and with one tile only where a CTA has at most two units; the tcgen05 kernel's 16 dequant warps
MEASURED_FINAL_SUM_WARPS = [((4096, 4096, 1), 8), ((4096, 4096, 16), 8), ((11008, 4096, 1), 2),
                            ((11008, 4096, 16), 8), ((8192, 8192, 8), 2), ((18432, 73728, 1), 2),
                            ((18432, 73728, 16), 8), ((2048, 7168, 1), 8), ((18432, 73728, 32), 16)]


@pytest.mark.parametrize("shape,warps", MEASURED_FINAL_SUM_WARPS,
                         ids=[f"{k}x{n}_m{m}" for (k, n, m), _ in MEASURED_FINAL_SUM_WARPS])
def test_split_strip_sum_build_is_the_measured_one(w, shape, warps):
    K, N, M = shape
    assert w.w4a16_plan(M, K, N, 128, 152)["final_sum_warps"] == warps


@pytest.mark.parametrize("M", [17, 32, 48, 64, 80, 128, 129, 256, 1000])
@pytest.mark.parametrize("K,N", [(11008, 4096), (2816, 4096), (18432, 73728), (8192, 28672), (384, 384), (128, 640)])
@pytest.mark.parametrize("force", [2, 3, 4])
def test_tensor_memory_plans_stay_inside_the_modelled_protocol(w, M, K, N, force):
    """The ring depths the planner picks are those the host protocol model checks: one-chunk
    units (K an odd multiple of 128) need an even weight ring; the A buffers per strip and the
    accumulators fit the 512 tensor-memory columns (checked again before launch).  The wide mode
    has four-chunk units, four A buffers and one strip per unit."""
    try:
        w.w4a16_debug_force_path(force)
        p = w.w4a16_plan(M, K, N, 128, 152)
    finally:
        w.w4a16_debug_force_path(0)
    ch = p["k_tile"] // 128
    mb = p["m_chunk"]
    assert mb % 16 == 0 and mb >= 16 and p["stages"] >= 2
    wide = K % 512 == 0 and (force == 4 or (force == 2 and M >= 129))
    if wide:
        assert p["n_tile"] == 128 and ch == 4 and mb <= 256 and 4 * 64 + mb <= 512
        launches = -(-M // mb)
        assert launches == -(-M // 256) and mb >= -(-M // launches)
    else:
        assert p["n_tile"] == 256
        assert ch in (1, 2, 4) and ch == (4 if K % 512 == 0 else 2 if K % 256 == 0 else 1)
        assert ch == 2 or p["stages"] % 2 == 0
        assert mb <= 128
        na = min(3, (256 - mb) // 64)
        assert na >= 2 and 2 * (na * 64 + mb) <= 512


def _split_reduction_check(units, T, grid, KU):
    """The kernels' split-strip bookkeeping against brute force.  A CTA c owns units
    [c*T, min(units, (c+1)*T)); strip j owns units [j*KU, (j+1)*KU).  For a strip, the kernels
    take the contributing CTAs as c_first = j*KU // T .. c_last = min(((j+1)*KU - 1) // T, grid - 1);
    a CTA writes its partial of the strip into slot 2c if the strip is the CTA's first, else
    2c + 1, and the last arriver reads slot 2c if j == (c*T) // KU, else 2c + 1."""
    assert (grid - 1) * T < units <= grid * T
    for j in range(units // KU):
        lo, hi = j * KU, (j + 1) * KU
        brute = [c for c in range(grid) if c * T < hi and min(units, (c + 1) * T) > lo]
        c_first, c_last = (j * KU) // T, min(((j + 1) * KU - 1) // T, grid - 1)
        assert brute == list(range(c_first, c_last + 1)), (units, T, KU, j)
        if c_first == c_last:
            continue  # one CTA holds the whole strip and writes C directly
        slots = []
        for c in brute:
            first_col = (c * T) // KU
            last_col = (min(units, (c + 1) * T) - 1) // KU
            assert j in (first_col, last_col), "a split strip is a CTA's first or last strip"
            written = 2 * c if j == first_col else 2 * c + 1
            read = 2 * c if j == (c * T) // KU else 2 * c + 1
            assert written == read
            slots.append(written)
        assert len(set(slots)) == len(slots) and max(slots) < 2 * grid


@pytest.mark.parametrize("M", [1, 16, 32, 128, 256, 1000])
def test_split_strip_slots_and_counters_cover_each_strip_once(w, M):
    for K, N in [(1024, 1024), (4096, 4096), (4096, 22016), (11008, 4096), (2816, 4096), (8192, 57344),
                 (28672, 8192), (18432, 73728), (384, 640), (128, 128), (7168, 4096)]:
        for G in (128, -1):
            p = w.w4a16_plan(M, K, N, G, 152)
            _split_reduction_check(p["units"], p["units_per_cta"], p["grid"], K // p["k_tile"])


def test_split_strip_bookkeeping_brute_force_small_grids():
    for KU in range(1, 13):
        for strips in range(1, 9):
            units = KU * strips
            for sms in range(1, 40):
                T = (units + sms - 1) // sms
                _split_reduction_check(units, T, (units + T - 1) // T, KU)
