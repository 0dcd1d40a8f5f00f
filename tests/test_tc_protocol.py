"""The tensor-memory GEMM kernel's barrier protocol under random interleavings (host only).

tc_protocol_model restates the roles of gemm_tc_kernel and checks, at every step of many random
schedules, that no parity wait passes on the wrong phase, that no barrier over-arrives, and that
no stage, A buffer or accumulator is read or overwritten out of turn.  The configurations are the
ones the planner produces (A buffers per strip, activation stages, unit depth, weight stages, CTA
ranges that start inside a strip pair and end just past a strip-pair boundary).  Orderings that
are wrong must be caught."""
import pytest

from tc_protocol_model import Config, explore

# (name, config) as planned: M <= 64 -> 3 A buffers per strip, M = 65..128 -> 2; unit depth two
# chunks (K a multiple of 256) or one; activation and weight stages from the shared-memory budget.
PLANNED = [
    ("m32_ch4", Config(NA=3, NS=8, CH=4, SW=2, nunits=8, KU=36, kt0=33)),
    ("m64_ch4", Config(NA=3, NS=4, CH=4, SW=2, nunits=8, KU=36, kt0=33)),
    ("m64_ch4_short", Config(NA=3, NS=5, CH=4, SW=2, nunits=10, KU=3, kt0=1)),
    ("m128_ch4", Config(NA=2, NS=2, CH=4, SW=2, nunits=8, KU=16, kt0=13)),
    ("m32_ch2", Config(NA=3, NS=8, CH=2, SW=4, nunits=12, KU=43, kt0=38)),
    ("m64_ch2", Config(NA=3, NS=6, CH=2, SW=3, nunits=12, KU=43, kt0=38)),
    ("m128_ch2", Config(NA=2, NS=4, CH=2, SW=2, nunits=12, KU=43, kt0=38)),
    ("m32_ch1", Config(NA=3, NS=8, CH=1, SW=4, nunits=9, KU=3, kt0=1)),
    ("m128_ch1", Config(NA=2, NS=4, CH=1, SW=6, nunits=7, KU=5, kt0=2)),
    ("one_unit_per_cta", Config(NA=3, NS=6, CH=2, SW=3, nunits=1, KU=43, kt0=5)),
    ("short_segments", Config(NA=3, NS=6, CH=2, SW=3, nunits=9, KU=2, kt0=1)),
    # wide mode (M > 128): one strip per unit, each of the four warpgroups owns one of four A
    # buffers and one chunk of every four-chunk unit; one issuer; 256 / 192 / 128 token rows
    ("wide_mb256", Config(NA=4, NS=2, CH=4, SW=2, nunits=24, KU=16, kt0=8, US=1)),
    ("wide_mb192", Config(NA=4, NS=3, CH=4, SW=2, nunits=24, KU=16, kt0=8, US=1)),
    ("wide_mb128_big_layer", Config(NA=4, NS=4, CH=4, SW=2, nunits=20, KU=36, kt0=30, US=1)),
    ("wide_short_segments", Config(NA=4, NS=2, CH=4, SW=2, nunits=9, KU=2, kt0=1, US=1)),
    ("wide_one_unit_per_cta", Config(NA=4, NS=2, CH=4, SW=2, nunits=1, KU=16, kt0=3, US=1)),
    # fewer token rows leave room for more A buffers (up to seven): a warpgroup's buffer then
    # last held another warpgroup's chunk
    ("wide_mb192_na5", Config(NA=5, NS=3, CH=4, SW=2, nunits=24, KU=16, kt0=8, US=1)),
    ("wide_mb128_na6", Config(NA=6, NS=4, CH=4, SW=2, nunits=20, KU=36, kt0=30, US=1)),
    ("wide_mb64_na7", Config(NA=7, NS=8, CH=4, SW=3, nunits=20, KU=36, kt0=30, US=1)),
    ("wide_mb32_na7_short", Config(NA=7, NS=8, CH=4, SW=4, nunits=9, KU=2, kt0=1, US=1)),
]


@pytest.mark.parametrize("name,cfg", PLANNED, ids=[n for n, _ in PLANNED])
def test_planned_protocol_has_no_race(name, cfg):
    err = explore(cfg, seeds=120)
    assert err is None, f"{name}: {err}"


def test_one_chunk_units_with_an_odd_weight_ring_are_caught():
    # units of one chunk are read by two of the four warpgroups, alternately; with an odd number
    # of weight stages a warpgroup meets a stage whose previous unit it never waited for, and its
    # parity wait can pass while that copy is still in flight (the planner keeps the ring even)
    err = explore(Config(NA=3, NS=8, CH=1, SW=3, nunits=12, KU=40, kt0=3), seeds=400)
    assert err is not None


def test_decode_without_the_buffer_wait_is_caught():
    err = explore(Config(NA=3, NS=6, CH=2, SW=3, nunits=10, KU=72, kt0=66, dequant_consumed_wait=False), seeds=400)
    assert err is not None


def test_idle_warpgroups_touching_the_stage_are_caught():
    # with one chunk per unit, warpgroups without a chunk must not arrive on the unit's stage
    err = explore(Config(NA=3, NS=8, CH=1, SW=4, nunits=9, KU=3, kt0=1, idle_wempty=False), seeds=200)
    assert err is not None


def test_odd_activation_ring_is_safe():
    # a warpgroup that waits for a stage shared with the other warpgroup's chunks has itself
    # waited for the stage's use two phases back (its own chunk gs - 2 NS), so the barrier is
    # never more than one phase behind
    err = explore(Config(NA=3, NS=7, CH=2, SW=3, nunits=12, KU=43, kt0=38), seeds=200)
    assert err is None, err


def test_dequant_waiting_for_the_activations_instead_is_safe_too():
    err = explore(Config(NA=3, NS=7, CH=2, SW=3, nunits=10, KU=43, kt0=38, dequant_afull_wait=True), seeds=120)
    assert err is None, err


def test_wide_mode_with_three_buffers_is_caught():
    # four warpgroups round-robin over three A buffers: a warpgroup's wait for a buffer's previous
    # multiplies can name a phase two behind (the kernel requires four buffers in the wide mode)
    err = explore(Config(NA=3, NS=2, CH=4, SW=2, nunits=24, KU=16, kt0=8, US=1), seeds=200)
    assert err is not None


def test_wide_mode_without_the_buffer_wait_is_caught():
    err = explore(Config(NA=4, NS=2, CH=4, SW=2, nunits=24, KU=16, kt0=8, US=1, dequant_consumed_wait=False),
                  seeds=200)
    assert err is not None
