"""The tensor-memory GEMM kernel's barrier protocol under random interleavings (host only).

tc_protocol_model restates the roles of gemm_tc_kernel and checks, at every step of many random
schedules, that no parity wait passes on the wrong phase, that no barrier over-arrives, and that
no stage, A buffer or accumulator is read or overwritten out of turn.  The configurations are the
ones the planner produces (A buffers, issuers, unit depth, weight stages, CTA ranges that start
inside a strip and end just past a strip boundary).  Three orderings that are wrong (each once
considered for the kernel) must be caught."""
import pytest

from tc_protocol_model import Config, explore

# (name, config) as planned: M = 17..32 -> 6 A buffers, 4 issuers; M = 33..64 -> 4, 4;
# M >= 80 -> 4 A buffers, 2 issuers.  Unit depth 4 chunks unless K is not a multiple of 512.
PLANNED = [
    ("m32_ch4", Config(NA=6, NI=4, CH=4, SW=5, nunits=12, KU=36, kt0=30)),
    ("m32_ch2_short_segment", Config(NA=6, NI=4, CH=2, SW=9, nunits=10, KU=43, kt0=34)),
    ("m32_ch1", Config(NA=6, NI=4, CH=1, SW=12, nunits=7, KU=3, kt0=1)),
    ("m64_ch4", Config(NA=4, NI=4, CH=4, SW=4, nunits=10, KU=36, kt0=33)),
    ("m64_ch2_short_segment", Config(NA=4, NI=4, CH=2, SW=9, nunits=10, KU=43, kt0=34)),
    ("m128_ch4", Config(NA=4, NI=2, CH=4, SW=2, nunits=10, KU=36, kt0=33)),
    ("m128_ch1", Config(NA=4, NI=2, CH=1, SW=10, nunits=7, KU=3, kt0=2)),
    ("one_unit_per_cta", Config(NA=6, NI=4, CH=2, SW=9, nunits=1, KU=43, kt0=5)),
]


@pytest.mark.parametrize("name,cfg", PLANNED, ids=[n for n, _ in PLANNED])
def test_planned_protocol_has_no_race(name, cfg):
    err = explore(cfg, seeds=120)
    assert err is None, f"{name}: {err}"


def test_activation_wait_first_is_caught():
    # 6 A buffers shared round-robin by 4 issuers: waiting for the activation stage before the
    # A chunk can pass on the copy of the chunk that used the slot before
    err = explore(Config(NA=6, NI=4, CH=4, SW=5, nunits=12, KU=36, kt0=30, afull_first=True), seeds=400)
    assert err is not None


def test_idle_issuer_without_readout_wait_is_caught():
    # a 2-chunk segment after a strip boundary leaves two of four issuers without a chunk
    err = explore(Config(NA=6, NI=4, CH=2, SW=9, nunits=10, KU=43, kt0=34, idle_wait=False), seeds=400)
    assert err is not None


def test_activation_ring_not_a_multiple_of_the_issuers_is_caught():
    # a separate activation ring of 11 stages: stages shared by chunks of different issuers and
    # producers, so a producer's wait can pass two phases early and re-arm a pending stage
    err = explore(Config(NA=6, NI=4, CH=4, SW=4, nunits=16, KU=36, kt0=30, NAS=11, decoupled=True), seeds=400)
    assert err is not None


def test_activation_ring_multiple_of_the_issuers_has_no_race():
    err = explore(Config(NA=6, NI=4, CH=4, SW=4, nunits=12, KU=36, kt0=30, NAS=8, decoupled=True), seeds=120)
    assert err is None, err
