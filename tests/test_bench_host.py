"""bench.py's host-side arithmetic and parsing (no GPU): the roofline byte and FLOP counts, the
lookup of profiled DRAM traffic by kernel-source hash, the oracle's timing child, and the clock
reader's parsing of nvidia-smi output (a stand-in script on PATH)."""
import os
import stat

import pytest

import bench


def test_algorithmic_bytes_and_flops():
    # 2MK (A) + KN/2 (4-bit codes) + 2(K/G)N (FP16 scales) + 2MN (C)
    assert bench.gemm_bytes(1, 18432, 73728, 128) == 2 * 18432 + 18432 * 73728 // 2 + 2 * 144 * 73728 + 2 * 73728
    # per-column scales: one row of N
    assert bench.gemm_bytes(32, 8192, 8192, -1) == 2 * 32 * 8192 + 8192 * 8192 // 2 + 2 * 8192 + 2 * 32 * 8192
    assert bench.gemm_bytes(32, 8192, 8192, 8192) == bench.gemm_bytes(32, 8192, 8192, -1)
    assert bench.gemm_flops(128, 18432, 73728) == 2 * 128 * 18432 * 73728


def test_big_layer_roofline_point_matches_the_metric_definition():
    # the big layer at M = 1 is memory-bound at any plausible peak pair
    by = bench.gemm_bytes(1, 18432, 73728, 128)
    fl = bench.gemm_flops(1, 18432, 73728)
    assert by / 6788e9 > fl / 1903e12
    tb, tf = bench.workload_totals(bench.WORKLOADS["big"][1])
    assert tb == sum(bench.gemm_bytes(M, 18432, 73728, 128) for M in (1, 2, 4, 8, 16, 32, 64, 128))
    assert tf == sum(bench.gemm_flops(M, 18432, 73728) for M in (1, 2, 4, 8, 16, 32, 64, 128))


def test_profiled_traffic_is_used_only_for_the_profiled_sources(monkeypatch):
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0000000000000000")
    assert bench.profiled_traffic("gemm_big_layer_traffic.md") is None
    assert bench.profiled_traffic("no_such_profile.md") is None
    monkeypatch.undo()
    t = bench.profiled_traffic("gemm_big_layer_traffic.md")
    if t is None:
        pytest.skip("the committed traffic summary was taken on other kernel sources (refresh the profiles)")
    assert {(k, m) for k, m, _ in t} == {("gemm_mma_kernel", m) for m in (1, 2, 4, 8, 16)} | \
        {("gemm_tc_kernel", m) for m in (32, 64, 128)}
    for (k, m, _), v in t.items():  # DRAM bytes per launch within 2 % of the algorithmic bytes
        assert abs(v / bench.gemm_bytes(m, 18432, 73728, 128) - 1) < 0.02, (k, m, v)


def test_kernel_source_hash_follows_code_not_comments():
    srcs = {}
    for name in bench.GEMM_SOURCES:
        with open(os.path.join(bench.ROOT, "mixed_precision_w4a16_gb300", "csrc", name), encoding="utf-8") as f:
            srcs[name] = f.read()
    h = bench.kernel_source_hash(srcs)
    assert h == bench.kernel_source_hash()
    commented = dict(srcs)
    commented["gemm_tc.cu"] = "// a new comment line\n/* and a block */\n" + srcs["gemm_tc.cu"].replace("\n", "  \n", 3)
    assert bench.kernel_source_hash(commented) == h
    changed = dict(srcs)
    changed["gemm_launch.cu"] = srcs["gemm_launch.cu"].replace("kTcMinRows = 17", "kTcMinRows = 33", 1)
    assert changed["gemm_launch.cu"] != srcs["gemm_launch.cu"]
    assert bench.kernel_source_hash(changed) != h
    assert bench._code_only('x = "// kept"; // dropped') == 'x = "// kept";'


def test_oracle_timing_child_reports_gemm_and_repack():
    r = bench.run_cpu_sample("pr1", 1024, repack=True)
    assert r["seconds"] > 0 and r["scaled_seconds"] == pytest.approx(r["seconds"])  # 1024 of 1024 columns
    assert r["repack"]["shape"] == "K=1024 N=1024 G=128" and r["repack"]["scaled_seconds"] > 0
    assert bench.run_cpu_sample("pr1", 1024)["repack"] is None


def _fake_smi(tmp_path, once_line, sample_line):
    p = tmp_path / "nvidia-smi"
    p.write_text("#!/bin/sh\ncase \"$*\" in\n"
                 f"  *clocks.mem*) echo \"{once_line}\" ;;\n"
                 f"  *) while true; do echo \"{sample_line}\"; sleep 0.05; done ;;\nesac\n")
    p.chmod(p.stat().st_mode | stat.S_IEXEC)
    return str(tmp_path)


def test_clock_reader_parses_nvidia_smi(tmp_path, monkeypatch):
    import time
    assert bench.ClockSampler.read_once(None) == {} or "mem_mhz" in bench.ClockSampler.read_once(None)
    d = _fake_smi(tmp_path, "3996, 3996, Enabled",
                  "0, 1980, 2070, 700.5, 0x4, Not Active, Not Active, Not Active, Active")
    monkeypatch.setenv("PATH", d + os.pathsep + os.environ["PATH"])
    assert bench.ClockSampler.read_once("GPU-x") == {"mem_mhz": 3996.0, "mem_max_mhz": 3996.0, "ecc": "Enabled"}
    cs = bench.ClockSampler(None)
    time.sleep(0.3)
    cs.start_timing()
    time.sleep(0.3)
    cs.stop_timing()
    out = cs.finish()
    assert out["sm_mhz"] == 1980.0 and out["sm_max_mhz"] == 2070.0 and out["reasons"] == ["sw_power_cap"]
    assert out["ecc"] == "Enabled" and out["samples"] >= 1
