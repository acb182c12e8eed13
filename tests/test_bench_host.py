"""Host-side arithmetic of the benchmark (CPU only): the algorithmic byte and flop counts
the roofline divides by, the whole-job throughput, the clock-sample summary, the traffic
record's source check, and the reference arm's JSON line."""
import hashlib
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_decode_bytes_count_every_row_once_plus_queries_outputs_and_tables():
    lens, B, H, L, R = [1, 64, 65], 3, 2, 4, 2
    E = L + R
    rows = 1 + 64 + 65
    pages = 1 + 1 + 2                       # pages of 64 rows in use
    want = rows * E * 2 + B * H * E * 2 + B * H * L * 2 + pages * 4 + B * 4
    assert bench.decode_algorithmic_bytes(lens, B, H, L, R, max_blocks=2) == want


def test_decode_flops_are_qk_over_the_entry_and_pv_over_the_latent():
    # per cached row and head: 2 * (L + R) for the scores, 2 * L for the output
    assert bench.decode_algorithmic_flops([3, 5], H=2, L=4, R=2) == 8 * 2 * 2 * (6 + 4)


def test_fp8_cache_rows_count_one_byte_an_element():
    lens, B, H, L, R = [64, 65], 2, 2, 4, 2
    bf16 = bench.decode_algorithmic_bytes(lens, B, H, L, R, 2)
    fp8 = bench.decode_algorithmic_bytes(lens, B, H, L, R, 2, cache_es=1)
    assert bf16 - fp8 == (64 + 65) * (L + R)


def test_roofline_follows_the_tighter_bound():
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 100.0, "bf16_tflops_sustained": 50.0}
    # 1 GB at 1000 GB/s = 1 ms; 10 GFLOP at 100 TFLOP/s = 0.1 ms: HBM is tighter
    r = bench.roofline(1e9, 1e10, 2.0, peaks)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(500.0) and r["frac"] == pytest.approx(0.5)
    # 1 GB (1 ms) against 200 GFLOP (2 ms at burst, 4 ms sustained): tensor is tighter
    r = bench.roofline(1e9, 2e11, 8.0, peaks)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] == 100.0
    assert r["frac"] == pytest.approx(0.25)
    r = bench.roofline(1e9, 2e11, 8.0, peaks, sustained=True)
    assert r["peak"] == 50.0 and r["frac"] == pytest.approx(0.5)
    # frac is the bound's time over the measured time either way
    for nbytes, flops, ms in ((3e9, 1e10, 7.0), (1e8, 5e11, 9.0)):
        r = bench.roofline(nbytes, flops, ms, peaks)
        t_bound = max(nbytes / 1e12, flops / 1e14) * 1e3
        assert r["frac"] == pytest.approx(t_bound / ms)


def test_job_throughput_is_all_ranks_bytes_over_the_slowest_step():
    assert bench.job_throughput(1e9, 1.0, 1) == pytest.approx(1000.0)
    assert bench.job_throughput(1e9, 2.0, 4) == pytest.approx(2000.0)


def test_clock_summary_takes_the_loaded_half_and_flags_throttle_reasons():
    c = bench.ClockSampler("0")
    c.lines = [
        "0, 1200, 2070, 300.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 950.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2050, 2070, 940.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    s = c.summary()
    assert s["samples"] == 4
    assert s["sm_max_mhz"] == 2070.0
    assert s["sm_mhz"] == pytest.approx(2070.0)   # median of the busier half: 2070, 2070
    assert s["reasons"] == ["sw_power_cap"]


def test_traffic_record_is_used_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    csrc = tmp_path / "mla_latent_kv_11_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cu").write_bytes(b"// kernel source\n")
    (csrc / "c.cu").write_bytes(b"// combine source\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench._sources_sha(("k.cu", "c.cu"))
    (tmp_path / "profiles" / "traffic.json").write_text(
        json.dumps({"decode": {"source_sha": sha, "bytes_per_launch": 1234.0}}))
    assert bench._traffic_for(("k.cu", "c.cu")) == 1234.0
    (csrc / "c.cu").write_bytes(b"// combine source, changed\n")
    assert bench._traffic_for(("k.cu", "c.cu")) is None
    assert bench._traffic_for(("k.cu", "missing.cu")) is None


def test_decode_v_up_counts_weights_and_out_instead_of_o_lat():
    lens, B, H, L, R, V = [3, 70], 2, 4, 8, 2, 5
    nbytes, flops = bench.decode_v_up_algorithmic(lens, B, H, L, R, V)
    assert nbytes == bench.decode_algorithmic_bytes(lens, B, H, L, R, 0) - B * H * L * 2 + H * L * V * 2 + B * H * V * 2
    assert flops == bench.decode_algorithmic_flops(lens, H, L, R) + 2 * B * H * L * V


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == bench.WORKLOAD
