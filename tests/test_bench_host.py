"""Host logic of bench.py, no GPU needed: the reference arm's JSON line (the
fp64 oracle timed on the host cores), the rank rule under torchrun, the
warm-up floor, the flop count, the gate that drops profiled DRAM traffic once
a kernel's sources change, and the clock summary."""

import json
import os
import subprocess
import sys

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(args, env=None):
    return subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True,
                          text=True, timeout=900, env=env)


def test_reference_arm_prints_one_contract_line():
    r = _bench(["--impl", "reference", "--steps", "1", "--warmup", "3", "--seed", "5"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["higher_is_better"] is True and d["value"] > 0
    assert d["steps"] == 1 and d["warmup"] == 3
    assert d["config"]["workload"] == "train_B8_H12_T512"
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = _bench(["--impl", "reference", "--steps", "1", "--warmup", "3"], env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_warmup_floor_is_enforced_before_any_work():
    r = _bench(["--warmup", "2"])
    assert r.returncode == 2
    assert "--warmup" in r.stderr


def test_flop_count():
    # 4D flop per causal pair forward (QK^T, PV) and 10D backward (S again,
    # dP, dV, dQ, dK): 14 * 64 per pair; T = 2 has three causal pairs.
    assert bench.pairs_causal(1, 1, 2) == 3
    assert bench.train_flops(1, 1, 2) == 3 * 14 * 64
    assert bench.pairs_causal(8, 12, 512) == 8 * 12 * 512 * 513 // 2


def test_kernel_hashes_are_per_source_set():
    # Kernels built from the same files (the two forward kernels share fwd.cu)
    # share a hash; different source sets, and the whole tree, differ.
    hs = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
    by_sources = {}
    for k, h in hs.items():
        by_sources.setdefault(bench.KERNEL_SOURCES[k], set()).add(h)
    assert all(len(v) == 1 for v in by_sources.values())
    distinct = {next(iter(v)) for v in by_sources.values()} | {bench.kernel_source_hash()}
    assert len(distinct) == len(by_sources) + 1
    for h in distinct:
        assert len(h) == 16 and int(h, 16) >= 0


def test_traffic_is_dropped_once_the_sources_change(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    os.symlink(os.path.join(ROOT, "transformer_attention_ggd_gb300"),
               tmp_path / "transformer_attention_ggd_gb300")
    current = bench.kernel_source_hash("bam_bwd_kernel")
    entries = {
        "bam_bwd_kernel": {"source_hash": current, "dram_bytes_per_launch": 123},
        "bam_bwd_kernel@other_workload": {"source_hash": current,
                                          "dram_bytes_per_launch": 456},
        "bam_fwd_kernel": {"source_hash": "0" * 16, "dram_bytes_per_launch": 789},
    }
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(entries))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("bam_bwd_kernel") == 123
    assert bench.profiled_traffic("bam_bwd_kernel@other_workload") == 456
    assert bench.profiled_traffic("bam_fwd_kernel") is None      # taken on other sources
    assert bench.profiled_traffic("bam_decode_kernel") is None   # never captured


def test_traffic_is_matched_to_its_workload(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    os.symlink(os.path.join(ROOT, "transformer_attention_ggd_gb300"),
               tmp_path / "transformer_attention_ggd_gb300")
    h = bench.kernel_source_hash("bam_fwd_kernel")
    entries = {
        "bam_fwd_kernel": {"workload": "prefill_A", "source_hash": h,
                           "dram_bytes_per_launch": 1},
        "bam_fwd_kernel@train_B": {"workload": "train_B", "source_hash": h,
                                   "dram_bytes_per_launch": 2},
    }
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(entries))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("bam_fwd_kernel", "prefill_A") == 1
    assert bench.traffic_for("bam_fwd_kernel", "train_B") == 2
    assert bench.traffic_for("bam_fwd_kernel", "prefill_C") is None
    assert bench.traffic_for("bam_bwd_kernel", "train_B") is None


def test_clock_summary():
    cs = bench.ClockSampler(0)
    cs.lines = [
        "0, 1995, 2070, 900.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1010.0, 0x0000000000000000, Not Active, Not Active, Not Active, "
        "Not Active",
        "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "short line",
    ]
    s = cs.summary()
    assert s == {"sm_mhz": 2032.5, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                 "samples": 2}
    cs.lines = ["0, 1500, 2070, 700, 0x8, Not Active, Active, Not Active, Not Active"]
    assert cs.summary()["reasons"] == ["hw_thermal_slowdown"]
    cs.lines = []
    assert cs.summary()["reasons"] == ["unsampled"]


@pytest.mark.parametrize("case", bench.PROFILE_CASES)
def test_profile_cases_are_accepted(case):
    """Every profile case parses (the run itself needs a GPU)."""
    r = _bench(["--profile-case", case, "--warmup", "2"])
    assert r.returncode == 2 and "--warmup" in r.stderr
