"""Host-side pieces of bench.py (no GPU): the choice of the tensor peak from the
sampled clock state, the traffic record's source-hash check, and the
workload lists."""
from __future__ import annotations

import os
import shutil

import bench

PK = {"hbm_gbs": 6784.2, "bf16_tflops": 1937.2, "bf16_tflops_sustained": 1701.9}


def test_peak_is_burst_only_when_the_clock_held_its_maximum():
    held = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 40, "reason_samples": {}}
    assert bench.tensor_peak(PK, "measured", held)[0] == PK["bf16_tflops"]
    # the power cap in a few samples: the clock still held; in a quarter or more: sustained
    rare = dict(held, reasons=["sw_power_cap"], reason_samples={"sw_power_cap": 3})
    assert bench.tensor_peak(PK, "measured", rare)[0] == PK["bf16_tflops"]
    capped = dict(held, reasons=["sw_power_cap"], reason_samples={"sw_power_cap": 10})
    assert bench.tensor_peak(PK, "measured", capped)[0] == PK["bf16_tflops_sustained"]
    slow = dict(held, sm_mhz=1800.0)
    assert bench.tensor_peak(PK, "measured", slow)[0] == PK["bf16_tflops_sustained"]
    unsampled = {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
    assert bench.tensor_peak(PK, "measured", unsampled)[0] == PK["bf16_tflops_sustained"]


def test_traffic_record_follows_the_kernel_sources(tmp_path, monkeypatch):
    """The committed dK/dV traffic figure is reported only while the listed
    kernel sources hash to the recorded value."""
    rel = bench.TRAFFIC_PROFILES["dkv"]
    assert os.path.exists(os.path.join(bench.ROOT, rel))
    root = tmp_path / "repo"
    csrc = root / "long_context_masked_attention_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (root / "profiles").mkdir()
    shutil.copy(os.path.join(bench.ROOT, rel), root / rel)
    src = os.path.join(bench.ROOT, "long_context_masked_attention_gb300", "csrc")
    for f in os.listdir(src):
        shutil.copy(os.path.join(src, f), csrc / f)
    monkeypatch.setattr(bench, "ROOT", str(root))
    first = bench.measured_traffic("dkv")
    with open(csrc / "lca_bwd.cu", "a") as fh:
        fh.write("\n// changed\n")
    assert bench.measured_traffic("dkv") is None
    if first is not None:
        assert first > 324e6  # above the algorithmic bytes of one launch


def test_workload_lists():
    assert len(bench.workload_problems()) == 12
    assert len(bench.workload_problems(workload="sweep8k_dropout")) == 12
    assert len(bench.workload_problems(workload="dense48k")) == 28
    assert len(bench.workload_problems(workload="blocksparse")) == 18
    assert len(bench.workload_problems(workload="shards512k")) == 1
    assert [p.mask.kind for p in bench.workload_problems(only="CAUSAL,FULL")] == ["FULL", "CAUSAL"]
    assert set(bench.DROPOUT) <= set(bench.WORKLOADS)


def test_clock_samples_parsed_with_reason_counts():
    out = "\n".join([
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1980, 2070, 1395.0, 0x4, Not Active, Not Active, Not Active, Active",
        "garbage line",
    ])
    clk = bench.parse_clock_samples(out)
    assert clk["samples"] == 3 and clk["sm_mhz"] == 2070.0 and clk["sm_max_mhz"] == 2070.0
    assert clk["reasons"] == ["sw_power_cap"] and clk["reason_samples"] == {"sw_power_cap": 2}
