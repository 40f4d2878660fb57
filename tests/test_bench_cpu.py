"""Host-side pieces of bench.py (no GPU): the choice of the tensor peak from the
sampled clock state, the traffic record's source-hash check, and the
workload lists."""
from __future__ import annotations

import os
import shutil

import bench

PK = {"hbm_gbs": 6784.2, "bf16_tflops": 1937.2, "bf16_tflops_sustained": 1701.9}


def test_peak_is_burst_only_when_the_clock_held_its_maximum():
    held = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3}
    assert bench.tensor_peak(PK, "measured", held)[0] == PK["bf16_tflops"]
    capped = dict(held, reasons=["sw_power_cap"])
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
