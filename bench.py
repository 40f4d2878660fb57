#!/usr/bin/env python
"""Benchmark: masked attention forward + backward on one GB300 (N replicas
under torchrun), effective TFLOP/s counting only attended score entries.

Workload (the 8K static-mask sweep): batch 1, sequence 8192, 64 query heads /
8 KV heads, head dim 128, bf16 Q, K, V, dO drawn i.i.d. N(0,1); one step runs
forward + backward once per static mask family (12 masks; document families
use seeded log-uniform document lengths over [128, 8192]).

FLOPs: 4*d*nnz for the forward and 10*d*nnz for the backward, nnz = attended
(query, key) cells summed over query heads, counted exactly on the device by
lca_mask_nnz (checked against the oracle by the tests).

Other workloads (--workload; each prints its own JSON line, with the same
per-problem forward/backward breakdown; the default line above is the
headline):
  dense48k     sequence lengths 1K..48K at 48K tokens per step, MHA 64:64 and
               GQA 64:8, CAUSAL and CAUSAL_DOC (70/30 document-length mixture)
  blocksparse  32K/64K/128K tokens, MHA and GQA, uniform 64/128 blocks keeping
               half of each block row (diagonal included) and variable blocks
               U{32..256} keeping half of the block pairs
  shards512k   524,288 tokens of Pareto(1.2) documents cut into U{1K..32K}
               token shards, shuffled and packed into one launch, GQA 64:8
  sweep8k_dropout  the 8K static-mask sweep with attention dropout p = 0.1
               fused into the forward and backward kernels

Arms:
  default            the CUDA library; prints one JSON line (rank 0)
  --impl reference   the fp64 CPU oracle on the host cores, on a bounded sample
                     of the same workload (rank 0 only)
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "masked attn fwd+bwd effective TFLOP/s (unmasked FLOPs), % of GB300 BF16 peak"
WORKLOAD = "static_mask_sweep_8k_gqa64x8_d128"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def tensor_peak(pk, pk_src, clk):
    """The bf16 peak that matches the clocks sampled during the timed region:
    the burst figure when the median SM clock stayed within 5% of its maximum
    and the power cap was active in under a quarter of the samples, else the
    sustained (power-capped) one."""
    sm, mx, n = clk.get("sm_mhz"), clk.get("sm_max_mhz"), clk.get("samples") or 0
    capped = clk.get("reason_samples", {}).get("sw_power_cap", 0)
    held = n > 0 and sm and mx and sm >= 0.95 * mx and capped < 0.25 * n
    if held:
        return pk["bf16_tflops"], (f"{pk_src} bf16 burst (median SM clock at its maximum; power cap in {capped} of "
                                   f"{n} samples)")
    return pk["bf16_tflops_sustained"], (f"{pk_src} bf16 sustained (power cap in {capped} of {n} samples, or clock "
                                         f"below its maximum)")


WORKLOADS = {
    "sweep8k": "static_mask_sweep_8k_gqa64x8_d128",
    "dense48k": "dense_length_sweep_1k_48k_48k_tokens_mha64_gqa64x8_d128",
    "blocksparse": "block_sparse_32k_64k_128k_mha64_gqa64x8_d128",
    "shards512k": "shard_batch_512k_pareto_docs_gqa64x8_d128",
    "sweep8k_dropout": "static_mask_sweep_8k_gqa64x8_d128_dropout0.1",
}
DROPOUT = {"sweep8k_dropout": (0x5EED, 0.1)}


def workload_problems(only=None, workload="sweep8k"):
    from gen import STATIC_KINDS, config2, config3, config4, config5

    if workload == "dense48k":
        probs = [config3(S * 1024, h, kind) for S in (1, 2, 4, 8, 16, 32, 48) for h in ("mha", "gqa")
                 for kind in ("CAUSAL", "CAUSAL_DOC")]
    elif workload == "blocksparse":
        probs = [config4(S * 1024, h, var) for S in (32, 64, 128) for h in ("mha", "gqa")
                 for var in ("uniform64", "uniform128", "variable")]
    elif workload == "shards512k":
        probs = [config5()]
    else:  # sweep8k, sweep8k_dropout
        kinds = [k for k in STATIC_KINDS if only is None or k in only.split(",")]
        return [config2(k) for k in kinds]
    return [p for p in probs if only is None or p.name in only.split(",")]


def time_problem(lca, p, ws, flush, steps, warmup, tensors=None, dropout=None):
    """Median forward and backward milliseconds of one problem (L2 flushed
    before every timed call pair), with its attended-cell count."""
    import torch

    from gen import make_tensors

    dev = ws.device
    q, k, v, do = tensors if tensors is not None else make_tensors(p, device=dev)
    call = lca.marshal(p.Tq, p.Tk, p.Hq, p.Hkv, p.d, p.segments, p.mask, p.scale)
    nnz = int(lca.mask_nnz(call).sum().item())
    o = torch.empty_like(q)
    lse = torch.empty((p.Hq, p.Tq), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for s in range(warmup + steps):
        flush.zero_()
        e = ev[s - warmup] if s >= warmup else None
        if e:
            e[0].record(stream)
        lca.attn_fwd(q, k, v, p.segments, p.mask, p.scale, out=o, lse=lse, workspace=ws, call=call, dropout=dropout)
        if e:
            e[1].record(stream)
        lca.attn_bwd(do, q, k, v, o, lse, p.segments, p.mask, p.scale, dq=dq, dk=dk, dv=dv, workspace=ws,
                     call=call, dropout=dropout)
        if e:
            e[2].record(stream)
    torch.cuda.synchronize()
    st = lca.read_status(ws)
    if st != (0, 0):
        raise RuntimeError(f"device status after {p.name}: {st}")
    f_ms = statistics.median(a.elapsed_time(b) for a, b, _ in ev)
    b_ms = statistics.median(b.elapsed_time(c) for _, b, c in ev)
    fl_f, fl_b = 4.0 * p.d * nnz, 10.0 * p.d * nnz
    return {"nnz": nnz, "fwd_ms": f_ms, "bwd_ms": b_ms, "fwd_tflops": fl_f / (f_ms * 1e-3) / 1e12,
            "bwd_tflops": fl_b / (b_ms * 1e-3) / 1e12,
            "tflops": (fl_f + fl_b) / ((f_ms + b_ms) * 1e-3) / 1e12}


# ------------------------------------------------------------------ spec targets
def target_problems():
    """Dense GQA 64:8 CAUSAL and FULL at 8K, 16K, 32K and 48K (48K tokens per
    problem: floor(49152 / S) sequences of S tokens) and MHA 64:64 CAUSAL at
    8K, for the ">= 60% of peak for dense causal/full at 8K-48K" reading."""
    from gen import MaskSpec, Problem, config3

    out = []
    for S in (8192, 16384, 32768, 49152):
        c = config3(S, "gqa", "CAUSAL")
        out.append(c)
        out.append(Problem(c.name.replace("causal", "full"), c.Tq, c.Tk, c.Hq, c.Hkv, c.d, c.segments,
                           MaskSpec("FULL"), c.seed))
    out.append(config3(8192, "mha", "CAUSAL"))
    return out


def run_targets(lca, ws_dev, flush, pk, pk_src, gpu_index, steps=3, warmup=2):
    """Forward, backward and combined effective TFLOP/s of the target
    problems, each as a fraction of the bf16 peak matching the clocks sampled
    while they ran (a few steps each, L2 flushed before every step)."""
    import torch

    clocks = ClockSampler(gpu_index)
    clocks.start()
    rows = {}
    for p in target_problems():
        call = lca.marshal(p.Tq, p.Tk, p.Hq, p.Hkv, p.d, p.segments, p.mask, p.scale)
        ws = torch.empty(lca.workspace_size(call, True), dtype=torch.uint8, device=ws_dev)
        rows[p.name] = time_problem(lca, p, ws, flush, steps, warmup)
        del ws
        torch.cuda.empty_cache()
    clk = clocks.stop()
    peak, src = tensor_peak(pk, pk_src, clk)
    for r in rows.values():
        r["frac_of_peak"] = r["tflops"] / peak
        r["frac_of_sustained"] = r["tflops"] / pk["bf16_tflops_sustained"]
    return {"peak_tflops": peak, "peak_source": src, "clocks": clk, "steps": steps, "warmup": warmup,
            "problems": rows}


def run_balance(lca, probs, calls, ws, tensors):
    """Per-CTA balance of the attention kernels: one profiled forward and
    backward per problem (outside every timed region); for each kernel the
    slowest CTA's busy time over the mean (max_over_mean) and the share of
    CTA-time spent idle before the kernel's last CTA finished (idle)."""
    import torch

    prof = lca.CtaProfile(ws.device)
    q, k, v, do = tensors
    out = {}
    for p, c in zip(probs, calls):
        prof.start()
        try:
            o, lse = lca.attn_fwd(q, k, v, p.segments, p.mask, p.scale, workspace=ws, call=c)
            torch.cuda.synchronize()
            rec = {"fwd": prof.records()["fwd"]}
            lca.attn_bwd(do, q, k, v, o, lse, p.segments, p.mask, p.scale, workspace=ws, call=c)
            torch.cuda.synchronize()
            rec.update({kk: vv for kk, vv in prof.records().items() if kk != "fwd"})
        finally:
            prof.stop()
        row = {}
        for name, r in rec.items():
            busy = (r[:, 1] - r[:, 0]).astype(float)
            span = float(r[:, 1].max() - r[:, 0].min())
            row[name] = {"max_over_mean": float(busy.max() / busy.mean()), "idle": float(1.0 - busy.mean() / span),
                         "ctas": int(r.shape[0])}
        out[p.mask.kind] = row
    return out


# ------------------------------------------------------------------ measured traffic
TRAFFIC_PROFILES = {"dkv": "profiles/dkv_kernel_traffic_sweep8k_gqa64x8.md"}


def measured_traffic(kernel):
    """DRAM bytes per launch of `kernel` from its committed ncu summary, or None
    when there is none or the kernel's sources changed since the capture."""
    import hashlib
    import re

    rel = TRAFFIC_PROFILES.get(kernel)
    if rel is None or not os.path.exists(os.path.join(ROOT, rel)):
        return None
    text = open(os.path.join(ROOT, rel)).read()
    b = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    srcs = re.search(r"kernel_sources:\s*(.+)", text)
    sha = re.search(r"kernel_sources_sha256:\s*([0-9a-f]{64})", text)
    if not (b and srcs and sha):
        return None
    h = hashlib.sha256()
    for f in srcs.group(1).split():
        path = os.path.join(ROOT, "long_context_masked_attention_gb300", "csrc", f)
        if not os.path.exists(path):
            return None
        with open(path, "rb") as fh:
            h.update(fh.read())
    return float(b.group(1)) if h.hexdigest() == sha.group(1) else None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 25):
        self.proc = None
        self.gpu = gpu_index
        self.interval_ms = interval_ms

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms",
                 str(self.interval_ms), "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return parse_clock_samples(out)


def parse_clock_samples(out: str):
    """Median SM clock, maximum clock, the throttle reasons seen and, per
    reason, the number of samples it was active in."""
    sm, mx, counts = [], [], {}
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in out.splitlines():
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            mx.append(float(parts[2]))
        except ValueError:
            continue
        for n, v in zip(names, parts[5:9]):
            if v.lower().startswith("active"):
                counts[n] = counts.get(n, 0) + 1
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
            "reasons": sorted(counts), "samples": len(sm), "reason_samples": counts}


# ------------------------------------------------------------------ host placement
def gpu_local_cpus(dev_index: int):
    """(CPUs local to the GPU, its NUMA node) from sysfs, or (None, None).
    On a Grace host the pinned buffers of the end-to-end leg should live in
    the memory of the CPU the GPU hangs off (NVLink-C2C), so the process is
    bound to those CPUs before it allocates them (first touch places pages)."""
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=pci.bus_id", "--format=csv,noheader", "-i",
                              str(dev_index)], capture_output=True, text=True, timeout=20).stdout.strip()
        dom, rest = out.split(":", 1)
        addr = f"{int(dom, 16):04x}:{rest.lower()}"
        base = f"/sys/bus/pci/devices/{addr}"
        cpus = set()
        with open(f"{base}/local_cpulist") as f:
            for part in f.read().strip().split(","):
                if "-" in part:
                    a, b = part.split("-")
                    cpus.update(range(int(a), int(b) + 1))
                elif part:
                    cpus.add(int(part))
        with open(f"{base}/numa_node") as f:
            node = int(f.read().strip())
        return (cpus or None), node
    except (OSError, ValueError, subprocess.SubprocessError):
        return None, None


# ------------------------------------------------------------------ distributed helpers
def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def aggregate(local_ms: float, local_units: float, world: int, device=None):
    """(max time over ranks, sum of units over ranks).  Weak scaling: each
    rank runs the full workload as a replica."""
    if world == 1:
        return local_ms, local_units
    import torch
    import torch.distributed as dist

    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    u = torch.tensor([local_units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ------------------------------------------------------------------ oracle (CPU) sample
def oracle_sample(kinds, heads=(0,)):
    """Runs the oracle, as it stands, fwd + bwd on the given masks and query
    heads of the workload; returns (effective flops, seconds)."""
    import numpy as np

    import oracle
    from gen import config2, make_tensors

    flops, secs = 0.0, 0.0
    for kind in kinds:
        prob = config2(kind)
        q, k, v, do = make_tensors(prob)
        G = prob.Hq // prob.Hkv
        for h in heads:
            g = h // G
            qf = q[:, h:h + 1].float().numpy().astype(np.float64)
            dof = do[:, h:h + 1].float().numpy().astype(np.float64)
            kf = k[:, g:g + 1].float().numpy().astype(np.float64)
            vf = v[:, g:g + 1].float().numpy().astype(np.float64)
            from gen import Problem

            p1 = Problem(prob.name, prob.Tq, prob.Tk, 1, 1, prob.d, prob.segments, prob.mask, prob.seed)
            nnz = int(oracle.mask_row_counts(p1, 0).sum())
            t0 = time.perf_counter()
            oracle.attention_forward(p1, qf, kf, vf)
            oracle.attention_backward(p1, qf, kf, vf, dof)
            secs += time.perf_counter() - t0
            flops += 14.0 * prob.d * nnz
    return flops, secs


def run_oracle_subprocess(kinds, threads, heads="0"):
    env = dict(os.environ)
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), "--_oracle_sample", ",".join(kinds), "--_oracle_heads", heads]
    out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=1800)
    if out.returncode != 0:
        raise RuntimeError(out.stderr[-2000:])
    return json.loads(out.stdout.strip().splitlines()[-1])


BASELINE_SAMPLE = ("CAUSAL", "SLIDING", "CAUSAL_DOC", "SHARED_QUESTION")


def cpu_baseline(kinds=BASELINE_SAMPLE):
    kinds = list(kinds)
    threads = os.cpu_count() or 1
    r = run_oracle_subprocess(kinds, threads, heads="0,8")
    return {"value": r["flops"] / r["seconds"] / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"fp64 oracle fwd+bwd, query heads 0 and 8 (KV heads 0 and 1), {len(kinds)} static masks at "
                      f"8192 tokens ({r['seconds']:.1f} s, numpy BLAS threads={threads})"}


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from gen import STATIC_KINDS

    kinds = list(STATIC_KINDS)
    per_step = 4  # masks per step, round robin over the 12
    threads = os.cpu_count() or 1
    flops = secs = 0.0
    for s in range(args.warmup + args.steps):
        sel = [kinds[(s * per_step + i) % len(kinds)] for i in range(per_step)]
        r = run_oracle_subprocess(sel, threads)
        if s >= args.warmup:
            flops += r["flops"]
            secs += r["seconds"]
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": "query head 0, 4 static masks per step (round robin)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": "fp64 oracle fwd+bwd, query head 0, 4 of the 12 static masks per step at 8192 "
                                   "tokens"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm
def run_ours(args):
    import torch

    import long_context_masked_attention_gb300 as lca
    from gen import make_tensors

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    lca.load()
    if args.workload != "sweep8k":
        return run_workload(args, lca, dev, rank, world, barrier)
    probs = workload_problems(args.only)
    p0 = probs[0]
    q, k, v, do = make_tensors(p0, device=dev)
    calls = [lca.marshal(p.Tq, p.Tk, p.Hq, p.Hkv, p.d, p.segments, p.mask, p.scale) for p in probs]
    ws_bytes = max(lca.workspace_size(c, True) for c in calls)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    nnz = [int(lca.mask_nnz(c).sum().item()) for c in calls]
    d = p0.d
    f_fwd = [4.0 * d * n for n in nnz]
    f_bwd = [10.0 * d * n for n in nnz]
    step_flops = sum(f_fwd) + sum(f_bwd)
    o = torch.empty_like(q)
    lse = torch.empty((p0.Hq, p0.Tq), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(qq, kk, vv, dd, out_host=None):
        for i, (p, c) in enumerate(zip(probs, calls)):
            lca.attn_fwd(qq, kk, vv, p.segments, p.mask, p.scale, out=o, lse=lse, workspace=ws, call=c)
            lca.attn_bwd(dd, qq, kk, vv, o, lse, p.segments, p.mask, p.scale, dq=dq, dk=dk, dv=dv, workspace=ws,
                         call=c)
            if out_host is not None:
                for src, dst in zip((o, lse, dq, dk, dv), out_host):
                    dst.copy_(src, non_blocking=True)

    for _ in range(args.warmup):
        step(q, k, v, do)
    torch.cuda.synchronize()
    st = lca.read_status(ws)
    if st != (0, 0):
        raise RuntimeError(f"device status after warm-up: {st}")

    # ---- timed region: device-resident inputs, L2 flushed between steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0])
                          if os.environ.get("CUDA_VISIBLE_DEVICES", "").replace(",", "").isdigit() else local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    launches0 = lca.launch_count()
    for s in range(args.steps):
        flush.zero_()
        starts[s].record(stream)
        step(q, k, v, do)
        ends[s].record(stream)
    launches = lca.launch_count() - launches0
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    # ---- phase pass: the same steps again with the library's phase events on;
    # with them on the backward runs dK/dV and dQ one after another, so each
    # kernel's events bracket that kernel alone (the roofline's launch times)
    n_calls = 2 * len(probs) * args.steps
    kev = lca.KernelEvents(5 * n_calls + 8)
    torch.cuda.synchronize()
    kev.start()
    for s in range(args.steps):
        flush.zero_()
        step(q, k, v, do)
    kev.stop()
    torch.cuda.synchronize()
    st = lca.read_status(ws)
    if st != (0, 0):
        raise RuntimeError(f"device status after timed region: {st}")
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    local_ms = sum(step_ms)
    tot_ms, tot_flops = aggregate(local_ms, step_flops * args.steps, world, dev)
    value = tot_flops / (tot_ms * 1e-3) / 1e12
    phases = kev.durations()

    # ---- end to end: pinned host inputs and outputs, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        # Through the public API with host buffers: each step copies its inputs in
        # from pinned memory and brings every mask's O, LSE, dQ, dK, dV out to
        # pinned host memory.  The library is asynchronous on the caller's
        # streams, so the copies run on other streams: a step's inputs arrive in
        # the other of two input sets while the previous step computes.  With
        # --e2e-outputs copy (default) all five outputs go to device buffers and
        # are copied out; with mapped the backward stores dQ, dK, dV straight
        # into the pinned host tensors through their device mapping (the ABI
        # accepts mapped host outputs; on a GB300 the stores cross NVLink-C2C)
        # and only O and LSE, which the backward reads, are copied.  The copies of a
        # mask's outputs run on one of four streams while the next masks
        # compute (several streams let several copy engines work at once).  One
        # timed region covers all steps, from the first input copy to the last
        # output byte.
        local_cpus, numa_node = gpu_local_cpus(int(clocks.gpu))
        bound, saved_cpus = False, os.sched_getaffinity(0)
        if local_cpus:
            try:
                os.sched_setaffinity(0, local_cpus)
                bound = True
            except OSError:
                pass
        copy = torch.cuda.Stream()  # host -> device inputs
        outq = [torch.cuda.Stream() for _ in range(4)]  # device -> host outputs, round robin over masks
        hosts_in = [t.cpu().pin_memory() for t in (q, k, v, do)]
        dev_in = [[torch.empty_like(t) for t in (q, k, v, do)] for _ in range(2)]
        mapped = args.e2e_outputs == "mapped"
        dev_out = [(torch.empty_like(q), torch.empty_like(lse)) +
                   (() if mapped else (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))) for _ in probs]
        host_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (q, lse, q, k, v)] for _ in probs]
        h2d = sum(t.numel() * t.element_size() for t in hosts_in)
        d2h = sum(t.numel() * t.element_size() for outs in host_out for t in outs)
        # the copy rates of these very buffers, alone, just before the timed
        # region: the leg can only hide its copies when they run near the
        # host link's rate (pinned pages of a VM whose host memory has been
        # churned sometimes copy at well under it)
        link = {}
        for name, pairs in (("d2h", [(dst, src) for i in range(len(probs)) for src, dst in zip(dev_out[i], host_out[i])]),
                            ("h2d", list(zip(dev_in[0], hosts_in)))):
            nbytes = sum(dst.numel() * dst.element_size() for dst, _ in pairs)
            a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            with torch.cuda.stream(copy):
                a_ev.record(copy)
                for dst, src in pairs:
                    dst.copy_(src, non_blocking=True)
                b_ev.record(copy)
            torch.cuda.synchronize()
            link[name] = round(nbytes / (a_ev.elapsed_time(b_ev) * 1e-3) / 1e9, 1)
        ev_in_ready = [torch.cuda.Event() for _ in range(2)]
        ev_in_free = [torch.cuda.Event() for _ in range(2)]
        ev_out_ready = [torch.cuda.Event() for _ in probs]
        ev_out_free = [torch.cuda.Event() for _ in probs]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        t0.record(stream)
        copy.wait_stream(stream)
        for oq in outq:
            oq.wait_stream(stream)
        for s in range(args.steps):
            b = s % 2
            with torch.cuda.stream(copy):
                if s >= 2:
                    copy.wait_event(ev_in_free[b])
                for src, dst in zip(hosts_in, dev_in[b]):
                    dst.copy_(src, non_blocking=True)
                ev_in_ready[b].record(copy)
            flush.zero_()
            stream.wait_event(ev_in_ready[b])
            qq, kk, vv, dd = dev_in[b]
            for i, (p, c) in enumerate(zip(probs, calls)):
                oo, ll = dev_out[i][:2]
                gq, gk, gv = host_out[i][2:] if mapped else dev_out[i][2:]
                if s >= 1:
                    stream.wait_event(ev_out_free[i])  # last step's copy of these buffers is done
                lca.attn_fwd(qq, kk, vv, p.segments, p.mask, p.scale, out=oo, lse=ll, workspace=ws, call=c)
                lca.attn_bwd(dd, qq, kk, vv, oo, ll, p.segments, p.mask, p.scale, dq=gq, dk=gk, dv=gv,
                             workspace=ws, call=c)
                ev_out_ready[i].record(stream)
                oq = outq[i % len(outq)]
                with torch.cuda.stream(oq):
                    oq.wait_event(ev_out_ready[i])
                    for src, dst in zip(dev_out[i], host_out[i]):
                        dst.copy_(src, non_blocking=True)
                    ev_out_free[i].record(oq)
            ev_in_free[b].record(stream)
        stream.wait_stream(copy)
        for oq in outq:
            stream.wait_stream(oq)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier()
        if bound:
            os.sched_setaffinity(0, saved_cpus)  # the CPU baseline below uses every core again
        e_ms, e_flops = aggregate(t0.elapsed_time(t1), step_flops * args.steps, world, dev)
        e2e = {"value": e_flops / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms / args.steps,
               "outputs": args.e2e_outputs,
               "copy_gbps_alone": link,
               "host_binding": ({"cpus": len(local_cpus), "gpu_numa_node": numa_node} if bound else
                                "not bound (GPU's local CPUs unknown)"),
               "copies": ("inputs on one copy stream, double-buffered across steps; dQ, dK, dV stored by the "
                          "kernels into mapped pinned host memory, " if mapped else
                          "inputs on one copy stream, double-buffered across steps; ") +
                         "each mask's O and LSE" + ("" if mapped else ", dQ, dK, dV") +
                         " copied out on one of four copy streams (round robin), overlapped with compute; one timed "
                         "region from the first input copy to the last output byte"}

    pk, pk_src = peaks()
    peak, peak_src = tensor_peak(pk, pk_src, clk)
    # dominant kernel and its roofline (algorithmic FLOPs per launch / launch time)
    alg = {"fwd": 4.0, "dkv": 8.0, "dq": 6.0}  # executed matmul FLOPs per attended cell / d
    kern = {ph: sum(v) for ph, v in phases.items() if ph in alg}
    dom = max(kern, key=kern.get) if kern else None
    roofline = None
    if dom:
        n_launch = len(phases[dom])
        flops_dom = alg[dom] * d * sum(nnz) * args.steps
        achieved = flops_dom / (sum(phases[dom]) * 1e-3) / 1e12
        roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                    "unit": "TFLOP/s", "frac": achieved / peak,
                    "traffic": measured_traffic(dom), "traffic_unit": "bytes per launch (ncu, cold L2)",
                    "launches": n_launch, "peak_source": peak_src,
                    "frac_of_sustained": achieved / pk["bf16_tflops_sustained"]}
    phase_ms = {ph: sum(v) / args.steps for ph, v in phases.items()}
    per_mask = {}
    for p in probs:
        per_mask[p.mask.kind] = time_problem(lca, p, ws, flush, args.steps, 1, tensors=(q, k, v, do))
    causal = per_mask.get("CAUSAL", {}).get("tflops")
    if causal:
        for r in per_mask.values():
            r["rel_to_causal"] = r["tflops"] / causal
    balance = run_balance(lca, probs, calls, ws, (q, k, v, do)) if not args.no_balance else None
    targets = None
    if not args.no_targets and args.only is None:
        targets = run_targets(lca, dev, flush, *peaks(), clocks.gpu)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": tot_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16; seeded document lengths)",
        "config": {"workload": WORKLOAD, "seq_len": 8192, "batch": 1, "heads": "64:8", "head_dim": 128,
                   "masks": [p.mask.kind for p in probs], "l2": "flushed between steps (256 MiB write)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "pct_of_peak": 100.0 * value / peak, "peak_tflops": peak, "peak_source": peak_src,
        "roofline": roofline, "phase_ms_per_step": phase_ms, "gpu_launches": launches,
        "clocks": clk, "e2e": e2e, "per_mask": per_mask, "balance": balance, "targets": targets,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            line["cpu_baseline"] = cpu_baseline()
        except Exception as exc:  # noqa: BLE001
            line["cpu_baseline"] = {"value": None, "error": str(exc)[:200]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def run_workload(args, lca, dev, rank, world, barrier):
    """One JSON line for a non-default workload: every problem timed on its
    own (fwd and bwd medians), value = all FLOPs / sum of per-problem times."""
    import torch

    probs = workload_problems(args.only, args.workload)
    calls = [lca.marshal(p.Tq, p.Tk, p.Hq, p.Hkv, p.d, p.segments, p.mask, p.scale) for p in probs]
    ws = torch.empty(max(lca.workspace_size(c, True) for c in calls), dtype=torch.uint8, device=dev)
    del calls
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clocks = ClockSampler(dev.index or 0)
    barrier()
    clocks.start()
    launches0 = lca.launch_count()
    rows = {}
    for p in probs:
        rows[p.name] = time_problem(lca, p, ws, flush, args.steps, args.warmup, dropout=DROPOUT.get(args.workload))
        torch.cuda.empty_cache()
    launches = lca.launch_count() - launches0
    clk = clocks.stop()
    flops = sum(14.0 * 128 * r["nnz"] for r in rows.values())
    ms = sum(r["fwd_ms"] + r["bwd_ms"] for r in rows.values())
    tot_ms, tot_flops = aggregate(ms, flops, world, dev)
    pk, pk_src = peaks()
    peak, peak_src = tensor_peak(pk, pk_src, clk)
    value = tot_flops / (tot_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": tot_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16; seeded lengths and maps)",
        "config": {"workload": WORKLOADS[args.workload], "problems": [p.name for p in probs], "head_dim": 128,
                   "dropout_p": DROPOUT[args.workload][1] if args.workload in DROPOUT else 0.0,
                   "l2": "flushed before every timed forward+backward (256 MiB write)",
                   "timing": "per problem: median of the timed steps; a step = every problem once",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "pct_of_peak": 100.0 * value / peak, "peak_tflops": peak,
        "peak_source": peak_src, "gpu_launches": launches * world, "clocks": clk, "e2e": None,
        "per_problem": rows,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-outputs", choices=["copy", "mapped"], default="copy",
                    help="end-to-end leg: outputs copied out (default), or gradients stored by the kernels into "
                         "mapped pinned host memory (slower on a GB300: the stores stall the backward)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-targets", action="store_true", help="skip the dense 8K-48K target problems")
    ap.add_argument("--no-balance", action="store_true", help="skip the per-CTA balance profile")
    ap.add_argument("--only", default=None, help="comma-separated mask kinds or problem names (partial runs)")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="sweep8k")
    ap.add_argument("--_oracle_sample", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--_oracle_heads", default="0", help=argparse.SUPPRESS)
    args = ap.parse_args(argv)
    if args._oracle_sample is not None:
        flops, secs = oracle_sample(args._oracle_sample.split(","), tuple(int(h) for h in args._oracle_heads.split(",")))
        print(json.dumps({"flops": flops, "seconds": secs}))
        return 0
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
