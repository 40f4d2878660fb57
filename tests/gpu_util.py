"""Helpers for the GPU parity tests: run the CUDA path through the binding and
compare with the fp64 oracle under the stated tolerances."""
from __future__ import annotations

import numpy as np

# Tolerances for bf16 inputs with fp32 accumulation.
FWD_MAX_ABS = 1e-2
FWD_MEAN_ABS = 1e-3
LSE_ABS = 1e-3
BWD_REL_L2 = 2e-2


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_fwd(lib, prob, q, k, v, device="cuda"):
    import torch

    qd, kd, vd = (t.to(device) for t in (q, k, v))
    o, lse = lib.attn_fwd(qd, kd, vd, prob.segments, prob.mask, prob.scale)
    torch.cuda.synchronize()
    return o, lse


def run_bwd(lib, prob, q, k, v, do, o, lse, device="cuda"):
    import torch

    qd, kd, vd, dod = (t.to(device) for t in (q, k, v, do))
    dq, dk, dv = lib.attn_bwd(dod, qd, kd, vd, o, lse, prob.segments, prob.mask, prob.scale)
    torch.cuda.synchronize()
    return dq, dk, dv


def check_fwd(O_gpu, L_gpu, O_ref, L_ref, heads=None, rows=None, what=""):
    """Element-wise forward parity.  `heads`/`rows` restrict the comparison."""
    O_gpu = to_np(O_gpu) if not isinstance(O_gpu, np.ndarray) else O_gpu
    L_gpu = to_np(L_gpu) if not isinstance(L_gpu, np.ndarray) else L_gpu
    if heads is not None:
        O_gpu, O_ref = O_gpu[:, heads], O_ref[:, heads]
        L_gpu, L_ref = L_gpu[heads], L_ref[heads]
    if rows is not None:
        O_gpu, O_ref = O_gpu[rows], O_ref[rows]
        L_gpu, L_ref = L_gpu[..., rows], L_ref[..., rows]
    assert np.all(np.isfinite(O_gpu)), f"{what}: non-finite O"
    err = np.abs(O_gpu - O_ref)
    assert err.max() <= FWD_MAX_ABS, f"{what}: max|O-O_ref| = {err.max():.3e}"
    assert err.mean() <= FWD_MEAN_ABS, f"{what}: mean|O-O_ref| = {err.mean():.3e}"
    ninf_ref, ninf_gpu = np.isneginf(L_ref), np.isneginf(L_gpu)
    assert np.array_equal(ninf_ref, ninf_gpu), f"{what}: -inf LSE rows differ ({(ninf_ref != ninf_gpu).sum()})"
    fin = ~ninf_ref
    assert np.all(np.isfinite(L_gpu[fin])), f"{what}: non-finite LSE"
    if fin.any():
        lerr = np.abs(L_gpu[fin] - L_ref[fin]).max()
        assert lerr <= LSE_ABS, f"{what}: max|LSE-LSE_ref| = {lerr:.3e}"
    return float(err.max()), float(err.mean())


def rel_l2(a, b):
    a = to_np(a) if not isinstance(a, np.ndarray) else a
    assert np.all(np.isfinite(a)), "non-finite gradient"
    nb = np.linalg.norm(b)
    if nb == 0.0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / nb)


def check_bwd(grads, refs, what=""):
    out = {}
    for name, g, r in zip(("dq", "dk", "dv"), grads, refs):
        e = rel_l2(g, r)
        out[name] = e
        assert e <= BWD_REL_L2, f"{what}: rel L2 {name} = {e:.3e}"
    return out
