"""Attention dropout on the GPU kernels (FlashAttention review page,
FlashAttention-1 核心优化, 算子融合: dropout fused into the attention kernel).

The keep decisions Z are integers, so they are checked bit-exactly against
the oracle's Philox draws in each of the three kernels that regenerate them:
with one-hot V the forward's O exposes Z row by row; with one-hot dO the dK/dV
kernel's dV exposes Z key by key (through its transposed bit layout); with
one-hot K, constant V and dO, the sign of dQ exposes Z.  Then forward and
backward values are checked against the fp64 oracle with the same dropout on
every static mask family and the block-sparse maps, on split dK/dV units, and at the 8K sweep's full
size on sampled rows and the last key tile."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from gen import MaskSpec, Problem, Segment, config2, make_tensors
from oracle.dropout import drop_threshold, keep_mask
from tests import cases
from tests.gpu_util import BWD_REL_L2, FWD_MAX_ABS, FWD_MEAN_ABS, LSE_ABS, check_bwd, to_np

pytestmark = pytest.mark.gpu


def check_fwd_dropout(O_gpu, L_gpu, O_ref, L_ref, p, what=""):
    """Forward bar under dropout.  O = (sum of kept P_ij v_j) / kp is rounded
    to bf16 once; its values reach 1/kp times the plain outputs' range, so
    binades whose half-ulp (up to 2^-8 |O|) exceeds the plain bar occur where
    plain outputs (convex combinations of bf16 values) cannot reach them.  The
    bar is the plain one plus that half-ulp: |dO| <= 1e-2 + 2^-8 |O_ref|, the
    mean scaled by 1/kp; LSE (independent of the dropout) keeps its bar."""
    O_gpu = to_np(O_gpu) if not isinstance(O_gpu, np.ndarray) else O_gpu
    L_gpu = to_np(L_gpu) if not isinstance(L_gpu, np.ndarray) else L_gpu
    kp = (256 - drop_threshold(p)) / 256
    assert np.all(np.isfinite(O_gpu)), what
    err = np.abs(O_gpu - O_ref)
    excess = err - (FWD_MAX_ABS + 2.0 ** -8 * np.abs(O_ref))
    assert excess.max() <= 0, f"{what}: |dO| over the bar by {excess.max():.3e} (max |dO| {err.max():.3e})"
    assert err.mean() <= FWD_MEAN_ABS / kp, f"{what}: mean |dO| = {err.mean():.3e}"
    assert np.array_equal(np.isneginf(L_ref), np.isneginf(L_gpu)), what
    fin = ~np.isneginf(L_ref)
    if fin.any():
        assert np.abs(L_gpu[fin] - L_ref[fin]).max() <= LSE_ABS, what

SEED = 0x0123456789ABCDEF

# three 128-row segments, 256 keys each; the last one at a high global row
SEGS = [Segment(0, 128, 0, 256), Segment(128, 128, 256, 256), Segment(70016, 128, 512, 256)]
TQ, TK, H, D = 70144, 768, 2, 128


def _onehot_keys(which_half, scale=1.0):
    """[TK, H, D] with key j (relative to its segment) = scale * e_{j - 128 * half}
    in the chosen half of every segment and 0 in the other half."""
    import torch

    x = torch.zeros(TK, H, D)
    for seg in SEGS:
        for c in range(128):
            x[seg.k_off + 128 * which_half + c, :, c] = scale
    return x


def _expected_z(p, h, seg):
    return keep_mask(SEED, p, h, seg.q_off + np.arange(seg.q_len), np.arange(seg.k_len))


@pytest.mark.parametrize("p", [0.1, 0.5])
def test_keep_bits_bit_exact_in_every_kernel(lca, p):
    import torch

    g = torch.Generator().manual_seed(5)
    q = (0.3 * torch.randn(TQ, H, D, generator=g)).bfloat16().cuda()
    k = (0.3 * torch.randn(TK, H, D, generator=g)).bfloat16().cuda()
    mask = MaskSpec("FULL")
    drop = (SEED, p)
    # forward: one-hot V over each half of the keys
    o_half = []
    for half in (0, 1):
        v = _onehot_keys(half).bfloat16().cuda()
        o, lse = lca.attn_fwd(q, k, v, SEGS, mask, dropout=drop)
        o_half.append(o)
    # dK/dV: dO_i = e_i (segment-relative row) makes dV_j[i] = P~_ij
    do = torch.zeros(TQ, H, D)
    for seg in SEGS:
        for r in range(128):
            do[seg.q_off + r, :, r] = 1.0
    do = do.bfloat16().cuda()
    v0 = _onehot_keys(0).bfloat16().cuda()
    o0, lse0 = lca.attn_fwd(q, k, v0, SEGS, mask, dropout=drop)
    _, _, dv = lca.attn_bwd(do, q, k, v0, o0, lse0, SEGS, mask, dropout=drop)
    # dQ: K_j = e_j on one half, V_j = e_0, dO_i = 1: dS_ij = P_ij (Z_ij / kp - D_i) > 0 iff kept
    vc = torch.zeros(TK, H, D)
    vc[:, :, 0] = 1.0
    vc = vc.bfloat16().cuda()
    ones = torch.ones(TQ, H, D).bfloat16().cuda()
    dq_half = []
    for half in (0, 1):
        kk = _onehot_keys(half, 2.0).bfloat16().cuda()
        oc, lc = lca.attn_fwd(q, kk, vc, SEGS, mask, dropout=drop)
        dq, _, _ = lca.attn_bwd(ones, q, kk, vc, oc, lc, SEGS, mask, dropout=drop)
        dq_half.append(dq)
    torch.cuda.synchronize()
    for h in range(H):
        for seg in SEGS:
            z = _expected_z(p, h, seg)  # [128 rows, 256 keys]
            rows = slice(seg.q_off, seg.q_off + 128)
            got_fwd = np.concatenate([to_np(o_half[half][rows, h]) != 0 for half in (0, 1)], axis=1)
            assert np.array_equal(got_fwd, z), ("forward", h, seg)
            got_dkv = to_np(dv[seg.k_off:seg.k_off + 256, h]).T != 0  # [row i, key j]
            assert np.array_equal(got_dkv, z), ("dK/dV", h, seg)
            got_dq = np.concatenate([to_np(dq_half[half][rows, h]) > 0 for half in (0, 1)], axis=1)
            assert np.array_equal(got_dq, z), ("dQ", h, seg)
            assert 0.3 < z.mean() / (1 - p) < 1.7


def _run(lca, prob, drop):
    import torch

    q, k, v, do = (t.cuda() for t in make_tensors(prob, device="cuda"))
    o, lse = lca.attn_fwd(q, k, v, prob.segments, prob.mask, prob.scale, dropout=drop)
    dq, dk, dv = lca.attn_bwd(do, q, k, v, o, lse, prob.segments, prob.mask, prob.scale, dropout=drop)
    torch.cuda.synchronize()
    return (q, k, v, do), (o, lse, dq, dk, dv)


def _parity(lca, prob, drop):
    (q, k, v, do), (o, lse, dq, dk, dv) = _run(lca, prob, drop)
    qc, kc, vc, doc = (t.cpu() for t in (q, k, v, do))
    O, L = oracle.attention_forward(prob, qc, kc, vc, dropout=drop)
    check_fwd_dropout(o, lse, O, L, drop[1], what=prob.name)
    check_bwd((dq, dk, dv), oracle.attention_backward(prob, qc, kc, vc, doc, dropout=drop), what=prob.name)


SMALL = cases.gpu_small_all() + [p for p in cases.edge_cases() if p.name in ("edge_q_gt_k", "edge_gaps")]


@pytest.mark.parametrize("prob", SMALL, ids=[p.name for p in SMALL])
def test_dropout_parity_families(lca, prob):
    _parity(lca, prob, (977 + len(prob.name), 0.1))


def test_dropout_parity_flashmask_descriptor(lca):
    from tests.flashmask_inputs import as_flashmask

    prob = cases.gpu_small_all()[5]
    fm = as_flashmask(prob)
    drop = (31337, 0.2)
    (q, k, v, do), outs = _run(lca, fm, drop)
    _, outs_family = _run(lca, prob, drop)
    for a, b in zip(outs, outs_family):
        assert np.array_equal(to_np(a), to_np(b))
    qc, kc, vc, doc = (t.cpu() for t in (q, k, v, do))
    O, L = oracle.attention_forward(prob, qc, kc, vc, dropout=drop)
    check_fwd_dropout(outs[0], outs[1], O, L, drop[1], what=fm.name)


def test_dropout_parity_split_units(lca):
    """dK/dV units cut into chunks: the reduction applies 1/kp as well."""
    prob = cases.single(2048, "GLOBAL_SLIDING", 8, 1, 128, 41, num_global=16, window_left=100, window_right=100)
    _parity(lca, prob, (4242, 0.15))


def test_same_seed_same_result_other_seed_other_result(lca):
    prob = cases.gpu_small_all()[1]
    _, a = _run(lca, prob, (1, 0.1))
    _, b = _run(lca, prob, (1, 0.1))
    _, c = _run(lca, prob, (2, 0.1))
    for x, y in zip(a, b):
        assert np.array_equal(to_np(x), to_np(y))
    assert not np.array_equal(to_np(a[0]), to_np(c[0]))
    assert np.array_equal(to_np(a[1]), to_np(c[1]))  # LSE does not depend on Z


@pytest.mark.parametrize("p", [0.0, 0.001])
def test_zero_threshold_is_the_plain_path(lca, p):
    """t = floor(256 p + 1/2) = 0 keeps every entry: results equal the call
    without dropout bit for bit."""
    prob = cases.gpu_small_all()[1]
    _, a = _run(lca, prob, (9, p))
    _, b = _run(lca, prob, None)
    for x, y in zip(a, b):
        assert np.array_equal(to_np(x), to_np(y))


def test_dropout_8k_causal_full_size(lca):
    """The 8K causal sweep case (GQA 64:8) with dropout 0.1: O, LSE, dQ on
    the first, middle and last 64 rows of three query heads, dK/dV of the last
    key tile (attended only by the last rows), and sum_j dK_j = 0."""
    prob = config2("CAUSAL")
    drop = (0xC0FFEE, 0.1)
    (q, k, v, do), (o, lse, dq, dk, dv) = _run(lca, prob, drop)
    seg = prob.segments[0]
    n = seg.q_len
    rows = np.unique(np.concatenate([np.arange(64), np.arange(n // 2 - 32, n // 2 + 32), np.arange(n - 64, n)]))
    G = prob.Hq // prob.Hkv
    num, den = 0.0, 0.0
    for h in (0, G + 1, prob.Hq - 1):
        O_ref, L_ref = oracle.forward_rows(prob, q, k, v, 0, h, rows, dropout=drop)
        check_fwd_dropout(o[rows, h], lse[h, rows], O_ref, L_ref, drop[1], what=f"8k head {h}")
        dQ_ref = oracle.backward_rows(prob, q, k, v, do, 0, h, rows, dropout=drop)
        num += float(np.sum((to_np(dq[rows, h]) - dQ_ref) ** 2))
        den += float(np.sum(dQ_ref ** 2))
    assert np.sqrt(num / den) <= BWD_REL_L2
    last = np.arange(n - 128, n)
    for g in (0, prob.Hkv - 1):
        dK_ref = np.zeros((128, prob.d))
        dV_ref = np.zeros((128, prob.d))
        for h in range(g * G, (g + 1) * G):
            a, b = oracle.key_grads_from_rows(prob, q, k, v, do, 0, h, last, last, dropout=drop)
            dK_ref += a
            dV_ref += b
        for name, x, r in (("dK", to_np(dk[last, g]), dK_ref), ("dV", to_np(dv[last, g]), dV_ref)):
            rel = np.linalg.norm(x - r) / np.linalg.norm(r)
            assert rel <= BWD_REL_L2, (name, g, rel)
        sk = dk[:, g].double().sum(0)
        ak = dk[:, g].double().abs().sum(0)
        assert float(sk.norm()) <= 1e-2 * float(ak.norm())
