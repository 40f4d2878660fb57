"""Masked attention forward and backward in fp64 — TEST INFRASTRUCTURE ONLY.

Definition (FlashAttention review page, FlashAttention-1 问题和瓶颈):
    S = tau * Q K^T,  tau = 1/sqrt(d)
    P = softmax(S) over the attended keys of each row
    O = P V
The forward also returns the one row statistic that the backward needs
(FlashAttention-2 核心优化, 合并反向传播统计量): LSE_i = log sum_j exp(S_ij),
natural log.  A row with no attended key has O_i = 0 and LSE_i = -inf.

Backward (FlashAttention-2 核心优化, 反向传播: dQ_i = sum_j dS_ij K_j), with
dO the upstream gradient:
    dP = dO V^T,  D_i = sum_j P_ij dP_ij,  dS = P * (dP - D)
    dQ = tau dS K,  dK = tau dS^T Q,  dV = P^T dO
dK and dV of a KV head are summed over the query heads that share it
(grouped-query attention, the GQA 64:8 setting of the benchmark review), and
over every segment that reads that key.  Masked cells have P = dS = 0.

Head h reads KV head h // (Hq // Hkv).

Dropout (FlashAttention review page, FlashAttention-1 核心优化, 算子融合):
with `dropout` = (seed, p), the forward uses P~ = P * Z / k (Z from
``oracle.dropout``) in O = P~ V, LSE stays that of P, and the backward is
    dP~ = dO V^T,  D_i = sum_j P~_ij dP~_ij = dO_i . O_i,
    dS = P * (Z/k * dP~ - D),  dV = P~^T dO,  dQ, dK as above.
"""
from __future__ import annotations

import numpy as np

from .dropout import scaled_keep
from .masks import segment_mask


def _f64(x):
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().float().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def segment_head_forward(q_s, k_s, v_s, mask, scale, zk=None):
    """One segment, one head.  q_s [n_q, d], k_s/v_s [n_k, d], mask [n_q, n_k];
    zk [n_q, n_k] = Z / k of dropout, or None.  Returns O, LSE and P (the
    undropped probabilities)."""
    s = scale * (q_s @ k_s.T)
    s = np.where(mask, s, -np.inf)
    has = mask.any(axis=1)
    m = np.where(has, np.max(s, axis=1, initial=-np.inf), 0.0)
    e = np.where(mask, np.exp(s - m[:, None]), 0.0)
    l = e.sum(axis=1)
    lse = np.where(has, m + np.log(np.where(has, l, 1.0)), -np.inf)
    p = np.where(mask, np.exp(s - np.where(has, lse, 0.0)[:, None]), 0.0)
    o = (p if zk is None else p * zk) @ v_s
    return o, lse, p


def segment_head_backward(q_s, k_s, v_s, do_s, mask, scale, zk=None):
    """Returns dq_s, dk_s, dv_s, D (and O) for one segment and one head."""
    o, lse, p = segment_head_forward(q_s, k_s, v_s, mask, scale, zk)
    pt = p if zk is None else p * zk  # the probabilities O was made from
    dpt = do_s @ v_s.T
    D = (pt * dpt).sum(axis=1)
    # the identity D_i = dO_i . O_i (FlashAttention-2's row statistic)
    assert np.allclose(D, (do_s * o).sum(axis=1), rtol=1e-9, atol=1e-9 * (1 + np.abs(D).max(initial=0)))
    dp = dpt if zk is None else zk * dpt
    ds = p * (dp - D[:, None])
    dq = scale * (ds @ k_s)
    dk = scale * (ds.T @ q_s)
    dv = pt.T @ do_s
    return dq, dk, dv, D, o, lse


def _kv_head(prob, h):
    return h // (prob.Hq // prob.Hkv)


def _zk(dropout, seg, h, rows=None):
    """Z / k of segment `seg`'s rows (segment-relative; all when None) and
    all of its keys, or None without dropout."""
    if dropout is None:
        return None
    rows = np.arange(seg.q_len) if rows is None else np.asarray(rows)
    return scaled_keep(dropout, h, seg.q_off + rows, np.arange(seg.k_len))


def attention_forward(prob, q, k, v, heads=None, dropout=None):
    """Full forward.  Returns O [Tq, Hq, d] and LSE [Hq, Tq] (fp64); rows of
    heads not in `heads` are left at 0 / -inf.  `dropout` = (seed, p)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    scale = prob.softmax_scale
    O = np.zeros((prob.Tq, prob.Hq, prob.d))
    LSE = np.full((prob.Hq, prob.Tq), -np.inf)
    for h in (range(prob.Hq) if heads is None else heads):
        g = _kv_head(prob, h)
        for s, seg in enumerate(prob.segments):
            qs = slice(seg.q_off, seg.q_off + seg.q_len)
            ks = slice(seg.k_off, seg.k_off + seg.k_len)
            mask = segment_mask(prob.mask, s, seg, h)
            o, lse, _ = segment_head_forward(q[qs, h], k[ks, g], v[ks, g], mask, scale, _zk(dropout, seg, h))
            O[qs, h] = o
            LSE[h, qs] = lse
    return O, LSE


def attention_backward(prob, q, k, v, do, heads=None, dropout=None):
    """Full backward.  Returns dQ [Tq, Hq, d], dK/dV [Tk, Hkv, d] (fp64).
    With `heads`, only those query heads contribute (dK/dV of a KV head are
    complete only when all of its query heads are listed)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    scale = prob.softmax_scale
    dQ = np.zeros((prob.Tq, prob.Hq, prob.d))
    dK = np.zeros((prob.Tk, prob.Hkv, prob.d))
    dV = np.zeros((prob.Tk, prob.Hkv, prob.d))
    for h in (range(prob.Hq) if heads is None else heads):
        g = _kv_head(prob, h)
        for s, seg in enumerate(prob.segments):
            qs = slice(seg.q_off, seg.q_off + seg.q_len)
            ks = slice(seg.k_off, seg.k_off + seg.k_len)
            mask = segment_mask(prob.mask, s, seg, h)
            dq, dk, dv, _, _, _ = segment_head_backward(
                q[qs, h], k[ks, g], v[ks, g], do[qs, h], mask, scale, _zk(dropout, seg, h)
            )
            dQ[qs, h] = dq
            dK[ks, g] += dk
            dV[ks, g] += dv
    return dQ, dK, dV


def forward_rows(prob, q, k, v, seg_index, head, rows, dropout=None):
    """Forward for selected rows (segment-relative) of one segment and head:
    returns O [len(rows), d], LSE [len(rows)]."""
    seg = prob.segments[seg_index]
    g = _kv_head(prob, head)
    scale = prob.softmax_scale
    rows = np.asarray(rows)
    qr = _f64(q[seg.q_off + rows, head]) if not hasattr(q, "detach") else _f64(q[seg.q_off + rows, head])
    kk = _f64(k[seg.k_off:seg.k_off + seg.k_len, g])
    vv = _f64(v[seg.k_off:seg.k_off + seg.k_len, g])
    mask = segment_mask(prob.mask, seg_index, seg, head, rows)
    o, lse, _ = segment_head_forward(qr, kk, vv, mask, scale, _zk(dropout, seg, head, rows))
    return o, lse


def backward_rows(prob, q, k, v, do, seg_index, head, rows, dropout=None):
    """dQ for selected rows (segment-relative) of one segment and head: a
    row's softmax, D_i and dS_ij depend on that row alone."""
    seg = prob.segments[seg_index]
    g = _kv_head(prob, head)
    scale = prob.softmax_scale
    rows = np.asarray(rows)
    qr = _f64(q[seg.q_off + rows, head])
    dor = _f64(do[seg.q_off + rows, head])
    kk = _f64(k[seg.k_off:seg.k_off + seg.k_len, g])
    vv = _f64(v[seg.k_off:seg.k_off + seg.k_len, g])
    mask = segment_mask(prob.mask, seg_index, seg, head, rows)
    dq, _, _, _, _, _ = segment_head_backward(qr, kk, vv, dor, mask, scale, _zk(dropout, seg, head, rows))
    return dq


def key_grads_from_rows(prob, q, k, v, do, seg_index, head, rows, key_cols, dropout=None):
    """Contribution of the given query rows of one segment and head to dK and
    dV of the given key columns (segment-relative): dK_j = tau sum_i dS_ij q_i,
    dV_j = sum_i P_ij dO_i over the listed rows only."""
    seg = prob.segments[seg_index]
    g = _kv_head(prob, head)
    scale = prob.softmax_scale
    rows = np.asarray(rows)
    key_cols = np.asarray(key_cols)
    qr = _f64(q[seg.q_off + rows, head])
    dor = _f64(do[seg.q_off + rows, head])
    kk = _f64(k[seg.k_off:seg.k_off + seg.k_len, g])
    vv = _f64(v[seg.k_off:seg.k_off + seg.k_len, g])
    mask = segment_mask(prob.mask, seg_index, seg, head, rows)
    zk = _zk(dropout, seg, head, rows)
    _, _, p = segment_head_forward(qr, kk, vv, mask, scale)
    pt = p if zk is None else p * zk
    dpt = dor @ vv.T
    D = (pt * dpt).sum(axis=1)
    dp = dpt if zk is None else zk * dpt
    ds = p * (dp - D[:, None])
    return scale * (ds[:, key_cols].T @ qr), pt[:, key_cols].T @ dor
