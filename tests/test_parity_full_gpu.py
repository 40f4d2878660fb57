"""Parity at the workloads' full sizes, in the launch configuration the
benchmark uses (one call over the whole packed batch), on outputs the oracle
can compute row by row, plus properties that hold at any size.

Sampled, not exhaustive: for a few segments (largest, a middle one, the
smallest) and query heads spread over the KV groups, the first, middle and
last 64 rows get O, LSE and dQ checked; dK/dV are checked on the last key
tile of causal segments (attended only by the segment's last rows, so the
oracle can compute them exactly) and, everywhere, through the identities
sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i (over the query heads of each KV
head), which hold for any mask because every softmax row sums to one."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from gen import config3, config4, config5, make_tensors
from tests.gpu_util import FWD_MAX_ABS, FWD_MEAN_ABS, LSE_ABS, BWD_REL_L2, to_np

pytestmark = pytest.mark.gpu


def _run(lca, prob):
    import torch

    q, k, v, do = make_tensors(prob, device="cuda")
    call = lca.marshal(prob.Tq, prob.Tk, prob.Hq, prob.Hkv, prob.d, prob.segments, prob.mask, prob.scale)
    o, lse = lca.attn_fwd(q, k, v, prob.segments, prob.mask, prob.scale, call=call)
    dq, dk, dv = lca.attn_bwd(do, q, k, v, o, lse, prob.segments, prob.mask, prob.scale, call=call)
    torch.cuda.synchronize()
    return (q, k, v, do), (o, lse, dq, dk, dv)


def _sample_segments(prob):
    order = sorted(range(len(prob.segments)), key=lambda s: -prob.segments[s].q_len)
    order = [s for s in order if prob.segments[s].q_len > 0 and prob.segments[s].k_len > 0]
    return sorted({order[0], order[len(order) // 2], order[-1]})


def _sample_rows(q_len, n=64):
    mid = max(0, q_len // 2 - n // 2)
    return np.unique(np.concatenate([np.arange(min(n, q_len)), np.arange(mid, min(q_len, mid + n)),
                                     np.arange(max(0, q_len - n), q_len)]))


def _check_rows(lca, prob, inputs, outputs, heads):
    q, k, v, do = inputs
    o, lse, dq, _, _ = outputs
    errs_o, errs_l, dq_num, dq_den = [], [], 0.0, 0.0
    for s in _sample_segments(prob):
        seg = prob.segments[s]
        rows = _sample_rows(seg.q_len)
        for h in heads:
            O_ref, L_ref = oracle.forward_rows(prob, q, k, v, s, h, rows)
            O_gpu = to_np(o[seg.q_off + rows, h])
            L_gpu = lse[h, seg.q_off + rows].double().cpu().numpy()
            e = np.abs(O_gpu - O_ref)
            errs_o.append(e)
            assert np.array_equal(np.isneginf(L_ref), np.isneginf(L_gpu)), (prob.name, s, h)
            fin = np.isfinite(L_ref)
            errs_l.append(np.abs(L_gpu[fin] - L_ref[fin]))
            dQ_ref = oracle.backward_rows(prob, q, k, v, do, s, h, rows)
            dQ_gpu = to_np(dq[seg.q_off + rows, h])
            dq_num += float(np.sum((dQ_gpu - dQ_ref) ** 2))
            dq_den += float(np.sum(dQ_ref ** 2))
    e = np.concatenate([x.ravel() for x in errs_o])
    assert e.max() <= FWD_MAX_ABS and e.mean() <= FWD_MEAN_ABS, (prob.name, e.max(), e.mean())
    le = np.concatenate(errs_l)
    assert le.size == 0 or le.max() <= LSE_ABS, (prob.name, le.max())
    rel = np.sqrt(dq_num / max(dq_den, 1e-30))
    assert rel <= BWD_REL_L2, (prob.name, "dQ", rel)


def _check_last_key_tile(lca, prob, inputs, outputs, g=0):
    """Causal segments: the last 128 keys are attended only by the last 128
    rows (bottom-right diagonal), so the oracle computes their dK/dV exactly."""
    q, k, v, do = inputs
    _, _, _, dk, dv = outputs
    G = prob.Hq // prob.Hkv
    # the segment reaching furthest into its keys: for a shard batch, the last
    # shard of the largest document (no other shard reads past its end)
    s = max((i for i, x in enumerate(prob.segments) if x.q_len > 0), key=lambda i: prob.segments[i].k_len)
    seg = prob.segments[s]
    n = min(128, seg.k_len, seg.q_len)
    rows = np.arange(seg.q_len - n, seg.q_len)
    cols = np.arange(seg.k_len - n, seg.k_len)
    dK_ref = np.zeros((n, prob.d))
    dV_ref = np.zeros((n, prob.d))
    # every segment sharing this key range contributes (shards of one document)
    for s2, seg2 in enumerate(prob.segments):
        if seg2.k_off != seg.k_off or seg2.k_len < seg.k_len:
            continue
        r2 = np.arange(max(0, seg2.q_len - n), seg2.q_len)
        c2 = cols  # same key positions (same k_off)
        for h in range(g * G, (g + 1) * G):
            a, b = oracle.key_grads_from_rows(prob, q, k, v, do, s2, h, r2, c2)
            dK_ref += a
            dV_ref += b
    dK_gpu = to_np(dk[seg.k_off + cols, g])
    dV_gpu = to_np(dv[seg.k_off + cols, g])
    for name, x, r in (("dK", dK_gpu, dK_ref), ("dV", dV_gpu, dV_ref)):
        rel = np.linalg.norm(x - r) / max(np.linalg.norm(r), 1e-30)
        assert rel <= BWD_REL_L2, (prob.name, name, rel)


def _check_gradient_sums(prob, inputs, outputs):
    import torch

    _, _, _, do = inputs
    _, _, _, dk, dv = outputs
    G = prob.Hq // prob.Hkv
    # every query row of these workloads attends at least one key, so the
    # expected sum of dV runs over all rows
    for g in range(prob.Hkv):
        sk = dk[:, g].double().sum(0)
        ak = dk[:, g].double().abs().sum(0)
        assert float(sk.norm()) <= 1e-2 * float(ak.norm()) + 1e-6, (prob.name, "sum dK", g)
        want = torch.zeros(prob.d, dtype=torch.float64, device=dv.device)
        for h in range(g * G, (g + 1) * G):
            want += do[:, h].double().sum(0)
        got = dv[:, g].double().sum(0)
        rel = float((got - want).norm() / max(float(want.norm()), 1e-30))
        assert rel <= 2e-2, (prob.name, "sum dV", g, rel)


def _heads(prob):
    G = prob.Hq // prob.Hkv
    return sorted({0, G + 1 if prob.Hq > G + 1 else 0, prob.Hq - 1})


DENSE = [config3(S, heads, kind) for S in (8192, 49152) for heads in ("gqa", "mha") for kind in ("CAUSAL", "CAUSAL_DOC")]


@pytest.mark.parametrize("prob", DENSE, ids=[p.name for p in DENSE])
def test_dense_sweep_full_size(lca, prob):
    inputs, outputs = _run(lca, prob)
    _check_rows(lca, prob, inputs, outputs, _heads(prob))
    _check_last_key_tile(lca, prob, inputs, outputs, g=0)
    _check_last_key_tile(lca, prob, inputs, outputs, g=prob.Hkv - 1)
    _check_gradient_sums(prob, inputs, outputs)


SPARSE = [config4(32768, "gqa", "uniform64"), config4(32768, "mha", "uniform128"), config4(32768, "gqa", "variable"),
          config4(131072, "gqa", "uniform128")]


@pytest.mark.parametrize("prob", SPARSE, ids=[p.name for p in SPARSE])
def test_block_sparse_full_size(lca, prob):
    inputs, outputs = _run(lca, prob)
    _check_rows(lca, prob, inputs, outputs, _heads(prob))
    _check_gradient_sums(prob, inputs, outputs)


def test_shard_batch_512k(lca):
    """512K tokens of Pareto-length documents cut into U{1K..32K} shards,
    rebatched into one launch; checked against the oracle on sampled rows and
    the largest document's last key tile, and against the same documents as
    one causal-document launch."""
    import torch

    prob = config5()
    inputs, outputs = _run(lca, prob)
    _check_rows(lca, prob, inputs, outputs, _heads(prob))
    _check_last_key_tile(lca, prob, inputs, outputs, g=0)
    _check_gradient_sums(prob, inputs, outputs)
    # same documents, one segment each, queries in document order
    from gen import MaskSpec, Problem, docs_to_segments

    docs = prob.extra["doc_lengths"]
    doc_prob = Problem("c5_docs", prob.Tq, prob.Tk, prob.Hq, prob.Hkv, prob.d, docs_to_segments(docs),
                       MaskSpec("CAUSAL_DOC"), prob.seed)
    q, k, v, do = inputs
    rows = np.empty(prob.Tq, dtype=np.int64)
    for seg, src in zip(prob.segments, prob.extra["shard_src"]):
        rows[seg.q_off:seg.q_off + seg.q_len] = src + np.arange(seg.q_len)
    inv = np.empty_like(rows)
    inv[rows] = np.arange(prob.Tq)
    ridx = torch.from_numpy(inv).cuda()  # document-order row -> packed shard row
    qd, dod = q[ridx], do[ridx]
    o_doc, lse_doc = lca.attn_fwd(qd, k, v, doc_prob.segments, doc_prob.mask)
    torch.cuda.synchronize()
    o, lse = outputs[0], outputs[1]
    assert float((o[ridx].float() - o_doc.float()).abs().max()) <= 1e-2
    assert float((lse[:, ridx] - lse_doc).abs().max()) <= 1e-3


def test_split_key_tile_full_size_global_sliding(lca):
    """8K global-sliding sweep case, GQA 64:8: key tile 0 holds the 64 global
    keys every query attends, so its dK/dV units are far longer than the rest
    and run as chunks whose f32 partials are reduced.  That tile's dK/dV (KV
    head 0, all 8192 rows of its 8 query heads) is checked exactly."""
    from gen import config2

    prob = config2("GLOBAL_SLIDING")
    inputs, outputs = _run(lca, prob)
    _check_rows(lca, prob, inputs, outputs, _heads(prob))
    _check_gradient_sums(prob, inputs, outputs)
    q, k, v, do = inputs
    _, _, _, dk, dv = outputs
    G = prob.Hq // prob.Hkv
    cols = np.arange(128)
    dK_ref = np.zeros((128, prob.d))
    dV_ref = np.zeros((128, prob.d))
    seg = prob.segments[0]
    for h in range(G):
        for r0 in range(0, seg.q_len, 2048):
            rows = np.arange(r0, min(seg.q_len, r0 + 2048))
            a, b = oracle.key_grads_from_rows(prob, q, k, v, do, 0, h, rows, cols)
            dK_ref += a
            dV_ref += b
    for name, x, r in (("dK", to_np(dk[cols, 0]), dK_ref), ("dV", to_np(dv[cols, 0]), dV_ref)):
        rel = np.linalg.norm(x - r) / max(np.linalg.norm(r), 1e-30)
        assert rel <= BWD_REL_L2, (name, rel)
