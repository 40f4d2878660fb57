"""Parity at the workloads' full sizes, in the launch configuration the
benchmark uses (one call over the whole packed batch), on outputs the oracle
can compute row by row, plus properties that hold at any size.

Sampled, not exhaustive: for a few segments (largest, a middle one, the
smallest) and query heads spread over the KV groups, the first, middle and
last 64 rows get O, LSE and dQ checked.  dK/dV are checked element-wise on
chosen key tiles -- the first, an interior one, the last and one the mask
makes partial -- against the oracle summed over every query head of the KV
group and every row (of every segment) that attends those keys; at 48K and
512K on documents no longer than 32K.  Everywhere, the identities
sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i (over the query heads of each KV
head) hold for any mask because every softmax row sums to one."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from gen import STATIC_KINDS, config2, config3, config4, config5, make_tensors
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


def _one_head_per_group(prob):
    """One query head of every KV group, at a different place in each group."""
    G = prob.Hq // prob.Hkv
    return [g * G + g % G for g in range(prob.Hkv)]


def _oracle_key_tiles(prob, inputs, s, g, kts, chunk=1024):
    """Oracle dK, dV of key tiles `kts` (128 keys each, relative to segment
    s's keys) of KV head g: the sum over every segment that reads those keys
    (the same k_off: shards of one document), every query head of the group
    and every query row that attends at least one of the keys.  Rows that
    attend none of them contribute nothing, so they are left out."""
    seg = prob.segments[s]
    cols = np.concatenate([np.arange(kt * 128, min(seg.k_len, kt * 128 + 128)) for kt in kts])
    dK = np.zeros((cols.size, prob.d))
    dV = np.zeros((cols.size, prob.d))
    G = prob.Hq // prob.Hkv
    for s2, seg2 in enumerate(prob.segments):
        if seg2.k_off != seg.k_off or seg2.q_len == 0:
            continue
        sel = np.nonzero(cols < seg2.k_len)[0]
        if sel.size == 0:
            continue
        for h in range(g * G, (g + 1) * G):
            for r0 in range(0, seg2.q_len, chunk):
                rows = np.arange(r0, min(seg2.q_len, r0 + chunk))
                m = oracle.segment_mask(prob.mask, s2, seg2, h, rows)[:, cols[sel]]
                att = rows[m.any(axis=1)]
                if att.size == 0:
                    continue
                a, b = oracle.key_grads_from_rows(prob, *inputs, s2, h, att, cols[sel])
                dK[sel] += a
                dV[sel] += b
    out, at = [], 0
    for kt in kts:
        n = min(seg.k_len, kt * 128 + 128) - kt * 128
        out.append((dK[at:at + n], dV[at:at + n]))
        at += n
    return out


def _check_key_tiles(prob, inputs, outputs, s, g, kts, what=""):
    """dK/dV of the given key tiles of segment s, KV head g, element-wise
    (relative L2 per tile) against the oracle."""
    _, _, _, dk, dv = outputs
    seg = prob.segments[s]
    refs = _oracle_key_tiles(prob, inputs, s, g, kts)
    for kt, (dK_ref, dV_ref) in zip(kts, refs):
        rows = seg.k_off + np.arange(kt * 128, min(seg.k_len, kt * 128 + 128))
        for name, x, r in (("dK", to_np(dk[rows, g]), dK_ref), ("dV", to_np(dv[rows, g]), dV_ref)):
            assert np.linalg.norm(r) > 0, (prob.name, what, s, g, kt, name, "no attending row")
            rel = np.linalg.norm(x - r) / np.linalg.norm(r)
            assert rel <= BWD_REL_L2, (prob.name, what, s, g, kt, name, rel)


def _partial_key_tiles(prob, s, h):
    """Key tiles of segment s holding at least one 128x128 (query tile, key
    tile) block that the oracle's mask for head h makes PARTIAL: some cells
    attended, not all (a block cut by the segment's end counts as partial
    when anything in it is attended, as the kernels treat it)."""
    seg = prob.segments[s]
    nk = -(-seg.k_len // 128)
    part = np.zeros(nk, dtype=bool)
    for r0 in range(0, seg.q_len, 128):
        rows = np.arange(r0, min(seg.q_len, r0 + 128))
        m = np.zeros((128, nk * 128), dtype=bool)
        m[:rows.size, :seg.k_len] = oracle.segment_mask(prob.mask, s, seg, h, rows)
        blk = m.reshape(128, nk, 128).transpose(1, 0, 2).reshape(nk, -1)
        part |= blk.any(axis=1) & ~blk.all(axis=1)
    return np.nonzero(part)[0]


def _tiles_to_check(prob, s, h):
    """The first, a middle and the last key tile of segment s, plus the
    partial tile nearest three quarters of the way (if the mask has one)."""
    nk = -(-prob.segments[s].k_len // 128)
    kts = {0, nk // 2, nk - 1}
    part = [kt for kt in _partial_key_tiles(prob, s, h) if kt not in kts]
    if part:
        kts.add(min(part, key=lambda kt: abs(kt - 3 * nk // 4)))
    return sorted(kts)


@pytest.mark.parametrize("kind", STATIC_KINDS)
def test_static_sweep_8k_full_size(lca, kind):
    """The benchmark's 8K static-mask sweep (GQA 64:8), each family in its own
    full-size launch: O, LSE and dQ of one query head per KV group on the
    first, middle and last 64 rows of three segments; dK/dV element-wise on
    the first, a middle, the last and a partial key tile of the largest
    segment (and, for document families, of a middle-sized and the smallest
    document), in a different KV group per family; gradient sums everywhere."""
    import torch

    prob = config2(kind)
    inputs, outputs = _run(lca, prob)
    cpu_inputs = tuple(t.cpu() for t in inputs)
    _check_rows(lca, prob, cpu_inputs, outputs, _one_head_per_group(prob))
    g = STATIC_KINDS.index(kind) % prob.Hkv
    G = prob.Hq // prob.Hkv
    segs = _sample_segments(prob)
    big = max(segs, key=lambda s: prob.segments[s].k_len)
    _check_key_tiles(prob, cpu_inputs, outputs, big, g, _tiles_to_check(prob, big, g * G), "largest segment")
    for s in segs:
        if s != big:
            nk = -(-prob.segments[s].k_len // 128)
            _check_key_tiles(prob, cpu_inputs, outputs, s, g, sorted({0, nk - 1}), "other document")
    _check_gradient_sums(prob, inputs, outputs)
    torch.cuda.synchronize()


def _check_document_key_tiles(prob, inputs, outputs, g, max_len=32768, budget=1 << 26):
    """Interior key tiles of one document (key group) no longer than
    `max_len`, element-wise against the oracle.  The oracle's cost is the
    attending rows times the document's keys per head, kept near `budget`:
    causal tiles move towards the document's end until at most
    budget / k_len rows attend them.  For a shard batch the document is one
    cut into several shards, and one tile lies just before its last shard, so
    rows of two or more shards (segments sharing the key range) add up in it;
    among such documents the cheapest is taken.  Otherwise the longest
    document within the limit is taken (the smallest one if none is)."""
    groups = {}
    for s, seg in enumerate(prob.segments):
        if seg.q_len > 0 and seg.k_len > 0:
            groups.setdefault(seg.k_off, []).append(s)

    def last(members):
        return max(members, key=lambda i: prob.segments[i].k_len)

    multi = [m for m in groups.values() if len(m) > 1 and prob.segments[last(m)].k_len <= max_len]
    if multi:
        members = min(multi, key=lambda m: prob.segments[last(m)].k_len * (prob.segments[last(m)].q_len + 256))
    else:
        fit = [m for m in groups.values() if prob.segments[last(m)].k_len <= max_len]
        members = (max(fit, key=lambda m: prob.segments[last(m)].k_len) if fit
                   else min(groups.values(), key=lambda m: prob.segments[last(m)].k_len))
    s = last(members)
    seg = prob.segments[s]
    nk = -(-seg.k_len // 128)
    max_rows = max(256, budget // seg.k_len)
    kts = set()
    for kt in (nk // 2, 2 * nk // 3):
        while kt < nk - 1 and seg.k_len - kt * 128 > max_rows:
            kt += 1
        kts.add(kt)
    if len(members) > 1:
        first_row = seg.k_len - seg.q_len  # the last shard's first query position in its document
        kts.add(max(0, first_row // 128 - 1))
    _check_key_tiles(prob, inputs, outputs, s, g, sorted(kts), f"document of {seg.k_len} keys, {len(members)} segments")


DENSE = [config3(S, heads, kind) for S in (8192, 49152) for heads in ("gqa", "mha") for kind in ("CAUSAL", "CAUSAL_DOC")]


@pytest.mark.parametrize("prob", DENSE, ids=[p.name for p in DENSE])
def test_dense_sweep_full_size(lca, prob):
    inputs, outputs = _run(lca, prob)
    _check_rows(lca, prob, inputs, outputs, _heads(prob))
    _check_last_key_tile(lca, prob, inputs, outputs, g=0)
    _check_last_key_tile(lca, prob, inputs, outputs, g=prob.Hkv - 1)
    _check_document_key_tiles(prob, inputs, outputs, g=prob.Hkv // 2)
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
    _check_document_key_tiles(prob, inputs, outputs, g=3)
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
