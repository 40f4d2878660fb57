"""Small problem builders shared by the oracle pins and the GPU parity tests.

Every mask family gets a tiny instance with parameters scaled down so the
structure (windows, parts, prefixes, blocks, documents) still shows inside a
few tiles, with ragged tails.
"""
from __future__ import annotations

import numpy as np

from gen import MaskSpec, Problem, Segment, docs_to_segments, uniform_block_map, variable_block_map, _rng


def single(S, kind, Hq=2, Hkv=1, d=8, seed=11, **kw):
    return Problem(f"tiny_{kind.lower()}_{S}", S, S, Hq, Hkv, d, [Segment(0, S, 0, S)], MaskSpec(kind, **kw), seed)


def docs(lengths, kind, Hq=2, Hkv=1, d=8, seed=12, **kw):
    segs = docs_to_segments(lengths)
    T = sum(lengths)
    spec = MaskSpec(kind, **kw)
    if kind == "PREFIX_LM_DOC" and spec.seg_prefix is None:
        spec.seg_prefix = [min(spec.prefix_len, n) for n in lengths]
    return Problem(f"tiny_{kind.lower()}_docs", T, T, Hq, Hkv, d, segs, spec, seed)


def block_uniform(S, b, Hq=2, Hkv=1, d=8, seed=13, heads_in_map=None):
    n = -(-S // b)
    hm = Hq if heads_in_map is None else heads_in_map
    rp, ci = uniform_block_map(n, n, hm, _rng(seed))
    spec = MaskSpec("BLOCK_SPARSE_UNIFORM", q_block=b, kv_block=b, heads_in_map=hm, blk_row_ptr=rp, blk_col_idx=ci)
    return Problem(f"tiny_bsu_{S}_{b}", S, S, Hq, Hkv, d, [Segment(0, S, 0, S)], spec, seed)


def block_variable(qb_bounds, kb_bounds, Hq=2, Hkv=1, d=8, seed=14):
    qb = np.asarray(qb_bounds, dtype=np.int32)
    kb = np.asarray(kb_bounds, dtype=np.int32)
    rp, ci = variable_block_map(len(qb) - 1, len(kb) - 1, Hq, _rng(seed))
    spec = MaskSpec("BLOCK_SPARSE_VARIABLE", qb_bounds=qb, kb_bounds=kb, heads_in_map=Hq, blk_row_ptr=rp, blk_col_idx=ci)
    S = int(qb[-1])
    return Problem(f"tiny_bsv_{S}", S, int(kb[-1]), Hq, Hkv, d, [Segment(0, S, 0, int(kb[-1]))], spec, seed)


def tiny_all(S=16, d=8, Hq=2, Hkv=1):
    """One tiny instance per family (S around 16)."""
    return [
        single(S, "FULL", Hq, Hkv, d),
        single(S, "CAUSAL", Hq, Hkv, d),
        single(S, "SLIDING", Hq, Hkv, d, window_left=3, window_right=3),
        single(S, "CAUSAL_SLIDING", Hq, Hkv, d, window_left=5),
        docs([5, 7, 4], "DOC", Hq, Hkv, d),
        docs([5, 7, 4], "CAUSAL_DOC", Hq, Hkv, d),
        single(S, "SHARED_QUESTION", Hq, Hkv, d, part_bounds=[0, 4, 8, 12, S]),
        single(S, "GLOBAL_SLIDING", Hq, Hkv, d, num_global=2, window_left=3, window_right=3),
        single(S, "CAUSAL_BLOCKWISE", Hq, Hkv, d, block=5),
        single(S, "PREFIX_LM_CAUSAL", Hq, Hkv, d, prefix_len=6),
        docs([5, 7, 4], "PREFIX_LM_DOC", Hq, Hkv, d, prefix_len=3),
        docs([5, 7, 4], "BLOCK_CAUSAL_DOC", Hq, Hkv, d, block=3),
        block_uniform(S, 4, Hq, Hkv, d),
        block_variable([0, 3, 7, 12, S], [0, 5, 6, 11, S], Hq, Hkv, d),
    ]


def shard_problem(doc_lengths, shards_per_doc, Hq=2, Hkv=1, d=8, seed=15, shuffle_seed=3):
    """Documents cut at given shard lengths; shards packed in a shuffled order.
    Returns the shard problem and the CAUSAL_DOC problem on the same documents."""
    shards = []
    off = 0
    for n, cuts in zip(doc_lengths, shards_per_doc):
        assert sum(cuts) == n
        a = 0
        for L in cuts:
            shards.append((off, a, L))
            a += L
        off += n
    order = np.random.Generator(np.random.PCG64(shuffle_seed)).permutation(len(shards))
    segs, src, qpos = [], [], 0
    for idx in order:
        doc_start, a, L = shards[idx]
        segs.append(Segment(qpos, L, doc_start, a + L))
        src.append(doc_start + a)
        qpos += L
    T = sum(doc_lengths)
    shard = Problem("tiny_shards", T, T, Hq, Hkv, d, segs, MaskSpec("CAUSAL"), seed)
    shard.extra["shard_src"] = np.asarray(src)
    docp = Problem("tiny_shard_docs", T, T, Hq, Hkv, d, docs_to_segments(doc_lengths), MaskSpec("CAUSAL_DOC"), seed)
    return shard, docp


def shard_row_map(prob):
    """packed query row -> row in document order, for a shard problem."""
    rows = np.empty(prob.Tq, dtype=np.int64)
    for seg, src in zip(prob.segments, prob.extra["shard_src"]):
        rows[seg.q_off:seg.q_off + seg.q_len] = src + np.arange(seg.q_len)
    return rows
