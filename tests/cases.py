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


def gpu_small_all(Hq=8, Hkv=2, S=700, seed=21):
    """One instance per family with head dim 128, several 128-tiles and ragged
    tails, for element-wise GPU parity against the full oracle."""
    d = 128
    docs_l = [300, 257, 143]
    r = np.random.Generator(np.random.PCG64(seed))
    n = -(-S // 64)
    rp64, ci64 = uniform_block_map(n, n, Hq, r)
    n2 = -(-S // 128)
    rp128, ci128 = uniform_block_map(n2, n2, Hq, r)
    from gen import variable_block_bounds

    qb = variable_block_bounds(S, 32, 256, r)
    kb = variable_block_bounds(S, 32, 256, r)
    rpv, civ = variable_block_map(len(qb) - 1, len(kb) - 1, Hq, r)
    probs = [
        single(S, "FULL", Hq, Hkv, d, seed),
        single(S, "CAUSAL", Hq, Hkv, d, seed),
        single(S, "SLIDING", Hq, Hkv, d, seed, window_left=100, window_right=100),
        single(S, "CAUSAL_SLIDING", Hq, Hkv, d, seed, window_left=150),
        docs(docs_l, "DOC", Hq, Hkv, d, seed),
        docs(docs_l, "CAUSAL_DOC", Hq, Hkv, d, seed),
        single(S, "SHARED_QUESTION", Hq, Hkv, d, seed, part_bounds=[0, 100, 300, 500, S]),
        single(S, "GLOBAL_SLIDING", Hq, Hkv, d, seed, num_global=16, window_left=100, window_right=100),
        single(S, "CAUSAL_BLOCKWISE", Hq, Hkv, d, seed, block=200),
        single(S, "PREFIX_LM_CAUSAL", Hq, Hkv, d, seed, prefix_len=250),
        docs(docs_l, "PREFIX_LM_DOC", Hq, Hkv, d, seed, prefix_len=100),
        docs(docs_l, "BLOCK_CAUSAL_DOC", Hq, Hkv, d, seed, block=64),
        Problem("small_bsu64", S, S, Hq, Hkv, d, [Segment(0, S, 0, S)],
                MaskSpec("BLOCK_SPARSE_UNIFORM", q_block=64, kv_block=64, heads_in_map=Hq, blk_row_ptr=rp64,
                         blk_col_idx=ci64), seed),
        Problem("small_bsu128", S, S, Hq, Hkv, d, [Segment(0, S, 0, S)],
                MaskSpec("BLOCK_SPARSE_UNIFORM", q_block=128, kv_block=128, heads_in_map=Hq, blk_row_ptr=rp128,
                         blk_col_idx=ci128), seed),
        Problem("small_bsv", S, S, Hq, Hkv, d, [Segment(0, S, 0, S)],
                MaskSpec("BLOCK_SPARSE_VARIABLE", qb_bounds=qb, kb_bounds=kb, heads_in_map=Hq, blk_row_ptr=rpv,
                         blk_col_idx=civ), seed),
    ]
    for p in probs:
        p.name = "g_" + p.name
    return probs


def edge_cases(d=128):
    """Degenerate and boundary layouts."""
    out = []
    out.append(Problem("edge_single_token", 1, 1, 2, 1, d, [Segment(0, 1, 0, 1)], MaskSpec("CAUSAL"), 31))
    out.append(Problem("edge_tiny", 5, 5, 2, 2, d, [Segment(0, 5, 0, 5)], MaskSpec("CAUSAL"), 32))
    # more queries than keys: the first rows of the segment see nothing
    out.append(Problem("edge_q_gt_k", 300, 140, 4, 2, d, [Segment(0, 300, 0, 140)], MaskSpec("CAUSAL"), 33))
    # rows and keys outside every segment, a segment with no keys, a segment with no queries
    out.append(Problem("edge_gaps", 600, 600, 4, 1, d,
                       [Segment(10, 200, 0, 200), Segment(300, 50, 250, 0), Segment(360, 0, 250, 90),
                        Segment(400, 170, 400, 170)], MaskSpec("CAUSAL"), 34))
    # exact tile multiples and one past
    out.append(Problem("edge_tile_exact", 512, 512, 2, 1, d, [Segment(0, 256, 0, 256), Segment(256, 256, 256, 256)],
                       MaskSpec("FULL"), 35))
    out.append(Problem("edge_tile_plus1", 257, 257, 2, 1, d, [Segment(0, 257, 0, 257)], MaskSpec("CAUSAL"), 36))
    # MHA
    out.append(Problem("edge_mha", 333, 333, 3, 3, d, [Segment(0, 333, 0, 333)], MaskSpec("CAUSAL"), 37))
    # a block-sparse row that keeps nothing (fully masked rows inside a partial map)
    rp = np.array([0, 1, 1, 3], dtype=np.int32)
    ci = np.array([0, 1, 2], dtype=np.int32)
    out.append(Problem("edge_bs_empty_row", 300, 300, 2, 1, d, [Segment(0, 300, 0, 300)],
                       MaskSpec("BLOCK_SPARSE_UNIFORM", q_block=100, kv_block=100, heads_in_map=1, blk_row_ptr=rp,
                                blk_col_idx=ci), 38))
    return out
