"""Mask predicates, one per family — TEST INFRASTRUCTURE ONLY.

The LongCA-bench review ("Long-Context Attention Benchmark", section 三 技术架构,
掩码模式分类) names 12 static masks (FULL, CAUSAL, FULL/CAUSAL SLIDING WINDOW,
FULL/CAUSAL DOCUMENT, SHARED QUESTION, GLOBAL SLIDING, CAUSAL BLOCKWISE,
PREFIX LM CAUSAL, PREFIX LM DOCUMENT, BLOCK CAUSAL DOCUMENT) and 2 dynamic
block masks (uniform blocks such as 64x64; variable-size blocks), but defines
none of them.  The predicates below (one branch per family in segment_mask)
are the plainest readings of the family names and their parameters.

Positions are relative to a segment: query row i in [0, q_len), key j in
[0, k_len).  When q_len != k_len the causal diagonal is aligned bottom-right:
query i sits at key position ie = i + (k_len - q_len).  Documents are
segments, so the document families evaluate per segment.
"""
from __future__ import annotations

import numpy as np


def _block_keep_rows(spec, head: int, q_pos: np.ndarray, k_pos: np.ndarray) -> np.ndarray:
    """keep[h][qb(q)][kb(k)] for global token positions (block-sparse maps)."""
    hm = head if spec.heads_in_map > 1 else 0
    if spec.kind == "BLOCK_SPARSE_UNIFORM":
        qb = q_pos // spec.q_block
        kb = k_pos // spec.kv_block
        n_kb = int(k_pos.max()) // spec.kv_block + 1 if k_pos.size else 0
        n_kb = max(n_kb, int(spec.blk_col_idx.max()) + 1 if spec.blk_col_idx.size else 0)
    else:
        qb = np.searchsorted(spec.qb_bounds, q_pos, side="right") - 1
        kb = np.searchsorted(spec.kb_bounds, k_pos, side="right") - 1
        n_kb = len(spec.kb_bounds) - 1
    n_qb = (len(spec.blk_row_ptr) - 1) // spec.heads_in_map
    out = np.zeros((q_pos.size, k_pos.size), dtype=bool)
    for r, b in enumerate(qb):
        row = hm * n_qb + int(b)
        cols = spec.blk_col_idx[spec.blk_row_ptr[row]:spec.blk_row_ptr[row + 1]]
        keep = np.zeros(n_kb, dtype=bool)
        keep[cols] = True
        out[r] = keep[kb]
    return out


def segment_mask(spec, seg_index: int, seg, head: int = 0, rows=None) -> np.ndarray:
    """Boolean mask M[i, j] (True = attend) for rows `rows` (default all) of
    one segment and one query head."""
    q_len, k_len = seg.q_len, seg.k_len
    i = np.arange(q_len) if rows is None else np.asarray(rows)
    i = i[:, None]
    j = np.arange(k_len)[None, :]
    ie = i + (k_len - q_len)  # query position on the key axis
    kind = spec.kind
    if kind in ("FULL", "DOC"):
        m = np.ones((i.shape[0], k_len), dtype=bool)
    elif kind in ("CAUSAL", "CAUSAL_DOC"):
        m = j <= ie
    elif kind == "SLIDING":
        m = (j >= ie - spec.window_left) & (j <= ie + spec.window_right)
    elif kind == "CAUSAL_SLIDING":
        m = (j >= ie - spec.window_left) & (j <= ie)
    elif kind == "SHARED_QUESTION":
        # part(x): index of the part (0 = question, 1.. = answers) holding key position x
        b = np.asarray(spec.part_bounds)
        part_q = np.searchsorted(b, ie, side="right") - 1
        part_k = np.searchsorted(b, j, side="right") - 1
        m = (j <= ie) & ((part_k == 0) | (part_k == part_q))
    elif kind == "GLOBAL_SLIDING":
        g = spec.num_global
        m = (ie < g) | (j < g) | ((j >= ie - spec.window_left) & (j <= ie + spec.window_right))
    elif kind == "CAUSAL_BLOCKWISE":
        blk_q = ie // spec.block
        blk_k = j // spec.block
        last = (k_len - 1) // spec.block
        m = (j <= ie) & ((blk_k == blk_q) | (blk_q == last))
    elif kind == "PREFIX_LM_CAUSAL":
        m = (j < spec.prefix_len) | (j <= ie)
    elif kind == "PREFIX_LM_DOC":
        p = spec.seg_prefix[seg_index]
        m = (j < p) | (j <= ie)
    elif kind == "BLOCK_CAUSAL_DOC":
        m = (j // spec.block) <= (ie // spec.block)
    elif kind == "FLASHMASK":
        # column-wise form (FlashMask, named by the LongCA-bench review): key
        # column j of the segment (global position k_off + j) is hidden from
        # the segment rows [lts, lte) and [uts, ute)
        cb = np.asarray(spec.col_bounds)[seg.k_off + j[0]]
        lts, lte, uts, ute = (cb[:, t][None, :] for t in range(4))
        m = ~(((i >= lts) & (i < lte)) | ((i >= uts) & (i < ute)))
    elif kind in ("BLOCK_SPARSE_UNIFORM", "BLOCK_SPARSE_VARIABLE"):
        q_pos = seg.q_off + i[:, 0]
        k_pos = seg.k_off + j[0]
        m = _block_keep_rows(spec, head, q_pos, k_pos)
    else:
        raise ValueError(f"unknown mask kind {kind}")
    return np.broadcast_to(m, (i.shape[0], k_len)).copy()


def dense_mask(prob, head: int = 0) -> np.ndarray:
    """Global [Tq, Tk] boolean mask of one head (small problems only)."""
    M = np.zeros((prob.Tq, prob.Tk), dtype=bool)
    for s, seg in enumerate(prob.segments):
        M[seg.q_off:seg.q_off + seg.q_len, seg.k_off:seg.k_off + seg.k_len] |= segment_mask(prob.mask, s, seg, head)
    return M


def mask_row_counts(prob, head: int = 0) -> np.ndarray:
    """Number of attended keys per query row (global row index)."""
    out = np.zeros(prob.Tq, dtype=np.int64)
    for s, seg in enumerate(prob.segments):
        rows = np.arange(seg.q_len)
        step = max(1, (1 << 22) // max(1, seg.k_len))
        for r0 in range(0, seg.q_len, step):
            r = rows[r0:r0 + step]
            out[seg.q_off + r] += segment_mask(prob.mask, s, seg, head, r).sum(axis=1)
    return out
