"""Constructive mask builders, written independently of the oracle's
predicates: each family is filled from its description (bands, triangles,
blocks, document squares, question/answer parts) with numpy tril/triu or
explicit loops, never by evaluating a per-cell formula shared with
oracle/masks.py.  Small sizes only."""
from __future__ import annotations

import numpy as np


def _square_causal(n):
    return np.tril(np.ones((n, n), dtype=bool))


def _segment_block(spec, s_index, seg, head):
    q, k = seg.q_len, seg.k_len
    kind = spec.kind
    # Build on a square k x k key canvas, then keep the last q rows
    # (bottom-right alignment of queries onto key positions).
    n = k
    if kind in ("FULL", "DOC"):
        C = np.ones((n, n), dtype=bool)
    elif kind in ("CAUSAL", "CAUSAL_DOC"):
        C = _square_causal(n)
    elif kind == "SLIDING":
        C = np.tril(np.ones((n, n), dtype=bool), spec.window_right) & np.triu(np.ones((n, n), dtype=bool),
                                                                               -spec.window_left)
    elif kind == "CAUSAL_SLIDING":
        C = _square_causal(n) & np.triu(np.ones((n, n), dtype=bool), -spec.window_left)
    elif kind == "SHARED_QUESTION":
        C = np.zeros((n, n), dtype=bool)
        b = list(spec.part_bounds)
        b = [min(x, n) for x in b]
        lq = b[1]
        C[:lq, :lq] = _square_causal(lq)  # the question, causal
        for a0, a1 in zip(b[1:-1], b[2:]):
            if a1 <= a0:
                continue
            C[a0:a1, :lq] = True  # every answer reads the whole question
            C[a0:a1, a0:a1] = _square_causal(a1 - a0)  # and itself causally
    elif kind == "GLOBAL_SLIDING":
        g = spec.num_global
        C = np.tril(np.ones((n, n), dtype=bool), spec.window_right) & np.triu(np.ones((n, n), dtype=bool),
                                                                               -spec.window_left)
        C[:g, :] = True
        C[:, :g] = True
    elif kind == "CAUSAL_BLOCKWISE":
        b = spec.block
        C = np.zeros((n, n), dtype=bool)
        starts = list(range(0, n, b))
        for s0 in starts[:-1]:
            e0 = min(n, s0 + b)
            C[s0:e0, s0:e0] = _square_causal(e0 - s0)
        last = starts[-1]
        C[last:, :] = _square_causal(n)[last:, :]
    elif kind == "PREFIX_LM_CAUSAL":
        C = _square_causal(n)
        C[:, :min(spec.prefix_len, n)] = True
    elif kind == "PREFIX_LM_DOC":
        C = _square_causal(n)
        C[:, :min(spec.seg_prefix[s_index], n)] = True
    elif kind == "BLOCK_CAUSAL_DOC":
        b = spec.block
        C = np.zeros((n, n), dtype=bool)
        for r0 in range(0, n, b):
            for c0 in range(0, r0 + 1, b):
                C[r0:r0 + b, c0:c0 + b] = True
    elif kind in ("BLOCK_SPARSE_UNIFORM", "BLOCK_SPARSE_VARIABLE"):
        return _block_sparse_segment(spec, seg, head)
    elif kind == "FLASHMASK":
        out = np.ones((q, k), dtype=bool)
        for jj in range(k):
            lts, lte, uts, ute = (int(x) for x in spec.col_bounds[seg.k_off + jj])
            for r in range(q):
                if lts <= r < lte or uts <= r < ute:
                    out[r, jj] = False
        return out
    else:
        raise ValueError(kind)
    if q <= k:
        return C[k - q:, :]
    out = np.zeros((q, k), dtype=bool)  # more queries than keys: first rows see nothing of C
    out[q - k:] = C
    if kind in ("FULL", "DOC"):
        out[:] = True
    return out


def _block_sparse_segment(spec, seg, head):
    hm = head if spec.heads_in_map > 1 else 0
    if spec.kind == "BLOCK_SPARSE_UNIFORM":
        Tq_end = seg.q_off + seg.q_len
        Tk_end = seg.k_off + seg.k_len
        qb = list(range(0, Tq_end + spec.q_block, spec.q_block))
        kb = list(range(0, Tk_end + spec.kv_block, spec.kv_block))
    else:
        qb = list(spec.qb_bounds)
        kb = list(spec.kb_bounds)
    n_qb = (len(spec.blk_row_ptr) - 1) // spec.heads_in_map
    G = np.zeros((max(qb[-1], seg.q_off + seg.q_len), max(kb[-1], seg.k_off + seg.k_len)), dtype=bool)
    for r in range(n_qb):
        row = hm * n_qb + r
        for c in spec.blk_col_idx[spec.blk_row_ptr[row]:spec.blk_row_ptr[row + 1]]:
            G[qb[r]:qb[r + 1], kb[c]:kb[c + 1]] = True
    return G[seg.q_off:seg.q_off + seg.q_len, seg.k_off:seg.k_off + seg.k_len]


def brute_dense_mask(prob, head=0):
    M = np.zeros((prob.Tq, prob.Tk), dtype=bool)
    for s, seg in enumerate(prob.segments):
        M[seg.q_off:seg.q_off + seg.q_len, seg.k_off:seg.k_off + seg.k_len] |= _segment_block(prob.mask, s, seg, head)
    return M
