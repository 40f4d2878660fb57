"""FlashMask descriptors for the tests: a static mask family re-expressed in
the column-wise form the LongCA-bench review names ("Long-Context Attention
Benchmark", 掩码模式分类: FlashMask covers all the static masks), used as input
to both the oracle and the CUDA path.  Test input only: the conversion is
checked against the oracle's family predicates and a brute-force column fill
(tests/test_oracle_masks.py)."""
from __future__ import annotations

import numpy as np

from gen import MaskSpec, Problem


def flashmask_columns(spec: MaskSpec, segments, Tk: int) -> np.ndarray:
    """A static mask family re-expressed in FlashMask's column-wise form:
    int32 [Tk, 4] = {lts, lte, uts, ute} per global key position, the segment
    rows that key masks being [lts, lte) U [uts, ute).  Segments must own
    disjoint key ranges.  With shift = k_len - q_len, a key column j of a
    segment is attended by row i when j <= i + shift (causal), etc.; the row
    ranges below are those conditions solved for i."""
    out = np.zeros((Tk, 4), dtype=np.int64)
    owner = np.full(Tk, -1)
    for s, seg in enumerate(segments):
        ks = slice(seg.k_off, seg.k_off + seg.k_len)
        assert (owner[ks] < 0).all(), "FlashMask columns need disjoint key ranges"
        owner[ks] = s
        Lq, Lk = seg.q_len, seg.k_len
        sh = Lk - Lq
        j = np.arange(Lk)
        z = np.zeros(Lk, dtype=np.int64)
        lts, lte, uts, ute = z.copy(), z.copy(), z.copy(), z.copy()
        kind = spec.kind
        if kind in ("FULL", "DOC"):
            pass
        elif kind in ("CAUSAL", "CAUSAL_DOC"):
            lte = j - sh
        elif kind == "SLIDING":
            lte = j - spec.window_right - sh
            uts, ute = j + spec.window_left - sh + 1, np.full(Lk, Lq)
        elif kind == "CAUSAL_SLIDING":
            lte = j - sh
            uts, ute = j + spec.window_left - sh + 1, np.full(Lk, Lq)
        elif kind == "GLOBAL_SLIDING":
            g = spec.num_global
            far = j >= g  # the global keys are attended by every row
            lts = np.where(far, g - sh, 0)
            lte = np.where(far, j - spec.window_right - sh, 0)
            uts = np.where(far, j + spec.window_left - sh + 1, 0)
            ute = np.where(far, Lq, 0)
        elif kind == "CAUSAL_BLOCKWISE":
            b = spec.block
            last = (Lk - 1) // b
            blk = j // b
            lte = j - sh
            inner = blk != last  # a block's keys are also hidden from later blocks but the last
            uts = np.where(inner, (blk + 1) * b - sh, 0)
            ute = np.where(inner, last * b - sh, 0)
        elif kind in ("PREFIX_LM_CAUSAL", "PREFIX_LM_DOC"):
            p = spec.prefix_len if kind == "PREFIX_LM_CAUSAL" else spec.seg_prefix[s]
            lte = np.where(j < p, 0, j - sh)
        elif kind == "BLOCK_CAUSAL_DOC":
            lte = (j // spec.block) * spec.block - sh
        elif kind == "SHARED_QUESTION":
            bnd = np.asarray(spec.part_bounds)
            part = np.searchsorted(bnd, j, side="right") - 1
            lte = j - sh
            ans = part > 0  # an answer's keys are hidden from the later answers
            end = bnd[np.minimum(part + 1, len(bnd) - 1)]
            uts = np.where(ans, end - sh, 0)
            ute = np.where(ans, Lq, 0)
        else:
            raise ValueError(f"no FlashMask form for {kind}")
        cols = np.stack([lts, lte, uts, ute], axis=1)
        out[ks] = np.clip(cols, 0, Lq)
    return out.astype(np.int32)


def as_flashmask(prob: Problem) -> Problem:
    """The same problem with its static mask given in FlashMask form."""
    spec = MaskSpec("FLASHMASK", col_bounds=flashmask_columns(prob.mask, prob.segments, prob.Tk))
    return Problem(prob.name + "_fm", prob.Tq, prob.Tk, prob.Hq, prob.Hkv, prob.d, prob.segments, spec, prob.seed,
                   prob.scale, dict(prob.extra))

