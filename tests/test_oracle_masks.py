"""Oracle mask predicates vs the independent constructive masks, cell by
cell: tiny instances of every family, then every static family at the 8K
sweep's full size and parameters, and the block-sparse generators."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from gen import STATIC_KINDS, config2, config4
from tests import cases
from tests.brute_masks import brute_dense_mask

TINY = cases.tiny_all() + cases.tiny_all(S=37, d=4) + [
    cases.single(23, "SLIDING", window_left=2, window_right=5),
    cases.single(23, "CAUSAL_SLIDING", window_left=0),
    cases.single(23, "SHARED_QUESTION", part_bounds=[0, 7, 9, 16, 23]),
    cases.docs([1, 9, 2, 11], "BLOCK_CAUSAL_DOC", block=4),
    cases.docs([1, 9, 2, 11], "PREFIX_LM_DOC", prefix_len=5),
    cases.block_uniform(30, 8, Hq=3, heads_in_map=1),
]


@pytest.mark.parametrize("prob", TINY, ids=[f"{p.name}_{i}" for i, p in enumerate(TINY)])
def test_tiny_masks_cell_by_cell(prob):
    for h in range(prob.Hq):
        np.testing.assert_array_equal(oracle.dense_mask(prob, h), brute_dense_mask(prob, h))


@pytest.mark.parametrize("kind", STATIC_KINDS)
def test_static_masks_at_8k(kind):
    p = config2(kind, Hq=1, Hkv=1)
    np.testing.assert_array_equal(oracle.dense_mask(p, 0), brute_dense_mask(p, 0))


@pytest.mark.parametrize("variant", ["uniform64", "uniform128", "variable"])
def test_block_sparse_generators_small(variant):
    p = config4(2048, "gqa", variant)
    for h in (0, 37):
        np.testing.assert_array_equal(oracle.dense_mask(p, h), brute_dense_mask(p, h))
        counts = oracle.mask_row_counts(p, h)
        # half of the blocks of every block row are kept
        assert 0.3 < counts.sum() / (p.Tq * p.Tk) < 0.7


# ---------------------------------------------------------------- FlashMask form
FM_CASES = (cases.tiny_all(S=16)[:12] + cases.tiny_all(S=37)[:12]
            + [p for p in cases.edge_cases(d=8) if p.name in ("edge_q_gt_k", "edge_tile_plus1")])


@pytest.mark.parametrize("prob", FM_CASES, ids=[f"{p.name}_{i}" for i, p in enumerate(FM_CASES)])
def test_flashmask_form_equals_family(prob):
    """Each static family written in FlashMask's column form (test input)
    gives, through the oracle's column predicate, the family's own mask, and
    the brute-force column fill agrees cell by cell."""
    from tests.flashmask_inputs import as_flashmask

    fm = as_flashmask(prob)
    want = oracle.dense_mask(prob)
    assert np.array_equal(oracle.dense_mask(fm), want)
    assert np.array_equal(brute_dense_mask(fm), want)


def test_flashmask_worked_example():
    """Hand-set columns of one 4x4 segment: key 0 hides no row; key 1 hides
    row 0; key 2 hides rows 0-1 and 3; key 3 hides rows 1-2.  Rows read
    keys {0,3}, {0,1}, {0,1,2}, {0,1,3}."""
    from gen import MaskSpec, Problem, Segment

    cb = np.array([[0, 0, 0, 0], [0, 1, 0, 0], [0, 2, 3, 4], [1, 3, 0, 0]], dtype=np.int32)
    p = Problem("fm4", 4, 4, 1, 1, 8, [Segment(0, 4, 0, 4)], MaskSpec("FLASHMASK", col_bounds=cb), 1)
    want = np.array([[1, 0, 0, 1], [1, 1, 0, 0], [1, 1, 1, 0], [1, 1, 0, 1]], dtype=bool)
    assert np.array_equal(oracle.dense_mask(p), want)


def test_small_parity_cases_have_empty_tile_halves():
    """The small GPU parity cases include partial 128x128 tiles one of whose
    64-row halves attends nothing (the halves the backward's dK/dV pass
    skips), so that element-wise parity covers the skip."""
    found = {}
    for prob in cases.gpu_small_all():
        n = 0
        for s, seg in enumerate(prob.segments):
            if seg.q_len == 0 or seg.k_len == 0:
                continue
            M = oracle.segment_mask(prob.mask, s, seg, 0)
            for q0 in range(0, seg.q_len, 128):
                for k0 in range(0, seg.k_len, 128):
                    blk = M[q0:q0 + 128, k0:k0 + 128]
                    if blk.any() and not blk.all() and blk.shape[0] > 64:
                        n += int(not blk[:64].any()) + int(not blk[64:].any())
        found[prob.name] = n
    assert found["g_small_bsu64"] > 0
    assert found["g_small_bsv"] > 0
