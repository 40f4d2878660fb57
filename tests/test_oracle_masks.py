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
