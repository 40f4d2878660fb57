"""GPU mask machinery vs the oracle: the device predicate (materialized) must
match the oracle's dense boolean mask bit-exactly in every cell, head and
segment; the mask compiler's tile classes must be exact (EMPTY = no attended
cell, FULL = every cell attended and inside the segment); the nnz counts
must match the oracle's."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from gen import STATIC_KINDS, config2, config4
from tests import cases

pytestmark = pytest.mark.gpu

# the tiny block-sparse instances use 4-wide blocks, below the library's 32-key minimum
SMALL = [p for p in cases.tiny_all(S=40, d=128) if not p.mask.kind.startswith("BLOCK_SPARSE")] + \
    cases.gpu_small_all() + cases.edge_cases()


def _call(lib, prob):
    return lib.marshal(prob.Tq, prob.Tk, prob.Hq, prob.Hkv, prob.d, prob.segments, prob.mask, prob.scale)


def _heads(prob):
    return sorted({0, prob.Hq - 1, prob.Hq // 2})


def _check_masks(lib, prob, heads):
    call = _call(lib, prob)
    for h in heads:
        for s, seg in enumerate(prob.segments):
            if seg.q_len == 0 or seg.k_len == 0:
                continue
            got = lib.mask_materialize(call, h, s, seg.q_len, seg.k_len).cpu().numpy().astype(bool)
            want = oracle.segment_mask(prob.mask, s, seg, h)
            assert np.array_equal(got, want), f"{prob.name} head {h} seg {s}: {(got != want).sum()} cells differ"


def _want_class(blk, inside):
    """Class byte of one 128x128 tile of the oracle mask: 0 empty, 1 full,
    2 partial, plus 4 / 8 on a partial tile whose first / second 64 query rows
    attend nothing."""
    if not blk.any():
        return 0
    if blk.all() and inside:
        return 1
    return 2 | (0 if blk[:64].any() else 4) | (0 if blk[64:].any() else 8)


def _check_classes(lib, prob, heads):
    call = _call(lib, prob)
    for h in heads:
        for s, seg in enumerate(prob.segments):
            if seg.q_len == 0 or seg.k_len == 0:
                continue
            cls = lib.mask_tile_classes(call, h, s, seg.q_len, seg.k_len).cpu().numpy()
            M = oracle.segment_mask(prob.mask, s, seg, h)
            for qt in range(cls.shape[0]):
                for kt in range(cls.shape[1]):
                    blk = M[qt * 128:(qt + 1) * 128, kt * 128:(kt + 1) * 128]
                    inside = (qt + 1) * 128 <= seg.q_len and (kt + 1) * 128 <= seg.k_len
                    want = _want_class(blk, inside)
                    assert cls[qt, kt] == want, f"{prob.name} h{h} s{s} tile ({qt},{kt}): {cls[qt, kt]} != {want}"


@pytest.mark.parametrize("prob", SMALL, ids=[p.name for p in SMALL])
def test_small_masks_bit_exact(lca, prob):
    _check_masks(lca, prob, range(prob.Hq))
    _check_classes(lca, prob, _heads(prob))


@pytest.mark.parametrize("prob", SMALL, ids=[p.name for p in SMALL])
def test_small_nnz(lca, prob):
    got = lca.mask_nnz(_call(lca, prob)).cpu().numpy()
    want = np.array([oracle.mask_row_counts(prob, h).sum() for h in range(prob.Hq)])
    assert np.array_equal(got, want)


@pytest.mark.parametrize("kind", STATIC_KINDS)
def test_static_masks_8k_bit_exact(lca, kind):
    prob = config2(kind)
    _check_masks(lca, prob, [0, prob.Hq - 1])
    _check_classes(lca, prob, [0])
    got = lca.mask_nnz(_call(lca, prob)).cpu().numpy()
    assert np.all(got == oracle.mask_row_counts(prob, 0).sum())


@pytest.mark.parametrize("variant", ["uniform64", "uniform128", "variable"])
def test_block_sparse_masks_bit_exact(lca, variant):
    prob = config4(32768, "gqa", variant)
    # cell-by-cell on a 8K corner is what fits in host memory; tile classes and
    # nnz are checked over the whole 32K map for sampled heads
    call = _call(lca, prob)
    heads = [0, 33, 63]
    for h in heads:
        got_cls = lca.mask_tile_classes(call, h, 0, prob.Tq, prob.Tk).cpu().numpy()
        rows = np.arange(0, 8192)
        M = oracle.segment_mask(prob.mask, 0, prob.segments[0], h, rows)
        full = lca.mask_materialize(call, h, 0, prob.Tq, prob.Tk)[:8192].cpu().numpy().astype(bool)
        assert np.array_equal(full, M)
        for qt in range(0, 64, 7):
            for kt in range(0, 256, 5):
                blk = M[qt * 128:(qt + 1) * 128, kt * 128:(kt + 1) * 128]
                assert got_cls[qt, kt] == _want_class(blk, True)
    nnz = lca.mask_nnz(call).cpu().numpy()
    for h in heads:
        assert nnz[h] == oracle.mask_row_counts(prob, h).sum()
