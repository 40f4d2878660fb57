"""lca_attn_merge: forward calls over disjoint key chunks, merged, against the
fp64 oracle (forward over all keys, and the oracle's own merge of the same
pieces), with the forward tolerances.  Covers FULL split into key chunks, a
causal mask assembled ring-style (FULL below the diagonal + CAUSAL on it),
per-head block-sparse maps split by key range, rows no part attends, one part,
and the output written over part 0."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from gen import MaskSpec, Problem, Segment, make_tensors
from tests import cases
from tests.gpu_util import check_fwd, to_np

pytestmark = pytest.mark.gpu

T, HQ, HKV, D = 700, 8, 2, 128


def _fwd(lca, q, k, v, segs, spec):
    import torch

    o, lse = lca.attn_fwd(q, k, v, segs, spec)
    torch.cuda.synchronize()
    return o, lse


def _inputs(seed=61):
    prob = Problem("merge", T, T, HQ, HKV, D, [Segment(0, T, 0, T)], MaskSpec("FULL"), seed)
    q, k, v, _ = (t.cuda() if t is not None else None for t in make_tensors(prob))
    return prob, q, k, v


@pytest.mark.parametrize("cuts", [[0, 700], [0, 300, 700], [0, 129, 256, 511, 700]])
def test_full_split_into_key_chunks(lca, cuts):
    prob, q, k, v = _inputs()
    parts = [_fwd(lca, q, k, v, [Segment(0, T, a, b - a)], MaskSpec("FULL")) for a, b in zip(cuts[:-1], cuts[1:])]
    o, lse = lca.attn_merge([p[0] for p in parts], [p[1] for p in parts])
    O, L = oracle.attention_forward(prob, q, k, v)
    check_fwd(o, lse, O, L, what=f"FULL merged from {len(parts)} chunks")
    # the oracle's merge of the GPU pieces agrees with the GPU merge
    Om, Lm = oracle.merge_partials([to_np(p[0]) for p in parts], [to_np(p[1]) for p in parts])
    check_fwd(o, lse, Om, Lm, what="oracle merge of the same pieces")


def test_causal_ring_decomposition(lca):
    """Causal over three query/key chunks: chunk i attends chunks j < i fully
    and its own chunk causally (equal lengths, so the alignment is the
    diagonal); chunk 0 has no below-diagonal part (its rows come back with
    LSE = -inf from that call)."""
    bounds = [0, 233, 466, 700]
    prob, q, k, v = _inputs(62)
    full_segs = [Segment(a, b - a, 0, a) for a, b in zip(bounds[1:-1], bounds[2:])]
    diag_segs = [Segment(a, b - a, a, b - a) for a, b in zip(bounds[:-1], bounds[1:])]
    below = _fwd(lca, q, k, v, full_segs, MaskSpec("FULL"))
    diag = _fwd(lca, q, k, v, diag_segs, MaskSpec("CAUSAL"))
    assert bool(np.isneginf(to_np(below[1])[:, :233]).all())
    o, lse = lca.attn_merge([below[0], diag[0]], [below[1], diag[1]])
    ref = Problem("causal", T, T, HQ, HKV, D, [Segment(0, T, 0, T)], MaskSpec("CAUSAL"), 62)
    O, L = oracle.attention_forward(ref, q, k, v)
    check_fwd(o, lse, O, L, what="causal from ring pieces")
    o1, l1 = _fwd(lca, q, k, v, [Segment(0, T, 0, T)], MaskSpec("CAUSAL"))
    np.testing.assert_allclose(to_np(o), to_np(o1), atol=1e-2)


def test_block_sparse_split_by_key_range(lca):
    """Per-head uniform 64-block map: block indices are global positions, so
    the same map restricted to two key ranges gives disjoint pieces."""
    bs = cases.block_uniform(640, 64, Hq=HQ, Hkv=HKV, d=D, seed=63)
    q, k, v = (t.cuda() for t in make_tensors(bs)[:3])
    pieces = [_fwd(lca, q, k, v, [Segment(0, 640, a, b - a)], bs.mask) for a, b in ((0, 256), (256, 640))]
    o, lse = lca.attn_merge([p[0] for p in pieces], [p[1] for p in pieces])
    O, L = oracle.attention_forward(bs, q, k, v)
    check_fwd(o, lse, O, L, what="block-sparse merged")


def test_rows_no_part_attends_and_in_place(lca):
    """Queries outside every segment: O = 0 and LSE = -inf in each part and in
    the merge.  The merge written over part 0's tensors equals the merge into
    fresh ones."""
    import torch

    prob, q, k, v = _inputs(64)
    segs_a = [Segment(100, 300, 0, 350)]
    segs_b = [Segment(100, 300, 350, 350), Segment(450, 150, 350, 350)]
    a = _fwd(lca, q, k, v, segs_a, MaskSpec("FULL"))
    b = _fwd(lca, q, k, v, segs_b, MaskSpec("FULL"))
    o, lse = lca.attn_merge([a[0], b[0]], [a[1], b[1]])
    L = to_np(lse)
    assert np.isneginf(L[:, :100]).all() and np.isneginf(L[:, 600:]).all()
    assert float(o[:100].abs().max()) == 0.0 and float(o[600:].abs().max()) == 0.0
    Om, Lm = oracle.merge_partials([to_np(a[0]), to_np(b[0])], [to_np(a[1]), to_np(b[1])])
    check_fwd(o, lse, Om, Lm, what="merge with empty rows")
    o_in, l_in = a[0].clone(), a[1].clone()
    lca.attn_merge([o_in, b[0]], [l_in, b[1]], out=o_in, lse=l_in)
    torch.cuda.synchronize()
    assert torch.equal(o_in, o) and torch.equal(l_in, lse)


def test_single_part_is_identity(lca):
    import torch

    prob, q, k, v = _inputs(65)
    o1, l1 = _fwd(lca, q, k, v, [Segment(0, T, 0, T)], MaskSpec("CAUSAL"))
    o, lse = lca.attn_merge([o1], [l1])
    torch.cuda.synchronize()
    np.testing.assert_allclose(to_np(o), to_np(o1), atol=4e-3)
    np.testing.assert_allclose(to_np(lse), to_np(l1), atol=1e-5)
