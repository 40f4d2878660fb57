"""FlashMask column-wise descriptor (LCA_MASK_FLASHMASK) on the GPU: every
static family written in column form must give, through the device
predicate, the oracle's mask bit-exactly, exact tile classes and nnz, and
attention outputs within the parity bar -- and, since the mask and hence the
tile classes are the same, the same outputs as the family's own descriptor.
Covers the 12 static families at 700 tokens (several tiles, ragged tails,
documents), more queries than keys, and the 8K sweep's CAUSAL and SHARED
QUESTION at full size."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from gen import config2, make_tensors
from tests import cases
from tests.flashmask_inputs import as_flashmask
from tests.gpu_util import check_bwd, check_fwd, run_bwd, run_fwd, to_np
from tests.test_masks_gpu import _call, _check_classes, _check_masks

pytestmark = pytest.mark.gpu

STATIC_SMALL = cases.gpu_small_all()[:12] + [p for p in cases.edge_cases() if p.name == "edge_q_gt_k"]


@pytest.mark.parametrize("prob", STATIC_SMALL, ids=[p.name for p in STATIC_SMALL])
def test_flashmask_masks_bit_exact(lca, prob):
    fm = as_flashmask(prob)
    _check_masks(lca, fm, [0])
    _check_classes(lca, fm, [0])
    got = lca.mask_nnz(_call(lca, fm)).cpu().numpy()
    assert np.all(got == oracle.mask_row_counts(prob, 0).sum())


@pytest.mark.parametrize("prob", STATIC_SMALL, ids=[p.name for p in STATIC_SMALL])
def test_flashmask_attention_parity_and_same_as_family(lca, prob):
    fm = as_flashmask(prob)
    q, k, v, do = make_tensors(prob)
    o, lse = run_fwd(lca, fm, q, k, v)
    O, L = oracle.attention_forward(prob, q, k, v)
    check_fwd(o, lse, O, L, what=fm.name)
    o2, lse2 = run_fwd(lca, prob, q, k, v)
    assert np.array_equal(to_np(o), to_np(o2)) and np.array_equal(to_np(lse), to_np(lse2))
    grads = run_bwd(lca, fm, q, k, v, do, o, lse)
    check_bwd(grads, oracle.attention_backward(prob, q, k, v, do), what=fm.name)
    grads2 = run_bwd(lca, prob, q, k, v, do, o2, lse2)
    for a, b in zip(grads, grads2):
        assert np.array_equal(to_np(a), to_np(b))


@pytest.mark.parametrize("kind", ["CAUSAL", "SHARED_QUESTION", "SLIDING", "GLOBAL_SLIDING", "CAUSAL_DOC"])
def test_flashmask_8k_full_size(lca, kind):
    """Full-size masks bit-exact on the first and last heads' segment, and the
    outputs equal to the family descriptor's.  The windowed and document
    families run the forward with paired query heads (two heads of one KV
    head per item) and the column descriptor with one head per item, so the
    equality also checks the pairing."""
    prob = config2(kind)
    fm = as_flashmask(prob)
    _check_masks(lca, fm, [0])
    q, k, v, do = (t.cuda() for t in make_tensors(prob, device="cuda"))
    o, lse = lca.attn_fwd(q, k, v, fm.segments, fm.mask)
    o2, lse2 = lca.attn_fwd(q, k, v, prob.segments, prob.mask)
    assert np.array_equal(to_np(o), to_np(o2)) and np.array_equal(to_np(lse), to_np(lse2))
