"""The per-CTA profile of the attention kernels (lca_set_cta_profile) counts
exactly the work the mask compiler planned: summed over CTAs, the forward
and dQ kernels ran every non-empty 128x128 tile of every query head once, as
FULL or PARTIAL per its class, and the dK/dV kernel every 64-row query step
(both halves of a FULL tile inside the segment; the halves of a PARTIAL tile
that are inside the segment and not flagged empty).  The counts are taken
from the tile-class test hook, which the mask-compiler tests pin to the
oracle.  Stamps are ordered and the grid is one CTA per SM at most."""
from __future__ import annotations

import numpy as np
import pytest

from gen import make_tensors
from tests import cases

pytestmark = pytest.mark.gpu

PROBS = [p for p in cases.gpu_small_all() if p.name in ("g_tiny_sliding_700", "g_tiny_causal_doc_docs", "g_small_bsu64")]


# Families whose forward items pair two query heads of one KV head (128 rows
# each) instead of taking 256 rows of one head, when G is even and the mask
# map is shared by all heads.
PAIRED = {"SLIDING", "CAUSAL_SLIDING", "GLOBAL_SLIDING", "DOC", "CAUSAL_DOC", "SHARED_QUESTION",
          "CAUSAL_BLOCKWISE", "PREFIX_LM_DOC", "BLOCK_CAUSAL_DOC"}


def _fwd_paired(prob):
    return prob.mask.kind in PAIRED and (prob.Hq // prob.Hkv) % 2 == 0


def _expected(lca, prob):
    call = lca.marshal(prob.Tq, prob.Tk, prob.Hq, prob.Hkv, prob.d, prob.segments, prob.mask, prob.scale)
    full = part = steps_full = steps_part = 0
    fwd_items = dq_items = 0
    for h in range(prob.Hq):
        for s, seg in enumerate(prob.segments):
            if seg.q_len == 0 or seg.k_len == 0:
                continue
            cls = lca.mask_tile_classes(call, h, s, seg.q_len, seg.k_len).cpu().numpy()
            c = cls & 3
            full += int((c == 1).sum())
            part += int((c == 2).sum())
            nq = cls.shape[0]
            for qt in range(nq):
                halves_in = 1 + (qt * 128 + 64 < seg.q_len)
                steps_full += halves_in * int((c[qt] == 1).sum())
                for b in cls[qt][c[qt] == 2]:
                    steps_part += int(not (b & 4)) + int(halves_in == 2 and not (b & 8))
            if not _fwd_paired(prob):
                fwd_items += -(-seg.q_len // 256)
            elif h % 2 == 0:  # one item per 128 rows of a head pair
                fwd_items += -(-seg.q_len // 128)
            dq_items += nq
    return dict(full=full, part=part, steps_full=steps_full, steps_part=steps_part, fwd_items=fwd_items,
                dq_items=dq_items)


@pytest.mark.parametrize("prob", PROBS, ids=[p.name for p in PROBS])
def test_cta_profile_counts_planned_work(lca, prob):
    import torch

    q, k, v, do = (t.cuda() for t in make_tensors(prob))
    exp = _expected(lca, prob)
    prof = lca.CtaProfile()
    prof.start()
    try:
        o, lse = lca.attn_fwd(q, k, v, prob.segments, prob.mask, prob.scale)
        torch.cuda.synchronize()
        rf = prof.records()["fwd"]
        lca.attn_bwd(do, q, k, v, o, lse, prob.segments, prob.mask, prob.scale)
        torch.cuda.synchronize()
        rb = prof.records()
    finally:
        prof.stop()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for name, r in (("fwd", rf), ("dkv", rb["dkv"]), ("dq", rb["dq"])):
        assert 1 <= r.shape[0] <= sms, name
        assert np.all(r[:, 1] >= r[:, 0]) and np.all(r[:, 0] > 0), name
        assert np.all(r[:, 6] < sms), name
    assert int(rf[:, 3].sum()) == exp["full"] and int(rf[:, 4].sum()) == exp["part"]
    assert int(rf[:, 2].sum()) == exp["fwd_items"]
    assert int(rb["dq"][:, 3].sum()) == exp["full"] and int(rb["dq"][:, 4].sum()) == exp["part"]
    assert int(rb["dq"][:, 2].sum()) == exp["dq_items"]
    assert int(rb["dkv"][:, 3].sum()) == exp["steps_full"] and int(rb["dkv"][:, 4].sum()) == exp["steps_part"]
    # profiling off: a later call writes no records
    prof.buf.zero_()
    lca.attn_fwd(q, k, v, prob.segments, prob.mask, prob.scale)
    torch.cuda.synchronize()
    assert int(prof.buf.abs().sum()) == 0
