"""Core-attention disaggregation on the GPU kernels: a 64K-token set of
heavy-tailed documents is planned onto 4 attention servers (lca_cad_plan);
each server's shards run as one packed CAUSAL batch through lca_attn_fwd and
lca_attn_bwd over the documents' keys read in place.  Scattered back (O, LSE,
dQ) and summed over servers (dK, dV: shards of one document on different
servers each add their share), the results match one causal-document call
over all documents."""
from __future__ import annotations

import numpy as np
import pytest

import long_context_masked_attention_gb300 as lca
from gen import MaskSpec, Problem, docs_to_segments, make_tensors
from tests.gpu_util import BWD_REL_L2, to_np

pytestmark = pytest.mark.gpu


def _docs(total=65536, lo=1024, seed=5):
    rng = np.random.Generator(np.random.PCG64(seed))
    out, left = [], total
    while left > 0:
        n = min(left, int(min(total, lo * rng.random() ** (-1 / 1.2))))
        out.append(n)
        left -= n
    return out


def _rel(a, b):
    a, b = to_np(a), to_np(b)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def test_cad_server_batches_match_one_call():
    import torch

    docs = _docs()
    T, Hq, Hkv, d = sum(docs), 8, 2, 128
    prob = Problem("cad64k", T, T, Hq, Hkv, d, docs_to_segments(docs), MaskSpec("CAUSAL_DOC"), 95)
    q, k, v, do = (t.cuda() for t in make_tensors(prob, device="cuda"))
    o_ref, lse_ref = lca.attn_fwd(q, k, v, prob.segments, prob.mask)
    dq_ref, dk_ref, dv_ref = lca.attn_bwd(do, q, k, v, o_ref, lse_ref, prob.segments, prob.mask)

    plan = lca.cad_plan(docs, 4, 1024, 8192, 0.05)
    assert len({s for *_, s in plan.shards}) == 4
    o = torch.zeros_like(q)
    lse = torch.full_like(lse_ref, float("nan"))
    dq = torch.zeros_like(q)
    dk = torch.zeros(k.shape, dtype=torch.float32, device="cuda")
    dv = torch.zeros_like(dk)
    served = torch.zeros(T, dtype=torch.int32, device="cuda")
    for server in range(4):
        segs, rows = plan.server_batch(server, docs)
        r = torch.from_numpy(rows).cuda()
        qs, dos = q[r].contiguous(), do[r].contiguous()
        mask = MaskSpec("CAUSAL")
        o_s, l_s = lca.attn_fwd(qs, k, v, segs, mask)
        dq_s, dk_s, dv_s = lca.attn_bwd(dos, qs, k, v, o_s, l_s, segs, mask)
        o[r], lse[:, r], dq[r] = o_s, l_s, dq_s
        dk += dk_s.float()
        dv += dv_s.float()
        served[r] += 1
    torch.cuda.synchronize()
    assert bool((served == 1).all()), "every token served exactly once"
    np.testing.assert_allclose(to_np(o), to_np(o_ref), atol=1e-2)
    np.testing.assert_allclose(to_np(lse), to_np(lse_ref), atol=1e-3)
    for name, x, ref in (("dQ", dq, dq_ref), ("dK", dk, dk_ref), ("dV", dv, dv_ref)):
        assert _rel(x, ref) <= BWD_REL_L2, (name, _rel(x, ref))
