"""The static-workspace forward (lca_attn_fwd_static_workspace) serves
callers that cannot allocate device memory — a process whose device-memory
pool was reserved up front and may not grow, or code running where
allocation is not allowed.  It must give the same result as the regular
forward with a caller-provided workspace, call after call, and reject shapes
whose workspace does not fit its fixed array before launching anything.

This file is collected last on purpose: the static array keeps the previous
call's contents, so these tests also show that a call clears what it needs."""
from __future__ import annotations

import ctypes as C

import numpy as np
import pytest

from gen import Segment, make_tensors
from tests import cases
from tests.gpu_util import check_fwd, to_np

pytestmark = pytest.mark.gpu


def _static_fwd(lca, call, q, k, v):
    import torch

    Tq, Hq, _ = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((Hq, Tq), dtype=torch.float32, device=q.device)
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    code = lca.load().lca_attn_fwd_static_workspace(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                                    lse.data_ptr(), C.byref(call.shape), C.byref(call.mask), stream)
    assert code == 0, (code, lca.load().lca_last_error_detail())
    torch.cuda.synchronize()
    return o, lse


@pytest.mark.parametrize("idx", [5, 12])  # causal documents; uniform 64-block sparse map
def test_static_workspace_forward_matches_regular_forward(lca, idx):
    import torch

    prob = cases.gpu_small_all()[idx]
    q, k, v, _ = (t.cuda() if t is not None else None for t in make_tensors(prob))
    call = lca.marshal(prob.Tq, prob.Tk, prob.Hq, prob.Hkv, prob.d, prob.segments, prob.mask, prob.scale)
    o_ref, lse_ref = lca.attn_fwd(q, k, v, prob.segments, prob.mask, prob.scale, call=call)
    torch.cuda.synchronize()
    O_ref, L_ref = to_np(o_ref), to_np(lse_ref)
    for _ in range(2):  # two calls in a row share the one static array
        o, lse = _static_fwd(lca, call, q, k, v)
        check_fwd(o, lse, O_ref, L_ref, what=f"static workspace {prob.name}")


def test_static_workspace_rejects_oversized_shape(lca):
    from gen import MaskSpec

    T = 1 << 20  # one FULL segment of 1M tokens: 4096 x 8192 forward list entries, far beyond the fixed array
    call = lca.marshal(T, T, 1, 1, 128, [Segment(0, T, 0, T)], MaskSpec("FULL"))
    need = lca.workspace_size(call, False)
    L = lca.load()
    assert need > 16 << 20
    fake = C.c_void_p(0x1000)
    code = L.lca_attn_fwd_static_workspace(fake, fake, fake, fake, fake, C.byref(call.shape), C.byref(call.mask),
                                           None)
    assert code == 3
    assert b"static workspace" in L.lca_last_error_detail()
