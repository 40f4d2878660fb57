"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, sizes workspaces on the host, and rejects malformed arguments
before launching anything (all calls below fail validation, so no CUDA call
is made)."""
from __future__ import annotations

import ctypes as C
import os
import re

import numpy as np
import pytest

import long_context_masked_attention_gb300 as lib
from long_context_masked_attention_gb300 import binding as B
from gen import MaskSpec, Segment, config1, config2, config3, config4, config5

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lca_attn.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(B.LIB_PATH):
        lib.build()
    return lib.load()


def test_exports_every_declared_symbol(L):
    declared = re.findall(r"LCA_API\s+[\w\s\*]+?\b(lca_\w+)\s*\(", open(HEADER).read())
    assert sorted(declared) == sorted(B.EXPORTED)
    for name in declared:
        assert hasattr(L, name), name


def test_status_strings(L):
    for code in range(7):
        assert L.lca_status_string(code)
    assert L.lca_version() >= 100


def _ws(L, Tq, Tk, Hq, Hkv, segs, mask, bwd=False, d=128, scale=0.0):
    call = B.marshal(Tq, Tk, Hq, Hkv, d, segs, mask, scale)
    n = C.c_size_t(0)
    code = L.lca_workspace_size(C.byref(call.shape), C.byref(call.mask), int(bwd), C.byref(n))
    return code, n.value


@pytest.mark.parametrize("prob", [config1("FULL"), config1("CAUSAL"), config2("CAUSAL_DOC"), config2("SHARED_QUESTION"),
                                  config3(1024, "gqa", "CAUSAL_DOC"), config5()], ids=lambda p: p.name)
def test_workspace_sizes(L, prob):
    code, f = _ws(L, prob.Tq, prob.Tk, prob.Hq, prob.Hkv, prob.segments, prob.mask, False)
    assert code == 0 and f > 0
    code, b = _ws(L, prob.Tq, prob.Tk, prob.Hq, prob.Hkv, prob.segments, prob.mask, True)
    assert code == 0 and b > f
    # the backward needs D and LSE in base 2 (2 x 4 bytes per query row and head) on top
    assert b - f >= 8 * prob.Tq * prob.Hq


BAD = [
    ("d != 128", dict(d=64), 2),
    ("Hq % Hkv", dict(Hq=6, Hkv=4), 1),
    ("negative scale", dict(scale=-1.0), 1),
    ("segment past Tq", dict(segs=[Segment(0, 300, 0, 256)]), 1),
    ("segment past Tk", dict(segs=[Segment(0, 256, 10, 256)]), 1),
    ("overlapping queries", dict(segs=[Segment(0, 128, 0, 128), Segment(100, 100, 128, 100)]), 1),
    ("overlapping key groups", dict(segs=[Segment(0, 128, 0, 128), Segment(128, 128, 64, 128)]), 1),
    ("negative window", dict(mask=MaskSpec("SLIDING", window_left=-1)), 1),
    ("block 0", dict(mask=MaskSpec("CAUSAL_BLOCKWISE", block=0)), 1),
    ("parts not starting at 0", dict(mask=MaskSpec("SHARED_QUESTION", part_bounds=[1, 100, 256])), 1),
    ("parts too short", dict(mask=MaskSpec("SHARED_QUESTION", part_bounds=[0, 100, 200])), 1),
    ("prefix doc without prefixes", dict(mask=MaskSpec("PREFIX_LM_DOC")), 1),
    ("unknown kind", dict(mask=MaskSpec(99)), 1),
    ("key block below 32", dict(mask=MaskSpec("BLOCK_SPARSE_UNIFORM", q_block=64, kv_block=16)), 1),
]


@pytest.mark.parametrize("name,over,code", BAD, ids=[b[0] for b in BAD])
def test_invalid_arguments_rejected_before_launch(L, name, over, code):
    args = dict(Tq=256, Tk=256, Hq=4, Hkv=2, segs=[Segment(0, 256, 0, 256)], mask=MaskSpec("CAUSAL"), d=128,
                scale=0.0)
    args.update(over)
    c, _ = _ws(L, args["Tq"], args["Tk"], args["Hq"], args["Hkv"], args["segs"], args["mask"], False, args["d"],
               args["scale"])
    assert c == code, (name, c)
    # the entry points return the same code without touching the (fake) device pointers
    call = B.marshal(args["Tq"], args["Tk"], args["Hq"], args["Hkv"], args["d"], args["segs"], args["mask"],
                     args["scale"])
    fake = C.c_void_p(0x1000)
    r = L.lca_attn_fwd(fake, fake, fake, fake, fake, C.byref(call.shape), C.byref(call.mask), C.c_void_p(0x10000),
                       1 << 30, None)
    assert r == code
    r = L.lca_attn_bwd(fake, fake, fake, fake, fake, fake, fake, fake, fake, C.byref(call.shape), C.byref(call.mask),
                       C.c_void_p(0x10000), 1 << 30, None)
    assert r == code


def test_block_sparse_validation(L):
    base = dict(kind="BLOCK_SPARSE_VARIABLE", heads_in_map=1)

    class M:
        pass

    m = M()
    m.kind = "BLOCK_SPARSE_VARIABLE"
    m.heads_in_map = 1
    m.qb_bounds = np.array([0, 100, 256])
    m.kb_bounds = np.array([0, 20, 256])  # a 20-wide inner key block: unsupported
    m.blk_row_ptr = None
    m.blk_col_idx = None
    call = B.marshal(256, 256, 2, 1, 128, [Segment(0, 256, 0, 256)], m)
    call.mask.blk_row_ptr = 0x1000  # fake device pointers; validation fails first
    call.mask.blk_col_idx = 0x1000
    call.mask.blk_nnz = 2
    n = C.c_size_t(0)
    assert L.lca_workspace_size(C.byref(call.shape), C.byref(call.mask), 0, C.byref(n)) == 2
    m.kb_bounds = np.array([0, 40, 200])  # does not cover Tk
    call2 = B.marshal(256, 256, 2, 1, 128, [Segment(0, 256, 0, 256)], m)
    call2.mask.blk_row_ptr = 0x1000
    call2.mask.blk_col_idx = 0x1000
    call2.mask.blk_nnz = 2
    assert L.lca_workspace_size(C.byref(call2.shape), C.byref(call2.mask), 0, C.byref(n)) == 1
    call2.mask.heads_in_map = 3  # neither 1 nor Hq
    assert L.lca_workspace_size(C.byref(call2.shape), C.byref(call2.mask), 0, C.byref(n)) == 1


def test_workspace_too_small_is_rejected(L):
    call = B.marshal(256, 256, 4, 2, 128, [Segment(0, 256, 0, 256)], MaskSpec("CAUSAL"))
    n = C.c_size_t(0)
    assert L.lca_workspace_size(C.byref(call.shape), C.byref(call.mask), 0, C.byref(n)) == 0
    fake = C.c_void_p(0x1000)
    assert L.lca_attn_fwd(fake, fake, fake, fake, fake, C.byref(call.shape), C.byref(call.mask), C.c_void_p(0x10000),
                          n.value - 1, None) == 3
    assert L.lca_attn_fwd(fake, fake, fake, fake, fake, C.byref(call.shape), C.byref(call.mask), C.c_void_p(0x10001),
                          n.value, None) == 3  # misaligned


@pytest.mark.parametrize("p", [-0.1, 1.0, 1.5, float("nan"), float("inf")])
def test_dropout_probability_out_of_range_rejected(L, p):
    call = B.marshal(256, 256, 4, 2, 128, [Segment(0, 256, 0, 256)], MaskSpec("CAUSAL"))
    fake = C.c_void_p(0x1000)
    drop = B.Dropout_t(p, 7)
    assert L.lca_attn_fwd_dropout(fake, fake, fake, fake, fake, C.byref(call.shape), C.byref(call.mask),
                                  C.byref(drop), C.c_void_p(0x10000), 1 << 30, None) == 1
    assert L.lca_attn_bwd_dropout(fake, fake, fake, fake, fake, fake, fake, fake, fake, C.byref(call.shape),
                                  C.byref(call.mask), C.byref(drop), C.c_void_p(0x10000), 1 << 30, None) == 1


def test_dropout_entry_points_validate_like_the_plain_ones(L):
    """A valid probability passes on to the same shape and workspace checks."""
    call = B.marshal(256, 256, 4, 2, 128, [Segment(0, 256, 0, 256)], MaskSpec("CAUSAL"))
    n = C.c_size_t(0)
    assert L.lca_workspace_size(C.byref(call.shape), C.byref(call.mask), 1, C.byref(n)) == 0
    fake = C.c_void_p(0x1000)
    drop = B.Dropout_t(0.1, 7)
    assert L.lca_attn_fwd_dropout(fake, fake, fake, fake, fake, C.byref(call.shape), C.byref(call.mask),
                                  C.byref(drop), C.c_void_p(0x10000), 16, None) == 3
    assert L.lca_attn_bwd_dropout(fake, fake, fake, fake, fake, fake, fake, fake, fake, C.byref(call.shape),
                                  C.byref(call.mask), C.byref(drop), C.c_void_p(0x10000), n.value - 1, None) == 3
    bad = B.marshal(256, 256, 6, 4, 128, [Segment(0, 256, 0, 256)], MaskSpec("CAUSAL"))  # Hq % Hkv != 0
    assert L.lca_attn_fwd_dropout(fake, fake, fake, fake, fake, C.byref(bad.shape), C.byref(bad.mask),
                                  C.byref(drop), C.c_void_p(0x10000), 1 << 30, None) == 1


def test_binding_rejects_unsuitable_tensors_before_calling_the_library():
    """The binding hands raw device pointers to the library, so host, wrongly
    typed, misshapen or strided tensors are rejected first (no CUDA needed)."""
    import torch

    segs, mask = [Segment(0, 8, 0, 8)], MaskSpec("CAUSAL")
    q = torch.zeros(8, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        lib.attn_fwd(q, q[:, :1], q[:, :1], segs, mask)
    with pytest.raises(ValueError, match="CUDA"):
        lib.attn_bwd(q, q, q[:, :1], q[:, :1], q, torch.zeros(2, 8), segs, mask)
    with pytest.raises(ValueError, match="CUDA"):
        lib.attn_merge([q], [torch.zeros(2, 8)])
    with pytest.raises(TypeError):
        lib.attn_fwd(np.zeros((8, 2, 128)), q, q, segs, mask)
    # the checks themselves, on tensor metadata only
    meta = torch.empty(8, 2, 128, dtype=torch.bfloat16, device="meta")
    with pytest.raises(ValueError, match="CUDA"):
        B._require(meta, "q", (8, 2, 128), torch.bfloat16)
    # outputs may be pinned host tensors, never pageable ones
    with pytest.raises(ValueError, match="pinned"):
        B._require(q, "dq", (8, 2, 128), torch.bfloat16, host_ok=True)
