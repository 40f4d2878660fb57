"""Forward and backward parity of the CUDA path against the fp64 oracle,
element by element, on every mask family (several tiles, ragged tails),
GQA and MHA, token-level shard batches, and the degenerate layouts.

Bar: forward max|O - O_ref| <= 1e-2 and mean <= 1e-3, LSE within 1e-3 with
-inf matching exactly; backward relative L2 error <= 2e-2 on dQ, dK, dV."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from gen import config1, make_tensors
from tests import cases
from tests.gpu_util import check_bwd, check_fwd, run_bwd, run_fwd, to_np

pytestmark = pytest.mark.gpu

SMALL = [config1("FULL"), config1("CAUSAL")] + cases.gpu_small_all() + cases.edge_cases()


def _parity(lib, prob, bwd=True):
    q, k, v, do = make_tensors(prob)
    o, lse = run_fwd(lib, prob, q, k, v)
    O, L = oracle.attention_forward(prob, q, k, v)
    check_fwd(o, lse, O, L, what=prob.name)
    if bwd:
        grads = run_bwd(lib, prob, q, k, v, do, o, lse)
        refs = oracle.attention_backward(prob, q, k, v, do)
        check_bwd(grads, refs, what=prob.name)


@pytest.mark.parametrize("prob", SMALL, ids=[p.name for p in SMALL])
def test_fwd_bwd_parity(lca, prob):
    _parity(lca, prob)


def test_shard_batch_parity_and_equivalence(lca):
    """Token-level shards of two documents in shuffled packed order: parity with
    the oracle, and equality with the causal-document result re-ordered."""
    shard, docp = cases.shard_problem([700, 300], [[130, 256, 200, 114], [77, 223]], Hq=8, Hkv=2, d=128)
    q, k, v, do = make_tensors(docp)
    rows = cases.shard_row_map(shard)
    qs, dos = q[rows], do[rows]
    o, lse = run_fwd(lca, shard, qs, k, v)
    O, L = oracle.attention_forward(shard, qs, k, v)
    check_fwd(o, lse, O, L, what="shards")
    grads = run_bwd(lca, shard, qs, k, v, dos, o, lse)
    refs = oracle.attention_backward(shard, qs, k, v, dos)
    check_bwd(grads, refs, what="shards")
    # same documents as one causal-document launch
    od, lsed = run_fwd(lca, docp, q, k, v)
    np.testing.assert_allclose(to_np(o), to_np(od)[rows], atol=1e-2)
    gd = run_bwd(lca, docp, q, k, v, do, od, lsed)
    np.testing.assert_allclose(to_np(grads[1]), to_np(gd[1]), atol=3e-2, rtol=3e-2)


def test_repeated_calls_are_deterministic(lca):
    prob = cases.gpu_small_all()[5]  # causal documents
    q, k, v, do = make_tensors(prob)
    o1, l1 = run_fwd(lca, prob, q, k, v)
    o2, l2 = run_fwd(lca, prob, q, k, v)
    assert np.array_equal(to_np(o1), to_np(o2)) and np.array_equal(to_np(l1), to_np(l2))
    g1 = run_bwd(lca, prob, q, k, v, do, o1, l1)
    g2 = run_bwd(lca, prob, q, k, v, do, o1, l1)
    for a, b in zip(g1, g2):
        assert np.array_equal(to_np(a), to_np(b))


@pytest.mark.parametrize("which", [5, 2])
def test_outputs_16_byte_aligned(lca, which):
    """Outputs that are 16- but not 32-byte aligned take 16-byte row stores
    instead of 32-byte ones: parity with the oracle, and the same bits as
    outputs at a 32-byte boundary (forward O; backward dQ, dK, dV)."""
    import torch

    prob = cases.gpu_small_all()[which]
    q, k, v, do = (t.cuda() for t in make_tensors(prob))
    segs, mask, sc = prob.segments, prob.mask, prob.scale
    o, lse = lca.attn_fwd(q, k, v, segs, mask, sc)
    grads = lca.attn_bwd(do, q, k, v, o, lse, segs, mask, sc)

    def off16(t):
        buf = torch.full((t.numel() + 8,), 7.0, dtype=t.dtype, device="cuda")
        u = buf[8:].view(t.shape)
        assert t.data_ptr() % 32 == 0 and u.data_ptr() % 32 == 16
        return u

    o16 = off16(o)
    lca.attn_fwd(q, k, v, segs, mask, sc, out=o16)
    g16 = [off16(g) for g in grads]
    lca.attn_bwd(do, q, k, v, o, lse, segs, mask, sc, dq=g16[0], dk=g16[1], dv=g16[2])
    torch.cuda.synchronize()
    assert torch.equal(o16, o)
    for a, b in zip(g16, grads):
        assert torch.equal(a, b)
    O, L = oracle.attention_forward(prob, *(t.cpu() for t in (q, k, v)))
    check_fwd(o16, lse, O, L, what=prob.name + "_o16")
    refs = oracle.attention_backward(prob, *(t.cpu() for t in (q, k, v, do)))
    check_bwd(g16, refs, what=prob.name + "_g16")


def test_misaligned_lse_refused_before_launch(lca):
    """An LSE pointer that is not 4-byte aligned (the row statistics are f32)
    makes both calls return LCA_ERR_INVALID_ARG with nothing launched."""
    import ctypes as C

    import torch

    prob = cases.gpu_small_all()[1]
    q, k, v, do = (t.cuda() for t in make_tensors(prob))
    call = lca.marshal(prob.Tq, prob.Tk, prob.Hq, prob.Hkv, prob.d, prob.segments, prob.mask, prob.scale)
    ws = torch.empty(max(lca.workspace_size(call, True), 256), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    lse_buf = torch.empty(prob.Hq * prob.Tq + 1, dtype=torch.float32, device="cuda")
    bad = lse_buf.data_ptr() + 2
    lib = lca.binding.load()
    torch.cuda.synchronize()
    n0 = lib.lca_launch_count()
    st = lib.lca_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), bad, C.byref(call.shape),
                          C.byref(call.mask), ws.data_ptr(), ws.numel(), None)
    assert st == 1
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    st = lib.lca_attn_bwd(do.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), bad,
                          dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), C.byref(call.shape), C.byref(call.mask),
                          ws.data_ptr(), ws.numel(), None)
    assert st == 1
    assert lib.lca_launch_count() == n0
    torch.cuda.synchronize()


def test_status_word_clean_after_calls(lca):
    import torch

    prob = config1("CAUSAL")
    q, k, v, do = (t.cuda() for t in make_tensors(prob))
    call = lca.marshal(prob.Tq, prob.Tk, prob.Hq, prob.Hkv, prob.d, prob.segments, prob.mask)
    ws = torch.empty(lca.workspace_size(call, True), dtype=torch.uint8, device="cuda")
    o, lse = lca.attn_fwd(q, k, v, prob.segments, prob.mask, workspace=ws, call=call)
    assert lca.read_status(ws) == (0, 0)
    lca.attn_bwd(do, q, k, v, o, lse, prob.segments, prob.mask, workspace=ws, call=call)
    assert lca.read_status(ws) == (0, 0)


def test_bounded_wait_reports_timeout(lca):
    """A barrier nothing arrives at: the wait gives up after its limit and the
    status word says LCA_ERR_TIMEOUT; the context stays usable."""
    import torch

    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    lca.probe_wait_timeout(ws, 50)
    code, where = lca.read_status(ws)
    assert code == 5 and where == 900
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum()) == 8.0


def _split_cases():
    """Layouts where some dK/dV units are far longer than the per-SM share,
    so the planner cuts them into chunks whose partial sums are reduced:
    keys every query attends (global tokens), every unit long (FULL with all
    query heads on one KV head), per-head block maps, one long document.  In
    all of them the last units of the cost order are also cut in two (the
    tail cut), so whole, long-unit and tail chunks meet in one launch."""
    from gen import MaskSpec, Problem, Segment

    out = [
        cases.single(2048, "GLOBAL_SLIDING", 8, 1, 128, 41, num_global=16, window_left=100, window_right=100),
        cases.single(1024, "FULL", 8, 1, 128, 42),
        cases.block_uniform(1536, 128, Hq=4, Hkv=1, d=128, seed=43),
        cases.docs([1800, 150, 98], "CAUSAL_DOC", 8, 2, 128, 44),
        Problem("q_gt_k", 1500, 700, 8, 1, 128, [Segment(0, 1500, 0, 700)], MaskSpec("FULL"), 45),
    ]
    for p in out:
        p.name = "split_" + p.name
    return out


SPLIT = _split_cases()


@pytest.mark.parametrize("prob", SPLIT, ids=[p.name for p in SPLIT])
def test_split_dkv_parity(lca, prob):
    _parity(lca, prob)


def test_split_dkv_deterministic(lca):
    prob = SPLIT[0]
    q, k, v, do = make_tensors(prob)
    o, lse = run_fwd(lca, prob, q, k, v)
    g1 = run_bwd(lca, prob, q, k, v, do, o, lse)
    g2 = run_bwd(lca, prob, q, k, v, do, o, lse)
    for a, b in zip(g1, g2):
        assert np.array_equal(to_np(a), to_np(b))


def test_binding_rejects_wrong_cuda_tensors(lca):
    """Wrong dtype, shape, layout or device of a CUDA tensor is refused before
    the library sees its pointer."""
    import torch

    from gen import MaskSpec, Segment

    segs, mask = [Segment(0, 256, 0, 256)], MaskSpec("CAUSAL")
    q = torch.randn(256, 4, 128, device="cuda").bfloat16()
    k = torch.randn(256, 2, 128, device="cuda").bfloat16()
    with pytest.raises(ValueError, match="dtype"):
        lca.attn_fwd(q.float(), k, k, segs, mask)
    with pytest.raises(ValueError, match="shape"):
        lca.attn_fwd(q, k, k[:128], segs, mask)
    with pytest.raises(ValueError, match="contiguous"):
        lca.attn_fwd(q, k, k.transpose(0, 1).contiguous().transpose(0, 1), segs, mask)
    with pytest.raises(ValueError, match="CUDA"):
        lca.attn_fwd(q, k, k.cpu(), segs, mask)
    o, lse = lca.attn_fwd(q, k, k, segs, mask)
    with pytest.raises(ValueError, match="dtype"):
        lca.attn_bwd(q, q, k, k, o, lse.double(), segs, mask)
    torch.cuda.synchronize()


HOST_OUT = [(p, None) for p in cases.edge_cases() + cases.gpu_small_all() if p.name in ("edge_gaps", "g_small_bsv")]
HOST_OUT += [(SPLIT[0], None), (SPLIT[0], (5, 0.1))]


@pytest.mark.parametrize("prob,drop", HOST_OUT, ids=[p.name + ("_drop" if d else "") for p, d in HOST_OUT])
def test_outputs_in_pinned_host_memory(lca, prob, drop):
    """Outputs may be page-locked host tensors: the kernels store into them
    through their device mapping (rows outside every segment, which a
    zero-fill kernel writes, and the reduced chunks of split dK/dV units
    included), bit for bit what device outputs receive.  A pageable host
    output is refused, by the binding and by the library."""
    import ctypes as C

    import torch

    q, k, v, do = (t.cuda() for t in make_tensors(prob))
    segs, mask, sc = prob.segments, prob.mask, prob.scale
    o, lse = lca.attn_fwd(q, k, v, segs, mask, sc, dropout=drop)
    dq, dk, dv = lca.attn_bwd(do, q, k, v, o, lse, segs, mask, sc, dropout=drop)
    torch.cuda.synchronize()

    def pinned(t):
        return torch.full(t.shape, 7, dtype=t.dtype, pin_memory=True)  # 7: stale contents must be overwritten

    oh, lh = pinned(o), pinned(lse)
    lca.attn_fwd(q, k, v, segs, mask, sc, out=oh, lse=lh, dropout=drop)
    gh = [pinned(t) for t in (dq, dk, dv)]
    lca.attn_bwd(do, q, k, v, o, lse, segs, mask, sc, dq=gh[0], dk=gh[1], dv=gh[2], dropout=drop)
    torch.cuda.synchronize()
    assert torch.equal(oh, o.cpu()) and torch.equal(lh, lse.cpu())
    for h, d in zip(gh, (dq, dk, dv)):
        assert torch.equal(h, d.cpu())

    pageable = torch.empty(dq.shape, dtype=dq.dtype)
    with pytest.raises(ValueError, match="pinned"):
        lca.attn_bwd(do, q, k, v, o, lse, segs, mask, sc, dq=pageable)
    call = lca.marshal(prob.Tq, prob.Tk, prob.Hq, prob.Hkv, prob.d, segs, mask, sc)
    ws = torch.empty(max(lca.workspace_size(call, True), 256), dtype=torch.uint8, device="cuda")
    st = lca.binding.load().lca_attn_bwd(do.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), pageable.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                         C.byref(call.shape), C.byref(call.mask), ws.data_ptr(), ws.numel(), None)
    assert st == 1  # LCA_ERR_INVALID_ARG, returned before any launch
    torch.cuda.synchronize()


def test_pointer_of_another_device_refused(lca):
    """With cuda:0 current, a call whose tensors live on cuda:1 is refused
    with LCA_ERR_INVALID_ARG before anything is launched (the kernels would
    run on cuda:0 and read another GPU's memory); through the binding, which
    makes the tensors' device current, the same call runs on cuda:1."""
    import ctypes as C

    import torch

    if torch.cuda.device_count() < 2:
        pytest.skip("needs two visible GPUs")
    from gen import MaskSpec, Segment

    segs, mask = [Segment(0, 256, 0, 256)], MaskSpec("CAUSAL")
    dev1 = torch.device("cuda", 1)
    q = torch.randn(256, 4, 128, device=dev1).bfloat16()
    k = torch.randn(256, 2, 128, device=dev1).bfloat16()
    o, lse = torch.empty_like(q), torch.empty((4, 256), dtype=torch.float32, device=dev1)
    call = lca.marshal(256, 256, 4, 2, 128, segs, mask)
    ws = torch.empty(max(lca.workspace_size(call, False), 256), dtype=torch.uint8, device=dev1)
    L = lca.binding.load()
    with torch.cuda.device(0):
        before = L.lca_launch_count()
        code = L.lca_attn_fwd(q.data_ptr(), k.data_ptr(), k.data_ptr(), o.data_ptr(), lse.data_ptr(),
                              C.byref(call.shape), C.byref(call.mask), ws.data_ptr(), ws.numel(), None)
        assert code == 1
        assert L.lca_launch_count() == before
        o1, lse1 = lca.attn_fwd(q, k, k, segs, mask)
    torch.cuda.synchronize(dev1)
    assert o1.device == dev1 and torch.isfinite(lse1).all()


def test_backward_on_a_side_stream_is_ordered(lca):
    """The backward forks its dK/dV pass onto the library's own stream and
    joins it back: work queued on the caller's (non-default) stream right
    after the call sees the finished dK and dV, and a second call reusing
    the same output buffers gives the same bits."""
    import torch

    prob = SPLIT[1]
    q, k, v, do = (t.cuda() for t in make_tensors(prob))
    o, lse = lca.attn_fwd(q, k, v, prob.segments, prob.mask, prob.scale)
    dq0, dk0, dv0 = lca.attn_bwd(do, q, k, v, o, lse, prob.segments, prob.mask, prob.scale)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        dq, dk, dv = torch.full_like(dq0, 3.0), torch.full_like(dk0, 3.0), torch.full_like(dv0, 3.0)
        lca.attn_bwd(do, q, k, v, o, lse, prob.segments, prob.mask, prob.scale, dq=dq, dk=dk, dv=dv)
        copies = [t.clone() for t in (dq, dk, dv)]  # queued right after the call on the same stream
    torch.cuda.synchronize()
    for c, ref in zip(copies, (dq0, dk0, dv0)):
        assert torch.equal(c, ref)


def _aligned_block_cases():
    """Uniform block maps whose blocks and segment starts are multiples of 32
    (the forward's per-warp keep-bit form), with ragged tails and several
    segments, and the same map with a segment start off the 32 grid (the
    per-row mask-word form)."""
    from gen import MaskSpec, Problem, Segment, uniform_block_map

    r = np.random.Generator(np.random.PCG64(71))
    out = []
    for b, T, segs, name in [
        (32, 1000, [(0, 1000, 0, 1000)], "b32_one"),
        (96, 960, [(0, 480, 0, 480), (512, 448, 512, 448)], "b96_two_aligned"),
        (96, 960, [(0, 470, 0, 470), (490, 470, 490, 470)], "b96_two_unaligned"),
        (64, 1100, [(64, 700, 0, 1100)], "b64_offset_q"),
    ]:
        n = -(-T // b)
        rp, ci = uniform_block_map(n, n, 4, r)
        spec = MaskSpec("BLOCK_SPARSE_UNIFORM", q_block=b, kv_block=b, heads_in_map=4, blk_row_ptr=rp, blk_col_idx=ci)
        out.append(Problem("aligned_" + name, T, T, 4, 2, 128, [Segment(*s) for s in segs], spec, 72))
    return out


ALIGNED = _aligned_block_cases()


@pytest.mark.parametrize("prob", ALIGNED, ids=[p.name for p in ALIGNED])
def test_aligned_block_map_parity(lca, prob):
    _parity(lca, prob)


def test_aligned_block_map_matches_variable_form(lca):
    """The keep-bit form gives the same forward and backward, bit for bit, as
    the same map stated as variable blocks (which always takes per-row mask
    words): the masked 32-key chunks it skips contribute exact zeros there."""
    import copy

    from gen import MaskSpec

    for prob in ALIGNED[:2]:
        m = prob.mask
        n = (len(m.blk_row_ptr) - 1) // 4  # block rows per map head (4 heads in the map)
        bounds = (np.arange(n + 1) * m.q_block).astype(np.int32)
        var = copy.copy(prob)
        var.mask = MaskSpec("BLOCK_SPARSE_VARIABLE", qb_bounds=bounds, kb_bounds=bounds, heads_in_map=4,
                            blk_row_ptr=m.blk_row_ptr, blk_col_idx=m.blk_col_idx)
        q, k, v, do = make_tensors(prob)
        o1, l1 = run_fwd(lca, prob, q, k, v)
        o2, l2 = run_fwd(lca, var, q, k, v)
        assert np.array_equal(to_np(o1), to_np(o2)), prob.name
        assert np.array_equal(to_np(l1), to_np(l2)), prob.name
        g1 = run_bwd(lca, prob, q, k, v, do, o1, l1)
        g2 = run_bwd(lca, var, q, k, v, do, o1, l1)
        for name, x, y in zip(("dq", "dk", "dv"), g1, g2):
            assert np.array_equal(to_np(x), to_np(y)), (prob.name, name)


def _variable_block_cases():
    """Variable block maps over several segments: packed documents (one key
    group each), and two query segments reading one key range (one key group
    with two members), with ragged ends."""
    from gen import MaskSpec, Problem, Segment, variable_block_bounds, variable_block_map

    r = np.random.Generator(np.random.PCG64(81))
    out = []
    for T, segs, name in [
        (1033, [(0, 400, 0, 400), (400, 300, 400, 300), (700, 333, 700, 333)], "docs"),
        (1000, [(0, 260, 0, 700), (260, 440, 0, 700), (700, 300, 700, 300)], "shared_keys"),
    ]:
        qb = variable_block_bounds(T, 32, 256, r)
        kb = variable_block_bounds(T, 32, 256, r)
        rp, ci = variable_block_map(len(qb) - 1, len(kb) - 1, 4, r)
        spec = MaskSpec("BLOCK_SPARSE_VARIABLE", qb_bounds=qb, kb_bounds=kb, heads_in_map=4, blk_row_ptr=rp,
                        blk_col_idx=ci)
        out.append(Problem("variable_" + name, T, T, 4, 2, 128, [Segment(*s) for s in segs], spec, 82))
    return out


VARIABLE = _variable_block_cases()


@pytest.mark.parametrize("prob", VARIABLE, ids=[p.name for p in VARIABLE])
def test_variable_block_map_segments_parity(lca, prob):
    _parity(lca, prob)
