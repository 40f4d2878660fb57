"""Pins of the fp64 oracle against facts fixed outside it: hand-derived worked
examples, closed forms, invariants of softmax attention, equivalences
between mask families, finite differences and an independent library
routine.  CPU only."""
from __future__ import annotations

import math
import os

import numpy as np
import pytest

import oracle
from gen import MaskSpec, Problem, Segment
from tests import cases
from tests.brute_masks import brute_dense_mask

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, val = line.partition("=") if "=" in line else line.partition(" ")
        out[key.strip()] = np.array([float(x) for x in val.split()])
    return out


def _rand(prob, seed=0, scale=1.0):
    r = np.random.Generator(np.random.PCG64(seed))
    q = r.standard_normal((prob.Tq, prob.Hq, prob.d)) * scale
    k = r.standard_normal((prob.Tk, prob.Hkv, prob.d)) * scale
    v = r.standard_normal((prob.Tk, prob.Hkv, prob.d))
    do = r.standard_normal((prob.Tq, prob.Hq, prob.d))
    return q, k, v, do


# ------------------------------------------------------------ worked examples
def test_worked_example_a():
    g = _golden("worked_examples.txt")
    p = Problem("A", 1, 2, 1, 1, 2, [Segment(0, 1, 0, 2)], MaskSpec("FULL"), 0, scale=1.0)
    q = np.array([[[1.0, 0.0]]])
    k = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])
    v = k.copy()
    O, L = oracle.attention_forward(p, q, k, v)
    assert abs(L[0, 0] - g["A.lse0"][0]) < 1e-12
    np.testing.assert_allclose(O[0, 0], g["A.o0"], atol=1e-12)


def test_worked_example_b_forward_backward():
    g = _golden("worked_examples.txt")
    p = Problem("B", 2, 2, 1, 1, 2, [Segment(0, 2, 0, 2)], MaskSpec("CAUSAL"), 0, scale=1.0)
    q = np.array([[[1.0, 0.0]], [[0.0, 2.0]]])
    k = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])
    v = k.copy()
    do = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])
    O, L = oracle.attention_forward(p, q, k, v)
    np.testing.assert_allclose(L[0], g["B.lse"], atol=1e-12)
    np.testing.assert_allclose(O[0, 0], g["B.o0"], atol=1e-12)
    np.testing.assert_allclose(O[1, 0], g["B.o1"], atol=1e-12)
    dQ, dK, dV = oracle.attention_backward(p, q, k, v, do)
    for name, arr, row in [("dq0", dQ, 0), ("dq1", dQ, 1), ("dk0", dK, 0), ("dk1", dK, 1), ("dv0", dV, 0),
                           ("dv1", dV, 1)]:
        np.testing.assert_allclose(arr[row, 0], g["B." + name], atol=1e-12, err_msg=name)


# ------------------------------------------------------------ closed forms
ALL_TINY = cases.tiny_all()


@pytest.mark.parametrize("prob", ALL_TINY, ids=[p.name for p in ALL_TINY])
def test_constant_v_gives_that_row(prob):
    q, k, v, _ = _rand(prob, 1)
    c = np.linspace(-1, 1, prob.d)
    v[:] = c
    O, L = oracle.attention_forward(prob, q, k, v)
    for h in range(prob.Hq):
        nonempty = np.isfinite(L[h])
        np.testing.assert_allclose(O[nonempty, h], np.broadcast_to(c, O[nonempty, h].shape), atol=1e-12)


@pytest.mark.parametrize("prob", ALL_TINY, ids=[p.name for p in ALL_TINY])
def test_zero_q_gives_log_count_and_mean(prob):
    """Q = 0 -> all scores 0 -> LSE_i = ln(n_i), O_i = mean of attended v_j.
    n_i and the attended set come from the brute-force constructive masks."""
    _, k, v, _ = _rand(prob, 2)
    q = np.zeros((prob.Tq, prob.Hq, prob.d))
    O, L = oracle.attention_forward(prob, q, k, v)
    G = prob.Hq // prob.Hkv
    for h in range(prob.Hq):
        M = brute_dense_mask(prob, h)
        n = M.sum(axis=1)
        want_L = np.where(n > 0, np.log(np.maximum(n, 1)), -np.inf)
        np.testing.assert_allclose(L[h], want_L, atol=1e-12)
        mean = (M.astype(float) @ v[:, h // G]) / np.maximum(n, 1)[:, None]
        np.testing.assert_allclose(O[:, h], mean, atol=1e-12)


def test_single_token():
    p = Problem("s1", 1, 1, 1, 1, 4, [Segment(0, 1, 0, 1)], MaskSpec("CAUSAL"), 0)
    q, k, v, _ = _rand(p, 3)
    O, L = oracle.attention_forward(p, q, k, v)
    np.testing.assert_allclose(O[0, 0], v[0, 0], atol=1e-14)
    assert abs(L[0, 0] - (q[0, 0] @ k[0, 0]) / 2.0) < 1e-14


def test_fully_masked_rows_give_zero_and_neg_inf():
    # bottom-right causal with more queries than keys: the first q_len-k_len rows see nothing
    p = Problem("fm", 6, 3, 1, 1, 4, [Segment(0, 6, 0, 3)], MaskSpec("CAUSAL"), 0)
    q, k, v, do = _rand(p, 4)
    O, L = oracle.attention_forward(p, q, k, v)
    assert np.all(np.isneginf(L[0, :3])) and np.all(np.isfinite(L[0, 3:]))
    assert np.all(O[:3] == 0.0)
    dQ, dK, dV = oracle.attention_backward(p, q, k, v, do)
    assert np.all(dQ[:3] == 0.0)
    # keys only receive gradient from rows that see them
    dQ2, dK2, dV2 = oracle.attention_backward(p, q, k, v, np.concatenate([np.zeros_like(do[:3]), do[3:]]))
    np.testing.assert_allclose(dK, dK2, atol=1e-14)
    np.testing.assert_allclose(dV, dV2, atol=1e-14)


def test_one_hot_large_scale_selects_argmax():
    S, d = 6, 8
    p = Problem("oh", S, S, 1, 1, d, [Segment(0, S, 0, S)], MaskSpec("FULL"), 0, scale=50.0)
    r = np.random.Generator(np.random.PCG64(5))
    k = np.zeros((S, 1, d))
    for j in range(S):
        k[j, 0, j] = 1.0
    q = np.zeros((S, 1, d))
    target = r.permutation(S)
    for i in range(S):
        q[i, 0, target[i]] = 1.0
    v = r.standard_normal((S, 1, d))
    O, _ = oracle.attention_forward(p, q, k, v)
    np.testing.assert_allclose(O[:, 0], v[target, 0], atol=1e-18 + 1e-15 * S * 1e3)


# ------------------------------------------------------------ invariants
@pytest.mark.parametrize("prob", ALL_TINY, ids=[p.name for p in ALL_TINY])
def test_rows_sum_to_one_and_match_exp_minus_lse(prob):
    """With d >= k_len and V = identity rows, O_i is the probability row P_i."""
    S = prob.Tk
    p2 = Problem(prob.name, prob.Tq, prob.Tk, prob.Hq, prob.Hkv, S, prob.segments, prob.mask, prob.seed)
    q, k, _, _ = _rand(p2, 6)
    v = np.zeros((S, prob.Hkv, S))
    for j in range(S):
        v[j, :, j] = 1.0
    O, L = oracle.attention_forward(p2, q, k, v)
    G = prob.Hq // prob.Hkv
    for h in range(prob.Hq):
        M = brute_dense_mask(p2, h)
        nonempty = M.any(axis=1)
        np.testing.assert_allclose(O[nonempty, h].sum(axis=1), 1.0, atol=1e-12)
        s = p2.softmax_scale * q[:, h] @ k[:, h // G].T
        want = np.where(M, np.exp(s - np.where(nonempty, L[h], 0)[:, None]), 0.0)
        np.testing.assert_allclose(O[:, h], want, atol=1e-12)


@pytest.mark.parametrize("prob", ALL_TINY, ids=[p.name for p in ALL_TINY])
def test_key_shift_invariance(prob):
    q, k, v, do = _rand(prob, 7)
    u = np.random.Generator(np.random.PCG64(8)).standard_normal(prob.d)
    O1, L1 = oracle.attention_forward(prob, q, k, v)
    O2, L2 = oracle.attention_forward(prob, q, k + u, v)
    np.testing.assert_allclose(O1, O2, atol=1e-10)
    G = prob.Hq // prob.Hkv
    for h in range(prob.Hq):
        fin = np.isfinite(L1[h])
        np.testing.assert_allclose(L2[h, fin] - L1[h, fin], prob.softmax_scale * q[fin, h] @ u, atol=1e-10)
    dQ1, _, _ = oracle.attention_backward(prob, q, k, v, do)
    dQ2, _, _ = oracle.attention_backward(prob, q, k + u, v, do)
    np.testing.assert_allclose(dQ1, dQ2, atol=1e-10)


@pytest.mark.parametrize("prob", ALL_TINY, ids=[p.name for p in ALL_TINY])
def test_gradient_sums(prob):
    """sum_j dS_ij = 0 -> sum_j dK_j = 0;  sum_j dV_j = sum of dO over rows with keys."""
    q, k, v, do = _rand(prob, 9)
    _, L = oracle.attention_forward(prob, q, k, v)
    dQ, dK, dV = oracle.attention_backward(prob, q, k, v, do)
    np.testing.assert_allclose(dK.sum(axis=0), 0.0, atol=1e-10)
    G = prob.Hq // prob.Hkv
    for g in range(prob.Hkv):
        want = sum(do[np.isfinite(L[h]), h].sum(axis=0) for h in range(g * G, (g + 1) * G))
        np.testing.assert_allclose(dV[:, g].sum(axis=0), want, atol=1e-10)


def test_key_permutation_invariance_full():
    p = cases.single(12, "FULL", d=6)
    q, k, v, do = _rand(p, 10)
    perm = np.random.Generator(np.random.PCG64(11)).permutation(12)
    O1, L1 = oracle.attention_forward(p, q, k, v)
    O2, L2 = oracle.attention_forward(p, q, k[perm], v[perm])
    np.testing.assert_allclose(O1, O2, atol=1e-12)
    np.testing.assert_allclose(L1, L2, atol=1e-12)
    _, dK1, dV1 = oracle.attention_backward(p, q, k, v, do)
    _, dK2, dV2 = oracle.attention_backward(p, q, k[perm], v[perm], do)
    np.testing.assert_allclose(dK1[perm], dK2, atol=1e-12)
    np.testing.assert_allclose(dV1[perm], dV2, atol=1e-12)


# ------------------------------------------------------------ equivalences
def _same(pa, pb, seed=12):
    q, k, v, do = _rand(pa, seed)
    Oa, La = oracle.attention_forward(pa, q, k, v)
    Ob, Lb = oracle.attention_forward(pb, q, k, v)
    np.testing.assert_allclose(Oa, Ob, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(La), np.isneginf(Lb))
    fin = np.isfinite(La)
    np.testing.assert_allclose(La[fin], Lb[fin], atol=1e-12)
    ga = oracle.attention_backward(pa, q, k, v, do)
    gb = oracle.attention_backward(pb, q, k, v, do)
    for x, y in zip(ga, gb):
        np.testing.assert_allclose(x, y, atol=1e-12)


S = 14


@pytest.mark.parametrize("a,b", [
    (cases.docs([S], "DOC"), cases.single(S, "FULL")),
    (cases.docs([S], "CAUSAL_DOC"), cases.single(S, "CAUSAL")),
    (cases.single(S, "SLIDING", window_left=S, window_right=S), cases.single(S, "FULL")),
    (cases.single(S, "CAUSAL_SLIDING", window_left=S), cases.single(S, "CAUSAL")),
    (cases.single(S, "PREFIX_LM_CAUSAL", prefix_len=0), cases.single(S, "CAUSAL")),
    (cases.single(S, "PREFIX_LM_CAUSAL", prefix_len=S), cases.single(S, "FULL")),
    (cases.single(S, "GLOBAL_SLIDING", num_global=0, window_left=3, window_right=3),
     cases.single(S, "SLIDING", window_left=3, window_right=3)),
    (cases.docs([5, 9], "BLOCK_CAUSAL_DOC", block=1), cases.docs([5, 9], "CAUSAL_DOC")),
    (cases.docs([5, 9], "BLOCK_CAUSAL_DOC", block=9), cases.docs([5, 9], "DOC")),
    (cases.single(S, "SHARED_QUESTION", part_bounds=[0, 6, S]), cases.single(S, "CAUSAL")),
    (cases.docs([5, 9], "PREFIX_LM_DOC", prefix_len=0), cases.docs([5, 9], "CAUSAL_DOC")),
    (cases.single(S, "CAUSAL_BLOCKWISE", block=S), cases.single(S, "CAUSAL")),
], ids=["doc1", "cdoc1", "slide_wide", "cslide_wide", "prefix0", "prefixS", "global0", "bcd1", "bcd_big",
        "sq_one_answer", "prefixdoc0", "cblock_one"])
def test_family_equivalences(a, b):
    _same(a, b)


def test_block_sparse_all_kept_is_full():
    p = cases.block_uniform(12, 4)
    n = 3
    p.mask.blk_row_ptr = (np.arange(p.mask.heads_in_map * n + 1) * n).astype(np.int32)
    p.mask.blk_col_idx = np.tile(np.arange(n, dtype=np.int32), p.mask.heads_in_map * n)
    _same(p, cases.single(12, "FULL"))


def test_shard_batch_equals_causal_document():
    shard, docp = cases.shard_problem([7, 12, 5], [[3, 4], [5, 2, 5], [5]])
    q, k, v, do = _rand(docp, 13)
    rows = cases.shard_row_map(shard)  # packed shard row -> document-order row
    Od, Ld = oracle.attention_forward(docp, q, k, v)
    Os, Ls = oracle.attention_forward(shard, q[rows], k, v)
    np.testing.assert_allclose(Os, Od[rows], atol=1e-12)
    np.testing.assert_allclose(Ls, Ld[:, rows], atol=1e-12)
    dQd, dKd, dVd = oracle.attention_backward(docp, q, k, v, do)
    dQs, dKs, dVs = oracle.attention_backward(shard, q[rows], k, v, do[rows])
    np.testing.assert_allclose(dQs, dQd[rows], atol=1e-12)
    np.testing.assert_allclose(dKs, dKd, atol=1e-12)
    np.testing.assert_allclose(dVs, dVd, atol=1e-12)


def test_mha_equals_gqa_with_repeated_kv():
    G = 3
    pg = cases.single(10, "CAUSAL", Hq=6, Hkv=2, d=4)
    pm = cases.single(10, "CAUSAL", Hq=6, Hkv=6, d=4)
    q, k, v, do = _rand(pg, 14)
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    Og, Lg = oracle.attention_forward(pg, q, k, v)
    Om, Lm = oracle.attention_forward(pm, q, kr, vr)
    np.testing.assert_allclose(Og, Om, atol=1e-12)
    np.testing.assert_allclose(Lg, Lm, atol=1e-12)
    dQg, dKg, dVg = oracle.attention_backward(pg, q, k, v, do)
    dQm, dKm, dVm = oracle.attention_backward(pm, q, kr, vr, do)
    np.testing.assert_allclose(dQg, dQm, atol=1e-12)
    np.testing.assert_allclose(dKg, dKm.reshape(10, 2, G, 4).sum(axis=2), atol=1e-12)
    np.testing.assert_allclose(dVg, dVm.reshape(10, 2, G, 4).sum(axis=2), atol=1e-12)


# ------------------------------------------------------------ finite differences
FD_CASES = cases.tiny_all(S=10, d=4)


@pytest.mark.parametrize("prob", FD_CASES, ids=[p.name for p in FD_CASES])
def test_backward_matches_central_differences(prob):
    """L = sum(O * dO); dL/dQ, dL/dK, dL/dV by central differences, h = 1e-6."""
    if prob.Tq > 16 or prob.d > 8:
        pytest.skip("finite differences only on tiny shapes")
    q, k, v, do = _rand(prob, 15, scale=0.7)
    dQ, dK, dV = oracle.attention_backward(prob, q, k, v, do)

    def loss(qq, kk, vv):
        O, _ = oracle.attention_forward(prob, qq, kk, vv)
        return float((O * do).sum())

    h = 1e-6
    for arr, grad, which in [(q, dQ, 0), (k, dK, 1), (v, dV, 2)]:
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.linalg.norm(num - grad) / max(np.linalg.norm(grad), 1e-30)
        assert err < 1e-6, (which, err)


# ------------------------------------------------------------ library cross-check
@pytest.mark.parametrize("prob", ALL_TINY, ids=[p.name for p in ALL_TINY])
def test_against_torch_sdpa_fp64(prob):
    torch = pytest.importorskip("torch")
    q, k, v, do = _rand(prob, 16)
    O, L = oracle.attention_forward(prob, q, k, v)
    G = prob.Hq // prob.Hkv
    for h in range(prob.Hq):
        M = brute_dense_mask(prob, h)
        nonempty = M.any(axis=1)
        if not nonempty.any():
            continue
        tq = torch.from_numpy(q[nonempty, h])[None, None]
        tk = torch.from_numpy(k[:, h // G])[None, None]
        tv = torch.from_numpy(v[:, h // G])[None, None]
        tm = torch.from_numpy(M[nonempty])[None, None]
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=tm, scale=prob.softmax_scale)
        np.testing.assert_allclose(O[nonempty, h], ref[0, 0].numpy(), atol=1e-12)


# ------------------------------------------------------------ nnz at full size
def test_mask_counts_at_8k_match_hand_derived():
    from gen import config2

    want = {k: int(v[0]) for k, v in _golden("mask_nnz_8k.txt").items()}
    for kind, n in want.items():
        p = config2(kind, Hq=1, Hkv=1)
        got = int(oracle.mask_row_counts(p).sum())
        assert got == n, (kind, got, n)


# ------------------------------------------------------------ row-local helpers
@pytest.mark.parametrize("prob", ALL_TINY + [cases.shard_problem([7, 12], [[3, 4], [5, 7]])[0]],
                         ids=[p.name for p in ALL_TINY] + ["shards"])
def test_row_local_helpers_match_full_backward(prob):
    """forward_rows / backward_rows / key_grads_from_rows, summed over all rows
    and heads, reproduce the full forward and backward."""
    q, k, v, do = _rand(prob, 17)
    O, L = oracle.attention_forward(prob, q, k, v)
    dQ, dK, dV = oracle.attention_backward(prob, q, k, v, do)
    G = prob.Hq // prob.Hkv
    dK2, dV2 = np.zeros_like(dK), np.zeros_like(dV)
    for s, seg in enumerate(prob.segments):
        rows = np.arange(seg.q_len)
        if seg.q_len == 0:
            continue
        for h in range(prob.Hq):
            o, lse = oracle.forward_rows(prob, q, k, v, s, h, rows)
            np.testing.assert_allclose(o, O[seg.q_off:seg.q_off + seg.q_len, h], atol=1e-12)
            np.testing.assert_allclose(lse, L[h, seg.q_off:seg.q_off + seg.q_len], atol=1e-12)
            dq = oracle.backward_rows(prob, q, k, v, do, s, h, rows)
            np.testing.assert_allclose(dq, dQ[seg.q_off:seg.q_off + seg.q_len, h], atol=1e-12)
            cols = np.arange(seg.k_len)
            # split the rows in two halves to exercise partial sums
            for part in (rows[: len(rows) // 2], rows[len(rows) // 2:]):
                if len(part) == 0:
                    continue
                a, b = oracle.key_grads_from_rows(prob, q, k, v, do, s, h, part, cols)
                dK2[seg.k_off:seg.k_off + seg.k_len, h // G] += a
                dV2[seg.k_off:seg.k_off + seg.k_len, h // G] += b
    np.testing.assert_allclose(dK2, dK, atol=1e-12)
    np.testing.assert_allclose(dV2, dV, atol=1e-12)


# ---------------------------------------------------------------- partial merge
def _partition_forward(rng, nq=37, nk=50, d=8, parts=3, causal=False):
    q, k, v = (rng.standard_normal((n, d)) for n in (nq, nk, nk))
    mask = rng.random((nq, nk)) < 0.6
    if causal:
        mask &= np.tril(np.ones((nq, nk), dtype=bool), nk - nq)
    mask[3] = False  # a row that attends nothing
    owner = rng.integers(0, parts, nk)  # key j belongs to part owner[j]
    owner[: parts] = np.arange(parts)
    full = oracle.segment_head_forward(q, k, v, mask, 0.3)
    pieces = [oracle.segment_head_forward(q, k, v, mask & (owner == p)[None, :], 0.3) for p in range(parts)]
    return full, pieces


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("parts", [1, 2, 5])
def test_merge_of_a_key_partition_is_the_union(parts, causal):
    """Softmax over a union of disjoint key sets from each set's output and
    log-normaliser (exact up to rounding); rows empty in some parts, and a
    row empty in all, included."""
    rng = np.random.Generator(np.random.PCG64(200 + parts + 10 * causal))
    (o_full, l_full, _), pieces = _partition_forward(rng, parts=parts, causal=causal)
    o, l = oracle.merge_partials([p[0][:, None, :] for p in pieces], [p[1][None, :] for p in pieces])
    assert np.array_equal(np.isneginf(l[0]), np.isneginf(l_full))
    fin = np.isfinite(l_full)
    np.testing.assert_allclose(l[0][fin], l_full[fin], rtol=0, atol=1e-12)
    np.testing.assert_allclose(o[:, 0], o_full, rtol=0, atol=1e-12)
    assert np.all(o[3, 0] == 0.0) and np.isneginf(l[0, 3])


def test_merge_worked_example():
    """Two parts of one row, by hand: keys {a} with score 0 and value 1, keys
    {b, c} with scores ln 2, ln 2 and values 4, 7.  Union: weights 1, 2, 2 over
    5 -> O = (1 + 8 + 14) / 5 = 4.6, LSE = ln 5.  Part 1: O = 1, LSE = 0;
    part 2: O = 5.5, LSE = ln 4."""
    o, l = oracle.merge_partials([np.array([[[1.0]]]), np.array([[[5.5]]])],
                                 [np.array([[0.0]]), np.array([[np.log(4.0)]])])
    assert o[0, 0, 0] == pytest.approx(4.6, abs=1e-12)
    assert l[0, 0] == pytest.approx(np.log(5.0), abs=1e-12)
