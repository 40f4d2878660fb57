"""Pins of the oracle's attention dropout (FlashAttention review page,
FlashAttention-1 核心优化, 算子融合: dropout fused with the matmuls, the mask
and the softmax).

The random bits are pinned to the generator's published definition through
its known-answer vectors; the keep decision, its byte and word order and the
scaling are pinned by direct extraction, by exact frequencies and by
statistics; the forward by p = 0 reducing to plain attention and by the
dropout average converging to it; the backward by central differences and
by torch autograd through the dropped probabilities."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from gen import MaskSpec, Problem, Segment, docs_to_segments
from oracle.dropout import philox4x32_10, keep_mask, keep_scale, drop_threshold
from tests import cases

# Known-answer vectors of Philox4x32-10 distributed with the generator's
# reference implementation (Random123, kat_vectors: counter, key -> output).
PHILOX_KAT = [
    ((0x00000000, 0x00000000, 0x00000000, 0x00000000), (0x00000000, 0x00000000),
     (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF), (0xFFFFFFFF, 0xFFFFFFFF),
     (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,want", PHILOX_KAT)
def test_philox_known_answers(ctr, key, want):
    got = philox4x32_10(np.array(ctr, dtype=np.uint64), key)
    assert [int(x) for x in got] == list(want)


def test_philox_vectorised_equals_scalar_calls():
    rng = np.random.Generator(np.random.PCG64(3))
    ctr = rng.integers(0, 2**32, size=(7, 5, 4), dtype=np.uint64)
    out = philox4x32_10(ctr, (0x1234, 0xABCDEF))
    for idx in [(0, 0), (3, 2), (6, 4)]:
        assert np.array_equal(out[idx], philox4x32_10(ctr[idx], (0x1234, 0xABCDEF)))


def test_threshold_and_scale():
    assert drop_threshold(0.0) == 0 and keep_scale(0.0) == 1.0
    assert drop_threshold(0.1) == 26 and keep_scale(0.1) == 256.0 / 230
    assert drop_threshold(0.5) == 128 and keep_scale(0.5) == 2.0
    assert drop_threshold(0.999) == 255  # capped: at least 1/256 is kept
    assert drop_threshold(1.5 / 256) == 2  # half-way rounds up


def test_keep_bit_is_the_documented_byte():
    """Key j of row i, head h keeps iff byte j % 4 of word (j % 16) // 4 of
    Philox(counter = (j // 16, i, h, 0), key = seed words) is >= t."""
    seed, p, h = 0x0123456789ABCDEF, 0.3, 5
    t = drop_threshold(p)
    rows = np.array([0, 7, 1000, 123457])
    cols = np.arange(64)
    got = keep_mask(seed, p, h, rows, cols)
    for a, i in enumerate(rows):
        for j in cols:
            w = philox4x32_10(np.array([j // 16, i, h, 0], dtype=np.uint64),
                              (seed & 0xFFFFFFFF, seed >> 32))[(j % 16) // 4]
            byte = (int(w) >> (8 * (j % 4))) & 0xFF
            assert got[a, j] == (byte >= t)


def test_keep_mask_of_a_sub_block_is_the_slice():
    seed, p, h = 99, 0.2, 3
    rows, cols = np.arange(40, 90), np.arange(300)
    full = keep_mask(seed, p, h, rows, cols)
    sub = keep_mask(seed, p, h, rows[5:17], cols[37:211])
    assert np.array_equal(sub, full[5:17, 37:211])


@pytest.mark.parametrize("p", [0.05, 0.1, 0.5, 0.9])
def test_keep_frequency_and_independence(p):
    """Kept fraction within 5 sigma of k = (256 - t) / 256 over 2^20 draws;
    neighbouring keys, rows and heads are uncorrelated."""
    k = (256 - drop_threshold(p)) / 256
    z = keep_mask(2024, p, 0, np.arange(1024), np.arange(1024)).astype(np.float64)
    n = z.size
    assert abs(z.mean() - k) < 5 * np.sqrt(k * (1 - k) / n)
    z2 = keep_mask(2024, p, 1, np.arange(1024), np.arange(1024)).astype(np.float64)
    for a, b in [(z[:, :-1], z[:, 1:]), (z[:-1], z[1:]), (z, z2), (z[:, :-16], z[:, 16:])]:
        c = np.corrcoef(a.ravel(), b.ravel())[0, 1]
        assert abs(c) < 5 / np.sqrt(a.size), c


def test_bytes_are_uniform():
    """Chi-square of the 256 byte values over 2^18 bytes (p-value > 1e-4)."""
    from scipy.stats import chi2

    ctr = np.zeros((16384, 4), dtype=np.uint64)
    ctr[:, 0] = np.arange(16384)
    ctr[:, 1] = 77
    words = philox4x32_10(ctr, (5, 6)).ravel()
    b = np.concatenate([(words >> np.uint32(8 * s)) & np.uint32(0xFF) for s in range(4)])
    cnt = np.bincount(b.astype(np.int64), minlength=256)
    e = b.size / 256
    stat = ((cnt - e) ** 2 / e).sum()
    assert chi2.sf(stat, 255) > 1e-4


def _rand(prob, seed=0, scale=1.0):
    r = np.random.Generator(np.random.PCG64(seed))
    q = r.standard_normal((prob.Tq, prob.Hq, prob.d)) * scale
    k = r.standard_normal((prob.Tk, prob.Hkv, prob.d)) * scale
    v = r.standard_normal((prob.Tk, prob.Hkv, prob.d))
    do = r.standard_normal((prob.Tq, prob.Hq, prob.d))
    return q, k, v, do


TINY = cases.tiny_all(S=10, d=4)


@pytest.mark.parametrize("prob", TINY[:6], ids=[p.name for p in TINY[:6]])
def test_p_zero_is_plain_attention(prob):
    q, k, v, do = _rand(prob, 4)
    O, L = oracle.attention_forward(prob, q, k, v)
    Od, Ld = oracle.attention_forward(prob, q, k, v, dropout=(7, 0.0))
    assert np.array_equal(O, Od) and np.array_equal(L, Ld)
    for a, b in zip(oracle.attention_backward(prob, q, k, v, do),
                    oracle.attention_backward(prob, q, k, v, do, dropout=(7, 0.0))):
        assert np.array_equal(a, b)


def test_lse_unchanged_and_dropped_cells_are_exact():
    """LSE is that of the undropped softmax; O equals sum over kept keys of
    P_ij / k v_j, with P from the undropped softmax."""
    prob = Problem("drop_causal", 40, 40, 2, 1, 8, [Segment(0, 40, 0, 40)], MaskSpec("CAUSAL"), 1)
    q, k, v, _ = _rand(prob, 9)
    seed, p = 31, 0.25
    O, L = oracle.attention_forward(prob, q, k, v)
    Od, Ld = oracle.attention_forward(prob, q, k, v, dropout=(seed, p))
    assert np.array_equal(L, Ld)
    for h in range(2):
        z = keep_mask(seed, p, h, np.arange(40), np.arange(40))
        s = (q[:, h] @ k[:, 0].T) / np.sqrt(8)
        P = np.exp(s - L[h][:, None]) * np.tril(np.ones((40, 40)))
        want = (P * z * keep_scale(p)) @ v[:, 0]
        np.testing.assert_allclose(Od[:, h], want, rtol=1e-12, atol=1e-12)
        assert not np.allclose(Od[:, h], O[:, h])


def test_dropout_average_is_unbiased():
    """E over seeds of the dropped output is the undropped output: the mean
    of 600 seeds lies within 5 standard errors everywhere."""
    prob = Problem("drop_avg", 12, 12, 1, 1, 4, [Segment(0, 12, 0, 12)], MaskSpec("FULL"), 1)
    q, k, v, _ = _rand(prob, 2)
    O, _ = oracle.attention_forward(prob, q, k, v)
    outs = np.stack([oracle.attention_forward(prob, q, k, v, dropout=(s, 0.3))[0] for s in range(600)])
    se = outs.std(axis=0) / np.sqrt(len(outs))
    assert np.all(np.abs(outs.mean(axis=0) - O) <= 5 * se + 1e-12)


def test_rows_use_global_row_index_and_segment_keys():
    """Two documents packed in one batch: each document's Z is that of its
    own global rows and of keys counted from the document's first key."""
    segs = docs_to_segments([30, 50])
    prob = Problem("drop_docs", 80, 80, 1, 1, 8, segs, MaskSpec("CAUSAL_DOC"), 1)
    q, k, v, _ = _rand(prob, 6)
    seed, p = 5, 0.4
    Od, L = oracle.attention_forward(prob, q, k, v, dropout=(seed, p))
    rows = np.arange(30, 80)
    z = keep_mask(seed, p, 0, rows, np.arange(50))
    s = (q[30:, 0] @ k[30:, 0].T) / np.sqrt(8)
    P = np.exp(s - L[0, 30:][:, None]) * np.tril(np.ones((50, 50)))
    np.testing.assert_allclose(Od[30:, 0], (P * z * keep_scale(p)) @ v[30:, 0], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("prob", TINY[:8], ids=[p.name for p in TINY[:8]])
def test_backward_with_dropout_matches_central_differences(prob):
    if prob.Tq > 16 or prob.d > 8:
        pytest.skip("finite differences only on tiny shapes")
    drop = (11, 0.3)
    q, k, v, do = _rand(prob, 21, scale=0.7)
    dQ, dK, dV = oracle.attention_backward(prob, q, k, v, do, dropout=drop)

    def loss(qq, kk, vv):
        O, _ = oracle.attention_forward(prob, qq, kk, vv, dropout=drop)
        return float((O * do).sum())

    h = 1e-6
    for arr, grad, which in [(q, dQ, 0), (k, dK, 1), (v, dV, 2)]:
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            ap = [q.copy(), k.copy(), v.copy()]
            am = [q.copy(), k.copy(), v.copy()]
            ap[which][idx] += h
            am[which][idx] -= h
            num[idx] = (loss(*ap) - loss(*am)) / (2 * h)
        err = np.linalg.norm(num - grad) / max(np.linalg.norm(grad), 1e-30)
        assert err < 1e-6, (which, err)


def test_backward_with_dropout_matches_torch_autograd():
    """Autograd of O = (softmax(masked S) * Z / k) V in fp64 torch, with the
    oracle's Z, against the oracle's closed-form backward."""
    import torch

    segs = docs_to_segments([23, 41])
    prob = Problem("drop_autograd", 64, 64, 4, 2, 16, segs, MaskSpec("CAUSAL_DOC"), 1)
    q, k, v, do = _rand(prob, 13)
    drop = (0xDEADBEEF12345678, 0.15)
    dQ, dK, dV = oracle.attention_backward(prob, q, k, v, do, dropout=drop)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    out = torch.zeros(64, 4, 16, dtype=torch.float64)
    for h in range(4):
        g = h // 2
        for seg in segs:
            qs = slice(seg.q_off, seg.q_off + seg.q_len)
            ks = slice(seg.k_off, seg.k_off + seg.k_len)
            s = tq[qs, h] @ tk[ks, g].T / 4.0
            causal = torch.tril(torch.ones(seg.q_len, seg.k_len, dtype=torch.bool))
            P = torch.softmax(s.masked_fill(~causal, float("-inf")), dim=-1)
            z = keep_mask(drop[0], drop[1], h, seg.q_off + np.arange(seg.q_len), np.arange(seg.k_len))
            zk = torch.tensor(z * keep_scale(drop[1]))
            out[qs, h] = (P * zk) @ tv[ks, g]
    (out * torch.tensor(do)).sum().backward()
    for got, want in ((dQ, tq.grad), (dK, tk.grad), (dV, tv.grad)):
        np.testing.assert_allclose(got, want.numpy(), rtol=1e-10, atol=1e-12)


def test_row_helpers_with_dropout_match_full():
    prob = Problem("drop_rows", 50, 70, 2, 1, 8, [Segment(0, 50, 0, 70)], MaskSpec("CAUSAL"), 1)
    q, k, v, do = _rand(prob, 8)
    drop = (3, 0.2)
    O, L = oracle.attention_forward(prob, q, k, v, dropout=drop)
    dQ, dK, dV = oracle.attention_backward(prob, q, k, v, do, heads=[1], dropout=drop)
    rows = np.array([0, 7, 31, 49])
    o, l = oracle.forward_rows(prob, q, k, v, 0, 1, rows, dropout=drop)
    np.testing.assert_allclose(o, O[rows, 1], rtol=1e-12, atol=1e-12)
    dq = oracle.backward_rows(prob, q, k, v, do, 0, 1, rows, dropout=drop)
    np.testing.assert_allclose(dq, dQ[rows, 1], rtol=1e-12, atol=1e-12)
    dk, dv = oracle.key_grads_from_rows(prob, q, k, v, do, 0, 1, np.arange(50), np.array([0, 33, 69]), dropout=drop)
    np.testing.assert_allclose(dk, dK[[0, 33, 69], 0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, dV[[0, 33, 69], 0], rtol=1e-10, atol=1e-12)
