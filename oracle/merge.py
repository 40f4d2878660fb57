"""Merge of partial attention results in fp64 — TEST INFRASTRUCTURE ONLY.

Blockwise and ring attention ("长上下文能力：FlashAttention vs. RingAttention",
Blockwise Parallel Transformer and RingAttention sections) compute a query
block's attention one key block at a time and combine the pieces through the
softmax normalisers.  For disjoint key sets A_1..A_n of a row, with O_p and
LSE_p the attention output and natural-log normaliser over A_p alone, the
exponentials of the union split over the parts, so

    LSE = log sum_p exp(LSE_p)
    O   = sum_p exp(LSE_p - LSE) O_p

A row with every LSE_p = -inf attends no key: O = 0, LSE = -inf.
"""
from __future__ import annotations

import numpy as np


def merge_partials(o_parts, lse_parts):
    """o_parts: list of [Tq, H, d]; lse_parts: list of [H, Tq] -> (O [Tq, H, d], LSE [H, Tq])."""
    o = np.stack([np.asarray(x, dtype=np.float64) for x in o_parts])    # [n, Tq, H, d]
    lse = np.stack([np.asarray(x, dtype=np.float64) for x in lse_parts])  # [n, H, Tq]
    m = lse.max(axis=0)                                                    # [H, Tq]
    has = np.isfinite(m)
    w = np.where(np.isfinite(lse), np.exp(lse - np.where(has, m, 0.0)[None]), 0.0)
    tot = w.sum(axis=0)
    lse_out = np.where(has, np.where(has, m, 0.0) + np.log(np.where(has, tot, 1.0)), -np.inf)
    coef = np.where(has[None], w / np.where(has, tot, 1.0)[None], 0.0)    # [n, H, Tq]
    o_out = np.einsum("nht,nthd->thd", coef, o)
    return o_out, lse_out
