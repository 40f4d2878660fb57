"""CPU fp64 oracle for masked core attention — TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
this package.  The product path (the CUDA library and its binding) never
imports it and shares no code with it; the two meet only through the seeded
input generators in ``gen``.

What it computes is the plain definition of attention from the FlashAttention
review page ("长上下文能力：FlashAttention vs. RingAttention", FlashAttention-1
问题和瓶颈: Attention(Q,K,V) = softmax(QK^T/sqrt(d_k)) V), restricted by an
explicit dense boolean mask built from per-(i, j) predicates for the mask
families that the LongCA-bench review lists (section 三 技术架构, 掩码模式分类).
The backward pass is the textbook softmax-attention gradient (FlashAttention-2
核心优化: the single stored row statistic, and dQ_i = sum_j dS_ij K_j).

Precision: fp64 throughout; bf16 inputs are widened exactly.

Parity status: every function here is pinned by tests/test_oracle_*.py
(closed forms, invariants, equivalences between families, brute-force mask
constructions, finite differences and an independent library cross-check).
"""
from .masks import segment_mask, mask_row_counts, dense_mask  # noqa: F401
from .merge import merge_partials  # noqa: F401
from .dropout import philox4x32_10, keep_mask, keep_scale, drop_threshold  # noqa: F401
from .attention import (  # noqa: F401
    attention_forward,
    attention_backward,
    forward_rows,
    backward_rows,
    key_grads_from_rows,
    segment_head_forward,
    segment_head_backward,
)
