"""Seeded synthetic inputs for the masked-attention workloads.

This module is shared by the CPU oracle tests, the GPU parity tests and the
benchmark.  It draws random numbers and lays out documents, shards and block
maps; it holds none of the attention or mask arithmetic (no scores, no
softmax, no mask predicates).

Workloads follow the long-context attention benchmark review
("Long-Context Attention Benchmark: From Kernel Efficiency to Distributed
Context Parallelism", section 三 技术架构 / 评估设置: BF16, head dim 128,
GQA 64:8 and MHA 64:64, 1K-48K dense, 32K-128K sparse) and the
core-attention-disaggregation summary ("Efficient Long-context Language Model
Training by Core Attention Disaggregation", 方法详解: token-level shards of
arbitrary length rebatched into one fused launch).  The pages' datasets
(Pile, ProLong64K, ProLong512K) are not available; the seeded length
distributions below stand in for them.
"""
from __future__ import annotations

from dataclasses import dataclass, field
import math

import numpy as np

MASK_KINDS = (
    "FULL",
    "CAUSAL",
    "SLIDING",
    "CAUSAL_SLIDING",
    "DOC",
    "CAUSAL_DOC",
    "SHARED_QUESTION",
    "GLOBAL_SLIDING",
    "CAUSAL_BLOCKWISE",
    "PREFIX_LM_CAUSAL",
    "PREFIX_LM_DOC",
    "BLOCK_CAUSAL_DOC",
    "BLOCK_SPARSE_UNIFORM",
    "BLOCK_SPARSE_VARIABLE",
    "FLASHMASK",
)
STATIC_KINDS = MASK_KINDS[:12]
KIND_ID = {k: i for i, k in enumerate(MASK_KINDS)}


@dataclass
class Segment:
    """One packed unit of work: query rows [q_off, q_off+q_len) attend keys
    [k_off, k_off+k_len).  Causal families align the diagonal bottom-right."""

    q_off: int
    q_len: int
    k_off: int
    k_len: int


@dataclass
class MaskSpec:
    """Parameters of one mask family (the structure, not the predicate)."""

    kind: str
    window_left: int = 0
    window_right: int = 0
    num_global: int = 0
    prefix_len: int = 0
    seg_prefix: list | None = None  # PREFIX_LM_DOC: per-segment prefix length
    block: int = 0  # CAUSAL_BLOCKWISE, BLOCK_CAUSAL_DOC
    part_bounds: list | None = None  # SHARED_QUESTION, key positions in a segment
    # block-sparse maps (token positions are global packed positions)
    q_block: int = 0
    kv_block: int = 0
    qb_bounds: np.ndarray | None = None  # variable: int32 [n_qb + 1]
    kb_bounds: np.ndarray | None = None  # variable: int32 [n_kb + 1]
    heads_in_map: int = 1
    blk_row_ptr: np.ndarray | None = None  # int32 [heads_in_map * n_qb + 1]
    blk_col_idx: np.ndarray | None = None  # int32 [nnz blocks], sorted per row
    col_bounds: np.ndarray | None = None  # FLASHMASK: int32 [Tk, 4] {lts, lte, uts, ute}

    def n_qb(self, Tq: int) -> int:
        if self.kind == "BLOCK_SPARSE_UNIFORM":
            return -(-Tq // self.q_block)
        return len(self.qb_bounds) - 1

    def n_kb(self, Tk: int) -> int:
        if self.kind == "BLOCK_SPARSE_UNIFORM":
            return -(-Tk // self.kv_block)
        return len(self.kb_bounds) - 1


@dataclass
class Problem:
    name: str
    Tq: int
    Tk: int
    Hq: int
    Hkv: int
    d: int
    segments: list
    mask: MaskSpec
    seed: int
    scale: float = 0.0  # 0 -> 1/sqrt(d)
    extra: dict = field(default_factory=dict)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale != 0.0 else 1.0 / math.sqrt(self.d)


# ----------------------------------------------------------------- random values
def make_tensors(prob: Problem, device="cpu", with_grad_out=True):
    """Q, K, V (and dO) i.i.d. N(0,1) drawn in fp32 and rounded to bf16.

    Layout is token-major packed: Q/dO [Tq, Hq, d], K/V [Tk, Hkv, d].
    Seeds: 16*seed + {1: q, 2: k, 3: v, 4: dO}.  CPU and CUDA generators give
    different streams; a test that needs the same values on both sides draws
    them once and copies.
    """
    import torch

    def draw(shape, sub):
        g = torch.Generator(device=device)
        g.manual_seed(16 * prob.seed + sub)
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)

    q = draw((prob.Tq, prob.Hq, prob.d), 1)
    k = draw((prob.Tk, prob.Hkv, prob.d), 2)
    v = draw((prob.Tk, prob.Hkv, prob.d), 3)
    do = draw((prob.Tq, prob.Hq, prob.d), 4) if with_grad_out else None
    return q, k, v, do


# ----------------------------------------------------------------- length samplers
def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def fill_lengths(total: int, draw) -> list:
    """Draw lengths until `total` is covered; the last one is cut to fit."""
    out, used = [], 0
    while used < total:
        n = int(draw())
        n = max(1, min(n, total - used))
        out.append(n)
        used += n
    return out


def loguniform_docs(total: int, lo: int, hi: int, rng) -> list:
    """floor(exp(U(ln lo, ln hi))) per document."""
    return fill_lengths(total, lambda: math.floor(math.exp(rng.uniform(math.log(lo), math.log(hi)))))


def mixture_docs(total: int, S: int, rng) -> list:
    """70% U{256..4096}, 30% U{4096..S}; each clipped to the space left."""

    def draw():
        if rng.random() < 0.7:
            return rng.integers(256, 4096, endpoint=True)
        return rng.integers(min(4096, S), S, endpoint=True)

    return fill_lengths(total, draw)


def pareto_docs(total: int, alpha: float, xm: int, hi: int, rng) -> list:
    """floor(xm * U^(-1/alpha)) clipped to [xm, hi]."""

    def draw():
        u = 1.0 - rng.random()  # (0, 1]
        return min(hi, max(xm, math.floor(xm * u ** (-1.0 / alpha))))

    return fill_lengths(total, draw)


def docs_to_segments(lengths, base: int = 0) -> list:
    segs, off = [], base
    for n in lengths:
        segs.append(Segment(off, n, off, n))
        off += n
    return segs


# ----------------------------------------------------------------- block maps
def uniform_block_map(n_qb: int, n_kb: int, heads: int, rng):
    """Per (head, q-block): keep ceil(n_kb/2) kv blocks — the diagonal block
    (index min(qb, n_kb-1)) plus ceil(n_kb/2)-1 others drawn without
    replacement.  Returns CSR (row_ptr, col_idx) over heads*n_qb rows."""
    keep = -(-n_kb // 2)
    rows = []
    for _h in range(heads):
        keys = rng.random((n_qb, n_kb))
        diag = np.minimum(np.arange(n_qb), n_kb - 1)
        keys[np.arange(n_qb), diag] = -1.0  # always first
        sel = np.argpartition(keys, keep - 1, axis=1)[:, :keep]
        sel.sort(axis=1)
        rows.append(sel.astype(np.int32))
    col = np.concatenate([r.reshape(-1) for r in rows])
    row_ptr = (np.arange(heads * n_qb + 1, dtype=np.int64) * keep).astype(np.int32)
    return row_ptr, col


def variable_block_bounds(total: int, lo: int, hi: int, rng) -> np.ndarray:
    lengths = fill_lengths(total, lambda: rng.integers(lo, hi, endpoint=True))
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def variable_block_map(n_qb: int, n_kb: int, heads: int, rng):
    """Per (head, q-block): keep max(1, round(n_kb/2)) kv blocks drawn without
    replacement (no forced diagonal: q and kv boundaries differ)."""
    keep = max(1, int(round(n_kb / 2)))
    rows = []
    for _h in range(heads):
        keys = rng.random((n_qb, n_kb))
        sel = np.argpartition(keys, keep - 1, axis=1)[:, :keep]
        sel.sort(axis=1)
        rows.append(sel.astype(np.int32))
    col = np.concatenate([r.reshape(-1) for r in rows])
    row_ptr = (np.arange(heads * n_qb + 1, dtype=np.int64) * keep).astype(np.int32)
    return row_ptr, col


# ----------------------------------------------------------------- workloads
D_HEAD = 128


def static_mask_spec(kind: str, seg_lengths=None) -> MaskSpec:
    """Mask parameters of the 8K static sweep: windows of 1024 (full +-512,
    causal 1024 back), shared question 1024 + 4 answers of 1792, 64 global
    tokens, causal blockwise 1024, prefix 2048, block-causal-document 512."""
    if kind in ("FULL", "CAUSAL", "DOC", "CAUSAL_DOC"):
        return MaskSpec(kind)
    if kind == "SLIDING":
        return MaskSpec(kind, window_left=512, window_right=512)
    if kind == "CAUSAL_SLIDING":
        return MaskSpec(kind, window_left=1024, window_right=0)
    if kind == "SHARED_QUESTION":
        return MaskSpec(kind, part_bounds=[0, 1024, 2816, 4608, 6400, 8192])
    if kind == "GLOBAL_SLIDING":
        return MaskSpec(kind, num_global=64, window_left=512, window_right=512)
    if kind == "CAUSAL_BLOCKWISE":
        return MaskSpec(kind, block=1024)
    if kind == "PREFIX_LM_CAUSAL":
        return MaskSpec(kind, prefix_len=2048)
    if kind == "PREFIX_LM_DOC":
        return MaskSpec(kind, prefix_len=2048, seg_prefix=[min(2048, n) for n in seg_lengths])
    if kind == "BLOCK_CAUSAL_DOC":
        return MaskSpec(kind, block=512)
    raise ValueError(kind)


DOC_KINDS = ("DOC", "CAUSAL_DOC", "PREFIX_LM_DOC", "BLOCK_CAUSAL_DOC")


def config1(kind: str = "CAUSAL") -> Problem:
    """Smallest instance: one sequence of 1024, 8 q heads / 2 kv heads."""
    S = 1024
    return Problem(f"c1_{kind.lower()}", S, S, 8, 2, D_HEAD, [Segment(0, S, 0, S)], MaskSpec(kind), seed=1)


def config2(kind: str, S: int = 8192, Hq: int = 64, Hkv: int = 8) -> Problem:
    """Static-mask sweep at 8K, GQA 64:8.  Document families take documents
    from a log-uniform length law over [128, 8192] filling the sequence."""
    if kind in DOC_KINDS:
        lengths = loguniform_docs(S, 128, 8192, _rng(2))
        segs = docs_to_segments(lengths)
    else:
        lengths = [S]
        segs = [Segment(0, S, 0, S)]
    return Problem(f"c2_{kind.lower()}", S, S, Hq, Hkv, D_HEAD, segs, static_mask_spec(kind, lengths), seed=2)


def config3(S: int, heads: str = "gqa", kind: str = "CAUSAL", total: int = 49152) -> Problem:
    """Dense length sweep: B = floor(total/S) sequences of S tokens.  CAUSAL
    uses one segment per sequence; CAUSAL_DOC packs documents drawn from the
    70/30 mixture inside each sequence."""
    Hq, Hkv = (64, 8) if heads == "gqa" else (64, 64)
    B = max(1, total // S)
    rng = _rng(3 + 1000 * S)
    segs = []
    for b in range(B):
        if kind == "CAUSAL":
            segs.append(Segment(b * S, S, b * S, S))
        else:
            segs += docs_to_segments(mixture_docs(S, S, rng), base=b * S)
    T = B * S
    return Problem(f"c3_{kind.lower()}_{S // 1024}k_{heads}", T, T, Hq, Hkv, D_HEAD, segs, MaskSpec(kind), seed=3)


def config4(S: int, heads: str = "gqa", variant: str = "uniform128") -> Problem:
    """Block-sparse at 32K-128K: uniform block 64/128 keeping 50% of kv blocks
    per (head, q-block) including the diagonal, or variable blocks with
    boundaries from U{32..256} keeping 50% of block pairs."""
    Hq, Hkv = (64, 8) if heads == "gqa" else (64, 64)
    rng = _rng(4 + 1000 * S + (0 if variant.startswith("uniform") else 7))
    if variant.startswith("uniform"):
        b = int(variant[len("uniform"):])
        n = -(-S // b)
        row_ptr, col = uniform_block_map(n, n, Hq, rng)
        spec = MaskSpec("BLOCK_SPARSE_UNIFORM", q_block=b, kv_block=b, heads_in_map=Hq,
                        blk_row_ptr=row_ptr, blk_col_idx=col)
    else:
        qb = variable_block_bounds(S, 32, 256, rng)
        kb = variable_block_bounds(S, 32, 256, rng)
        row_ptr, col = variable_block_map(len(qb) - 1, len(kb) - 1, Hq, rng)
        spec = MaskSpec("BLOCK_SPARSE_VARIABLE", qb_bounds=qb, kb_bounds=kb, heads_in_map=Hq,
                        blk_row_ptr=row_ptr, blk_col_idx=col)
    return Problem(f"c4_{variant}_{S // 1024}k_{heads}", S, S, Hq, Hkv, D_HEAD, [Segment(0, S, 0, S)], spec, seed=4)


def shard_layout(doc_lengths, shard_lo: int, shard_hi: int, rng, shuffle: bool = True):
    """Cut each document into token-level shards of U{shard_lo..shard_hi}
    query tokens (last one cut to fit).  Shard [a, b) of a document starting
    at key offset s attends keys [s, s+b) bottom-right causally.  Shards are
    packed into the query buffer in a seeded shuffled order; K/V stay packed
    in document order (read in place)."""
    shards = []
    off = 0
    for n in doc_lengths:
        a = 0
        for L in fill_lengths(n, lambda: rng.integers(shard_lo, shard_hi, endpoint=True)):
            shards.append((off, a, L))  # doc start, start within doc, length
            a += L
        off += n
    order = rng.permutation(len(shards)) if shuffle else np.arange(len(shards))
    segs, qpos, src = [], 0, []
    for idx in order:
        doc_start, a, L = shards[idx]
        segs.append(Segment(qpos, L, doc_start, a + L))
        src.append(doc_start + a)  # where these query rows sit in document order
        qpos += L
    return segs, np.asarray(src, dtype=np.int64)


def config5(total: int = 524288, Hq: int = 64, Hkv: int = 8, shard_lo: int = 1024, shard_hi: int = 32768,
            doc_lo: int = 1024) -> Problem:
    """Core-attention shard batch: Pareto(1.2) documents clipped to
    [1K, total], cut into U{1K..32K} shards, rebatched into one launch."""
    rng = _rng(5 + total)
    docs = pareto_docs(total, 1.2, doc_lo, total, rng)
    segs, src = shard_layout(docs, shard_lo, shard_hi, rng)
    p = Problem(f"c5_shards_{total // 1024}k", total, total, Hq, Hkv, D_HEAD, segs, MaskSpec("CAUSAL"), seed=5)
    p.extra["doc_lengths"] = docs
    p.extra["shard_src"] = src
    return p
