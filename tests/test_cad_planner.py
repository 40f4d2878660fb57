"""Core-attention disaggregation planner (lca_cad_plan) on CPU.

The planner is host code: it cuts documents into token-level query shards and
assigns them to attention servers so that each server's causal attention work
is balanced ("Efficient Long-context Language Model Training by Core Attention
Disaggregation").  Checked here: a worked example, exact coverage of every
document, shard length bounds, the per-server cell accounting, the balance
rule, argument errors, and -- with gloo ranks standing for the servers, each
computing its own shards with the fp64 oracle -- that the servers' results
reassemble to causal-document attention over all documents."""
from __future__ import annotations

import datetime
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import long_context_masked_attention_gb300 as lca


def _cells(a, b):
    return (b * (b + 1) - a * (a + 1)) // 2


def test_worked_example_cost_midpoint():
    """One document of 10 tokens on 2 servers: rows 0..9 cost 1..10 cells
    (55 in all); the cut at row 7 gives 28 and 27."""
    plan = lca.cad_plan([10], 2, min_shard=1, max_shard=0, tolerance=0.05)
    assert plan.shards == [(0, 0, 7, 0), (0, 7, 3, 1)]
    assert plan.server_cells == [28, 27]


def _pareto_docs(rng, total, lo, hi):
    out, left = [], total
    while left > 0:
        n = int(min(hi, lo * rng.random() ** (-1 / 1.2)))
        n = min(n, left)
        out.append(n)
        left -= n
    return out


@pytest.mark.parametrize("n_servers", [1, 2, 4, 8])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_coverage_bounds_accounting_balance(n_servers, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    docs = _pareto_docs(rng, 200_000, 1024, 200_000) + [300, 0, 5]
    min_s, max_s, tol = 512, 8192, 0.05
    plan = lca.cad_plan(docs, n_servers, min_s, max_s, tol)
    by_doc = {}
    cells = [0] * n_servers
    for doc, start, n, srv in plan.shards:
        by_doc.setdefault(doc, []).append((start, n))
        cells[srv] += _cells(start, start + n)
        assert 0 <= srv < n_servers
        assert n <= max_s
        assert n >= min_s or n == docs[doc], (doc, start, n)  # short documents stay whole
    for d, L in enumerate(docs):
        pieces = sorted(by_doc.get(d, []))
        assert sum(n for _, n in pieces) == L
        pos = 0
        for start, n in pieces:
            assert start == pos
            pos += n
    assert cells == plan.server_cells
    # output order: by server, then document order
    keys = [(srv, doc, start) for doc, start, _, srv in plan.shards]
    assert keys == sorted(keys)
    # balance: within tolerance, or the hottest server holds only shards too short to cut
    mean = sum(cells) / n_servers
    hot = int(np.argmax(cells))
    if cells[hot] > mean * (1 + tol):
        assert all(n < 2 * min_s for _, _, n, srv in plan.shards if srv == hot)


def test_splitting_improves_balance_over_whole_documents():
    rng = np.random.Generator(np.random.PCG64(7))
    docs = _pareto_docs(rng, 500_000, 1024, 500_000)
    whole = lca.cad_plan(docs, 8, 1024, 0, 1e9)  # no cuts: documents only
    cut = lca.cad_plan(docs, 8, 1024, 32768, 0.02)
    ratio = lambda p: max(p.server_cells) / (sum(p.server_cells) / len(p.server_cells))  # noqa: E731
    assert ratio(cut) < ratio(whole)
    assert ratio(cut) <= 1.02 + 1e-9 or ratio(cut) < 1.2


def test_argument_errors():
    with pytest.raises(lca.LcaError):
        lca.cad_plan([100], 0, 1, 0, 0.1)
    with pytest.raises(lca.LcaError):
        lca.cad_plan([100], 2, 64, 100, 0.1)  # max_shard below 2 * min_shard
    with pytest.raises(lca.LcaError):
        lca.cad_plan([-5], 2, 1, 0, 0.1)


# ---------------------------------------------------------------- servers as CPU ranks
DOCS = [300, 257, 143, 500, 64]
HQ, HKV, D = 2, 1, 8


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem_inputs():
    from gen import MaskSpec, Problem, docs_to_segments, make_tensors

    T = sum(DOCS)
    prob = Problem("cad_docs", T, T, HQ, HKV, D, docs_to_segments(DOCS), MaskSpec("CAUSAL_DOC"), 91)
    return prob, make_tensors(prob)


def _server_worker(rank, world, port, out):
    import torch.distributed as dist

    import oracle
    from gen import MaskSpec, Problem, Segment

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=120))
    plan = lca.cad_plan(DOCS, world, 48, 128, 0.05)
    prob, (q, k, v, _) = _problem_inputs()
    segs, rows = plan.server_batch(rank, DOCS)
    mine = Problem("server", len(rows), prob.Tk, HQ, HKV, D, [Segment(*s) for s in segs], MaskSpec("CAUSAL"), 91)
    O, L = oracle.attention_forward(mine, q[rows], k, v)
    gathered = [None] * world
    dist.all_gather_object(gathered, (rows, O, L))
    if rank == 0:
        out["parts"] = gathered
    dist.destroy_process_group()


def test_servers_reassemble_causal_document_attention():
    import oracle

    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_server_worker, args=(3, _free_port(), out), nprocs=3, join=True, start_method="spawn")
    prob, (q, k, v, _) = _problem_inputs()
    O_ref, L_ref = oracle.attention_forward(prob, q, k, v)
    O = np.full_like(O_ref, np.nan)
    L = np.full_like(L_ref, np.nan)
    for rows, o, l in out["parts"]:
        assert np.all(np.isnan(O[rows])), "a row served twice"
        O[rows] = o
        L[:, rows] = l
    assert not np.isnan(O).any(), "a row not served"
    np.testing.assert_allclose(O, O_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, L_ref, rtol=0, atol=1e-12)
