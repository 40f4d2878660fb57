"""The binding makes the tensors' device current around every library call
and takes that device's current stream, whichever device the caller had
selected (the library launches on the current device and refuses pointers
into another device's memory).  Checked without a GPU: the library, the
device context and the stream lookup are replaced by recorders, and the
tensor checks by a pass-through, so the test sees which device each call
asked for and in which order."""
from __future__ import annotations

import contextlib

import pytest
import torch

from gen import MaskSpec, Segment
from long_context_masked_attention_gb300 import binding as B


class _FakeLib:
    def __init__(self, log):
        self.log = log

    def __getattr__(self, name):
        def call(*args):
            self.log.append(("call", name))
            return 0

        return call


@pytest.fixture
def recorder(monkeypatch):
    log = []

    @contextlib.contextmanager
    def on_device(dev):
        log.append(("enter", None if dev is None else str(dev)))
        yield
        log.append(("exit", None if dev is None else str(dev)))

    def stream(stream, device=None):
        log.append(("stream", None if device is None else str(device)))
        return None

    monkeypatch.setattr(B, "load", lambda path=B.LIB_PATH: _FakeLib(log))
    monkeypatch.setattr(B, "_on_device", on_device)
    monkeypatch.setattr(B, "_stream", stream)
    monkeypatch.setattr(B, "_require", lambda t, *a, **kw: t)
    monkeypatch.setattr(B, "workspace_size", lambda call, for_bwd: 256)
    return log


def _calls(log, name):
    """The device entered, and the device whose stream was taken, around
    library call `name`."""
    i = log.index(("call", name))
    enter = max(j for j in range(i) if log[j][0] == "enter")
    stream = max(j for j in range(i) if log[j][0] == "stream")
    assert enter < stream < i < log.index(("exit", log[enter][1]), i), log
    return log[enter][1], log[stream][1]


def test_fwd_bwd_run_on_the_tensors_device(recorder):
    T, segs, mask = 128, [Segment(0, 128, 0, 128)], MaskSpec("CAUSAL")
    q = torch.zeros(T, 2, 128, dtype=torch.bfloat16)
    k = torch.zeros(T, 1, 128, dtype=torch.bfloat16)
    o, lse = B.attn_fwd(q, k, k, segs, mask)
    assert _calls(recorder, "lca_attn_fwd") == (str(q.device), str(q.device))
    B.attn_bwd(q, q, k, k, o, lse, segs, mask)
    assert _calls(recorder, "lca_attn_bwd") == (str(q.device), str(q.device))
    B.attn_fwd(q, k, k, segs, mask, dropout=(1, 0.1))
    assert _calls(recorder, "lca_attn_fwd_dropout") == (str(q.device), str(q.device))


def test_merge_and_hooks_run_on_the_tensors_device(recorder):
    o = torch.zeros(64, 2, 128, dtype=torch.bfloat16)
    lse = torch.zeros(2, 64, dtype=torch.float32)
    B.attn_merge([o, o], [lse, lse])
    assert _calls(recorder, "lca_attn_merge") == (str(o.device), str(o.device))
    ws = torch.zeros(256, dtype=torch.uint8)
    B.probe_wait_timeout(ws, 10)
    assert _calls(recorder, "lca_probe_wait_timeout") == (str(ws.device), str(ws.device))


def test_device_context_selects_only_cuda_devices():
    assert isinstance(B._on_device(None), contextlib.nullcontext)
    assert isinstance(B._on_device(torch.device("cpu")), contextlib.nullcontext)
    ctx = B._on_device(torch.device("cuda", 1))
    assert isinstance(ctx, torch.cuda.device) and ctx.idx == 1
