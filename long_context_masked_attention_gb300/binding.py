"""Thin ctypes binding of liblca_attn.so (include/lca_attn.h).

Argument marshalling only: it builds the C structs, allocates outputs and the
workspace with PyTorch when the caller does not pass them, and calls the
library on the current CUDA stream.  Every step of the attention path runs in
the library's kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass, field

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liblca_attn.so")

MASK_KINDS = (
    "FULL", "CAUSAL", "SLIDING", "CAUSAL_SLIDING", "DOC", "CAUSAL_DOC", "SHARED_QUESTION", "GLOBAL_SLIDING",
    "CAUSAL_BLOCKWISE", "PREFIX_LM_CAUSAL", "PREFIX_LM_DOC", "BLOCK_CAUSAL_DOC", "BLOCK_SPARSE_UNIFORM",
    "BLOCK_SPARSE_VARIABLE", "FLASHMASK",
)
STATUS = {0: "LCA_OK", 1: "LCA_ERR_INVALID_ARG", 2: "LCA_ERR_UNSUPPORTED", 3: "LCA_ERR_WORKSPACE",
          4: "LCA_ERR_CUDA", 5: "LCA_ERR_TIMEOUT", 6: "LCA_ERR_DEVICE_ARG"}
EXPORTED = ("lca_workspace_size", "lca_attn_fwd", "lca_attn_bwd", "lca_mask_materialize", "lca_mask_tile_classes",
            "lca_mask_nnz", "lca_read_status", "lca_probe_wait_timeout", "lca_set_kernel_events", "lca_launch_count",
            "lca_last_error_detail", "lca_attn_fwd_static_workspace", "lca_status_string", "lca_version",
            "lca_attn_merge", "lca_cad_plan", "lca_attn_fwd_dropout", "lca_attn_bwd_dropout", "lca_set_cta_profile")
PHASES = ("fwd_plan", "fwd", "d_prepass", "dkv_plan", "dkv", "dq_plan", "dq")


class LcaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)}")
        self.code = code


class Segment_t(C.Structure):
    _fields_ = [("q_off", C.c_int32), ("q_len", C.c_int32), ("k_off", C.c_int32), ("k_len", C.c_int32)]


class MaskDesc_t(C.Structure):
    _fields_ = [
        ("kind", C.c_int32),
        ("window_left", C.c_int32), ("window_right", C.c_int32),
        ("num_global", C.c_int32),
        ("prefix_len", C.c_int32),
        ("seg_prefix", C.POINTER(C.c_int32)),
        ("block", C.c_int32),
        ("part_bounds", C.POINTER(C.c_int32)),
        ("n_part_bounds", C.c_int32),
        ("q_block", C.c_int32), ("kv_block", C.c_int32),
        ("qb_bounds", C.POINTER(C.c_int32)), ("kb_bounds", C.POINTER(C.c_int32)),
        ("n_qb", C.c_int32), ("n_kb", C.c_int32),
        ("heads_in_map", C.c_int32),
        ("blk_row_ptr", C.c_void_p), ("blk_col_idx", C.c_void_p),
        ("blk_nnz", C.c_int64),
        ("col_bounds", C.c_void_p),
    ]


class Shape_t(C.Structure):
    _fields_ = [("Tq", C.c_int32), ("Tk", C.c_int32), ("Hq", C.c_int32), ("Hkv", C.c_int32), ("d", C.c_int32),
                ("n_seg", C.c_int32), ("segs", C.POINTER(Segment_t)), ("scale", C.c_float)]


class Dropout_t(C.Structure):
    _fields_ = [("p", C.c_float), ("seed", C.c_uint64)]


_lib = None


def load(path: str = LIB_PATH):
    """Loads the library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with long_context_masked_attention_gb300._build.build()")
    lib = C.CDLL(path)
    st = C.c_int
    vp = C.c_void_p
    lib.lca_workspace_size.argtypes = [C.POINTER(Shape_t), C.POINTER(MaskDesc_t), C.c_int, C.POINTER(C.c_size_t)]
    lib.lca_attn_fwd.argtypes = [vp, vp, vp, vp, vp, C.POINTER(Shape_t), C.POINTER(MaskDesc_t), vp, C.c_size_t, vp]
    lib.lca_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, C.POINTER(Shape_t), C.POINTER(MaskDesc_t), vp,
                                 C.c_size_t, vp]
    lib.lca_attn_fwd_dropout.argtypes = [vp, vp, vp, vp, vp, C.POINTER(Shape_t), C.POINTER(MaskDesc_t),
                                         C.POINTER(Dropout_t), vp, C.c_size_t, vp]
    lib.lca_attn_bwd_dropout.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, C.POINTER(Shape_t),
                                         C.POINTER(MaskDesc_t), C.POINTER(Dropout_t), vp, C.c_size_t, vp]
    lib.lca_mask_materialize.argtypes = [C.POINTER(Shape_t), C.POINTER(MaskDesc_t), C.c_int32, C.c_int32, vp, vp,
                                         C.c_size_t, vp]
    lib.lca_mask_tile_classes.argtypes = lib.lca_mask_materialize.argtypes
    lib.lca_mask_nnz.argtypes = [C.POINTER(Shape_t), C.POINTER(MaskDesc_t), vp, vp, C.c_size_t, vp]
    lib.lca_read_status.argtypes = [vp, C.POINTER(C.c_int32), vp]
    lib.lca_probe_wait_timeout.argtypes = [vp, C.c_size_t, C.c_int32, vp]
    lib.lca_set_kernel_events.argtypes = [C.POINTER(C.c_void_p), C.c_int32, C.POINTER(C.c_int32)]
    lib.lca_set_cta_profile.argtypes = [vp, C.c_size_t]
    lib.lca_launch_count.restype = C.c_uint64
    lib.lca_launch_count.argtypes = []
    lib.lca_attn_fwd_static_workspace.argtypes = [vp, vp, vp, vp, vp, C.POINTER(Shape_t), C.POINTER(MaskDesc_t), vp]
    lib.lca_last_error_detail.restype = C.c_char_p
    lib.lca_last_error_detail.argtypes = []
    lib.lca_status_string.argtypes = [st]
    lib.lca_status_string.restype = C.c_char_p
    lib.lca_version.restype = C.c_int32
    for name in EXPORTED:
        if name not in ("lca_status_string", "lca_version", "lca_launch_count", "lca_last_error_detail"):
            getattr(lib, name).restype = st
    _lib = lib
    return lib


# ------------------------------------------------------------------ descriptors
@dataclass
class Mask:
    """Mask descriptor; attribute names match lca_mask_desc (any object with
    these attributes is accepted too)."""
    kind: str
    window_left: int = 0
    window_right: int = 0
    num_global: int = 0
    prefix_len: int = 0
    seg_prefix: list | None = None
    block: int = 0
    part_bounds: list | None = None
    q_block: int = 0
    kv_block: int = 0
    qb_bounds: np.ndarray | None = None
    kb_bounds: np.ndarray | None = None
    heads_in_map: int = 1
    blk_row_ptr: object = None
    blk_col_idx: object = None
    col_bounds: object = None  # FLASHMASK: int32 [Tk, 4] {lts, lte, uts, ute}


@dataclass
class Call:
    """Marshalled C arguments plus the Python objects they point into."""
    shape: Shape_t
    mask: MaskDesc_t
    keep: list = field(default_factory=list)


def _i32(seq):
    arr = np.ascontiguousarray(np.asarray(seq, dtype=np.int32))
    return arr, arr.ctypes.data_as(C.POINTER(C.c_int32))


def marshal(Tq, Tk, Hq, Hkv, d, segments, mask, scale=0.0, device=None) -> Call:
    """segments: iterable of objects with q_off/q_len/k_off/k_len or 4-tuples."""
    import torch

    segs = list(segments)
    seg_arr = (Segment_t * max(1, len(segs)))()
    for i, s in enumerate(segs):
        if isinstance(s, (tuple, list)):
            seg_arr[i] = Segment_t(*[int(x) for x in s])
        else:
            seg_arr[i] = Segment_t(int(s.q_off), int(s.q_len), int(s.k_off), int(s.k_len))
    shape = Shape_t(int(Tq), int(Tk), int(Hq), int(Hkv), int(d), len(segs), seg_arr, float(scale))
    md = MaskDesc_t()
    keep = [seg_arr]
    kind = mask.kind if isinstance(mask.kind, int) else MASK_KINDS.index(mask.kind)
    md.kind = kind
    md.window_left = int(getattr(mask, "window_left", 0) or 0)
    md.window_right = int(getattr(mask, "window_right", 0) or 0)
    md.num_global = int(getattr(mask, "num_global", 0) or 0)
    md.prefix_len = int(getattr(mask, "prefix_len", 0) or 0)
    md.block = int(getattr(mask, "block", 0) or 0)
    if getattr(mask, "seg_prefix", None) is not None:
        arr, ptr = _i32(mask.seg_prefix)
        keep.append(arr)
        md.seg_prefix = ptr
    if getattr(mask, "part_bounds", None) is not None:
        arr, ptr = _i32(mask.part_bounds)
        keep.append(arr)
        md.part_bounds = ptr
        md.n_part_bounds = len(arr)
    md.q_block = int(getattr(mask, "q_block", 0) or 0)
    md.kv_block = int(getattr(mask, "kv_block", 0) or 0)
    md.heads_in_map = int(getattr(mask, "heads_in_map", 1) or 1)
    for name, cnt in (("qb_bounds", "n_qb"), ("kb_bounds", "n_kb")):
        b = getattr(mask, name, None)
        if b is not None:
            arr, ptr = _i32(b)
            keep.append(arr)
            setattr(md, name, ptr)
            setattr(md, cnt, len(arr) - 1)
    rp = getattr(mask, "blk_row_ptr", None)
    ci = getattr(mask, "blk_col_idx", None)
    if rp is not None:
        dev = device if device is not None else torch.device("cuda")

        def to_dev(x):
            if isinstance(x, torch.Tensor):
                return x.to(device=dev, dtype=torch.int32).contiguous()
            return torch.from_numpy(np.ascontiguousarray(np.asarray(x, dtype=np.int32))).to(dev)

        trp, tci = to_dev(rp), to_dev(ci)
        keep += [trp, tci]
        md.blk_row_ptr = trp.data_ptr()
        md.blk_col_idx = tci.data_ptr() if tci.numel() else None
        md.blk_nnz = int(tci.numel())
    cb = getattr(mask, "col_bounds", None)
    if cb is not None:
        dev = device if device is not None else torch.device("cuda")
        tcb = (cb.to(device=dev, dtype=torch.int32) if isinstance(cb, torch.Tensor)
               else torch.from_numpy(np.ascontiguousarray(np.asarray(cb, dtype=np.int32))).to(dev)).contiguous()
        keep.append(tcb)
        md.col_bounds = tcb.data_ptr()
    return Call(shape, md, keep)


def _check(code, what):
    if code != 0:
        if code == 4:
            what += " (" + load().lca_last_error_detail().decode() + ")"
        raise LcaError(code, what)


def _stream(stream, device=None):
    """The stream handle for a call: the given one, else the current stream
    of `device` (the device the call's tensors live on)."""
    import torch

    if stream is None:
        stream = torch.cuda.current_stream(device)
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _on_device(device):
    """Context that makes `device` the current CUDA device for a library call:
    the library launches on the current device and refuses pointers into
    another device's memory, so every call runs with its tensors' device
    current, whichever device the caller had selected."""
    import contextlib

    import torch

    if device is None or torch.device(device).type != "cuda":
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def workspace_size(call: Call, for_bwd: bool) -> int:
    n = C.c_size_t(0)
    _check(load().lca_workspace_size(C.byref(call.shape), C.byref(call.mask), int(for_bwd), C.byref(n)),
           "lca_workspace_size")
    return n.value


def _workspace(call, for_bwd, workspace, device):
    import torch

    need = workspace_size(call, for_bwd)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    return workspace


# ------------------------------------------------------------------ entry points
def _require(t, name, shape, dtype, device=None, host_ok=False):
    """The library reads and writes raw device pointers, so every tensor is
    checked here: a CUDA tensor of the given dtype, shape and device, laid out
    densely (a host or strided tensor would be read as garbage).  With
    host_ok (outputs the kernels only store to), a pinned host tensor is
    accepted too: the kernels write it through its device mapping."""
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if host_ok and t.device.type == "cpu":
        if not t.is_pinned():
            raise ValueError(f"{name}: must be a CUDA tensor or a pinned host tensor (got unpinned {t.device})")
    elif t.device.type != "cuda":
        raise ValueError(f"{name}: must be a CUDA tensor (got {t.device})")
    elif device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t


def _dropout(dropout):
    """(seed, p) -> lca_dropout, or None."""
    if dropout is None:
        return None
    seed, p = dropout
    return Dropout_t(float(p), int(seed) & 0xFFFFFFFFFFFFFFFF)


def attn_fwd(q, k, v, segments, mask, scale=0.0, out=None, lse=None, workspace=None, stream=None, call=None,
             dropout=None):
    """q [Tq,Hq,128], k/v [Tk,Hkv,128] bf16 CUDA tensors -> (o, lse[Hq,Tq]).
    out / lse may be given as CUDA or pinned host tensors.
    dropout: (seed, p) for attention dropout with drop probability p."""
    import torch

    Tq, Hq, d = q.shape
    Tk, Hkv, _ = k.shape
    bf = torch.bfloat16
    _require(q, "q", (Tq, Hq, d), bf)
    _require(k, "k", (Tk, Hkv, d), bf, q.device)
    _require(v, "v", (Tk, Hkv, d), bf, q.device)
    call = call or marshal(Tq, Tk, Hq, Hkv, d, segments, mask, scale, q.device)
    out = torch.empty_like(q) if out is None else _require(out, "out", (Tq, Hq, d), bf, q.device, host_ok=True)
    lse = (torch.empty((Hq, Tq), dtype=torch.float32, device=q.device) if lse is None
           else _require(lse, "lse", (Hq, Tq), torch.float32, q.device, host_ok=True))
    workspace = _workspace(call, False, workspace, q.device)
    drop = _dropout(dropout)
    with _on_device(q.device):
        if drop is None:
            _check(load().lca_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                       C.byref(call.shape), C.byref(call.mask), workspace.data_ptr(),
                                       workspace.numel(), _stream(stream, q.device)), "lca_attn_fwd")
        else:
            _check(load().lca_attn_fwd_dropout(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                               lse.data_ptr(), C.byref(call.shape), C.byref(call.mask),
                                               C.byref(drop), workspace.data_ptr(), workspace.numel(),
                                               _stream(stream, q.device)), "lca_attn_fwd_dropout")
    return out, lse


class CadShard_t(C.Structure):
    _fields_ = [("doc", C.c_int32), ("start", C.c_int32), ("len", C.c_int32), ("server", C.c_int32)]


@dataclass
class CadPlan:
    """Shards (doc, start, len, server) ordered by server then document, and
    each server's causal attention cells per head."""
    shards: list
    server_cells: list

    def server_batch(self, server: int, doc_lengths):
        """The server's packed query batch: CAUSAL segments (q_off, q_len,
        k_off, k_len) over keys packed in document order, and for each packed
        query row its row in the document-ordered token buffer."""
        starts = np.concatenate([[0], np.cumsum(np.asarray(doc_lengths, dtype=np.int64))])
        segs, rows, q = [], [], 0
        for doc, start, n, srv in self.shards:
            if srv != server:
                continue
            segs.append((q, n, int(starts[doc]), start + n))
            rows.append(np.arange(starts[doc] + start, starts[doc] + start + n))
            q += n
        return segs, (np.concatenate(rows) if rows else np.zeros(0, dtype=np.int64))


def cad_plan(doc_lengths, n_servers, min_shard=1024, max_shard=32768, tolerance=0.05) -> CadPlan:
    """Core-attention disaggregation plan (host only, lca_cad_plan)."""
    arr, ptr = _i32(doc_lengths)
    n = C.c_int32(0)
    cells = (C.c_int64 * max(1, int(n_servers)))()
    cap = max(16, 4 * len(arr) + 4 * int(n_servers))
    while True:
        buf = (CadShard_t * cap)()
        code = load().lca_cad_plan(ptr, len(arr), int(n_servers), int(min_shard), int(max_shard),
                                   C.c_double(float(tolerance)), buf, cap, C.byref(n), cells)
        if code == 3 and n.value > cap:  # LCA_ERR_WORKSPACE: more shards than room
            cap = n.value
            continue
        _check(code, "lca_cad_plan")
        break
    shards = [(buf[i].doc, buf[i].start, buf[i].len, buf[i].server) for i in range(n.value)]
    return CadPlan(shards, [int(cells[i]) for i in range(int(n_servers))])


def attn_merge(o_parts, lse_parts, out=None, lse=None, stream=None):
    """Merges forward results of the same queries over disjoint key sets:
    o_parts [Tq,Hq,128] bf16 and lse_parts [Hq,Tq] f32 CUDA tensors ->
    (o, lse).  `out`/`lse` may be part 0's tensors."""
    import torch

    n = len(o_parts)
    if n != len(lse_parts):
        raise ValueError("o_parts and lse_parts differ in length")
    Tq, Hq, d = o_parts[0].shape
    dev = o_parts[0].device
    for p, (o_p, l_p) in enumerate(zip(o_parts, lse_parts)):
        _require(o_p, f"o_parts[{p}]", (Tq, Hq, d), torch.bfloat16, dev if p else None)
        _require(l_p, f"lse_parts[{p}]", (Hq, Tq), torch.float32, dev)
    out = torch.empty_like(o_parts[0]) if out is None else _require(out, "out", (Tq, Hq, d), torch.bfloat16, dev)
    lse = torch.empty_like(lse_parts[0]) if lse is None else _require(lse, "lse", (Hq, Tq), torch.float32, dev)
    optrs = (C.c_void_p * n)(*[t.data_ptr() for t in o_parts])
    lptrs = (C.c_void_p * n)(*[t.data_ptr() for t in lse_parts])
    with _on_device(dev):
        _check(load().lca_attn_merge(optrs, lptrs, n, C.c_void_p(out.data_ptr()), C.c_void_p(lse.data_ptr()), Tq, Hq,
                                     d, _stream(stream, dev)), "lca_attn_merge")
    return out, lse


def attn_bwd(do, q, k, v, o, lse, segments, mask, scale=0.0, dq=None, dk=None, dv=None, workspace=None, stream=None,
             call=None, dropout=None):
    """Returns (dq, dk, dv) bf16; given dq / dk / dv may be CUDA or pinned host
    tensors.  dropout: the (seed, p) the forward used."""
    import torch

    Tq, Hq, d = q.shape
    Tk, Hkv, _ = k.shape
    bf = torch.bfloat16
    _require(q, "q", (Tq, Hq, d), bf)
    for name, t in (("do", do), ("o", o)):
        _require(t, name, (Tq, Hq, d), bf, q.device)
    _require(k, "k", (Tk, Hkv, d), bf, q.device)
    _require(v, "v", (Tk, Hkv, d), bf, q.device)
    _require(lse, "lse", (Hq, Tq), torch.float32, q.device)
    call = call or marshal(Tq, Tk, Hq, Hkv, d, segments, mask, scale, q.device)
    dq = torch.empty_like(q) if dq is None else _require(dq, "dq", (Tq, Hq, d), bf, q.device, host_ok=True)
    dk = torch.empty_like(k) if dk is None else _require(dk, "dk", (Tk, Hkv, d), bf, q.device, host_ok=True)
    dv = torch.empty_like(v) if dv is None else _require(dv, "dv", (Tk, Hkv, d), bf, q.device, host_ok=True)
    workspace = _workspace(call, True, workspace, q.device)
    drop = _dropout(dropout)
    args = (do.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dq.data_ptr(),
            dk.data_ptr(), dv.data_ptr(), C.byref(call.shape), C.byref(call.mask))
    with _on_device(q.device):
        tail = (workspace.data_ptr(), workspace.numel(), _stream(stream, q.device))
        if drop is None:
            _check(load().lca_attn_bwd(*args, *tail), "lca_attn_bwd")
        else:
            _check(load().lca_attn_bwd_dropout(*args, C.byref(drop), *tail), "lca_attn_bwd_dropout")
    return dq, dk, dv


def mask_materialize(call: Call, head: int, seg: int, q_len: int, k_len: int, device="cuda", stream=None):
    import torch

    out = torch.empty((q_len, k_len), dtype=torch.uint8, device=device)
    ws = _workspace(call, False, None, device)
    with _on_device(out.device):
        _check(load().lca_mask_materialize(C.byref(call.shape), C.byref(call.mask), head, seg, out.data_ptr(),
                                           ws.data_ptr(), ws.numel(), _stream(stream, out.device)),
               "lca_mask_materialize")
    return out


def mask_tile_classes(call: Call, head: int, seg: int, q_len: int, k_len: int, device="cuda", stream=None):
    import torch

    nq, nk = -(-q_len // 128), -(-k_len // 128)
    out = torch.empty((max(nq, 0), max(nk, 0)), dtype=torch.uint8, device=device)
    ws = _workspace(call, False, None, device)
    with _on_device(out.device):
        _check(load().lca_mask_tile_classes(C.byref(call.shape), C.byref(call.mask), head, seg, out.data_ptr(),
                                            ws.data_ptr(), ws.numel(), _stream(stream, out.device)),
               "lca_mask_tile_classes")
    return out


def mask_nnz(call: Call, device="cuda", stream=None):
    import torch

    out = torch.zeros(call.shape.Hq, dtype=torch.int64, device=device)
    ws = _workspace(call, False, None, device)
    with _on_device(out.device):
        _check(load().lca_mask_nnz(C.byref(call.shape), C.byref(call.mask), out.data_ptr(), ws.data_ptr(),
                                   ws.numel(), _stream(stream, out.device)), "lca_mask_nnz")
    return out


def read_status(workspace, stream=None):
    buf = (C.c_int32 * 2)()
    with _on_device(workspace.device):
        _check(load().lca_read_status(workspace.data_ptr(), buf, _stream(stream, workspace.device)),
               "lca_read_status")
    return int(buf[0]), int(buf[1])


def probe_wait_timeout(workspace, limit_ms: int, stream=None):
    with _on_device(workspace.device):
        _check(load().lca_probe_wait_timeout(workspace.data_ptr(), workspace.numel(), int(limit_ms),
                                             _stream(stream, workspace.device)), "lca_probe_wait_timeout")


class KernelEvents:
    """Ring of CUDA event pairs the library records around each phase of its
    fwd/bwd calls (lca_set_kernel_events)."""

    def __init__(self, n_pairs: int):
        import torch

        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_pairs)]
        for e in self.events:  # torch creates the CUDA event lazily, on first record
            e.record()
        torch.cuda.synchronize()
        self._arr = (C.c_void_p * (2 * n_pairs))(*[e.cuda_event for e in self.events])
        self._ph = (C.c_int32 * n_pairs)(*([-1] * n_pairs))
        self.n_pairs = n_pairs

    def start(self):
        for i in range(self.n_pairs):
            self._ph[i] = -1
        _check(load().lca_set_kernel_events(self._arr, 2 * self.n_pairs, self._ph), "lca_set_kernel_events")

    def stop(self):
        _check(load().lca_set_kernel_events(None, 0, None), "lca_set_kernel_events")

    def durations(self):
        """{phase name: [ms, ...]} for every recorded pair (call after a sync)."""
        out = {}
        for i in range(self.n_pairs):
            ph = self._ph[i]
            if ph < 0:
                continue
            out.setdefault(PHASES[ph], []).append(self.events[2 * i].elapsed_time(self.events[2 * i + 1]))
        return out


def launch_count() -> int:
    return int(load().lca_launch_count())


CTA_PROFILE_BYTES = 3 * 1024 * 64
PROFILE_KERNELS = ("fwd", "dkv", "dq")


class CtaProfile:
    """Per-CTA records of the attention kernels (lca_set_cta_profile): after a
    call, records() gives for each kernel the rows (start_ns, end_ns, items,
    full, partial, grid, sm) of the CTAs it launched."""

    def __init__(self, device="cuda"):
        import torch

        self.buf = torch.zeros(CTA_PROFILE_BYTES // 8, dtype=torch.int64, device=device)

    def start(self):
        with _on_device(self.buf.device):
            _check(load().lca_set_cta_profile(self.buf.data_ptr(), CTA_PROFILE_BYTES), "lca_set_cta_profile")

    def stop(self):
        _check(load().lca_set_cta_profile(None, 0), "lca_set_cta_profile")

    def records(self):
        """{kernel: int64 array [grid, 7]} for every kernel slot the last call
        filled (call after a synchronize)."""
        r = self.buf.view(3, 1024, 8).cpu().numpy()
        out = {}
        for k, name in enumerate(PROFILE_KERNELS):
            grid = int(r[k, 0, 5])
            if grid > 0:
                out[name] = r[k, :grid, :7].copy()
        return out

