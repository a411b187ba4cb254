"""Batched multi-adapter LoRA branch for GB300 (sm_103a): Python binding.

Thin marshalling over the C ABI of include/lora_gemm.h: each ``lora_*``
function below has the C function's name, takes torch tensors (device memory
owned by the caller) and passes their addresses, leading dimensions and the
current CUDA stream.  All arithmetic runs in the library's CUDA kernels; there
is no CPU path.  A non-OK status raises :class:`LoraError`.

The helper classes at the end (``SlotTable``, ``TokenIndex``, ``Workspace``)
only allocate the caller-owned buffers the calls need.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import numpy as np

from ._lib import (LORA_ABI_VERSION, LORA_DECODE_MAX_SEG, LORA_MAX_RANK, LORA_MAX_SLICES, LORA_MAX_SLOTS,
                   LORA_NOALLOC_WS_BYTES, PATHS, LoraError, check, load, lora_shape_t, status_string)

__all__ = [
    "LORA_ABI_VERSION", "LORA_MAX_RANK", "LORA_MAX_SLICES", "LORA_MAX_SLOTS", "LORA_DECODE_MAX_SEG",
    "LORA_NOALLOC_WS_BYTES",
    "LoraError", "lora_shape_t", "make_shape", "lora_abi_version", "lora_status_string", "lora_scale",
    "lora_premultiply", "lora_premultiply_e4m3", "lora_slot_table_bytes", "lora_pack_slot_table", "lora_set_slot_table",
    "lora_slot_table_tma_bytes", "lora_set_slot_table_tma",
    "lora_build_index", "lora_build_index_seq", "lora_workspace_bytes", "lora_workspace_xa_offset", "lora_shrink", "lora_expand", "lora_apply", "lora_resolve_path",
    "apply", "lora_apply_noalloc", "lora_apply_overlap", "lora_moe_slot_pointers", "lora_build_index_moe", "lora_apply_moe",
    "lora_build_index_activated", "lora_plan_bytes", "lora_build_plan", "lora_apply_plan", "lora_build_plans", "Plan", "apply_with_base", "SlotTable", "TokenIndex", "Workspace",
]


def _torch():
    import torch
    return torch


def _p(t) -> Optional[ctypes.c_void_p]:
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return ctypes.c_void_p(t.ctypes.data)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t, name, dtype=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _rows(t, name):
    torch = _torch()
    _dev(t, name, torch.bfloat16)
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D bf16 tensor with unit column stride")
    return t.stride(0)


def make_shape(S: int, r_max: int, k: int, slice_widths: Sequence[int]) -> lora_shape_t:
    """Shape of one packed projection (lora_shape_t)."""
    widths = [int(w) for w in slice_widths]
    if not 1 <= len(widths) <= LORA_MAX_SLICES:
        raise ValueError("between 1 and LORA_MAX_SLICES output slices")
    sh = lora_shape_t()
    sh.S, sh.r_max, sh.k, sh.n_slices = int(S), int(r_max), int(k), len(widths)
    off = 0
    sh.slice_offsets[0] = 0
    for i, w in enumerate(widths):
        off += w
        sh.slice_offsets[i + 1] = off
    for i in range(len(widths) + 1, LORA_MAX_SLICES + 1):
        sh.slice_offsets[i] = off
    return sh


# ---------------------------------------------------------------------------
# C ABI, one wrapper per entry point
# ---------------------------------------------------------------------------
def lora_abi_version() -> int:
    return int(load().lora_abi_version())


def lora_status_string(status: int) -> str:
    return status_string(status)


def lora_scale(alpha: float, rank: int, rslora: bool = False, adapter_scale: float = 1.0) -> float:
    return float(load().lora_scale(float(alpha), int(rank), int(bool(rslora)), float(adapter_scale)))


def lora_premultiply(w, scale: float, stream=None) -> None:
    _dev(w, "w", _torch().bfloat16)
    if not w.is_contiguous():
        raise ValueError("w must be contiguous")
    check(load().lora_premultiply(_p(w), w.numel(), float(scale), _stream(stream)), "lora_premultiply")


def lora_premultiply_e4m3(w, scale: float, stream=None) -> None:
    """In-place load-time scale of float8_e4m3fn codes (a uint8 or float8_e4m3fn tensor)."""
    torch = _torch()
    if not isinstance(w, torch.Tensor) or not w.is_cuda or w.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError("w must be a CUDA uint8 or float8_e4m3fn tensor")
    if not w.is_contiguous():
        raise ValueError("w must be contiguous")
    check(load().lora_premultiply_e4m3(_p(w), w.numel(), float(scale), _stream(stream)), "lora_premultiply_e4m3")


def lora_slot_table_bytes(S: int, n_slices: int) -> int:
    return int(load().lora_slot_table_bytes(int(S), int(n_slices)))


def lora_pack_slot_table(host_buf, S, n_slices, r_max, ranks, scales, A_ptrs, B_ptrs) -> None:
    ranks = np.ascontiguousarray(ranks, dtype=np.int32)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    A_ptrs = np.ascontiguousarray(A_ptrs, dtype=np.uint64)
    B_ptrs = np.ascontiguousarray(B_ptrs, dtype=np.uint64)
    check(load().lora_pack_slot_table(_p(host_buf), int(S), int(n_slices), int(r_max), _p(ranks), _p(scales),
                                      _p(A_ptrs), _p(B_ptrs)), "lora_pack_slot_table")


def lora_set_slot_table(dev_table, host_staging, S, n_slices, r_max, ranks, scales, A_ptrs, B_ptrs,
                        stream=None) -> None:
    ranks = np.ascontiguousarray(ranks, dtype=np.int32)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    A_ptrs = np.ascontiguousarray(A_ptrs, dtype=np.uint64)
    B_ptrs = np.ascontiguousarray(B_ptrs, dtype=np.uint64)
    _dev(dev_table, "dev_table")
    check(load().lora_set_slot_table(_p(dev_table), _p(host_staging), int(S), int(n_slices), int(r_max),
                                     _p(ranks), _p(scales), _p(A_ptrs), _p(B_ptrs), _stream(stream)),
          "lora_set_slot_table")


def lora_slot_table_tma_bytes(S: int, shape: lora_shape_t) -> int:
    return int(load().lora_slot_table_tma_bytes(int(S), ctypes.byref(shape)))


def lora_set_slot_table_tma(dev_table, host_staging, shape, ranks, scales, A_ptrs, B_ptrs, stream=None) -> None:
    """The slot table plus TMA tensor maps of every A and B (for path "decode_tma")."""
    ranks = np.ascontiguousarray(ranks, dtype=np.int32)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    A_ptrs = np.ascontiguousarray(A_ptrs, dtype=np.uint64)
    B_ptrs = np.ascontiguousarray(B_ptrs, dtype=np.uint64)
    _dev(dev_table, "dev_table")
    check(load().lora_set_slot_table_tma(_p(dev_table), _p(host_staging), ctypes.byref(shape), _p(ranks),
                                         _p(scales), _p(A_ptrs), _p(B_ptrs), _stream(stream)),
          "lora_set_slot_table_tma")


def lora_build_index(slot_ids, S, dev_table, sorted_ids, seg_offsets, active, err, stream=None) -> None:
    torch = _torch()
    _dev(slot_ids, "slot_ids", torch.int32)
    T = int(slot_ids.numel())
    check(load().lora_build_index(_p(slot_ids), T, int(S), _p(dev_table), _p(sorted_ids), _p(seg_offsets),
                                  _p(active), _p(err), _stream(stream)), "lora_build_index")


def lora_workspace_bytes(T: int, shape: lora_shape_t) -> int:
    out = ctypes.c_size_t(0)
    check(load().lora_workspace_bytes(int(T), ctypes.byref(shape), ctypes.byref(out)), "lora_workspace_bytes")
    return int(out.value)


def lora_workspace_xa_offset(shape: lora_shape_t) -> int:
    """Byte offset of xa (float32 [n_slices][T][r_max]) inside the workspace."""
    return int(load().lora_workspace_xa_offset(ctypes.byref(shape)))


def lora_shrink(x, shape, dev_table, sorted_ids, seg_offsets, active, ws, err, stream=None) -> None:
    ldx = _rows(x, "x")
    check(load().lora_shrink(_p(x), ldx, int(x.shape[0]), ctypes.byref(shape), _p(dev_table), _p(sorted_ids),
                             _p(seg_offsets), _p(active), _p(ws), ws.numel() * ws.element_size(), _p(err),
                             _stream(stream)), "lora_shrink")


def lora_expand(ws, y, shape, dev_table, sorted_ids, seg_offsets, active, err, stream=None) -> None:
    ldy = _rows(y, "y")
    check(load().lora_expand(_p(ws), ws.numel() * ws.element_size(), _p(y), ldy, int(y.shape[0]),
                             ctypes.byref(shape), _p(dev_table), _p(sorted_ids), _p(seg_offsets), _p(active),
                             _p(err), _stream(stream)), "lora_expand")


def lora_apply(x, y, shape, dev_table, sorted_ids, seg_offsets, active, ws, err, max_seg_hint: int = 0,
               path: str = "auto", stream=None) -> None:
    ldx = _rows(x, "x")
    ldy = _rows(y, "y")
    if x.shape[0] != y.shape[0]:
        raise ValueError("x and y must have the same number of rows")
    args = (_p(x), ldx, _p(y), ldy, int(x.shape[0]), ctypes.byref(shape), _p(dev_table), _p(sorted_ids),
            _p(seg_offsets), _p(active), int(max_seg_hint))
    tail = (_p(ws), ws.numel() * ws.element_size(), _p(err), _stream(stream))
    if path == "auto":
        check(load().lora_apply(*args, *tail), "lora_apply")
    else:
        check(load().lora_apply_ex(*args, PATHS[path], *tail), "lora_apply_ex")


def apply(x, y, table, index, ws, shape, max_seg_hint: int = 0, path: str = "auto", stream=None) -> None:
    """y += the branch for x, with a SlotTable, a built TokenIndex and a Workspace
    (their device buffers passed to lora_apply / lora_apply_ex); raises on error."""
    lora_apply(x, y, shape, table.dev, index.sorted_ids, index.seg_offsets, index.active, ws.buf, index.err,
               max_seg_hint=max_seg_hint, path=path, stream=stream)


def lora_apply_overlap(x, y, shape, dev_table, sorted_ids, seg_offsets, active, ws, err, y_ready=None,
                       max_seg_hint: int = 0, path: str = "auto", stream=None) -> None:
    """lora_apply on `stream` whose y half waits for the event `y_ready`
    (a torch.cuda.Event recorded once y holds its input values)."""
    ldx = _rows(x, "x")
    ldy = _rows(y, "y")
    if x.shape[0] != y.shape[0]:
        raise ValueError("x and y must have the same number of rows")
    ev = ctypes.c_void_p(y_ready.cuda_event) if y_ready is not None else None
    check(load().lora_apply_overlap(_p(x), ldx, _p(y), ldy, int(x.shape[0]), ctypes.byref(shape), _p(dev_table),
                                    _p(sorted_ids), _p(seg_offsets), _p(active), int(max_seg_hint), PATHS[path],
                                    _p(ws), ws.numel() * ws.element_size(), _p(err), _stream(stream), ev),
          "lora_apply_overlap")


def apply_with_base(x, w0, y, shape, dev_table, index, ws, aux_stream, max_seg_hint: int = 0,
                    path: str = "auto") -> None:
    """y = x w0^T + branch, the base projection (a bf16 library GEMM) on the
    current stream and the branch on `aux_stream`: the branch's x-only half
    overlaps the GEMM, its y half runs once the GEMM has written y, and the
    current stream waits for the branch before it goes on."""
    torch = _torch()
    main = torch.cuda.current_stream()
    x_ready = torch.cuda.Event()
    x_ready.record(main)
    aux_stream.wait_event(x_ready)
    torch.matmul(x, w0.t(), out=y)
    y_ready = torch.cuda.Event()
    y_ready.record(main)
    lora_apply_overlap(x, y, shape, dev_table, index.sorted_ids, index.seg_offsets, index.active, ws, index.err,
                       y_ready=y_ready, max_seg_hint=max_seg_hint, path=path, stream=aux_stream)
    done = torch.cuda.Event()
    done.record(aux_stream)
    main.wait_event(done)


def lora_apply_noalloc(x, y, shape, dev_table, sorted_ids, seg_offsets, active, err, stream=None) -> None:
    """lora_apply with the library's built-in scratch instead of a workspace:
    for callers that cannot allocate device memory where they run the branch.
    Calls on one device share that scratch, so keep them on one stream."""
    ldx = _rows(x, "x")
    ldy = _rows(y, "y")
    if x.shape[0] != y.shape[0]:
        raise ValueError("x and y must have the same number of rows")
    check(load().lora_apply_noalloc(_p(x), ldx, _p(y), ldy, int(x.shape[0]), ctypes.byref(shape), _p(dev_table),
                                    _p(sorted_ids), _p(seg_offsets), _p(active), _p(err), _stream(stream)),
          "lora_apply_noalloc")


def lora_resolve_path(path: str, T: int, max_seg_hint: int = 0):
    """(path name lora_apply takes, kernel launches per call)."""
    launches = ctypes.c_int32(0)
    code = load().lora_resolve_path(PATHS[path], int(T), int(max_seg_hint), ctypes.byref(launches))
    name = {v: k for k, v in PATHS.items()}[int(code)]
    return name, int(launches.value)


# ---------------------------------------------------------------------------
# Caller-owned buffers (allocation only)
# ---------------------------------------------------------------------------
def lora_build_index_seq(seq_slot_ids, tokens_per_seq, S, dev_table, sorted_ids, seg_offsets, active, err,
                         stream=None) -> None:
    """Token index of n_seq sequences of tokens_per_seq tokens each (speculative decode)."""
    torch = _torch()
    _dev(seq_slot_ids, "seq_slot_ids", torch.int32)
    n_seq = int(seq_slot_ids.numel())
    check(load().lora_build_index_seq(_p(seq_slot_ids), n_seq, int(tokens_per_seq), int(S), _p(dev_table),
                                      _p(sorted_ids), _p(seg_offsets), _p(active), _p(err), _stream(stream)),
          "lora_build_index_seq")


def lora_moe_slot_pointers(n_adapters: int, E: int, shape: lora_shape_t, ranks, scales, A_base, B_base,
                           elem_bytes: int = 2):
    """Virtual slot entries (rank, scale, A and B pointers) of n_adapters * E
    routed-expert slots, from each adapter's [E][r][k] and [E][d_i][r] bases."""
    ranks = np.ascontiguousarray(ranks, dtype=np.int32)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    A_base = np.ascontiguousarray(A_base, dtype=np.uint64)
    B_base = np.ascontiguousarray(B_base, dtype=np.uint64)
    V, n = int(n_adapters) * int(E), int(shape.n_slices)
    v_ranks = np.zeros(V, np.int32)
    v_scales = np.zeros(V, np.float32)
    A_ptrs = np.zeros(V * n, np.uint64)
    B_ptrs = np.zeros(V * n, np.uint64)
    check(load().lora_moe_slot_pointers(int(n_adapters), int(E), ctypes.byref(shape), int(elem_bytes), _p(ranks),
                                        _p(scales), _p(A_base), _p(B_base), _p(v_ranks), _p(v_scales), _p(A_ptrs),
                                        _p(B_ptrs)), "lora_moe_slot_pointers")
    return v_ranks, v_scales, A_ptrs, B_ptrs


def lora_build_index_activated(seq_ids, positions, seq_slot, invocation_start, S, dev_table, sorted_ids,
                               seg_offsets, active, err, stream=None) -> None:
    """Token index with aLoRA enablement: token t takes its sequence's slot from
    the sequence's invocation start on, and no adapter before it."""
    torch = _torch()
    for t, name in ((seq_ids, "seq_ids"), (positions, "positions"), (seq_slot, "seq_slot"),
                    (invocation_start, "invocation_start")):
        _dev(t, name, torch.int32)
    T, n_seq = int(seq_ids.numel()), int(seq_slot.numel())
    if int(positions.numel()) != T or int(invocation_start.numel()) != n_seq:
        raise ValueError("positions must match seq_ids, invocation_start must match seq_slot")
    check(load().lora_build_index_activated(_p(seq_ids), _p(positions), T, _p(seq_slot), _p(invocation_start), n_seq,
                                            int(S), _p(dev_table), _p(sorted_ids), _p(seg_offsets), _p(active),
                                            _p(err), _stream(stream)), "lora_build_index_activated")


def lora_build_index_moe(slot_ids, expert_ids, K, E, S, dev_table, sorted_ids, seg_offsets, active, err,
                         stream=None) -> None:
    """Index of the T * K (token, choice) pairs over S = n_adapters * E virtual slots."""
    torch = _torch()
    _dev(slot_ids, "slot_ids", torch.int32)
    _dev(expert_ids, "expert_ids", torch.int32)
    T = int(slot_ids.numel())
    if int(expert_ids.numel()) != T * int(K):
        raise ValueError("expert_ids must hold K ids per token")
    check(load().lora_build_index_moe(_p(slot_ids), _p(expert_ids), T, int(K), int(E), int(S), _p(dev_table),
                                      _p(sorted_ids), _p(seg_offsets), _p(active), _p(err), _stream(stream)),
          "lora_build_index_moe")


def lora_apply_moe(x, y, K, shape, dev_table, sorted_ids, seg_offsets, active, ws, err, x_per_token: bool = True,
                   stream=None, plan=None, path: str = "decode_direct") -> None:
    """Routed-expert branch: y [T*K, d] per (token, choice) pair; x [T, k] shared
    by a token's experts (x_per_token) or [T*K, k] per pair.  `path` is
    "decode_direct" or "decode_tma" (dev_table then a tensor-map table of the
    virtual slots).  With `plan` (a Plan built for T*K rows on the virtual table
    and the pair index) the table and index arguments are not used and the
    plan's path is run."""
    ldx = _rows(x, "x")
    ldy = _rows(y, "y")
    P = int(y.shape[0])
    if P % int(K) != 0:
        raise ValueError("y must have T * K rows")
    T = P // int(K)
    if int(x.shape[0]) != (T if x_per_token else P):
        raise ValueError("x must have T rows (x_per_token) or T * K rows")
    if plan is not None:
        check(load().lora_apply_moe_plan_ex(_p(x), ldx, int(bool(x_per_token)), _p(y), ldy, T, int(K),
                                            ctypes.byref(shape), _p(plan.buf), plan.buf.numel(), PATHS[plan.path],
                                            _p(ws), ws.numel() * ws.element_size(), _p(err), _stream(stream)),
              "lora_apply_moe_plan_ex")
        return
    check(load().lora_apply_moe_ex(_p(x), ldx, int(bool(x_per_token)), _p(y), ldy, T, int(K), ctypes.byref(shape),
                                   _p(dev_table), _p(sorted_ids), _p(seg_offsets), _p(active), PATHS[path], _p(ws),
                                   ws.numel() * ws.element_size(), _p(err), _stream(stream)), "lora_apply_moe_ex")


def lora_plan_bytes(T: int, shape: lora_shape_t) -> int:
    return int(load().lora_plan_bytes(int(T), ctypes.byref(shape)))


def lora_build_plan(T, shape, dev_table, sorted_ids, seg_offsets, active, plan, err, path: str = "decode_direct",
                    stream=None) -> None:
    check(load().lora_build_plan(int(T), ctypes.byref(shape), _p(dev_table), _p(sorted_ids), _p(seg_offsets),
                                 _p(active), PATHS[path], _p(plan), plan.numel() * plan.element_size(), _p(err),
                                 _stream(stream)), "lora_build_plan")


def lora_apply_plan(x, y, shape, plan, ws, err, path: str = "decode_direct", stream=None) -> None:
    ldx = _rows(x, "x")
    ldy = _rows(y, "y")
    if x.shape[0] != y.shape[0]:
        raise ValueError("x and y must have the same number of rows")
    check(load().lora_apply_plan(_p(x), ldx, _p(y), ldy, int(x.shape[0]), ctypes.byref(shape), _p(plan),
                                 plan.numel() * plan.element_size(), PATHS[path], _p(ws), ws.numel() * ws.element_size(),
                                 _p(err), _stream(stream)), "lora_apply_plan")


def lora_build_plans(plans, tables, index, stream=None) -> None:
    """The plans of several slot tables of one shape and batch (e.g. every layer of
    a step), in one launch; plans[j] is built for tables[j]."""
    if len(plans) != len(tables):
        raise ValueError("one table per plan")
    if not plans:
        return
    p0 = plans[0]
    if any(p.T != p0.T or p.path != p0.path or p.buf.numel() != p0.buf.numel() for p in plans):
        raise ValueError("plans of one call share T, shape and path")
    tabs = (ctypes.c_void_p * len(plans))(*[t.dev.data_ptr() for t in tables])
    bufs = (ctypes.c_void_p * len(plans))(*[p.buf.data_ptr() for p in plans])
    check(load().lora_build_plans(p0.T, ctypes.byref(p0.shape), len(plans), tabs, bufs, p0.buf.numel(),
                                  _p(index.sorted_ids), _p(index.seg_offsets), _p(index.active), PATHS[p0.path],
                                  _p(index.err), _stream(stream)), "lora_build_plans")


class Plan:
    """The per-step tables of the warp-streaming kernels ("decode_direct",
    "decode_direct_fp8") or of the one-kernel TMA path ("decode_tma") for one
    batch and shape, built once (after the index) and used by every call of that
    shape."""

    def __init__(self, T: int, shape: lora_shape_t, path: str = "decode_direct", device="cuda"):
        torch = _torch()
        nbytes = lora_plan_bytes(T, shape)
        if nbytes == 0:
            raise ValueError("no plan for this T and shape")
        self.T, self.shape, self.path = int(T), shape, path
        self.buf = torch.zeros(nbytes, dtype=torch.uint8, device=device)

    def build(self, index, table, stream=None) -> None:
        lora_build_plan(self.T, self.shape, table.dev, index.sorted_ids, index.seg_offsets, index.active, self.buf,
                        index.err, self.path, stream)

    def apply(self, x, y, ws, err, stream=None) -> None:
        lora_apply_plan(x, y, self.shape, self.buf, ws.buf, err, self.path, stream)


class SlotTable:
    """Device slot table plus the pinned staging buffer its upload copies from.
    With ``shape`` the table also carries the TMA tensor maps of every A and B
    (lora_set_slot_table_tma), which path "decode_tma" needs; every path accepts it."""

    def __init__(self, S: int, n_slices: int, r_max: int, device="cuda", shape: Optional[lora_shape_t] = None):
        torch = _torch()
        self.S, self.n_slices, self.r_max, self.shape = int(S), int(n_slices), int(r_max), shape
        nbytes = lora_slot_table_tma_bytes(S, shape) if shape is not None else lora_slot_table_bytes(S, n_slices)
        if nbytes == 0:
            raise ValueError("no slot table for this S and shape")
        self.dev = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        self.staging = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()

    def set(self, ranks, scales, A_ptrs, B_ptrs, stream=None) -> None:
        if self.shape is not None:
            lora_set_slot_table_tma(self.dev, self.staging, self.shape, ranks, scales, A_ptrs, B_ptrs, stream)
        else:
            lora_set_slot_table(self.dev, self.staging, self.S, self.n_slices, self.r_max, ranks, scales,
                                A_ptrs, B_ptrs, stream)


class TokenIndex:
    """sorted_ids[T], seg_offsets[S+2], active[S+1] and the error word."""

    def __init__(self, T: int, S: int, device="cuda"):
        torch = _torch()
        self.T, self.S = int(T), int(S)
        self.sorted_ids = torch.zeros(max(T, 1), dtype=torch.int32, device=device)
        self.seg_offsets = torch.zeros(S + 2, dtype=torch.int32, device=device)
        self.active = torch.zeros(S + 1, dtype=torch.int32, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    def build(self, slot_ids, table: SlotTable, stream=None) -> None:
        lora_build_index(slot_ids, self.S, table.dev, self.sorted_ids, self.seg_offsets, self.active, self.err,
                         stream)

    def build_seq(self, seq_slot_ids, tokens_per_seq: int, table: SlotTable, stream=None) -> None:
        """Index for T = len(seq_slot_ids) * tokens_per_seq tokens, sequence-major."""
        assert int(seq_slot_ids.numel()) * int(tokens_per_seq) == self.T
        lora_build_index_seq(seq_slot_ids, tokens_per_seq, self.S, table.dev, self.sorted_ids, self.seg_offsets,
                             self.active, self.err, stream)


    def build_activated(self, seq_ids, positions, seq_slot, invocation_start, table: SlotTable,
                        stream=None) -> None:
        """Index of this index's T tokens with aLoRA enablement per sequence."""
        lora_build_index_activated(seq_ids, positions, seq_slot, invocation_start, self.S, table.dev,
                                   self.sorted_ids, self.seg_offsets, self.active, self.err, stream)

    def build_moe(self, slot_ids, expert_ids, K: int, E: int, table: SlotTable, stream=None) -> None:
        """Index of len(slot_ids) * K pairs over this index's S = n_adapters * E virtual slots."""
        assert int(slot_ids.numel()) * int(K) == self.T
        lora_build_index_moe(slot_ids, expert_ids, K, E, self.S, table.dev, self.sorted_ids, self.seg_offsets,
                             self.active, self.err, stream)


class Workspace:
    """fp32 workspace of lora_workspace_bytes(T, shape) bytes, zeroed once."""

    def __init__(self, T: int, shape: lora_shape_t, device="cuda"):
        torch = _torch()
        nbytes = lora_workspace_bytes(T, shape)
        self.buf = torch.zeros((nbytes + 3) // 4, dtype=torch.float32, device=device)
