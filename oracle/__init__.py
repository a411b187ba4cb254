"""CPU oracle for the batched multi-adapter LoRA branch (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The library's product path never does: it has no CPU
fallback.  The arithmetic lives in ``lora_oracle.c`` (plain C loops, fp64); this
file builds it with gcc and marshals numpy arrays into it.  It shares no code
with the CUDA library.

Every function below states the passage it follows; the header of
``lora_oracle.c`` has the full definitions.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liblora_oracle.so")

ERR_OK = 0
ERR_SLOT_RANGE = 1

_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, no fast-math) into _build/."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def configure(lib):
    """Declare the C signatures on a loaded oracle library and return it."""
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_round_bf16.restype = ctypes.c_uint16
    lib.oracle_round_bf16.argtypes = [f64]
    lib.oracle_bf16_to_double.restype = f64
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_scale.restype = f64
    lib.oracle_scale.argtypes = [f64, i32, i32, f64]
    lib.oracle_premultiply.restype = None
    lib.oracle_premultiply.argtypes = [P, i64, f64, P]
    lib.oracle_build_index.restype = ctypes.c_int
    lib.oracle_build_index.argtypes = [P, i32, i32, P, P, P, P]
    lib.oracle_shrink.restype = None
    lib.oracle_shrink.argtypes = [P, i64, i32, i32, P, i32, P, P, P, i32, i32, P, P]
    lib.oracle_apply.restype = ctypes.c_int
    lib.oracle_apply.argtypes = [P, i64, P, i64, i32, i32, P, P, i32, P, P, P, P, P, i32, P, P]
    lib.oracle_e4m3_to_double.restype = f64
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_round.restype = ctypes.c_uint8
    lib.oracle_e4m3_round.argtypes = [f64]
    lib.oracle_premultiply_e4m3.restype = None
    lib.oracle_premultiply_e4m3.argtypes = [P, i64, f64, P]
    lib.oracle_apply_e4m3.restype = ctypes.c_int
    lib.oracle_apply_e4m3.argtypes = [P, i64, P, i64, i32, i32, P, P, i32, P, P, P, P, P, i32, P]
    lib.oracle_apply_moe.restype = ctypes.c_int
    lib.oracle_apply_moe.argtypes = [P, i64, i32, P, i64, i32, i32, P, P, P, i32, i32, i32, P, P, P, P, P, i32, P]
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = configure(ctypes.CDLL(build()))
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _ptr_table(mats: Sequence[Sequence[Optional[np.ndarray]]], dtype=np.uint16):
    """[S][n] arrays -> (ctypes array of S*n pointers, keep-alive list)."""
    flat = [m for row in mats for m in row]
    keep = [np.ascontiguousarray(m, dtype=dtype) if m is not None else None for m in flat]
    arr = (ctypes.c_void_p * max(1, len(keep)))()
    for e, m in enumerate(keep):
        arr[e] = None if m is None else m.ctypes.data
    return arr, keep


# ----------------------------------------------------------------------------
# bf16 helpers
# ----------------------------------------------------------------------------
def round_bf16(v: float) -> int:
    """Nearest bf16 bit pattern of a double, ties to even."""
    return int(_load().oracle_round_bf16(float(v)))


def bf16_to_double(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.oracle_bf16_to_double(int(b)) for b in flat], dtype=np.float64).reshape(np.shape(bits))


# ----------------------------------------------------------------------------
# Scale rules
# ----------------------------------------------------------------------------
def scale(alpha: float, rank: int, rslora: bool = False, adapter_scale: float = 1.0) -> float:
    """llama.cpp get_scale (alpha/r, alpha==0 -> adapter_scale) or rsLoRA alpha/sqrt(r)."""
    return float(_load().oracle_scale(float(alpha), int(rank), int(bool(rslora)), float(adapter_scale)))


def slot_scales(ranks: np.ndarray, alphas: np.ndarray, scale_rule: str, premultiplied: bool) -> np.ndarray:
    """Runtime scale per slot: 1 when the rule's scale is already folded into B."""
    rs = scale_rule == "alpha_over_sqrt_r"
    out = np.ones(len(ranks), dtype=np.float64)
    if not premultiplied:
        for s in range(len(ranks)):
            out[s] = scale(alphas[s], int(ranks[s]), rs)
    return out


def premultiply(b_bits: np.ndarray, s: float) -> np.ndarray:
    """bf16(s * B) elementwise, nearest-even (vLLM's LoRALayerWeights.optimize)."""
    src = np.ascontiguousarray(b_bits, dtype=np.uint16)
    out = np.empty_like(src)
    _load().oracle_premultiply(_ptr(src), int(src.size), float(s), _ptr(out))
    return out


# ----------------------------------------------------------------------------
# FP8 (float8_e4m3fn) adapters
# ----------------------------------------------------------------------------
def e4m3_to_double(codes: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.oracle_e4m3_to_double(int(c)) for c in flat], dtype=np.float64).reshape(np.shape(codes))


def e4m3_round(values: np.ndarray) -> np.ndarray:
    """v.clamp(-448, 448).to(float8_e4m3fn) codes (nearest, ties to even)."""
    lib = _load()
    flat = np.asarray(values, dtype=np.float64).ravel()
    return np.array([lib.oracle_e4m3_round(float(v)) for v in flat], dtype=np.uint8).reshape(np.shape(values))


def premultiply_e4m3(b_codes: np.ndarray, s: float) -> np.ndarray:
    """The pages' load-time scale of FP8 B: (b.to(bf16) * s).clamp(+-448).to(fp8)."""
    src = np.ascontiguousarray(b_codes, dtype=np.uint8)
    out = np.empty_like(src)
    _load().oracle_premultiply_e4m3(_ptr(src), int(src.size), float(s), _ptr(out))
    return out


def apply_e4m3(x: np.ndarray, y_in: Optional[np.ndarray], slice_widths: Sequence[int],
               slot_ids: np.ndarray, ranks: np.ndarray, scales: np.ndarray,
               A: Sequence[Sequence[Optional[np.ndarray]]], B: Sequence[Sequence[Optional[np.ndarray]]],
               rows: Optional[np.ndarray] = None):
    """Branch rows (fp64) with x rounded to e4m3 and A, B given as e4m3 codes;
    returns (y[len(rows), d], status)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    slot_ids = np.ascontiguousarray(slot_ids, dtype=np.int32)
    ranks = np.ascontiguousarray(ranks, dtype=np.int32)
    scales = np.ascontiguousarray(scales, dtype=np.float64)
    T, k = x.shape
    widths = [int(w) for w in slice_widths]
    offs = np.zeros(len(widths) + 1, dtype=np.int32)
    offs[1:] = np.cumsum(widths)
    d = int(offs[-1])
    if y_in is not None:
        y_in = np.ascontiguousarray(y_in, dtype=np.uint16)
    rows = np.arange(T, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    out = np.zeros((len(rows), d), dtype=np.float64)
    ta, ka = _ptr_table(A, np.uint8)
    tb, kb = _ptr_table(B, np.uint8)
    st = _load().oracle_apply_e4m3(_ptr(x), k, _ptr(y_in), d, k, len(widths), _ptr(offs), _ptr(slot_ids),
                                   len(ranks), _ptr(ranks), _ptr(scales), ta, tb, _ptr(rows), len(rows), _ptr(out))
    del ka, kb
    return out, int(st)


# ----------------------------------------------------------------------------
# Routed-expert (MoE) LoRA
# ----------------------------------------------------------------------------
def apply_moe(x: np.ndarray, x_per_token: bool, y_in: Optional[np.ndarray], slice_widths: Sequence[int],
              slot_ids: np.ndarray, expert_ids: np.ndarray, E: int, ranks: np.ndarray, scales: np.ndarray,
              A: Sequence[Sequence[Optional[np.ndarray]]], B: Sequence[Sequence[Optional[np.ndarray]]],
              rows: Optional[np.ndarray] = None):
    """Rows (fp64) of the routed-expert branch for the pairs p = t K + j
    (llama.cpp's build_lora_mm_id, TensorRT-LLM's per-expert layout).  A[s][i] is
    [E, r_s, k] and B[s][i] [E, d_i, r_s]; expert_ids is [T, K]; y_in and the
    result have one row per pair.  Returns (y[len(rows), d], status)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    slot_ids = np.ascontiguousarray(slot_ids, dtype=np.int32)
    expert_ids = np.ascontiguousarray(expert_ids, dtype=np.int32)
    ranks = np.ascontiguousarray(ranks, dtype=np.int32)
    scales = np.ascontiguousarray(scales, dtype=np.float64)
    T, K = expert_ids.shape
    k = x.shape[1]
    widths = [int(w) for w in slice_widths]
    offs = np.zeros(len(widths) + 1, dtype=np.int32)
    offs[1:] = np.cumsum(widths)
    d = int(offs[-1])
    if y_in is not None:
        y_in = np.ascontiguousarray(y_in, dtype=np.uint16)
    rows = np.arange(T * K, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    out = np.zeros((len(rows), d), dtype=np.float64)
    ta, ka = _ptr_table(A)
    tb, kb = _ptr_table(B)
    st = _load().oracle_apply_moe(_ptr(x), k, int(bool(x_per_token)), _ptr(y_in), d, k, len(widths), _ptr(offs),
                                  _ptr(slot_ids), _ptr(expert_ids), int(K), int(E), len(ranks), _ptr(ranks),
                                  _ptr(scales), ta, tb, _ptr(rows), len(rows), _ptr(out))
    del ka, kb
    return out, int(st)


def activated_token_slots(seq_ids: np.ndarray, positions: np.ndarray, seq_slot: np.ndarray,
                          invocation_start: np.ndarray) -> np.ndarray:
    """Per-token slots with activated LoRA (llama.cpp's aLoRA: no adapter before
    the request's invocation point, its adapter from there on): token t of
    sequence q gets seq_slot[q] at positions >= invocation_start[q], else -1; a
    sequence id outside [0, n_seq) gives an out-of-range slot (reported)."""
    seq_ids = np.asarray(seq_ids, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    seq_slot = np.asarray(seq_slot, dtype=np.int64)
    start = np.asarray(invocation_start, dtype=np.int64)
    out = np.empty(len(seq_ids), dtype=np.int64)
    for t, q in enumerate(seq_ids):
        if q < 0 or q >= len(seq_slot):
            out[t] = np.iinfo(np.int32).max
        else:
            out[t] = seq_slot[q] if positions[t] >= start[q] else -1
    return out.astype(np.int32)


def moe_pair_slots(slot_ids: np.ndarray, expert_ids: np.ndarray, E: int, n_adapters: int) -> np.ndarray:
    """Slot of each pair p = t K + j over n_adapters * E virtual slots: s E + e for
    a token with adapter s routed to expert e, -1 without an adapter, and
    n_adapters * E (out of range, reported) for an id outside its range."""
    slot_ids = np.asarray(slot_ids, dtype=np.int64)
    expert_ids = np.asarray(expert_ids, dtype=np.int64)
    T, K = expert_ids.shape
    s = np.repeat(slot_ids, K)
    e = expert_ids.reshape(-1)
    ok = (s >= 0) & (s < n_adapters) & (e >= 0) & (e < E)
    bad = (s < -1) | (s >= n_adapters) | ((s >= 0) & ~ok)
    return np.where(ok, s * E + e, np.where(bad, n_adapters * E, -1)).astype(np.int32)


# ----------------------------------------------------------------------------
# Index
# ----------------------------------------------------------------------------
def build_index(slot_ids: np.ndarray, S: int, ranks: np.ndarray):
    """Returns (sorted_ids[T], seg_offsets[S+2], active[S+1], status)."""
    slot_ids = np.ascontiguousarray(slot_ids, dtype=np.int32)
    ranks = np.ascontiguousarray(ranks, dtype=np.int32)
    T = int(slot_ids.shape[0])
    sorted_ids = np.zeros(max(T, 1), dtype=np.int32)
    seg = np.zeros(S + 2, dtype=np.int32)
    active = np.zeros(S + 1, dtype=np.int32)
    st = _load().oracle_build_index(_ptr(slot_ids), T, int(S), _ptr(ranks), _ptr(sorted_ids),
                                    _ptr(seg), _ptr(active))
    return sorted_ids[:T], seg, active, int(st)


def build_index_seq(seq_slot_ids: np.ndarray, tokens_per_seq: int, S: int, ranks: np.ndarray):
    """Token index of sequences of tokens_per_seq tokens each (speculative decode).

    The definition: sequence b owns tokens b*tps .. b*tps + tps - 1, every one of
    them carrying the sequence's slot, so the index is the token index of the
    slot ids repeated tps times (TensorRT-LLM LoRA serving page, "一次 decode 批次
    的路由").  Returns (sorted_ids[n_seq*tps], seg_offsets[S+2], active[S+1], status)."""
    tok = np.repeat(np.ascontiguousarray(seq_slot_ids, dtype=np.int32), int(tokens_per_seq))
    return build_index(tok, S, ranks)


# ----------------------------------------------------------------------------
# Branch
# ----------------------------------------------------------------------------
def shrink(x: np.ndarray, slot_ids: np.ndarray, ranks: np.ndarray,
           A: Sequence[Sequence[Optional[np.ndarray]]], r_max: int,
           rows: Optional[np.ndarray] = None):
    """xa[q, i, j] for token rows[q] (default all), NaN where not defined; also MACs."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    slot_ids = np.ascontiguousarray(slot_ids, dtype=np.int32)
    ranks = np.ascontiguousarray(ranks, dtype=np.int32)
    T, k = x.shape
    n = len(A[0]) if len(A) else 1
    rows = np.arange(T, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    xa = np.full((len(rows), n, max(r_max, 1)), np.nan, dtype=np.float64)
    tab, keep = _ptr_table(A)
    macs = ctypes.c_int64(0)
    _load().oracle_shrink(_ptr(x), k, k, n, _ptr(slot_ids), len(ranks), _ptr(ranks), tab,
                          _ptr(rows), len(rows), max(r_max, 1), _ptr(xa), ctypes.byref(macs))
    del keep
    return xa, int(macs.value)


def apply(x: np.ndarray, y_in: Optional[np.ndarray], slice_widths: Sequence[int],
          slot_ids: np.ndarray, ranks: np.ndarray, scales: np.ndarray,
          A: Sequence[Sequence[Optional[np.ndarray]]], B: Sequence[Sequence[Optional[np.ndarray]]],
          rows: Optional[np.ndarray] = None):
    """Branch output rows (fp64, before rounding), MAC count and status.

    Returns (y[len(rows), d], macs, status)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    slot_ids = np.ascontiguousarray(slot_ids, dtype=np.int32)
    ranks = np.ascontiguousarray(ranks, dtype=np.int32)
    scales = np.ascontiguousarray(scales, dtype=np.float64)
    T, k = x.shape
    widths = [int(w) for w in slice_widths]
    offs = np.zeros(len(widths) + 1, dtype=np.int32)
    offs[1:] = np.cumsum(widths)
    d = int(offs[-1])
    if y_in is not None:
        y_in = np.ascontiguousarray(y_in, dtype=np.uint16)
        assert y_in.shape == (T, d)
    rows = np.arange(T, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    out = np.zeros((len(rows), d), dtype=np.float64)
    ta, ka = _ptr_table(A)
    tb, kb = _ptr_table(B)
    macs = ctypes.c_int64(0)
    st = _load().oracle_apply(_ptr(x), k, _ptr(y_in), d, k, len(widths), _ptr(offs),
                              _ptr(slot_ids), len(ranks), _ptr(ranks), _ptr(scales), ta, tb,
                              _ptr(rows), len(rows), _ptr(out), ctypes.byref(macs))
    del ka, kb
    return out, int(macs.value), int(st)
