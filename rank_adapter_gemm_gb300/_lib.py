"""ctypes view of the C ABI in include/lora_gemm.h.

Loads ``_build/librank_adapter_gemm.so`` (built by ``build.py``) and declares
every entry point's signature.  There is no fallback: if the library is not
built, or no CUDA device is present when a kernel is called, the call raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

LORA_ABI_VERSION = 1
LORA_MAX_SLICES = 4
LORA_MAX_RANK = 512
LORA_MAX_SLOTS = 1024
LORA_DECODE_MAX_SEG = 256
LORA_NOALLOC_WS_BYTES = 4 << 20

STATUS = {
    0: "LORA_OK",
    1: "LORA_ERR_INVALID_ARG",
    2: "LORA_ERR_ALIGNMENT",
    3: "LORA_ERR_RANK",
    4: "LORA_ERR_SLOT_RANGE",
    5: "LORA_ERR_NULL_WEIGHT",
    6: "LORA_ERR_WORKSPACE",
    7: "LORA_ERR_TIMEOUT",
    8: "LORA_ERR_CUDA",
    9: "LORA_ERR_UNSUPPORTED",
}
globals().update({name: code for code, name in STATUS.items()})

PATHS = {"auto": 0, "decode_fused": 1, "decode_split": 2, "prefill": 3, "decode_tc": 4, "decode_stream": 5,
         "decode_direct": 6, "decode_direct_fp8": 7, "decode_tma": 8, "decode_cluster": 9}

# Every function the header declares, for the export check.
EXPORTED = (
    "lora_abi_version", "lora_status_string", "lora_scale", "lora_premultiply",
    "lora_slot_table_bytes", "lora_pack_slot_table", "lora_set_slot_table", "lora_build_index",
    "lora_workspace_bytes", "lora_shrink", "lora_expand", "lora_apply", "lora_apply_ex",
    "lora_resolve_path", "lora_apply_noalloc", "lora_workspace_xa_offset", "lora_build_index_seq",
    "lora_apply_overlap", "lora_premultiply_e4m3", "lora_moe_slot_pointers", "lora_build_index_moe",
    "lora_apply_moe", "lora_build_index_activated", "lora_plan_bytes", "lora_build_plan", "lora_apply_plan",
    "lora_build_plans", "lora_apply_moe_plan", "lora_slot_table_tma_bytes", "lora_set_slot_table_tma",
    "lora_apply_moe_ex", "lora_apply_moe_plan_ex",
)


class lora_shape_t(ctypes.Structure):
    _fields_ = [
        ("S", ctypes.c_int32),
        ("r_max", ctypes.c_int32),
        ("k", ctypes.c_int32),
        ("n_slices", ctypes.c_int32),
        ("slice_offsets", ctypes.c_int32 * (LORA_MAX_SLICES + 1)),
    ]


class LoraError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {status_string(status)}")


_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Load the built library (fails loudly if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA library not built ({path} missing): run `python -c 'import __graft_entry__ as g; g.build()'` "
            "or `python rank_adapter_gemm_gb300/build.py`")
    lib = ctypes.CDLL(path)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    ST = ctypes.c_int
    SH = ctypes.POINTER(lora_shape_t)
    sig = {
        "lora_abi_version": (I32, []),
        "lora_status_string": (ctypes.c_char_p, [ST]),
        "lora_scale": (ctypes.c_double, [ctypes.c_double, I32, I32, ctypes.c_double]),
        "lora_premultiply": (ST, [P, I64, ctypes.c_float, P]),
        "lora_premultiply_e4m3": (ST, [P, I64, ctypes.c_float, P]),
        "lora_slot_table_bytes": (SZ, [I32, I32]),
        "lora_pack_slot_table": (ST, [P, I32, I32, I32, P, P, P, P]),
        "lora_set_slot_table": (ST, [P, P, I32, I32, I32, P, P, P, P, P]),
        "lora_build_index": (ST, [P, I32, I32, P, P, P, P, P, P]),
        "lora_build_index_seq": (ST, [P, I32, I32, I32, P, P, P, P, P, P]),
        "lora_workspace_bytes": (ST, [I32, SH, ctypes.POINTER(SZ)]),
        "lora_workspace_xa_offset": (SZ, [SH]),
        "lora_shrink": (ST, [P, I64, I32, SH, P, P, P, P, P, SZ, P, P]),
        "lora_expand": (ST, [P, SZ, P, I64, I32, SH, P, P, P, P, P, P]),
        "lora_apply": (ST, [P, I64, P, I64, I32, SH, P, P, P, P, I32, P, SZ, P, P]),
        "lora_apply_ex": (ST, [P, I64, P, I64, I32, SH, P, P, P, P, I32, ST, P, SZ, P, P]),
        "lora_apply_overlap": (ST, [P, I64, P, I64, I32, SH, P, P, P, P, I32, ST, P, SZ, P, P, P]),
        "lora_resolve_path": (ST, [ST, I32, I32, ctypes.POINTER(I32)]),
        "lora_apply_noalloc": (ST, [P, I64, P, I64, I32, SH, P, P, P, P, P, P]),
        "lora_moe_slot_pointers": (ST, [I32, I32, SH, I32, P, P, P, P, P, P, P, P]),
        "lora_build_index_moe": (ST, [P, P, I32, I32, I32, I32, P, P, P, P, P, P]),
        "lora_apply_moe": (ST, [P, I64, I32, P, I64, I32, I32, SH, P, P, P, P, P, SZ, P, P]),
        "lora_build_index_activated": (ST, [P, P, I32, P, P, I32, I32, P, P, P, P, P, P]),
        "lora_plan_bytes": (SZ, [I32, SH]),
        "lora_build_plan": (ST, [I32, SH, P, P, P, P, ST, P, SZ, P, P]),
        "lora_apply_plan": (ST, [P, I64, P, I64, I32, SH, P, SZ, ST, P, SZ, P, P]),
        "lora_build_plans": (ST, [I32, SH, I32, P, P, SZ, P, P, P, ST, P, P]),
        "lora_apply_moe_plan": (ST, [P, I64, I32, P, I64, I32, I32, SH, P, SZ, P, SZ, P, P]),
        "lora_slot_table_tma_bytes": (SZ, [I32, SH]),
        "lora_set_slot_table_tma": (ST, [P, P, SH, P, P, P, P, P]),
        "lora_apply_moe_ex": (ST, [P, I64, I32, P, I64, I32, I32, SH, P, P, P, P, ST, P, SZ, P, P]),
        "lora_apply_moe_plan_ex": (ST, [P, I64, I32, P, I64, I32, I32, SH, P, SZ, ST, P, SZ, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.lora_abi_version() != LORA_ABI_VERSION:
        raise RuntimeError("library ABI version does not match the binding")
    _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().lora_status_string(int(status)).decode()
    except RuntimeError:
        return STATUS.get(int(status), f"status {status}")


def check(status: int, where: str) -> None:
    if status != 0:
        raise LoraError(status, where)
