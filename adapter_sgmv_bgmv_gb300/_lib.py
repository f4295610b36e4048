"""ctypes declarations of the C ABI in include/lora.h (marshalling only)."""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblora.so")

P = ctypes.c_void_p
I = ctypes.c_int
I64 = ctypes.c_int64
F = ctypes.c_float


class PlanView(ctypes.Structure):
    _fields_ = [("n_active", I64), ("active_rows", ctypes.POINTER(ctypes.c_int32)),
                ("perm", ctypes.POINTER(ctypes.c_int32)), ("n_segments", I64),
                ("seg_offsets", ctypes.POINTER(ctypes.c_int32)),
                ("seg_adapter", ctypes.POINTER(ctypes.c_int32)),
                ("row_items", I64), ("tile_items", I64), ("rows_per_item", I64),
                ("tile_min_run", I64)]


class FusedArgs(ctypes.Structure):
    """lora_fused_args (include/lora.h)."""
    _fields_ = [("ctx", P), ("table", P), ("ids", P), ("n", I64), ("x", P), ("ldx", I64),
                ("y", P), ("ldy", I64), ("d_in", I), ("d_out", I), ("stream", P)]


SIGNATURES = {
    "lora_version": ([], I),
    "lora_strerror": ([I], ctypes.c_char_p),
    "lora_last_cuda_error": ([P], ctypes.c_char_p),
    "lora_ctx_create": ([I, I64, I, ctypes.POINTER(P)], I),
    "lora_ctx_destroy": ([P], I),
    "lora_table_create": ([P, P, I64, I, P, I64, I, I, I, P, P, P, P, ctypes.POINTER(P)], I),
    "lora_table_destroy": ([P], I),
    "lora_table_invalidate": ([P, I], I),
    "lora_plan_build": ([P, P, P, I64, ctypes.POINTER(PlanView)], I),
    "lora_shrink": ([P, P, P, I64, P, I64, I, P, I64, P], I),
    "lora_expand": ([P, P, P, I64, P, I64, P, I64, I, P], I),
    "lora_fused": ([P, P, P, I64, P, I64, I, P, I64, I, P], I),
    "lora_fused_noalloc": ([P, P, P, I64, P, I64, I, P, I64, I, P], I),
    "lora_base_fused": ([P, P, P, I64, P, I64, I, P, I64, P, I64, I, P], I),
    "lora_merge": ([P, P, I, P, I64, I, I, P], I),
    "lora_unmerge": ([P, P, I, P, I64, I, I, P], I),
    "lora_page_in": ([P, P, I, P, I, P, I, P], I),
    "lora_fused_device_ids": ([P, P, P, I64, P, I64, I, P, I64, I, P], I),
    "lora_fused_args_call": ([ctypes.POINTER(FusedArgs)], I),
    "lora_fused_device_ids_args_call": ([ctypes.POINTER(FusedArgs)], I),
    "lora_selftest_timeout": ([P, I64, P], I),
    "lora_tiles_load": ([P, ctypes.c_char_p], I),
    "lora_tiles_save": ([P, ctypes.c_char_p], I),
    "lora_tiles_count": ([P], I64),
    "lora_tile_status": ([P], I),
    "lora_tune": ([P, ctypes.c_char_p, ctypes.c_char_p, P], I),
    "lora_tune_shape": ([P, P, I, P, I64, P, I64, I, P, I64, I, I, ctypes.POINTER(F), P], I),
    "lora_sync_status": ([P, P], I),
    "lora_last_path": ([P, ctypes.POINTER(I)], I),
    "lora_launch_count": ([P], I64),
    "lora_profile_begin": ([P, I], I),
    "lora_ctx_set_option": ([P, I, I], I),
    "lora_profile_end": ([P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(I64)], I),
}

_lib = None


def load(path: str = LIB_PATH):
    """Load liblora.so; raises if it is missing (there is no other implementation)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; "
            f"g.build()'` (needs nvcc); the package has no fallback implementation")
    lib = ctypes.CDLL(path)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def untyped(name: str):
    """A second foreign-function object for `name` with no argument types: called
    with ctypes instances, it passes them as they are, without the per-argument
    conversion that the typed object does on every call."""
    lib = load()
    fn = lib._FuncPtr((name, lib))
    fn.restype = SIGNATURES[name][1]
    return fn
