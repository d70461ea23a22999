"""ctypes loader for libqlora.so: declares the C ABI of include/qlora.h.  No fallback: if the
library is missing or cannot be loaded, every call raises."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqlora.so")
# the same library built with device-side bounds checks (build.build(checks=True)); a process
# selects it with QLORA_LIB=checked before the first call
CHECKED_LIB_PATH = os.path.join(HERE, "libqlora_checked.so")
if os.environ.get("QLORA_LIB") == "checked":
    LIB_PATH = CHECKED_LIB_PATH

QLORA_STATUS = {
    0: "QLORA_OK", 1: "QLORA_ERR_INVALID_ARG", 2: "QLORA_ERR_UNSUPPORTED_SHAPE", 3: "QLORA_ERR_MISALIGNED",
    4: "QLORA_ERR_WORKSPACE", 5: "QLORA_ERR_CUDA", 6: "QLORA_ERR_TIMEOUT", 7: "QLORA_ERR_DEVICE_CHECK",
}

# every function declared in include/qlora.h
EXPORTS = (
    "qlora_nf4_storage_bytes", "qlora_quantize_workspace_bytes", "qlora_fwd_workspace_bytes",
    "qlora_bwd_workspace_bytes", "nf4_quantize", "nf4_dequantize", "qlora_linear_fwd", "qlora_linear_bwd",
    "qlora_merge_workspace_bytes", "qlora_merge",
    "qlora_cat_fwd_workspace_bytes", "qlora_cat_bwd_workspace_bytes", "qlora_linear_fwd_cat", "qlora_linear_bwd_cat",
    "qlora_fwd_dropout_workspace_bytes", "qlora_bwd_dropout_workspace_bytes", "qlora_linear_fwd_dropout",
    "qlora_linear_bwd_dropout",
    "qlora_check_device_error", "qlora_test_inject", "qlora_status_string", "qlora_launch_count",
    "qlora_nf4_levels",
    "qlora_set_kernel_timer", "qlora_kernel_timer_count", "nf4_quantize_noalloc",
    "qlora_paged_alloc", "qlora_paged_free", "qlora_paged_prefetch", "qlora_adamw_step",
)

QLORA_PAGE_HOST = -1
QLORA_INJECT_SKIP_CODES = 1
QLORA_INJECT_BOUNDS = 2


class NF4TensorStruct(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("codes", ctypes.c_void_p),
                ("scale_codes", ctypes.c_void_p), ("scale_scales", ctypes.c_void_p),
                ("scale_offset", ctypes.c_void_p)]


class DropoutStruct(ctypes.Structure):
    _fields_ = [("p", ctypes.c_float), ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint64)]


class AdamWStruct(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float)]


class CatModuleStruct(ctypes.Structure):
    _fields_ = [("W", ctypes.POINTER(NF4TensorStruct)), ("A", ctypes.c_void_p), ("B", ctypes.c_void_p),
                ("r", ctypes.c_int32), ("alpha", ctypes.c_float)]


_lib = None


def load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libqlora.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    ST = ctypes.POINTER(NF4TensorStruct)
    sig = {
        "qlora_nf4_storage_bytes": (SZ, [I64, I64]),
        "qlora_quantize_workspace_bytes": (SZ, [I64, I64]),
        "qlora_fwd_workspace_bytes": (SZ, [I64, I64, I64, I32]),
        "qlora_bwd_workspace_bytes": (SZ, [I64, I64, I64, I32]),
        "qlora_merge_workspace_bytes": (SZ, [I64, I64, I32]),
        "qlora_merge": (ctypes.c_int, [ST, P, P, I32, ctypes.c_float, P, P, SZ, P]),
        "qlora_cat_fwd_workspace_bytes": (SZ, [P, P, I32, I64, I64]),
        "qlora_cat_bwd_workspace_bytes": (SZ, [P, P, I32, I64, I64]),
        "qlora_linear_fwd_cat": (ctypes.c_int, [P, I32, P, I64, P, P, P, SZ, P]),
        "qlora_linear_bwd_cat": (ctypes.c_int, [P, I32, P, I64, P, P, P, P, P, P, SZ, P]),
        "qlora_fwd_dropout_workspace_bytes": (SZ, [I64, I64, I64, I32]),
        "qlora_bwd_dropout_workspace_bytes": (SZ, [I64, I64, I64, I32]),
        "qlora_linear_fwd_dropout": (ctypes.c_int, [ST, P, I64, P, P, I32, ctypes.c_float, P, P, P, P, SZ, P]),
        "qlora_linear_bwd_dropout": (ctypes.c_int, [ST, P, I64, P, P, I32, ctypes.c_float, P, P, P, P, P, P, P, SZ,
                                                    P]),
        "nf4_quantize": (ctypes.c_int, [P, ST, P, SZ, P]),
        "nf4_dequantize": (ctypes.c_int, [ST, P, P]),
        "nf4_quantize_noalloc": (ctypes.c_int, [P, ST, P]),
        "qlora_linear_fwd": (ctypes.c_int, [ST, P, I64, P, P, I32, ctypes.c_float, P, P, P, SZ, P]),
        "qlora_linear_bwd": (ctypes.c_int, [ST, P, I64, P, P, I32, ctypes.c_float, P, P, P, P, P, P, SZ, P]),
        "qlora_check_device_error": (ctypes.c_int, [P]),
        "qlora_test_inject": (ctypes.c_int, [ctypes.c_uint32]),
        "qlora_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "qlora_launch_count": (ctypes.c_uint64, []),
        "qlora_nf4_levels": (None, [P]),
        "qlora_set_kernel_timer": (ctypes.c_int, [P, I32]),
        "qlora_kernel_timer_count": (I32, []),
        "qlora_paged_alloc": (ctypes.c_int, [SZ, ctypes.POINTER(ctypes.c_void_p)]),
        "qlora_paged_free": (ctypes.c_int, [P]),
        "qlora_paged_prefetch": (ctypes.c_int, [P, SZ, I32, P]),
        "qlora_adamw_step": (ctypes.c_int, [ctypes.POINTER(AdamWStruct), I64, I64, P, P, P, P, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L
