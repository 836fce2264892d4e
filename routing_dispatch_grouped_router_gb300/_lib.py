"""ctypes view of libmok.so (include/mok.h).  Argument marshalling only."""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libmok.so")

c_void_p = ctypes.c_void_p
c_size_t = ctypes.c_size_t
c_int64 = ctypes.c_int64
c_int32 = ctypes.c_int32


class MoeDesc(ctypes.Structure):
    _fields_ = [("T", c_int64), ("d", c_int64), ("E", c_int64), ("I", c_int64),
                ("k", c_int32), ("dtype", c_int32), ("mb_tokens", c_int32),
                ("ring_slots", c_int32), ("flags", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


class SavedLayout(ctypes.Structure):
    _fields_ = [(n, c_size_t) for n in (
        "status", "topk_idx", "topk_w", "counts", "offsets", "pos", "token_of_row",
        "padded_offsets", "padded_pos", "padded_token", "row_weight", "x_perm", "gate_up",
        "nv_weight_scales", "w_gate_up_t", "w_down_col", "rows_max", "mb_count", "mb_stride", "ring_slots", "ring_slot_bytes", "total")]


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", c_int32), ("total_ms", ctypes.c_double)]


# name -> (restype, argtypes)
_SIGS = {
    "mok_moe_workspace_size": (c_int32, [ctypes.POINTER(MoeDesc), ctypes.POINTER(c_size_t),
                                         ctypes.POINTER(c_size_t), ctypes.POINTER(c_size_t)]),
    "mok_moe_saved_layout": (c_int32, [ctypes.POINTER(MoeDesc), ctypes.POINTER(SavedLayout)]),
    "mok_moe_forward": (c_int32, [ctypes.POINTER(MoeDesc), c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_void_p, c_void_p, c_size_t, c_void_p, c_size_t,
                                  c_void_p]),
    "mok_moe_backward": (c_int32, [ctypes.POINTER(MoeDesc), c_void_p, c_void_p, c_void_p, c_void_p,
                                   c_void_p, c_void_p, c_void_p, c_size_t, c_void_p, c_void_p,
                                   c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "mok_moe_stage_workspace_size": (c_int32, [ctypes.POINTER(MoeDesc), ctypes.POINTER(c_size_t)]),
    "mok_moe_route": (c_int32, [ctypes.POINTER(MoeDesc), c_void_p, c_void_p, c_void_p, c_void_p,
                                c_void_p, c_void_p, c_size_t, c_void_p]),
    "mok_moe_dispatch_plan": (c_int32, [ctypes.POINTER(MoeDesc), c_void_p, c_void_p, c_void_p,
                                        c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "mok_moe_dispatch_plan_noalloc": (c_int32, [ctypes.POINTER(MoeDesc), c_void_p, c_void_p,
                                                c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "mok_mx_quantize": (c_int32, [c_void_p, c_int64, c_int64, c_int32, c_void_p, c_void_p,
                                  c_void_p, c_void_p]),
    "mok_gemm_bf16": (c_int32, [c_int64, c_int64, c_int64, c_void_p, c_int32, c_void_p, c_int32,
                                c_void_p, c_void_p, c_size_t, c_void_p]),
    "mok_gemm_mxfp8": (c_int32, [c_int64, c_int64, c_int64, c_void_p, c_void_p, c_void_p,
                                 c_void_p, c_void_p, c_int32, c_void_p, c_size_t, c_void_p]),
    "mok_nvfp4_tensor_scale": (c_int32, [c_void_p, c_int64, c_void_p, c_void_p]),
    "mok_nvfp4_quantize": (c_int32, [c_void_p, c_int64, c_int64, c_void_p, c_void_p, c_void_p,
                                     c_void_p]),
    "mok_nvfp4_quantize_cols": (c_int32, [c_void_p, c_int64, c_int64, c_int64, c_void_p,
                                          c_void_p, c_void_p, c_void_p]),
    "mok_gemm_nvfp4": (c_int32, [c_int64, c_int64, c_int64, c_void_p, c_void_p, c_void_p,
                                 c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                 c_void_p]),
    "mok_selftest_bounded_wait": (c_int32, [c_void_p, c_size_t, c_void_p]),
    "mok_fill_zero": (c_int32, [c_void_p, c_size_t, c_void_p]),
    "mok_get_device_status": (c_int32, [c_void_p, c_void_p, ctypes.POINTER(c_int32)]),
    "mok_status_string": (ctypes.c_char_p, [c_int32]),
    "mok_last_launch_count": (c_int32, []),
    "mok_profile_enable": (c_int32, [c_int32]),
    "mok_profile_reset": (c_int32, []),
    "mok_profile_collect": (c_int32, [ctypes.POINTER(KernelTime), c_int32, ctypes.POINTER(c_int32)]),
}

_lib = None


def load(path: str | None = None):
    """Loads libmok.so once.  Raises when it has not been built: there is no
    other implementation to fall back to."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with "
                           "`python -m routing_dispatch_grouped_router_gb300.build`")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def exported_names():
    return list(_SIGS)


class MokError(RuntimeError):
    def __init__(self, code: int, where: str):
        lib = load()
        super().__init__(f"{where}: {lib.mok_status_string(code).decode()} (code {code})")
        self.code = code


def check(code: int, where: str):
    if code != 0:
        raise MokError(code, where)
