"""ctypes binding of libattnres (include/attnres.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  There is no fallback: if the shared library is
missing or fails to load, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "libattnres.so")

ATTNRES_OK = 0
ATTNRES_EINVAL = -1
ATTNRES_EDTYPE = -2
ATTNRES_ERANGE = -4
ATTNRES_ECUDA = -5
ATTNRES_ESTATE = -6

ATTNRES_F32 = 0
ATTNRES_BF16 = 1

ATTNRES_DEVERR_WAIT_TIMEOUT = 0x1
ATTNRES_MAX_SOURCES = 128
ATTNRES_MAX_BLOCKS = ATTNRES_MAX_SOURCES - 1
ATTNRES_DEFAULT_EPS = 1e-5
ATTNRES_STATE_EARLY_LOADS = 0x1

# every function declared in include/attnres.h
EXPORTED = (
    "attnres_aggregate",
    "attnres_aggregate_fold",
    "attnres_aggregate_host",
    "attnres_aggregate_host_workspace_size",
    "attnres_aggregate_backward",
    "attnres_aggregate_backward_workspace_size",
    "attnres_aggregate_backward_noalloc",
    "attnres_interblock",
    "attnres_interblock_workspace_size",
    "attnres_intrablock_step",
    "attnres_state_init",
    "attnres_state_reset",
    "attnres_state_resume",
    "attnres_num_sources",
    "attnres_layer_sources",
    "attnres_block_step",
    "attnres_layer_step",
    "attnres_synthetic_layer",
    "attnres_synthetic_layer_backward",
    "attnres_fold",
    "attnres_debug_wait_test",
    "attnres_status_string",
    "attnres_last_error",
    "attnres_version",
)


class AttnresState(ctypes.Structure):
    """Mirror of `attnres_state` (natural C alignment)."""
    _fields_ = [
        ("h0", ctypes.c_void_p),
        ("block_reps", ctypes.c_void_p * ATTNRES_MAX_BLOCKS),
        ("partial", ctypes.c_void_p),
        ("T", ctypes.c_int64),
        ("d", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("num_layers", ctypes.c_int),
        ("block_size", ctypes.c_int),
        ("eps", ctypes.c_float),
        ("folded", ctypes.c_int),
        ("flags", ctypes.c_int),
    ]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libattnres.so not found at {LIB_PATH}; build it first "
            "(python depth_wise_attention_block_gb300/build.py). There is no CPU fallback.")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    sp = ctypes.POINTER(AttnresState)
    sig = {
        "attnres_aggregate": (i32, [ctypes.POINTER(vp), i32, i64, i32, i32, vp, f32, vp, i32, vp, vp, vp]),
        "attnres_aggregate_fold": (i32, [ctypes.POINTER(vp), i32, vp, vp, vp, i64, i32, i32, vp, f32, vp, vp, i32,
                                         vp, vp]),
        "attnres_aggregate_host": (i32, [ctypes.POINTER(vp), i32, i64, i32, i32, vp, f32, vp, i32, vp, i64, vp,
                                          i64, vp, vp]),
        "attnres_aggregate_host_workspace_size": (i64, [i32, i64, i32, i32, i32, i32, i32]),
        "attnres_aggregate_backward": (i32, [ctypes.POINTER(vp), i32, i64, i32, i32, vp, f32, vp,
                                              ctypes.POINTER(vp), i32, vp, vp, i64, vp, vp]),
        "attnres_aggregate_backward_workspace_size": (i64, [i64, i32]),
        "attnres_aggregate_backward_noalloc": (i32, [ctypes.POINTER(vp), i32, i64, i32, i32, vp, f32, vp,
                                                      ctypes.POINTER(vp), i32, vp, vp, vp]),
        "attnres_interblock": (i32, [ctypes.POINTER(vp), i32, i64, i32, i32, ctypes.POINTER(vp), i32, f32, vp, vp,
                                      vp, vp, vp, vp, i64, vp, vp]),
        "attnres_interblock_workspace_size": (i64, [i32, i64, i32, i32, i32]),
        "attnres_intrablock_step": (i32, [sp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp]),
        "attnres_state_init": (i32, [sp, vp, ctypes.POINTER(vp), i32, vp, i64, i32, i32, i32, i32, f32]),
        "attnres_state_reset": (i32, [sp]),
        "attnres_state_resume": (i32, [sp, i32]),
        "attnres_num_sources": (i32, [i32, i32, i32]),
        "attnres_layer_sources": (i32, [sp, i32, ctypes.POINTER(vp), ctypes.POINTER(i32)]),
        "attnres_block_step": (i32, [sp, vp, i32, vp, vp]),
        "attnres_layer_step": (i32, [sp, vp, vp, i32, vp, vp, vp, vp]),
        "attnres_synthetic_layer": (i32, [vp, vp, vp, vp, i64, i32, i32, vp]),
        "attnres_synthetic_layer_backward": (i32, [vp, vp, vp, vp, vp, vp, i64, i32, i32, vp]),
        "attnres_fold": (i32, [vp, vp, vp, i64, i32, i32, vp]),
        "attnres_debug_wait_test": (i32, [ctypes.c_uint64, i32]),
        "attnres_status_string": (ctypes.c_char_p, [i32]),
        "attnres_last_error": (ctypes.c_char_p, []),
        "attnres_version": (i32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class AttnresError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib.attnres_status_string(status).decode()
        detail = lib.attnres_last_error().decode()
        super().__init__(f"{where}: {msg}" + (f" ({detail})" if detail else ""))


def check(status: int, where: str) -> int:
    if status < 0:
        raise AttnresError(status, where)
    return status
