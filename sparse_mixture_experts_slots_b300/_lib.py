"""ctypes declarations of the C ABI in include/switch_moe.h (libswitch_moe.so).

Loading fails loudly when the library has not been built: there is no
fallback implementation behind this module.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_double, c_float, c_int, c_int32, c_int64, c_uint, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libswitch_moe.so")

SWITCH_OK = 0
SWITCH_ERR_INVALID_ARG = 1
SWITCH_ERR_UNSUPPORTED = 2
SWITCH_ERR_CUDA = 3
SWITCH_ERR_DEVICE_TIMEOUT = 4
SWITCH_ERR_OOM = 5
SWITCH_ERR_DEVICE_BOUNDS = 6

SWITCH_F32 = 0
SWITCH_BF16 = 1

FLAG_WRITE_PROBS = 0x1
FLAG_WRITE_LOGITS = 0x2
FLAG_DEBUG_BOUNDS = 0x4
FLAG_PROFILE = 0x8
FLAG_TOP2 = 0x10
FLAG_TRAINING = 0x20
FLAG_TEST_STALL = 0x40
FLAG_TEST_DISCARD = 0x80


class SwitchConfig(ctypes.Structure):
    _fields_ = [("G", c_int), ("T", c_int), ("d_model", c_int), ("d_ff", c_int), ("E", c_int),
                ("capacity_factor", c_double), ("capacity_override", c_int), ("alpha", c_float),
                ("dtype", c_int), ("flags", c_uint)]


ROUTE_FIELDS = ["expert", "slot", "keep", "gate", "row", "raw_count", "accepted_count", "P", "balance",
                "aux_loss_per_group", "aux_loss", "expert_rows", "probs", "logits", "z_loss_per_group", "z_loss",
                "expert2", "slot2", "keep2", "gate2", "row2", "raw2_count", "accepted2_count"]


class SwitchRouteOut(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ROUTE_FIELDS]


# name -> (restype, argtypes); every function declared in include/switch_moe.h
SIGNATURES = {
    "switch_capacity": (c_int64, [POINTER(SwitchConfig)]),
    "switch_expert_block_rows": (c_int64, [POINTER(SwitchConfig)]),
    "switch_status_string": (ctypes.c_char_p, [c_int]),
    "switch_create": (c_int, [POINTER(SwitchConfig), POINTER(c_void_p)]),
    "switch_destroy": (c_int, [c_void_p]),
    "switch_route": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, POINTER(SwitchRouteOut), c_void_p]),
    "switch_prepare_router": (c_int, [c_void_p, c_void_p, c_void_p]),
    "switch_dispatch": (c_int, [c_void_p, c_void_p, POINTER(SwitchRouteOut), c_void_p, c_void_p]),
    "switch_expert_ffn": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_void_p]),
    "switch_combine": (c_int, [c_void_p, c_void_p, POINTER(SwitchRouteOut), c_void_p, c_void_p, c_void_p]),
    "switch_forward": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                               c_void_p, POINTER(SwitchRouteOut), c_void_p, c_void_p, c_void_p]),
    "switch_backward": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, POINTER(SwitchRouteOut), c_void_p,
                                ctypes.c_float, ctypes.c_float, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                c_void_p, c_void_p, c_void_p, c_void_p]),
    "switch_forward_host": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_void_p, POINTER(SwitchRouteOut), c_int, c_void_p, c_void_p, c_void_p,
                                    c_void_p]),
    "switch_get_stats": (c_int, [c_void_p, POINTER(SwitchRouteOut), c_void_p, POINTER(c_float),
                                 POINTER(c_int32), POINTER(c_int32), POINTER(c_int64)]),
    "switch_sync_status": (c_int, [c_void_p, c_void_p]),
    "switch_stage_ms": (c_int, [c_void_p, POINTER(c_float), c_int]),
    "switch_last_launch_count": (c_int, [c_void_p]),
    "switch_set_sm_budget": (c_int, [c_void_p, c_int, c_int]),
    "switch_ep_regroup": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_void_p]),
    "switch_route_static": (c_int, [POINTER(SwitchConfig), c_void_p, c_void_p, c_void_p, POINTER(SwitchRouteOut),
                                    c_void_p]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libswitch_moe.so (once) and declare its signatures."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -m sparse_mixture_experts_slots_b300.build, or __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == LIB_PATH:
        _lib = lib
    return lib


class SwitchError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        lib = load()
        msg = lib.switch_status_string(status).decode()
        super().__init__(f"{what}: {msg} (status {status})" if what else msg)
        self.status = status


def check(status: int, what: str = "") -> None:
    if status != SWITCH_OK:
        raise SwitchError(status, what)
