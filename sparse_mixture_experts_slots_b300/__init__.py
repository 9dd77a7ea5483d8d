"""B300-native (sm_103a) top-1 Switch MoE layer forward pass.

The layer runs in libswitch_moe.so (hand-written CUDA, C ABI in
include/switch_moe.h); this package only loads it and marshals arguments.
"""
from ._lib import SwitchError, load as load_library, LIB_PATH
from .layer import RouteResult, SwitchMoE

__all__ = ["SwitchMoE", "RouteResult", "SwitchError", "load_library", "LIB_PATH"]
