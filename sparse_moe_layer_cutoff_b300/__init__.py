"""Stable LatentMoE layer forward for one B300 (sm_103a): a C-ABI CUDA library
(liblmoe.so, declared in include/lmoe.h) and its thin Python binding."""
from .lmoe import (DenseFFN, LatentMoE, LmoeError, lmoe_build_info, lmoe_create, lmoe_destroy, lmoe_forward,
                   lmoe_route, lmoe_status_string, lmoe_sync_status, lmoe_workspace, load_library)

__all__ = ["DenseFFN", "LatentMoE", "LmoeError", "lmoe_build_info", "lmoe_create", "lmoe_destroy", "lmoe_forward",
           "lmoe_route", "lmoe_status_string", "lmoe_sync_status", "lmoe_workspace", "load_library"]
