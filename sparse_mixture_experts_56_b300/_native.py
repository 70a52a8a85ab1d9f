"""ctypes loader for libmoe.so (the C ABI declared in include/moe.h).

The library must have been built (``python -m sparse_mixture_experts_56_b300.build``);
there is no fallback of any kind: a missing library raises at first use.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe.so")

MOE_F32 = 0
MOE_BF16 = 1

MOE_TC_FORM_AUTO = 0
MOE_TC_FORM_SINGLE = 1
MOE_TC_FORM_PAIR = 2
MOE_TC_FORM_SWAP = 3

STATUS_NAMES = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
    4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_DEVICE_INDEX",
}

# name -> (restype, argtypes); mirrors include/moe.h
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_F = ctypes.c_float
SIGNATURES = {
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_version": (_I, []),
    "moe_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "moe_router_topk": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    "moe_permute": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute_noalloc": (_I, [_P, _I, _I, _I, _P, _P, _P, _P]),
    "moe_grouped_swiglu": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "moe_expert_up": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "moe_expert_down": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "moe_combine": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "moe_rmsnorm": (_I, [_P, _I, _I, _F, _I, _P, _P]),
    "moe_layer_forward": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P,
                               _SZ, _P]),
    "moe_routing_stats": (_I, [_P, _I, _I, _I, _I, _P, _P, _P]),
    "moe_attention_gqa": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "moe_backward_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "moe_train_saved_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "moe_layer_forward_train": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ,
                                     _P, _SZ, _P]),
    "moe_layer_backward_saved": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _SZ, _P,
                                      _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_layer_backward": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P,
                                _P, _P, _P, _SZ, _P]),
    "moe_decoder_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "moe_decoder_layer_forward": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                       _I, _I, _I, _F, _I, _P, _P, _P, _SZ, _P]),
    "moe_ep_regroup": (_I, [_P, _I, _I, _I, _P, _P, _P, _P]),
    "moe_gather_rows": (_I, [_P, _I, _P, _I, _I, _SZ, _P, _P]),
    "moe_check_device_error": (_I, [_P, _SZ, _P]),
    "moe_set_wait_limit_ns": (None, [ctypes.c_ulonglong]),
    "moe_set_tc_form": (_I, [_I]),
}

_lib = None
_lock = threading.Lock()


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded library (loaded once).  Raises OSError if libmoe.so is missing."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise OSError(f"{LIB_PATH} is missing: build it with "
                                  "`python -m sparse_mixture_experts_56_b300.build`")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def check(fn: str, status: int) -> None:
    if status != 0:
        raise MoEError(fn, status)
