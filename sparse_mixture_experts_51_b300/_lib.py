"""ctypes loader for libmoe_b300.so (built in-tree by ``build.py``).

The library is the product: there is no fallback.  If it is missing or a
symbol cannot be resolved, loading raises immediately.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
                4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_TIMEOUT", 6: "MOE_ERR_BOUNDS"}
MOE_F32, MOE_BF16 = 0, 1
MOE_ACT_GELU, MOE_ACT_SWIGLU = 0, 1
MOE_ROUTE_TOKEN_CHOICE, MOE_ROUTE_EXPERT_CHOICE = 0, 1
MOE_GATES_RENORM, MOE_GATES_RAW = 0, 1
MOE_OVERFLOW_DROP, MOE_OVERFLOW_REROUTE = 0, 1


class MoeShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("d_ff", ctypes.c_int32), ("dtype", ctypes.c_int32), ("act", ctypes.c_int32),
                ("d_ff_shared", ctypes.c_int32), ("routing", ctypes.c_int32), ("gates", ctypes.c_int32),
                ("overflow", ctypes.c_int32)]


class MoeShared(ctypes.Structure):
    """moe_shared_t: the shared experts' weights (device pointers)."""
    _fields_ = [("W1s", ctypes.c_void_p), ("W3s", ctypes.c_void_p), ("W2s", ctypes.c_void_p),
                ("b1s", ctypes.c_void_p), ("b2s", ctypes.c_void_p)]


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where} failed: {STATUS_NAMES.get(status, status)}")


_P = ctypes.c_void_p
_SHAPE = ctypes.POINTER(MoeShape)

SIGNATURES = {
    "moe_capacity": (ctypes.c_int32, [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_double]),
    "moe_max_rows": (ctypes.c_int64, [_SHAPE, ctypes.c_int32]),
    "moe_workspace_size": (ctypes.c_int, [_SHAPE, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)]),
    "moe_route": (ctypes.c_int, [_SHAPE, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_route_expert_choice": (ctypes.c_int, [_SHAPE, ctypes.c_int32] + [_P] * 10 + [ctypes.c_size_t, _P]),
    "moe_dispatch": (ctypes.c_int, [_SHAPE, ctypes.c_int32, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                    ctypes.c_size_t, _P]),
    "moe_dispatch_noalloc": (ctypes.c_int, [_SHAPE, ctypes.c_int32] + [_P] * 10),
    "moe_expert_ffn": (ctypes.c_int, [_SHAPE, ctypes.c_int32, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                      ctypes.c_size_t, _P]),
    "moe_combine": (ctypes.c_int, [_SHAPE, ctypes.c_int32] + [_P] * 10),
    "moe_shared_ffn": (ctypes.c_int, [_SHAPE, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_forward": (ctypes.c_int, [_SHAPE, ctypes.c_double, ctypes.c_int32] + [_P] * 22
                    + [ctypes.c_size_t, _P]),
    "moe_forward_timed": (ctypes.c_int, [_SHAPE, ctypes.c_double, ctypes.c_int32] + [_P] * 22
                          + [ctypes.c_size_t, _P, ctypes.POINTER(ctypes.c_void_p)]),
    "moe_routing_stats": (ctypes.c_int, [_SHAPE] + [_P] * 8 + [ctypes.c_size_t, _P]),
    "moe_get_device_error": (ctypes.c_int, [_P, _P]),
    "moe_kernel_launches": (ctypes.c_ulonglong, []),
    "moe_testing_dispatch_stalled": (ctypes.c_int, [_SHAPE, ctypes.c_int32] + [_P] * 7
                                     + [ctypes.c_int32, _P, ctypes.c_size_t, _P]),
    "moe_testing_router_filter": (ctypes.c_int, [_SHAPE] + [_P] * 5 + [ctypes.c_size_t, _P]),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the shared library once and attach the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -m sparse_mixture_experts_51_b300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, where)
