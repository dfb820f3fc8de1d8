"""ctypes loader of libmoe_gb300.so and the C signatures of include/moe_gb300.h.

The library is built in-tree by build.py.  Loading fails loudly when it is
missing: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libmoe_gb300.so")

c_int, c_size_t, c_void_p, c_float = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float
c_ull = ctypes.c_ulonglong

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5

MOE_FMT_BF16 = 0
MOE_FMT_NVFP4 = 1
MOE_FMT_MXFP8 = 2
MOE_FMT_MXFP4 = 3

MOE_EPI_STORE_BF16 = 0
MOE_EPI_SWIGLU_BF16 = 1
MOE_EPI_SWIGLU_NVFP4 = 2
MOE_EPI_SWIGLU_MX = 3


class MoeLayerC(ctypes.Structure):
    """Mirror of the C struct moe_layer."""
    _fields_ = [
        ("H", c_int), ("E", c_int), ("k", c_int), ("I", c_int), ("I_s", c_int),
        ("w_fmt", c_int), ("act_fmt", c_int),
        ("w13", c_void_p), ("w13_sf", c_void_p), ("w13_g", c_void_p),
        ("w2", c_void_p), ("w2_sf", c_void_p), ("w2_g", c_void_p),
        ("ws13", c_void_p), ("ws13_sf", c_void_p), ("ws13_g", c_void_p),
        ("ws2", c_void_p), ("ws2_sf", c_void_p), ("ws2_g", c_void_p),
        ("g_h", c_void_p), ("g_hs", c_void_p),
        ("no_renorm", c_int), ("ws_gate", c_void_p),
    ]


# name -> (restype, argtypes)
SIGNATURES = {
    "moe_version": (c_int, []),
    "moe_status_string": (ctypes.c_char_p, [c_int]),
    "moe_last_cuda_error": (ctypes.c_char_p, []),
    "moe_set_wait_timeout_ns": (c_int, [c_ull]),
    "moe_sync_status": (c_int, [c_void_p]),
    "moe_selftest_wait_timeout": (c_int, [c_ull, c_void_p]),
    "moe_route": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "moe_route_ex": (c_int, [c_void_p, c_int, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "moe_permute_workspace_size": (c_size_t, [c_int, c_int, c_int]),
    "moe_permute": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_int, c_void_p, c_int,
                            c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                            c_void_p, c_size_t, c_void_p]),
    "moe_permute_noalloc": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_int, c_void_p, c_int,
                                    c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "moe_route_permute_workspace_size": (c_size_t, [c_int, c_int, c_int]),
    "moe_route_permute": (c_int, [c_void_p, c_int, c_int, c_int, c_int, c_void_p, c_void_p,
                                  c_void_p, c_int, c_void_p, c_int,
                                  c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_size_t, c_void_p]),
    "moe_selftest_grid_barrier_timeout": (c_int, [c_ull, c_void_p]),
    "moe_quant_nvfp4_workspace_size": (c_size_t, [c_int]),
    "moe_quant_nvfp4": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p,
                                c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_quant_mx": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "moe_grouped_gemm": (c_int, [c_int, c_int, c_int, c_int, c_void_p, c_int, c_int, c_int,
                                 c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                 c_void_p, c_void_p, c_void_p, c_void_p]),
    "moe_combine": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                            c_void_p, c_void_p]),
    "moe_combine_gated": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                                  c_void_p, c_void_p]),
    "moe_shared_gate": (c_int, [c_void_p, c_void_p, c_int, c_int, c_void_p, c_void_p]),
    "moe_forward_workspace_size": (c_size_t, [ctypes.POINTER(MoeLayerC), c_int]),
    "moe_forward": (c_int, [ctypes.POINTER(MoeLayerC), c_void_p, c_void_p, c_int, c_void_p,
                            c_void_p, c_size_t, c_void_p]),
    "moe_forward_profiled": (c_int, [ctypes.POINTER(MoeLayerC), c_void_p, c_void_p, c_int, c_void_p,
                                     c_void_p, c_size_t, c_void_p, c_void_p]),
    "moe_forward_host": (c_int, [ctypes.POINTER(MoeLayerC), c_void_p, c_void_p, c_int, c_void_p,
                                 c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_forward_host_pipelined": (c_int, [ctypes.POINTER(MoeLayerC), c_int, c_void_p, c_void_p, c_int, c_void_p,
                                           c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p, c_void_p]),
    "moe_forward_graph_create": (c_int, [ctypes.POINTER(MoeLayerC), c_void_p, c_void_p, c_int, c_void_p,
                                         c_void_p, c_size_t, c_void_p, ctypes.POINTER(c_void_p)]),
    "moe_graph_launch": (c_int, [c_void_p, c_void_p]),
    "moe_graph_destroy": (c_int, [c_void_p]),
}

_lib = None


def load(path: str = LIB_PATH):
    """Load (once) and return the ctypes handle; raises if the library is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()' "
            "or python mixture_experts_layer_fwd_gb300/build.py)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        msg = lib.moe_status_string(status).decode()
        if status == MOE_ERR_CUDA:
            msg += " (" + lib.moe_last_cuda_error().decode() + ")"
        super().__init__(f"{where}: {msg}")
        self.status = status


def check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoEError(status, where)
