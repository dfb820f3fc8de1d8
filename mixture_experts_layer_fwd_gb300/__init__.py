"""GB300 (sm_103a) top-k routed MoE FFN layer forward.

The compute runs in the C-ABI CUDA library libmoe_gb300.so (declared in
include/moe_gb300.h, built in-tree by build.py); this package is its thin
Python binding.  Importing the package does not load the library; the first
call does, and fails loudly if the library has not been built.
"""
from .api import (MOE_EPI_STORE_BF16, MOE_EPI_SWIGLU_BF16, MOE_EPI_SWIGLU_MX, MOE_EPI_SWIGLU_NVFP4, MOE_FMT_BF16,
                  MOE_FMT_MXFP4, MOE_FMT_MXFP8, MOE_FMT_NVFP4, ForwardGraph, moe_combine, moe_forward,
                  moe_forward_host, moe_forward_host_pipelined, moe_forward_profiled, moe_forward_workspace_size, moe_grouped_gemm, moe_permute,
                  moe_permute_noalloc, moe_quant_mx, moe_quant_nvfp4, moe_route, moe_route_permute,
                  moe_selftest_grid_barrier_timeout, moe_selftest_wait_timeout, moe_set_wait_timeout_ns,
                  moe_shared_gate, moe_sync_status, moe_version)
from .layer import MoELayer, NVFP4Tensor, quantize_weights

__all__ = ["MOE_EPI_STORE_BF16", "MOE_EPI_SWIGLU_BF16", "MOE_EPI_SWIGLU_MX", "MOE_EPI_SWIGLU_NVFP4", "MOE_FMT_BF16", "MOE_FMT_NVFP4",
           "MOE_FMT_MXFP8", "MOE_FMT_MXFP4", "moe_quant_mx",
           "ForwardGraph", "moe_combine", "moe_forward", "moe_forward_host", "moe_forward_host_pipelined", "moe_forward_profiled",
           "moe_forward_workspace_size", "moe_grouped_gemm", "moe_permute", "moe_permute_noalloc", "moe_quant_nvfp4",
           "moe_route", "moe_route_permute", "moe_selftest_grid_barrier_timeout", "moe_selftest_wait_timeout", "moe_set_wait_timeout_ns", "moe_shared_gate", "moe_sync_status",
           "moe_version", "MoELayer", "NVFP4Tensor", "quantize_weights"]
