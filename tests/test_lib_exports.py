"""The C-ABI library builds, loads without a GPU, and exports every function
declared in include/*.h; host-side argument checks reject bad input before
anything touches a device."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+\**\s*(moe_[a-z0-9_]+)\s*\(",
                             src, flags=re.M):
            names.append(m.group(1))
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from mixture_experts_layer_fwd_gb300 import _lib
    return _lib.load()


def test_header_declares_the_six_stage_calls():
    names = _declared_functions()
    for n in ["moe_route", "moe_permute", "moe_quant_nvfp4", "moe_grouped_gemm", "moe_combine", "moe_forward"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 10
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_symbol():
    from mixture_experts_layer_fwd_gb300 import _lib
    assert set(_declared_functions()) == set(_lib.SIGNATURES)


def test_version_and_status_strings(lib):
    assert lib.moe_version() == 100
    assert lib.moe_status_string(0) == b"MOE_OK"
    assert lib.moe_status_string(5) == b"MOE_ERR_TIMEOUT"


def test_host_argument_checks_without_gpu(lib):
    from mixture_experts_layer_fwd_gb300 import _lib as L
    # k > E, E too large, negative T: rejected on the host
    assert lib.moe_route(None, 4, 8, 9, None, None, None) == L.MOE_ERR_UNSUPPORTED
    assert lib.moe_route(None, 4, 2048, 2, None, None, None) == L.MOE_ERR_UNSUPPORTED
    assert lib.moe_route(None, -1, 8, 2, None, None, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_route(None, 4, 8, 2, None, None, None) == L.MOE_ERR_INVALID_ARG
    # T == 0 is a no-op
    assert lib.moe_route(None, 0, 8, 2, None, None, None) == L.MOE_OK
    assert lib.moe_combine(None, None, None, None, 0, 2, 256, None, None) == L.MOE_OK
    assert lib.moe_combine(None, None, None, None, 4, 2, 250, None, None) == L.MOE_ERR_UNSUPPORTED
    # quantiser: cols not a multiple of 16
    assert lib.moe_quant_nvfp4(None, 1, 4, 24, None, None, None, None, None, 0, None) == L.MOE_ERR_UNSUPPORTED
    # grouped GEMM: K not a multiple of 64
    assert lib.moe_grouped_gemm(0, 0, 0, 4, ctypes.c_void_p(256), 128, 256, 96, ctypes.c_void_p(256), None,
                                None, ctypes.c_void_p(256), None, None, ctypes.c_void_p(256), None, None,
                                None) == L.MOE_ERR_UNSUPPORTED
    # permute workspace grows with the number of chunks
    assert lib.moe_permute_workspace_size(0, 8, 128) == 0
    assert lib.moe_permute_workspace_size(16384, 8, 256) > lib.moe_permute_workspace_size(256, 8, 256)


def test_forward_layer_validation(lib):
    from mixture_experts_layer_fwd_gb300 import _lib as L
    c = L.MoeLayerC()
    c.H, c.E, c.k, c.I, c.I_s = 4096, 128, 8, 1536, 0
    c.w_fmt = c.act_fmt = L.MOE_FMT_BF16
    assert lib.moe_forward_workspace_size(ctypes.byref(c), 256) == 0  # no weights given
    c.w13, c.w2 = 4096, 8192
    n = lib.moe_forward_workspace_size(ctypes.byref(c), 256)
    # Xp + Y dominate: 2 * T*k*H*2 bytes
    assert n >= 2 * 256 * 8 * 4096 * 2
    assert lib.moe_forward_workspace_size(ctypes.byref(c), (1 << 27) // 8) == 0  # T*k past the limit
    c.H = 4000
    assert lib.moe_forward_workspace_size(ctypes.byref(c), 256) == 0
    c.H = 4096
    c.act_fmt = L.MOE_FMT_NVFP4  # NVFP4 activations need NVFP4 weights
    assert lib.moe_forward(ctypes.byref(c), None, None, 4, None, None, 0, None) == L.MOE_ERR_UNSUPPORTED


def test_quant_mx_checks_arguments_on_the_host(lib):
    from mixture_experts_layer_fwd_gb300 import _lib as L
    P = ctypes.c_void_p
    assert lib.moe_quant_mx(None, 0, 64, L.MOE_FMT_MXFP8, None, None, None) == L.MOE_OK  # no rows
    assert lib.moe_quant_mx(P(256), 4, 48, L.MOE_FMT_MXFP8, P(256), P(256), None) == L.MOE_ERR_UNSUPPORTED
    assert lib.moe_quant_mx(P(256), 4, 64, L.MOE_FMT_NVFP4, P(256), P(256), None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_quant_mx(P(264), 4, 64, L.MOE_FMT_MXFP4, P(256), P(256), None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_quant_mx(P(256), 4, 64, L.MOE_FMT_MXFP8, P(260), P(256), None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_quant_mx(P(256), -1, 64, L.MOE_FMT_MXFP8, P(256), P(256), None) == L.MOE_ERR_INVALID_ARG


def test_sizes_past_the_32_bit_thread_index_are_rejected(lib):
    """One warp per token (routing, shared gate) or per routed row
    (permutation, layer): 32 * rows threads must stay below 2^32."""
    from mixture_experts_layer_fwd_gb300 import _lib as L
    P = ctypes.c_void_p
    big = 1 << 27
    assert lib.moe_route(P(256), big, 8, 2, P(256), P(256), None) == L.MOE_ERR_UNSUPPORTED
    assert lib.moe_shared_gate(P(256), P(256), big, 256, P(256), None) == L.MOE_ERR_UNSUPPORTED
    assert lib.moe_permute(P(256), big // 4, 4, 8, None, 0, None, 0, P(256), P(256), P(256), P(256), None, None,
                           P(256), 1 << 40, None) == L.MOE_ERR_UNSUPPORTED


def test_mxfp4_grouped_gemm_checks_arguments_on_the_host(lib):
    from mixture_experts_layer_fwd_gb300 import _lib as L
    P = ctypes.c_void_p
    MX, NV = L.MOE_FMT_MXFP4, L.MOE_FMT_NVFP4

    def gemm(a_fmt, w_fmt, epi, K, sf=P(256)):
        return lib.moe_grouped_gemm(a_fmt, w_fmt, epi, 2, P(256), 256, 128, K, P(256), sf, None, P(256), sf, None,
                                    P(256), None, None, None)
    assert gemm(MX, NV, 0, 512) == L.MOE_ERR_UNSUPPORTED     # both operands MXFP4 or neither
    assert gemm(MX, MX, 2, 512) == L.MOE_ERR_UNSUPPORTED     # bf16 epilogues only
    assert gemm(MX, MX, 0, 768) == L.MOE_ERR_UNSUPPORTED     # K % 512 != 0
    assert gemm(MX, MX, 0, 512, sf=P(264)) == L.MOE_ERR_INVALID_ARG  # scales not 16-byte aligned
    assert gemm(MX, MX, 0, 512, sf=None) == L.MOE_ERR_INVALID_ARG
    M8 = L.MOE_FMT_MXFP8
    assert gemm(M8, MX, 0, 512) == L.MOE_ERR_UNSUPPORTED
    assert gemm(M8, M8, 0, 320) == L.MOE_ERR_UNSUPPORTED     # K % 256 != 0
    assert gemm(M8, M8, 0, 256, sf=P(260)) == L.MOE_ERR_INVALID_ARG  # scales not 8-byte aligned


def test_mx_layer_validation(lib):
    from mixture_experts_layer_fwd_gb300 import _lib as L
    c = L.MoeLayerC()
    c.H, c.E, c.k, c.I, c.I_s = 512, 8, 2, 512, 0
    c.w_fmt = c.act_fmt = L.MOE_FMT_MXFP4
    c.w13, c.w2, c.w13_sf, c.w2_sf = 4096, 8192, 12288, 16384
    assert lib.moe_forward_workspace_size(ctypes.byref(c), 64) > 0
    c.act_fmt = L.MOE_FMT_MXFP8  # weights and activations in the same MX format
    assert lib.moe_forward_workspace_size(ctypes.byref(c), 64) == 0
    c.act_fmt = L.MOE_FMT_MXFP4
    c.I = 256  # MXFP4 needs multiples of 512
    assert lib.moe_forward_workspace_size(ctypes.byref(c), 64) == 0
    c.w_fmt = c.act_fmt = L.MOE_FMT_MXFP8  # MXFP8: multiples of 256
    assert lib.moe_forward_workspace_size(ctypes.byref(c), 64) > 0
    c.w2_sf = None
    assert lib.moe_forward_workspace_size(ctypes.byref(c), 64) == 0
