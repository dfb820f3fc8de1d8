"""The Python binding refuses tensors that a kernel would read or write at
the wrong place before it calls into the library.  On a machine without a
GPU every tensor is a host tensor, so each wrapper must raise instead of
passing a host address to a launch."""
import pytest
import torch

import mixture_experts_layer_fwd_gb300 as m
from mixture_experts_layer_fwd_gb300._lib import MoeLayerC


def _layer_c(H=256, E=8, k=2, I=128):
    c = MoeLayerC()
    c.H, c.E, c.k, c.I, c.I_s = H, E, k, I, 0
    return c


def test_stage_calls_reject_host_tensors():
    bf = torch.bfloat16
    with pytest.raises(ValueError, match="CUDA"):
        m.moe_route(torch.zeros(4, 8), 2)
    with pytest.raises(ValueError, match="CUDA"):
        m.moe_permute(torch.zeros(4, 2, dtype=torch.int32), 8)
    with pytest.raises(ValueError, match="CUDA"):
        m.moe_permute_noalloc(torch.zeros(4, 2, dtype=torch.int32), 8)
    with pytest.raises(ValueError, match="CUDA"):
        m.moe_quant_nvfp4(torch.zeros(4, 16, dtype=bf))
    with pytest.raises(ValueError, match="CUDA"):
        m.moe_grouped_gemm(0, 0, 0, torch.tensor([0, 4], dtype=torch.int32), 128, 64,
                           torch.zeros(4, 64, dtype=bf), torch.zeros(1, 128, 64, dtype=bf))
    with pytest.raises(ValueError, match="CUDA"):
        m.moe_combine(torch.zeros(8, 256, dtype=bf), torch.zeros(4, 2, dtype=torch.int32),
                      torch.zeros(4, 2), None, 4, 2, 256)
    with pytest.raises(ValueError, match="CUDA"):
        m.moe_shared_gate(torch.zeros(4, 256, dtype=bf), torch.zeros(256, dtype=bf))


def test_layer_calls_reject_host_tensors():
    c = _layer_c()
    x = torch.zeros(4, 256, dtype=torch.bfloat16)
    logits = torch.zeros(4, 8)
    out = torch.zeros(4, 256, dtype=torch.bfloat16)
    ws = torch.zeros(1024, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA"):
        m.moe_forward(c, x, logits, out, ws)
    with pytest.raises(ValueError, match="CUDA"):
        m.moe_forward_profiled(c, x, logits, out, ws, [None] * 6)
    with pytest.raises(ValueError, match="CUDA"):
        # the device-side buffers of the host entry point must be on a GPU
        m.moe_forward_host(c, x, logits, out, x, logits, out, ws)
    with pytest.raises(ValueError, match="CUDA"):
        m.api.ForwardGraph(c, x, logits, out, ws)  # and its destructor has nothing to free
    x2, lg2, out2 = x.expand(2, 4, 256).contiguous(), logits.expand(2, 4, 8).contiguous(), out.expand(2, 4, 256).contiguous()
    with pytest.raises(ValueError, match="CUDA"):
        m.moe_forward_host_pipelined(c, [x], [logits], [out], x2, lg2, out2, ws)
    with pytest.raises(ValueError, match="n >= 1"):
        m.moe_forward_host_pipelined(c, [], [], [], x2, lg2, out2, ws)
    with pytest.raises(ValueError, match="6"):
        m.moe_forward_profiled(c, x, logits, out, ws, [None] * 7)


def test_layer_rejects_host_weights_and_unknown_formats():
    w13 = torch.zeros(4, 256, 256, dtype=torch.bfloat16)
    w2 = torch.zeros(4, 256, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        m.MoELayer(256, 4, 2, 128, 0, w13, w2)
    with pytest.raises(ValueError, match="formats"):
        m.MoELayer(256, 4, 2, 128, 0, w13, w2, w_fmt="fp8")


def test_missing_operand_is_named():
    with pytest.raises(ValueError, match="A: required"):
        m.moe_grouped_gemm(0, 0, 0, None, 128, 64, None, None)


def test_every_binding_is_exported_by_the_package():
    """What api.py binds is reachable as mixture_experts_layer_fwd_gb300.<name>,
    and every C entry point of the header that takes tensors has a wrapper."""
    from mixture_experts_layer_fwd_gb300 import _lib, api
    assert set(api.__all__) <= set(m.__all__)
    for name in api.__all__:
        assert getattr(m, name) is getattr(api, name)
    size_queries = {n for n in _lib.SIGNATURES if n.endswith("_workspace_size") or n.endswith("_size")}
    handled_elsewhere = {"moe_status_string", "moe_last_cuda_error", "moe_route_ex", "moe_combine_gated",
                         "moe_forward_graph_create", "moe_graph_launch", "moe_graph_destroy"}
    missing = set(_lib.SIGNATURES) - set(api.__all__) - size_queries - handled_elsewhere
    assert not missing, sorted(missing)
