"""MX layers (MXFP8 and MXFP4 weights and activations) through moe_forward
against the fp64 oracle on every token: x quantised in blocks of 32 along
H, h quantised the same way along I from its fp32 value, weights encoded by
the oracle's own MX codec from the bf16 masters.  Tolerance 1e-2 relative
Frobenius (as for the NVFP4 layers)."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from tests.helpers import OracleWeights, oracle_layer, require_gpu, to_np_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def mx_layer(fmt):
    """Small MX layers: Qwen3-235B-like (no shared expert) in MXFP8, the
    format the pages serve it in, and DeepSeek-V3-like (shared expert, the
    shared problem of the same launch) in MXFP8 and MXFP4."""
    if fmt == "mxfp8":
        base = synth.small_variant(synth.QWEN3_235B, H=512, E=16, k=4, I=256, name="qwen3-mxfp8-small")
        return dataclasses.replace(base, w_fmt=fmt, act_fmt=fmt)
    base = synth.small_variant(synth.DEEPSEEK_V3, H=512, E=16, k=4, I=512, I_s=512, name=f"ds-{fmt}-small")
    fmt = fmt.replace("-shared", "")
    return dataclasses.replace(base, w_fmt=fmt, act_fmt=fmt)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp8-shared", "mxfp4"])
@pytest.mark.parametrize("T", [1, 37, 300])
def test_mx_layer_all_tokens(fmt, T):
    from mixture_experts_layer_fwd_gb300 import MoELayer, moe_sync_status
    cfg = mx_layer(fmt)
    acts = synth.make_activations(cfg, T, seed=T)
    w = synth.make_weights(cfg, seed=0, device=DEV)
    layer = MoELayer.from_config(cfg, w)
    out = layer(acts.x.to(DEV), acts.logits.to(DEV))
    assert moe_sync_status() == 0
    got = to_np_f32(out)
    ref, *_ = oracle_layer(cfg, acts, OracleWeights(cfg, w))
    err = oracle.rel_frobenius(got, ref)
    assert err <= 1e-2, err
