"""Shared helpers of the GPU parity tests: oracle-side weight decoding and
the layer runner.  Every expected value here is computed by oracle/ from the
seeded inputs of synth/; nothing is read back from the CUDA path except the
results under test."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
from oracle import mx, nvfp4

F32 = np.float32


def require_gpu():
    import pytest
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g
    g.build()


def to_np_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float32).numpy()


class OracleWeights:
    """Oracle view of the master weights: fp64 dequantised per expert, with
    the oracle's own NVFP4 quantiser on the NVFP4 workloads (one global scale
    per expert and projection, like the CUDA path's weight preparation)."""

    def __init__(self, cfg: synth.LayerConfig, master: synth.MasterWeights, cache: bool = True,
                 zero_experts=()):
        """cache=False decodes each expert when asked and keeps nothing (host
        memory stays at one expert on the full-size workloads).
        zero_experts: experts whose master weights the caller has set to
        zero; the oracle skips them (expert() returns None, see
        oracle.forward)."""
        self.cfg, self.m = cfg, master
        self.cache = {}
        self.keep = cache
        self.zero = set(int(e) for e in zero_experts)

    def _decode(self, w: torch.Tensor):
        a = to_np_f32(w)
        if self.cfg.w_fmt == "bf16":
            return a.astype(np.float64), None
        if self.cfg.w_fmt.startswith("mx"):
            q, s = mx.quantize(a, self.cfg.w_fmt)
            return mx.dequantize(q, s, self.cfg.w_fmt), (q, s)
        q, s, g = nvfp4.quantize(a)
        return nvfp4.dequantize(q, s, g), (q, s, g)

    def expert(self, e: int):
        if e in self.zero:
            return None
        if e in self.cache:
            return self.cache[e]
        w13, _ = self._decode(self.m.w13[e])
        w2, _ = self._decode(self.m.w2[e])
        ew = oracle.ExpertWeights(w13, w2)
        if self.keep:
            self.cache[e] = ew
        return ew

    def expert_codes(self, e: int):
        """Oracle NVFP4 encoding of expert e: ((q13, s13, g13), (q2, s2, g2))."""
        return self._decode(self.m.w13[e])[1], self._decode(self.m.w2[e])[1]

    def shared(self):
        if self.cfg.I_s == 0:
            return None
        if "shared" not in self.cache:
            w13, _ = self._decode(self.m.ws13)
            w2, _ = self._decode(self.m.ws2)
            self.cache["shared"] = oracle.ExpertWeights(w13, w2)
        return self.cache["shared"]


def oracle_layer(cfg: synth.LayerConfig, acts: synth.Activations, ow: OracleWeights, tokens=None,
                 renorm: bool = True, shared_g=None):
    """Oracle output (fp64) for the given tokens, plus idx / w / perm over all T.
    renorm / shared_g select the router and shared-gate variants (the gate sees
    the bf16 activations)."""
    x = to_np_f32(acts.x)
    hq = None
    if cfg.act_fmt == "nvfp4":
        # one global scale over the whole input; every row is then quantised
        # on its own (blocks of 16 inside the row), so only the rows of the
        # requested tokens are encoded (the others are never read)
        g = nvfp4.global_scale(x)
        rows = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
        x_deq = np.zeros(x.shape, np.float64)
        if len(rows):
            q, s, _ = nvfp4.quantize(x[rows], g)
            x_deq[rows] = nvfp4.dequantize(q, s, g)
        gh = F32(cfg.g_h)
    elif cfg.act_fmt.startswith("mx"):
        x_deq = mx.fake_quant(x, cfg.act_fmt)  # blocks of 32 along H, no global scale
        gh = None
        hq = mx.h_quant(cfg.act_fmt)
    else:
        x_deq = x.astype(np.float64)
        gh = None
    return oracle.forward(x_deq, acts.logits.numpy(), cfg.k, cfg.E, ow.expert, ow.shared(), tokens=tokens,
                          h_quant_g=gh, hs_quant_g=gh, renorm=renorm, h_quant=hq, hs_quant=hq,
                          shared_g=None if shared_g is None else to_np_f32(shared_g).astype(np.float64),
                          x_gate=x.astype(np.float64))
