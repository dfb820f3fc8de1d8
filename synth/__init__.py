"""Seeded synthetic inputs for the MoE FFN layer forward.

This module serves both the oracle (tests) and the CUDA path (tests, bench).
It holds none of the layer's arithmetic: it only draws inputs.  The layer
shapes are those of the workloads the pages talk about:

  tiny        H=256,  E=8,   top-2,  I=512,  no shared expert, bf16
  qwen3-235b  H=4096, E=128, top-8,  I=1536, no shared expert, bf16
              ("Hosting Qwen on Blackwell": Qwen3 235B, 128 experts, top-8)
  qwen35-397b H=4096, E=512, top-10, I=1024, one shared expert (I_s=1024),
              NVFP4 weights, bf16 activations
              ("Como Servimos um Modelo MoE de 397B ...", MoE FFN description)
  deepseek-v3 H=7168, E=256, top-8,  I=2048, one shared expert (I_s=2048),
              NVFP4 weights and NVFP4 activations
              ("Driving vLLM WideEP ... on Blackwell (Part I)")
  qwen3-235b-mxfp8  the qwen3-235b shapes with MXFP8 weights and activations
              ("Hosting Qwen on Blackwell", section "Quantização")

Recipe (seed s):
  x       ~ N(0, 1) fp32 drawn with torch.Generator('cpu').manual_seed(s); on
            the NVFP4-activation workload a Bernoulli(0.001) mask (same
            generator) multiplies entries by 20; then rounded to bf16 (RNE).
  logits  = fp32( x @ W_r + bias ) evaluated in fp64, W_r [H, E] ~ N(0, 0.02)
            from the same generator; bias_e = -0.5 * z * ln(rank_e), rank a
            seeded permutation of 1..E and z the Zipf exponent (z=0: uniform).
  weights ~ N(0, 0.02) fp32 rounded to bf16, drawn per expert with
            torch.Generator(device).manual_seed(s + 1000) (device 'cuda' on the
            GPU, 'cpu' for CPU-only tests).  NVFP4 / MX weights are the bf16
            master passed through the format's quantiser by whoever consumes
            them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional, Tuple

import numpy as np
import torch


@dataclass(frozen=True)
class LayerConfig:
    name: str
    H: int
    E: int
    k: int
    I: int
    I_s: int            # 0: no shared expert
    w_fmt: str          # 'bf16' | 'nvfp4' | 'mxfp8' | 'mxfp4'
    act_fmt: str        # 'bf16' | 'nvfp4' | 'mxfp8' | 'mxfp4'
    zipf: float = 1.1
    outlier_p: float = 0.0
    Ts: Tuple[int, ...] = ()
    # static global scale of the SwiGLU output when it is quantised to NVFP4
    # (NVFP4-activation workload only): g_h = H_AMAX / 2688
    h_amax: float = 0.0

    @property
    def g_h(self) -> float:
        return float(np.float32(self.h_amax) / np.float32(2688.0)) if self.h_amax else 0.0

    def flops_per_token(self) -> int:
        return 6 * self.k * self.H * self.I + 6 * self.H * self.I_s


TINY = LayerConfig("tiny", 256, 8, 2, 512, 0, "bf16", "bf16", 1.1, 0.0, (64,))
QWEN3_235B = LayerConfig("qwen3-235b", 4096, 128, 8, 1536, 0, "bf16", "bf16", 1.1, 0.0, (256, 8192))
QWEN35_397B = LayerConfig("qwen35-397b", 4096, 512, 10, 1024, 1024, "nvfp4", "bf16", 1.1, 0.0,
                          (64, 512, 4096))
DEEPSEEK_V3 = LayerConfig("deepseek-v3", 7168, 256, 8, 2048, 2048, "nvfp4", "nvfp4", 1.1, 0.001,
                          (256, 16384), h_amax=128.0)

# the Qwen3-235B-shaped layer in MXFP8 weights and activations (E4M3 elements,
# one E8M0 scale per 32), the format "Hosting Qwen on Blackwell" (section
# "Quantização") serves that model in
QWEN3_235B_MXFP8 = LayerConfig("qwen3-235b-mxfp8", 4096, 128, 8, 1536, 0, "mxfp8", "mxfp8", 1.1, 0.0,
                               (256, 8192))

CONFIGS = {c.name: c for c in (TINY, QWEN3_235B, QWEN35_397B, DEEPSEEK_V3, QWEN3_235B_MXFP8)}

# size / imbalance sweep on the DeepSeek-V3 shapes
SWEEP_TS = tuple(2 ** i for i in range(17))
SWEEP_ZIPF = (0.0, 1.1, 2.0)


def sweep_config(w_fmt: str, zipf: float) -> LayerConfig:
    """DeepSeek-V3 shapes with bf16 weights (bf16 activations) or NVFP4
    weights and activations, and the given Zipf exponent of the router bias."""
    act = "nvfp4" if w_fmt == "nvfp4" else "bf16"
    return replace(DEEPSEEK_V3, name=f"deepseek-v3-sweep-{w_fmt}-z{zipf}", w_fmt=w_fmt,
                   act_fmt=act, zipf=zipf, Ts=SWEEP_TS)


def small_variant(cfg: LayerConfig, H: int, E: int, k: int, I: int, I_s: Optional[int] = None,
                  name: Optional[str] = None) -> LayerConfig:
    """Same formats / distributions at reduced shapes (for oracle-speed tests)."""
    return replace(cfg, name=name or f"{cfg.name}-small", H=H, E=E, k=k, I=I,
                   I_s=(cfg.I_s and I) if I_s is None else I_s)


@dataclass
class Activations:
    x: torch.Tensor        # bf16 [T, H] (CPU)
    logits: torch.Tensor   # fp32 [T, E] (CPU)


def make_activations(cfg: LayerConfig, T: int, seed: int = 0) -> Activations:
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(T, cfg.H, generator=g, dtype=torch.float32)
    if cfg.outlier_p > 0:
        mask = torch.rand(T, cfg.H, generator=g) < cfg.outlier_p
        x = torch.where(mask, x * 20.0, x)
    xb = x.to(torch.bfloat16)
    w_r = torch.randn(cfg.H, cfg.E, generator=g, dtype=torch.float32) * 0.02
    rank = torch.randperm(cfg.E, generator=g).to(torch.float64) + 1.0
    bias = -0.5 * cfg.zipf * torch.log(rank)
    logits = (xb.to(torch.float64) @ w_r.to(torch.float64) + bias).to(torch.float32)
    return Activations(xb, logits.contiguous())


@dataclass
class MasterWeights:
    """bf16 master weights on `device`."""
    w13: torch.Tensor            # [E, 2I, H]
    w2: torch.Tensor             # [E, H, I]
    ws13: Optional[torch.Tensor]  # [2I_s, H]
    ws2: Optional[torch.Tensor]   # [H, I_s]


def make_weights(cfg: LayerConfig, seed: int = 0, device: str = "cpu") -> MasterWeights:
    g = torch.Generator(device=device).manual_seed(seed + 1000)
    E, H, I = cfg.E, cfg.H, cfg.I
    w13 = torch.empty(E, 2 * I, H, dtype=torch.bfloat16, device=device)
    w2 = torch.empty(E, H, I, dtype=torch.bfloat16, device=device)
    for e in range(E):
        w13[e] = (torch.randn(2 * I, H, generator=g, device=device) * 0.02).to(torch.bfloat16)
        w2[e] = (torch.randn(H, I, generator=g, device=device) * 0.02).to(torch.bfloat16)
    ws13 = ws2 = None
    if cfg.I_s:
        ws13 = (torch.randn(2 * cfg.I_s, H, generator=g, device=device) * 0.02).to(torch.bfloat16)
        ws2 = (torch.randn(H, cfg.I_s, generator=g, device=device) * 0.02).to(torch.bfloat16)
    return MasterWeights(w13, w2, ws13, ws2)


def sample_tokens(T: int, n: int, seed: int = 0) -> np.ndarray:
    """A seeded, sorted subsample of n distinct token ids (all of them if n >= T)."""
    if n >= T:
        return np.arange(T)
    rng = np.random.default_rng(seed + 77)
    return np.sort(rng.choice(T, size=n, replace=False))


def forced_one_token_per_expert_logits(cfg: LayerConfig) -> Tuple[int, torch.Tensor]:
    """Decode microbenchmark shape from "Hosting Qwen on Blackwell" (section
    "MoE GEMM": all experts active with a single token): T = E / k tokens
    whose logits make token t pick experts [t*k, (t+1)*k) in descending order."""
    assert cfg.E % cfg.k == 0
    T = cfg.E // cfg.k
    logits = torch.full((T, cfg.E), -10.0, dtype=torch.float32)
    for t in range(T):
        for j in range(cfg.k):
            logits[t, t * cfg.k + j] = float(cfg.k - j)
    return T, logits


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def log2_int(n: int) -> int:
    return int(math.log2(n))
