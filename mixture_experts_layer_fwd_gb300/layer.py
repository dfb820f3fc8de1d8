"""A ready-to-call MoE layer: owns the weights in the kernels' formats, the
workspace, and the C struct that describes them to moe_forward.

Weight preparation for the NVFP4 formats runs the library's own quantiser
(moe_quant_nvfp4, one global scale per expert and projection).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import api
from ._lib import MOE_FMT_BF16, MOE_FMT_MXFP4, MOE_FMT_MXFP8, MOE_FMT_NVFP4, MoeLayerC

_FMT = {"bf16": MOE_FMT_BF16, "nvfp4": MOE_FMT_NVFP4, "mxfp8": MOE_FMT_MXFP8, "mxfp4": MOE_FMT_MXFP4}


@dataclass
class NVFP4Tensor:
    codes: torch.Tensor  # uint8 [..., cols/2]
    sf: torch.Tensor     # uint8 [..., cols/16]
    g: torch.Tensor      # fp32 [groups]


def quantize_weights(w: torch.Tensor) -> NVFP4Tensor:
    """bf16 [groups, rows, cols] (or [rows, cols]) -> NVFP4 with one global
    scale per group."""
    codes, sf, g = api.moe_quant_nvfp4(w.contiguous())
    return NVFP4Tensor(codes, sf, g)


@dataclass
class MXTensor:
    codes: torch.Tensor  # uint8 [..., cols] (MXFP8) or [..., cols/2] (MXFP4)
    sf: torch.Tensor     # uint8 [..., cols/32] (E8M0)


def quantize_weights_mx(w: torch.Tensor, fmt: str) -> MXTensor:
    """bf16 [..., rows, cols] -> MXFP8 / MXFP4 along cols (moe_quant_mx)."""
    w = w.contiguous()
    codes, sf = api.moe_quant_mx(w.reshape(-1, w.shape[-1]), _FMT[fmt])
    return MXTensor(codes.reshape(w.shape[:-1] + (codes.shape[-1],)), sf.reshape(w.shape[:-1] + (sf.shape[-1],)))


def _check_weight(t: Optional[torch.Tensor], name: str, shape, device=None) -> None:
    if t is None:
        raise ValueError(f"{name}: required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name}: expected bf16 master weights, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")


class MoELayer:
    def __init__(self, H: int, E: int, k: int, I: int, I_s: int, w13: torch.Tensor, w2: torch.Tensor,
                 ws13: Optional[torch.Tensor] = None, ws2: Optional[torch.Tensor] = None,
                 w_fmt: str = "bf16", act_fmt: str = "bf16", g_h: float = 0.0, g_hs: Optional[float] = None,
                 renorm: bool = True, shared_gate: Optional[torch.Tensor] = None):
        """w13 bf16 [E, 2I, H], w2 bf16 [E, H, I], ws13 bf16 [2I_s, H], ws2 bf16
        [H, I_s] on one CUDA device.  With w_fmt='nvfp4' (or 'mxfp8' /
        'mxfp4', whose act_fmt must be the same format) they are quantised
        here; act_fmt='nvfp4' also needs the static global scale g_h of the
        SwiGLU output (g_hs for the shared expert, default g_h).
        renorm=False routes without renormalisation; shared_gate (bf16 [H])
        scales the shared expert by sigmoid(x . shared_gate)."""
        if w_fmt not in _FMT or act_fmt not in _FMT:
            raise ValueError(f"formats: expected one of {sorted(_FMT)}, got {w_fmt!r}, {act_fmt!r}")
        _check_weight(w13, "w13", (E, 2 * I, H))
        _check_weight(w2, "w2", (E, H, I), w13.device)
        if I_s:
            _check_weight(ws13, "ws13", (2 * I_s, H), w13.device)
            _check_weight(ws2, "ws2", (H, I_s), w13.device)
        self.H, self.E, self.k, self.I, self.I_s = H, E, k, I, I_s
        self.w_fmt, self.act_fmt = w_fmt, act_fmt
        self.device = w13.device
        self._keep = []
        c = MoeLayerC()
        c.H, c.E, c.k, c.I, c.I_s = H, E, k, I, I_s
        c.w_fmt, c.act_fmt = _FMT[w_fmt], _FMT[act_fmt]
        if w_fmt.startswith("mx"):
            if act_fmt != w_fmt:
                raise ValueError("MX layers take the same MX format for weights and activations")
            self.w13 = quantize_weights_mx(w13, w_fmt)
            self.w2 = quantize_weights_mx(w2, w_fmt)
            c.w13, c.w13_sf = self.w13.codes.data_ptr(), self.w13.sf.data_ptr()
            c.w2, c.w2_sf = self.w2.codes.data_ptr(), self.w2.sf.data_ptr()
            self._keep += [self.w13, self.w2]
            if I_s:
                self.ws13 = quantize_weights_mx(ws13, w_fmt)
                self.ws2 = quantize_weights_mx(ws2, w_fmt)
                c.ws13, c.ws13_sf = self.ws13.codes.data_ptr(), self.ws13.sf.data_ptr()
                c.ws2, c.ws2_sf = self.ws2.codes.data_ptr(), self.ws2.sf.data_ptr()
                self._keep += [self.ws13, self.ws2]
        elif w_fmt == "bf16":
            self.w13, self.w2 = w13.contiguous(), w2.contiguous()
            c.w13, c.w2 = self.w13.data_ptr(), self.w2.data_ptr()
            self._keep += [self.w13, self.w2]
            if I_s:
                self.ws13, self.ws2 = ws13.contiguous(), ws2.contiguous()
                c.ws13, c.ws2 = self.ws13.data_ptr(), self.ws2.data_ptr()
                self._keep += [self.ws13, self.ws2]
        else:
            self.w13 = quantize_weights(w13)
            self.w2 = quantize_weights(w2)
            c.w13, c.w13_sf, c.w13_g = (t.data_ptr() for t in (self.w13.codes, self.w13.sf, self.w13.g))
            c.w2, c.w2_sf, c.w2_g = (t.data_ptr() for t in (self.w2.codes, self.w2.sf, self.w2.g))
            self._keep += [self.w13, self.w2]
            if I_s:
                self.ws13 = quantize_weights(ws13)
                self.ws2 = quantize_weights(ws2)
                c.ws13, c.ws13_sf, c.ws13_g = (t.data_ptr() for t in (self.ws13.codes, self.ws13.sf, self.ws13.g))
                c.ws2, c.ws2_sf, c.ws2_g = (t.data_ptr() for t in (self.ws2.codes, self.ws2.sf, self.ws2.g))
                self._keep += [self.ws13, self.ws2]
        if act_fmt == "nvfp4" and w_fmt == "nvfp4":
            self.g_h = torch.tensor([g_h], dtype=torch.float32, device=self.device)
            self.g_hs = torch.tensor([g_h if g_hs is None else g_hs], dtype=torch.float32, device=self.device)
            c.g_h, c.g_hs = self.g_h.data_ptr(), self.g_hs.data_ptr()
        c.no_renorm = 0 if renorm else 1
        if shared_gate is not None:
            if not I_s:
                raise ValueError("a shared-expert gate needs a shared expert (I_s > 0)")
            if tuple(shared_gate.shape) != (H,):
                raise ValueError(f"shared_gate: expected shape ({H},), got {tuple(shared_gate.shape)}")
            self.shared_gate = shared_gate.to(device=self.device, dtype=torch.bfloat16).contiguous()
            c.ws_gate = self.shared_gate.data_ptr()
            self._keep.append(self.shared_gate)
        self.c = c
        self._ws = None

    @classmethod
    def from_config(cls, cfg, weights) -> "MoELayer":
        """From a synth.LayerConfig and synth.MasterWeights."""
        return cls(cfg.H, cfg.E, cfg.k, cfg.I, cfg.I_s, weights.w13, weights.w2, weights.ws13, weights.ws2,
                   cfg.w_fmt, cfg.act_fmt, cfg.g_h)

    def workspace_size(self, T: int) -> int:
        n = api.moe_forward_workspace_size(self.c, T)
        if n == 0 and T > 0:
            raise ValueError("layer description rejected by moe_forward_workspace_size")
        return n

    def workspace(self, T: int) -> torch.Tensor:
        n = self.workspace_size(T)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(max(n, 1), dtype=torch.uint8, device=self.device)
        return self._ws

    def forward(self, x: torch.Tensor, logits: torch.Tensor, out: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
        T = x.shape[0]
        if out is None:
            out = torch.empty(T, self.H, dtype=torch.bfloat16, device=self.device)
        return api.moe_forward(self.c, x, logits, out, self.workspace(T), stream)

    __call__ = forward

    def capture(self, x: torch.Tensor, logits: torch.Tensor, out: Optional[torch.Tensor] = None,
                stream=None) -> "api.ForwardGraph":
        """The forward on these buffers as a CUDA graph (one launch per replay)."""
        if out is None:
            out = torch.empty(x.shape[0], self.H, dtype=torch.bfloat16, device=self.device)
        return api.ForwardGraph(self.c, x, logits, out, self.workspace(x.shape[0]), stream)
