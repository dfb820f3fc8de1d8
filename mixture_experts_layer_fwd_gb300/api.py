"""Python binding of the C ABI (include/moe_gb300.h), same names.

Argument marshalling only: every step of the layer runs in the CUDA library.
PyTorch provides device memory and the current stream.  Outputs that are not
passed in are allocated with torch on the input's device.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib
from ._lib import (MOE_EPI_STORE_BF16, MOE_EPI_SWIGLU_BF16, MOE_EPI_SWIGLU_MX, MOE_EPI_SWIGLU_NVFP4, MOE_FMT_BF16, MOE_FMT_MXFP4,
                   MOE_FMT_MXFP8, MOE_FMT_NVFP4, check, load)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dev(t: torch.Tensor, name: str = "tensor", dtype=None, shape=None, device=None) -> None:
    """Reject what the kernels cannot take before any launch: a tensor that
    is missing, not on a CUDA device (its address would be read by a
    kernel), not contiguous, or of the wrong dtype, shape or device."""
    if t is None:
        raise ValueError(f"{name}: required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")


def _opt(t: Optional[torch.Tensor], name: str, **kw) -> None:
    if t is not None:
        _dev(t, name, **kw)


def _at_least(t: torch.Tensor, name: str, nbytes: int) -> None:
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{name}: {have} bytes, needs {nbytes}")


def _ws(nbytes: int, device) -> torch.Tensor:
    # 256-byte aligned by the caching allocator (allocations are 512-byte aligned)
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def moe_version() -> int:
    return load().moe_version()


def moe_sync_status(stream=None) -> int:
    return load().moe_sync_status(_stream(stream))


def moe_set_wait_timeout_ns(ns: int) -> None:
    check(load().moe_set_wait_timeout_ns(int(ns)), "moe_set_wait_timeout_ns")


def moe_selftest_wait_timeout(timeout_ns: int, stream=None) -> None:
    check(load().moe_selftest_wait_timeout(int(timeout_ns), _stream(stream)), "moe_selftest_wait_timeout")


def moe_route(logits: torch.Tensor, k: int, idx: Optional[torch.Tensor] = None,
              w: Optional[torch.Tensor] = None, stream=None, renorm: bool = True):
    """logits fp32 [T, E] -> (idx int32 [T, k], w fp32 [T, k]); renorm=False
    takes the full softmax over E at the picks (moe_route_ex)."""
    _dev(logits, "logits", dtype=torch.float32)
    if logits.dim() != 2:
        raise ValueError("logits: expected [T, E]")
    T, E = logits.shape
    if idx is None:
        idx = torch.empty(T, k, dtype=torch.int32, device=logits.device)
    if w is None:
        w = torch.empty(T, k, dtype=torch.float32, device=logits.device)
    _dev(idx, "idx", dtype=torch.int32, shape=(T, k), device=logits.device)
    _dev(w, "w", dtype=torch.float32, shape=(T, k), device=logits.device)
    if renorm:
        check(load().moe_route(_ptr(logits), T, E, k, _ptr(idx), _ptr(w), _stream(stream)), "moe_route")
    else:
        check(load().moe_route_ex(_ptr(logits), T, E, k, 0, _ptr(idx), _ptr(w), _stream(stream)), "moe_route_ex")
    return idx, w


def moe_permute(idx: torch.Tensor, E: int, x_rows: Optional[torch.Tensor] = None,
                x_sf: Optional[torch.Tensor] = None, stream=None):
    """Stable permutation into expert-contiguous order.

    idx int32 [T, k]; x_rows: [T, ...] any dtype (rows copied as bytes) or None;
    x_sf: uint8 [T, sf_bytes] or None.  Returns dict(counts, offsets, row_of,
    src_tok, xp, xp_sf)."""
    _dev(idx, "idx", dtype=torch.int32)
    if idx.dim() != 2:
        raise ValueError("idx: expected [T, k]")
    T, k = idx.shape
    dev = idx.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    row_of = torch.empty(T, k, dtype=torch.int32, device=dev)
    src_tok = torch.empty(T * k, dtype=torch.int32, device=dev)
    xp = xp_sf = None
    row_bytes = sf_bytes = 0
    if x_rows is not None:
        _dev(x_rows, "x_rows", device=dev)
        if x_rows.shape[0] != T:
            raise ValueError("x_rows: expected one row per token")
        row_bytes = x_rows[0].numel() * x_rows.element_size() if T else 0
        xp = torch.empty((T * k,) + tuple(x_rows.shape[1:]), dtype=x_rows.dtype, device=dev)
        if x_sf is not None:
            _dev(x_sf, "x_sf", dtype=torch.uint8, device=dev)
            if x_sf.dim() != 2 or x_sf.shape[0] != T:
                raise ValueError("x_sf: expected [T, sf_bytes]")
            sf_bytes = x_sf.shape[1]
            xp_sf = torch.empty(T * k, sf_bytes, dtype=torch.uint8, device=dev)
    lib = load()
    nbytes = lib.moe_permute_workspace_size(T, k, E)
    ws = _ws(nbytes, dev)
    check(lib.moe_permute(_ptr(idx), T, k, E, _ptr(x_rows), row_bytes, _ptr(x_sf), sf_bytes,
                          _ptr(counts), _ptr(offsets), _ptr(row_of), _ptr(src_tok), _ptr(xp),
                          _ptr(xp_sf), _ptr(ws), nbytes, _stream(stream)), "moe_permute")
    return dict(counts=counts, offsets=offsets, row_of=row_of, src_tok=src_tok, xp=xp, xp_sf=xp_sf)


def moe_permute_noalloc(idx: torch.Tensor, E: int, x_rows: Optional[torch.Tensor] = None,
                        x_sf: Optional[torch.Tensor] = None, out: Optional[dict] = None, stream=None):
    """moe_permute for callers that cannot allocate device memory when they
    dispatch: the library keeps the scratch in its own fixed device array
    (size limit ceil(T*k/1024) * E <= 131072).  Pass preallocated outputs in
    `out` (keys counts, offsets, row_of, src_tok, xp, xp_sf) to make the call
    allocation-free end to end; missing outputs are allocated here."""
    _dev(idx, "idx", dtype=torch.int32)
    if idx.dim() != 2:
        raise ValueError("idx: expected [T, k]")
    T, k = idx.shape
    dev = idx.device
    o = dict(out or {})

    def need(key, make):
        # allocate only what the caller did not pass (a setdefault would build
        # the default tensor, and so allocate, even when the key is present)
        if o.get(key) is None:
            o[key] = make()

    need("counts", lambda: torch.empty(E, dtype=torch.int32, device=dev))
    need("offsets", lambda: torch.empty(E + 1, dtype=torch.int32, device=dev))
    need("row_of", lambda: torch.empty(T, k, dtype=torch.int32, device=dev))
    need("src_tok", lambda: torch.empty(T * k, dtype=torch.int32, device=dev))
    row_bytes = sf_bytes = 0
    if x_rows is not None:
        _dev(x_rows, "x_rows", device=dev)
        if x_rows.shape[0] != T:
            raise ValueError("x_rows: expected one row per token")
        row_bytes = x_rows[0].numel() * x_rows.element_size() if T else 0
        need("xp", lambda: torch.empty((T * k,) + tuple(x_rows.shape[1:]), dtype=x_rows.dtype, device=dev))
        if x_sf is not None:
            _dev(x_sf, "x_sf", dtype=torch.uint8, device=dev)
            if x_sf.dim() != 2 or x_sf.shape[0] != T:
                raise ValueError("x_sf: expected [T, sf_bytes]")
            sf_bytes = x_sf.shape[1]
            need("xp_sf", lambda: torch.empty(T * k, sf_bytes, dtype=torch.uint8, device=dev))
    o.setdefault("xp", None)
    o.setdefault("xp_sf", None)
    # caller-given outputs are written by the kernels: check them like inputs
    _dev(o["counts"], "counts", dtype=torch.int32, shape=(E,), device=dev)
    _dev(o["offsets"], "offsets", dtype=torch.int32, shape=(E + 1,), device=dev)
    _dev(o["row_of"], "row_of", dtype=torch.int32, shape=(T, k), device=dev)
    _dev(o["src_tok"], "src_tok", dtype=torch.int32, shape=(T * k,), device=dev)
    if x_rows is not None:
        _dev(o["xp"], "xp", device=dev)
        _at_least(o["xp"], "xp", T * k * row_bytes)
        if x_sf is not None:
            _dev(o["xp_sf"], "xp_sf", device=dev)
            _at_least(o["xp_sf"], "xp_sf", T * k * sf_bytes)
    check(load().moe_permute_noalloc(_ptr(idx), T, k, E, _ptr(x_rows), row_bytes, _ptr(x_sf), sf_bytes,
                                     _ptr(o["counts"]), _ptr(o["offsets"]), _ptr(o["row_of"]), _ptr(o["src_tok"]),
                                     _ptr(o["xp"]), _ptr(o["xp_sf"]), _stream(stream)), "moe_permute_noalloc")
    return o


def moe_route_permute(logits: torch.Tensor, k: int, x_rows: Optional[torch.Tensor] = None,
                      x_sf: Optional[torch.Tensor] = None, renorm: bool = True, stream=None):
    """Fused dispatch: moe_route then moe_permute in one cooperative launch.
    logits fp32 [T, E]; x_rows / x_sf as for moe_permute.  Returns dict(idx,
    w, counts, offsets, row_of, src_tok, xp, xp_sf)."""
    _dev(logits, "logits", dtype=torch.float32)
    if logits.dim() != 2:
        raise ValueError("logits: expected [T, E]")
    T, E = logits.shape
    dev = logits.device
    o = dict(idx=torch.empty(T, k, dtype=torch.int32, device=dev), w=torch.empty(T, k, device=dev),
             counts=torch.empty(E, dtype=torch.int32, device=dev),
             offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
             row_of=torch.empty(T, k, dtype=torch.int32, device=dev),
             src_tok=torch.empty(T * k, dtype=torch.int32, device=dev), xp=None, xp_sf=None)
    row_bytes = sf_bytes = 0
    if x_rows is not None:
        _dev(x_rows, "x_rows", device=dev)
        if x_rows.shape[0] != T:
            raise ValueError("x_rows: expected one row per token")
        row_bytes = x_rows[0].numel() * x_rows.element_size() if T else 0
        o["xp"] = torch.empty((T * k,) + tuple(x_rows.shape[1:]), dtype=x_rows.dtype, device=dev)
        if x_sf is not None:
            _dev(x_sf, "x_sf", dtype=torch.uint8, device=dev)
            if x_sf.dim() != 2 or x_sf.shape[0] != T:
                raise ValueError("x_sf: expected [T, sf_bytes]")
            sf_bytes = x_sf.shape[1]
            o["xp_sf"] = torch.empty(T * k, sf_bytes, dtype=torch.uint8, device=dev)
    lib = load()
    nbytes = lib.moe_route_permute_workspace_size(T, k, E)
    ws = _ws(nbytes, dev)
    check(lib.moe_route_permute(_ptr(logits), T, E, k, 1 if renorm else 0, _ptr(o["idx"]), _ptr(o["w"]),
                                _ptr(x_rows), row_bytes, _ptr(x_sf), sf_bytes, _ptr(o["counts"]),
                                _ptr(o["offsets"]), _ptr(o["row_of"]), _ptr(o["src_tok"]), _ptr(o["xp"]),
                                _ptr(o["xp_sf"]), _ptr(ws), nbytes, _stream(stream)), "moe_route_permute")
    return o


def moe_selftest_grid_barrier_timeout(timeout_ns: int, stream=None) -> None:
    check(load().moe_selftest_grid_barrier_timeout(int(timeout_ns), _stream(stream)),
          "moe_selftest_grid_barrier_timeout")


def moe_quant_nvfp4(x: torch.Tensor, g_in: Optional[torch.Tensor] = None, stream=None):
    """x bf16 [rows, cols] or [groups, rows, cols] -> (codes uint8 [..., cols/2],
    sf uint8 [..., cols/16], g fp32 [groups])."""
    _dev(x, "x", dtype=torch.bfloat16)
    if x.dim() not in (2, 3):
        raise ValueError("x: expected [rows, cols] or [groups, rows, cols]")
    x3 = x if x.dim() == 3 else x.unsqueeze(0)
    G, R, Cc = x3.shape
    _opt(g_in, "g_in", dtype=torch.float32, shape=(G,), device=x.device)
    codes = torch.empty(x.shape[:-1] + (Cc // 2,), dtype=torch.uint8, device=x.device)
    sf = torch.empty(x.shape[:-1] + (Cc // 16,), dtype=torch.uint8, device=x.device)
    g = torch.empty(G, dtype=torch.float32, device=x.device)
    lib = load()
    nbytes = lib.moe_quant_nvfp4_workspace_size(G)
    ws = _ws(nbytes, x.device)
    check(lib.moe_quant_nvfp4(_ptr(x3), G, R, Cc, _ptr(g_in), _ptr(codes), _ptr(sf), _ptr(g),
                              _ptr(ws), nbytes, _stream(stream)), "moe_quant_nvfp4")
    return codes, sf, g


def moe_quant_mx(x: torch.Tensor, fmt: int, stream=None):
    """x bf16 [rows, cols] -> (codes, scales uint8 [rows, cols/32]): MXFP8
    codes uint8 [rows, cols], MXFP4 packed codes uint8 [rows, cols/2]."""
    _dev(x, "x", dtype=torch.bfloat16)
    if x.dim() != 2:
        raise ValueError("x: expected [rows, cols]")
    if fmt not in (MOE_FMT_MXFP8, MOE_FMT_MXFP4):
        raise ValueError("fmt: expected MOE_FMT_MXFP8 or MOE_FMT_MXFP4")
    R, Cc = x.shape
    codes = torch.empty(R, Cc if fmt == MOE_FMT_MXFP8 else Cc // 2, dtype=torch.uint8, device=x.device)
    scales = torch.empty(R, Cc // 32, dtype=torch.uint8, device=x.device)
    check(load().moe_quant_mx(_ptr(x), R, Cc, int(fmt), _ptr(codes), _ptr(scales), _stream(stream)), "moe_quant_mx")
    return codes, scales


def moe_grouped_gemm(a_fmt: int, w_fmt: int, epilogue: int, offsets: torch.Tensor, N: int, K: int,
                     A: torch.Tensor, W: torch.Tensor, A_sf=None, A_g=None, W_sf=None, W_g=None,
                     c_g=None, C=None, C_sf=None, stream=None):
    """Grouped GEMM over expert-contiguous rows; see include/moe_gb300.h.
    Every operand is checked for device, contiguity and size against
    (G, M, N, K) and the formats before the call."""
    _dev(A, "A")
    dev = A.device
    _dev(offsets, "offsets", dtype=torch.int32, device=dev)
    G = offsets.numel() - 1
    M = A.shape[0]
    wn = 2 * N if epilogue in (MOE_EPI_SWIGLU_BF16, MOE_EPI_SWIGLU_NVFP4, MOE_EPI_SWIGLU_MX) else N
    mx_c = N // 2 if a_fmt == MOE_FMT_MXFP4 else N  # bytes per row of MX-coded C
    _dev(W, "W", device=dev)
    if a_fmt == MOE_FMT_NVFP4:
        _at_least(A, "A", M * K // 2)
        _dev(A_sf, "A_sf", device=dev)
        _at_least(A_sf, "A_sf", M * K // 16)
        _dev(A_g, "A_g", dtype=torch.float32, device=dev)
        _at_least(A_g, "A_g", 4)
    elif a_fmt in (MOE_FMT_MXFP4, MOE_FMT_MXFP8):
        _at_least(A, "A", M * K // (2 if a_fmt == MOE_FMT_MXFP4 else 1))
        _dev(A_sf, "A_sf", device=dev)
        _at_least(A_sf, "A_sf", M * K // 32)
    else:
        _at_least(A, "A", M * K * 2)
    if w_fmt == MOE_FMT_NVFP4:
        _at_least(W, "W", G * wn * K // 2)
        _dev(W_sf, "W_sf", device=dev)
        _at_least(W_sf, "W_sf", G * wn * K // 16)
        _dev(W_g, "W_g", dtype=torch.float32, device=dev)
        _at_least(W_g, "W_g", 4 * G)
    elif w_fmt in (MOE_FMT_MXFP4, MOE_FMT_MXFP8):
        _at_least(W, "W", G * wn * K // (2 if w_fmt == MOE_FMT_MXFP4 else 1))
        _dev(W_sf, "W_sf", device=dev)
        _at_least(W_sf, "W_sf", G * wn * K // 32)
    else:
        _at_least(W, "W", G * wn * K * 2)
    if C is None:
        if epilogue == MOE_EPI_SWIGLU_NVFP4:
            C = torch.empty(M, N // 2, dtype=torch.uint8, device=dev)
            C_sf = torch.empty(M, N // 16, dtype=torch.uint8, device=dev)
        elif epilogue == MOE_EPI_SWIGLU_MX:
            C = torch.empty(M, mx_c, dtype=torch.uint8, device=dev)
            C_sf = torch.empty(M, N // 32, dtype=torch.uint8, device=dev)
        else:
            C = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    _dev(C, "C", device=dev)
    if epilogue == MOE_EPI_SWIGLU_NVFP4:
        _at_least(C, "C", M * N // 2)
        _dev(C_sf, "C_sf", device=dev)
        _at_least(C_sf, "C_sf", M * N // 16)
        _dev(c_g, "c_g", dtype=torch.float32, device=dev)
        _at_least(c_g, "c_g", 4)
    elif epilogue == MOE_EPI_SWIGLU_MX:
        _at_least(C, "C", M * mx_c)
        _dev(C_sf, "C_sf", device=dev)
        _at_least(C_sf, "C_sf", M * N // 32)
    else:
        _at_least(C, "C", M * N * 2)
    check(load().moe_grouped_gemm(a_fmt, w_fmt, epilogue, G, _ptr(offsets), M, N, K, _ptr(A), _ptr(A_sf),
                                  _ptr(A_g), _ptr(W), _ptr(W_sf), _ptr(W_g), _ptr(C), _ptr(C_sf), _ptr(c_g),
                                  _stream(stream)), "moe_grouped_gemm")
    return (C, C_sf) if epilogue in (MOE_EPI_SWIGLU_NVFP4, MOE_EPI_SWIGLU_MX) else C


def moe_combine(Y: torch.Tensor, row_of: torch.Tensor, w: torch.Tensor, Ys: Optional[torch.Tensor],
                T: int, k: int, H: int, out: Optional[torch.Tensor] = None, stream=None,
                ys_gate: Optional[torch.Tensor] = None):
    """ys_gate: fp32 [T] per-token factor of the shared row (moe_combine_gated)."""
    _dev(Y, "Y", dtype=torch.bfloat16)
    dev = Y.device
    _at_least(Y, "Y", T * k * H * 2)
    _dev(row_of, "row_of", dtype=torch.int32, device=dev)
    _at_least(row_of, "row_of", T * k * 4)
    _dev(w, "w", dtype=torch.float32, device=dev)
    _at_least(w, "w", T * k * 4)
    _opt(Ys, "Ys", dtype=torch.bfloat16, shape=(T, H), device=dev)
    _opt(ys_gate, "ys_gate", dtype=torch.float32, shape=(T,), device=dev)
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    _dev(out, "out", dtype=torch.bfloat16, shape=(T, H), device=dev)
    if ys_gate is None:
        check(load().moe_combine(_ptr(Y), _ptr(row_of), _ptr(w), _ptr(Ys), T, k, H, _ptr(out), _stream(stream)),
              "moe_combine")
    else:
        check(load().moe_combine_gated(_ptr(Y), _ptr(row_of), _ptr(w), _ptr(Ys), _ptr(ys_gate), T, k, H,
                                       _ptr(out), _stream(stream)), "moe_combine_gated")
    return out


def moe_shared_gate(x: torch.Tensor, g: torch.Tensor, gate: Optional[torch.Tensor] = None, stream=None):
    """x bf16 [T, H], g bf16 [H] -> gate fp32 [T] = sigmoid(x . g)."""
    _dev(x, "x", dtype=torch.bfloat16)
    if x.dim() != 2:
        raise ValueError("x: expected [T, H]")
    T, H = x.shape
    _dev(g, "g", dtype=torch.bfloat16, shape=(H,), device=x.device)
    if gate is None:
        gate = torch.empty(T, dtype=torch.float32, device=x.device)
    _dev(gate, "gate", dtype=torch.float32, shape=(T,), device=x.device)
    check(load().moe_shared_gate(_ptr(x), _ptr(g), T, H, _ptr(gate), _stream(stream)), "moe_shared_gate")
    return gate


def moe_forward_workspace_size(layer_c, T: int) -> int:
    import ctypes
    return int(load().moe_forward_workspace_size(ctypes.byref(layer_c), T))


def _host(t: torch.Tensor, name: str, dtype, shape) -> None:
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError(f"{name}: expected a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


def _forward_args(layer_c, x: torch.Tensor, logits: torch.Tensor, out: torch.Tensor, ws: torch.Tensor) -> int:
    """Checks the device buffers of a whole-layer call against the layer's
    H and E; returns T."""
    _dev(x, "x", dtype=torch.bfloat16)
    if x.dim() != 2 or x.shape[1] != layer_c.H:
        raise ValueError(f"x: expected [T, {layer_c.H}]")
    T = x.shape[0]
    dev = x.device
    _dev(logits, "logits", dtype=torch.float32, shape=(T, layer_c.E), device=dev)
    _dev(out, "out", dtype=torch.bfloat16, shape=(T, layer_c.H), device=dev)
    _dev(ws, "ws", device=dev)
    _at_least(ws, "ws", moe_forward_workspace_size(layer_c, T))
    return T


def moe_forward(layer_c, x: torch.Tensor, logits: torch.Tensor, out: torch.Tensor, ws: torch.Tensor,
                stream=None) -> torch.Tensor:
    import ctypes
    T = _forward_args(layer_c, x, logits, out, ws)
    check(load().moe_forward(ctypes.byref(layer_c), _ptr(x), _ptr(logits), T, _ptr(out), _ptr(ws),
                             ws.numel(), _stream(stream)), "moe_forward")
    return out


def moe_forward_profiled(layer_c, x: torch.Tensor, logits: torch.Tensor, out: torch.Tensor, ws: torch.Tensor,
                         events, stream=None) -> torch.Tensor:
    """moe_forward recording 6 torch.cuda.Event objects at the stage
    boundaries: start, after the activation quantisation, after the router
    top-k and permutation, after each grouped GEMM, after the combine (see
    include/moe_gb300.h)."""
    import ctypes
    if len(events) != 6:
        raise ValueError("events: expected 6 torch.cuda.Event objects")
    T = _forward_args(layer_c, x, logits, out, ws)
    handles = (ctypes.c_void_p * 6)(*[ev.cuda_event for ev in events])
    check(load().moe_forward_profiled(ctypes.byref(layer_c), _ptr(x), _ptr(logits), T, _ptr(out), _ptr(ws),
                                      ws.numel(), handles, _stream(stream)), "moe_forward_profiled")
    return out


def moe_forward_host(layer_c, x_host: torch.Tensor, logits_host: torch.Tensor, out_host: torch.Tensor,
                     x_dev: torch.Tensor, logits_dev: torch.Tensor, out_dev: torch.Tensor,
                     ws: torch.Tensor, stream=None) -> torch.Tensor:
    import ctypes
    T = _forward_args(layer_c, x_dev, logits_dev, out_dev, ws)
    _host(x_host, "x_host", torch.bfloat16, (T, layer_c.H))
    _host(logits_host, "logits_host", torch.float32, (T, layer_c.E))
    _host(out_host, "out_host", torch.bfloat16, (T, layer_c.H))
    check(load().moe_forward_host(ctypes.byref(layer_c), _ptr(x_host), _ptr(logits_host), T, _ptr(out_host),
                                  _ptr(x_dev), _ptr(logits_dev), _ptr(out_dev), _ptr(ws), ws.numel(),
                                  _stream(stream)), "moe_forward_host")
    return out_host


def moe_forward_host_pipelined(layer_c, x_host, logits_host, out_host, x_dev: torch.Tensor,
                               logits_dev: torch.Tensor, out_dev: torch.Tensor, ws: torch.Tensor, stream=None,
                               copy_stream=None):
    """n batches of T tokens through moe_forward_host_pipelined: x_host,
    logits_host, out_host are lists of n pinned host tensors (bf16 [T,H],
    fp32 [T,E], bf16 [T,H]); x_dev / logits_dev / out_dev hold two batches
    ([2,T,H], [2,T,E], [2,T,H]).  The layer runs on `stream`, the copies on
    `copy_stream` (a torch.cuda.Stream other than `stream`)."""
    import ctypes
    n = len(x_host)
    if n < 1 or len(logits_host) != n or len(out_host) != n:
        raise ValueError("x_host, logits_host, out_host: n >= 1 host tensors each")
    for nm, t, dt in (("x_dev", x_dev, torch.bfloat16), ("logits_dev", logits_dev, torch.float32),
                      ("out_dev", out_dev, torch.bfloat16)):
        _dev(t, nm, dtype=dt)
        if t.dim() != 3 or t.shape[0] != 2:
            raise ValueError(f"{nm}: expected two batches [2, T, ...]")
    T = _forward_args(layer_c, x_dev[0], logits_dev[0], out_dev[0], ws)
    for i in range(n):
        _host(x_host[i], f"x_host[{i}]", torch.bfloat16, (T, layer_c.H))
        _host(logits_host[i], f"logits_host[{i}]", torch.float32, (T, layer_c.E))
        _host(out_host[i], f"out_host[{i}]", torch.bfloat16, (T, layer_c.H))
    if copy_stream is None:
        raise ValueError("copy_stream: required (a stream other than the compute stream)")
    if stream is None:
        stream = torch.cuda.current_stream()
    if copy_stream.cuda_stream == stream.cuda_stream:
        raise ValueError("copy_stream: must differ from the compute stream")
    ptrs = lambda ts: (ctypes.c_void_p * n)(*[t.data_ptr() for t in ts])
    check(load().moe_forward_host_pipelined(ctypes.byref(layer_c), n, ptrs(x_host), ptrs(logits_host), T,
                                            ptrs(out_host), _ptr(x_dev), _ptr(logits_dev), _ptr(out_dev),
                                            _ptr(ws), ws.numel(), stream.cuda_stream, copy_stream.cuda_stream),
          "moe_forward_host_pipelined")
    return out_host


__all__ = ["MOE_FMT_BF16", "MOE_FMT_NVFP4", "MOE_FMT_MXFP8", "MOE_FMT_MXFP4", "moe_quant_mx", "MOE_EPI_STORE_BF16", "MOE_EPI_SWIGLU_BF16",
           "MOE_EPI_SWIGLU_NVFP4", "moe_version", "moe_sync_status", "moe_set_wait_timeout_ns",
           "moe_selftest_wait_timeout", "moe_selftest_grid_barrier_timeout", "moe_route", "moe_permute",
           "moe_route_permute", "moe_quant_nvfp4", "MOE_EPI_SWIGLU_MX",
           "moe_permute_noalloc", "moe_grouped_gemm", "moe_combine", "moe_shared_gate",
           "moe_forward_workspace_size", "moe_forward", "moe_forward_profiled", "moe_forward_host",
           "moe_forward_host_pipelined",
           "ForwardGraph"]


class ForwardGraph:
    """moe_forward captured as a CUDA graph on fixed buffers
    (moe_forward_graph_create): launch() replays the layer with one launch;
    the contents of x / logits may change between replays, the buffers may
    not.  Creating it runs the forward once."""

    def __init__(self, layer_c, x: torch.Tensor, logits: torch.Tensor, out: torch.Tensor, ws: torch.Tensor,
                 stream=None):
        import ctypes
        self._h = None
        T = _forward_args(layer_c, x, logits, out, ws)
        self._keep = (layer_c, x, logits, out, ws)
        h = ctypes.c_void_p()
        check(load().moe_forward_graph_create(ctypes.byref(layer_c), _ptr(x), _ptr(logits), T, _ptr(out),
                                              _ptr(ws), ws.numel(), _stream(stream), ctypes.byref(h)),
              "moe_forward_graph_create")
        self._h = h

    def launch(self, stream=None) -> None:
        check(load().moe_graph_launch(self._h, _stream(stream)), "moe_graph_launch")

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            load().moe_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
