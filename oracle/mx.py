"""Microscaling (MX) codec of the oracle -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
legs may import this package.  The product path never does.

The pages name the formats without defining them: Qwen3-235B is served with
MXFP8 weights converted once after fine-tuning, and MXFP4 was considered
("Hosting Qwen on Blackwell", section "Quantização"); abs-max reductions run
over 16 elements for NVFP4 and over 32 for MXFP8 / MXFP4 ("CuTeDSL at
Perplexity", section on Blackwell support).  The reading taken for what they
leave open is the Open Compute Project's microscaling definition:

  * block    : 32 consecutive elements along the reduction dimension share
               one scale X = 2^e stored as an E8M0 byte (unsigned exponent,
               bias 127, code 255 = NaN, no mantissa)
  * element  : MXFP8 -> E4M3 (max 448 = 1.75 * 2^8, emax 8);
               MXFP4 -> E2M1 (max 6 = 1.5 * 2^2, emax 2)
  * scale    : e = floor(log2(amax_block)) - emax(element), clamped to
               [-127, 127]; an all-zero block takes the smallest scale
               (code 0)
  * elements : q_i = element_RNE_satfinite(x_i / 2^e) (the division by a
               power of two is exact; values above the element's largest
               magnitude saturate to it, ties go to the even code, the sign
               of x_i is kept, as in the NVFP4 codec)

Decoded value = element(q) * 2^e.  There is no tensor-wide scale.  MXFP4
codes pack two per byte (element 2j in the low nibble); MXFP8 codes are one
byte each.  Scales are raw E8M0 bytes, row-major [rows, cols/32].
"""
from __future__ import annotations

import numpy as np

from .nvfp4 import e2m1_decode, e2m1_encode, e4m3_decode, e4m3_encode, unpack_codes

F32 = np.float32
BLOCK = 32
E8M0_BIAS = 127
# largest unbiased exponent of each element type's normal values
EMAX = {"mxfp8": 8, "mxfp4": 2}


def e8m0_decode(c: np.ndarray) -> np.ndarray:
    """E8M0 byte(s) -> fp64 2^(c - 127); code 255 -> NaN."""
    c = np.asarray(c, dtype=np.int64)
    v = np.ldexp(np.ones(c.shape), c - E8M0_BIAS)
    return np.where(c == 255, np.nan, v)


def floor_log2(a: np.ndarray) -> np.ndarray:
    """floor(log2(a)) for positive finite fp32 values, exactly (frexp gives
    a = m * 2^k with 0.5 <= m < 1, so floor(log2(a)) = k - 1)."""
    _, k = np.frexp(np.asarray(a, dtype=F32).astype(np.float64))
    return k.astype(np.int64) - 1


def shared_exponent(amax: np.ndarray, fmt: str) -> np.ndarray:
    """Unbiased scale exponent e of each block from its fp32 abs-max."""
    amax = np.asarray(amax, dtype=F32)
    pos = amax > 0
    e = np.where(pos, floor_log2(np.where(pos, amax, F32(1))) - EMAX[fmt], -E8M0_BIAS)
    return np.clip(e, -E8M0_BIAS, E8M0_BIAS)


def quantize(x: np.ndarray, fmt: str):
    """Quantise an fp32 matrix [rows, cols] (cols % 32 == 0) to MXFP8 or MXFP4.

    Returns (codes, scales): MXFP8 codes uint8 [rows, cols] (E4M3 bytes),
    MXFP4 codes uint8 [rows, cols/2] (packed E2M1), scales uint8
    [rows, cols/32] (E8M0 bytes)."""
    if fmt not in EMAX:
        raise ValueError(f"unknown MX format {fmt!r}")
    x = np.asarray(x, dtype=F32)
    rows, cols = x.shape
    assert cols % BLOCK == 0
    blocks = x.reshape(rows, cols // BLOCK, BLOCK)
    amax = np.max(np.abs(blocks), axis=2)                        # exact
    e = shared_exponent(amax, fmt)
    # x / 2^e: exact in fp64, and exact after rounding to fp32 unless it
    # falls below fp32's range, where every element type rounds to zero anyway
    scaled = np.ldexp(blocks.astype(np.float64), -e[:, :, None]).astype(F32)
    if fmt == "mxfp8":
        q = e4m3_encode(scaled).reshape(rows, cols)
    else:
        q = e2m1_encode(scaled).reshape(rows, cols)
        q = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return q.astype(np.uint8), (e + E8M0_BIAS).astype(np.uint8)


def dequantize(codes: np.ndarray, scales: np.ndarray, fmt: str) -> np.ndarray:
    """MX -> fp64 values element(q) * 2^e (exact in fp64)."""
    if fmt == "mxfp8":
        vals = e4m3_decode(np.asarray(codes, dtype=np.uint8)).astype(np.float64)
    elif fmt == "mxfp4":
        vals = e2m1_decode(unpack_codes(codes)).astype(np.float64)
    else:
        raise ValueError(f"unknown MX format {fmt!r}")
    rows, cols = vals.shape
    sc = e8m0_decode(scales)[:, :, None]
    return (vals.reshape(rows, cols // BLOCK, BLOCK) * sc).reshape(rows, cols)


def round_bf16(v: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 -> bf16 (round to nearest even, torch's cast) -> fp64."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(v, dtype=np.float64).astype(F32)))
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def fake_quant(v: np.ndarray, fmt: str) -> np.ndarray:
    """Values (fp64, last dimension a multiple of 32) through the MX codec
    along the last dimension: the decoded values, fp64."""
    v = np.asarray(v, dtype=np.float64)
    q, s = quantize(v.reshape(-1, v.shape[-1]).astype(F32), fmt)
    return dequantize(q, s, fmt).reshape(v.shape)


def round_f32(v: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 (round to nearest even) -> fp64."""
    return np.asarray(v, dtype=np.float64).astype(F32).astype(np.float64)


def h_quant(fmt: str):
    """The MX layers' step between the SwiGLU and the down projection.  The
    pages leave it open; reading taken (the same as for the NVFP4
    activations): h is the SwiGLU output in fp32, the precision of the
    gate/up GEMM's accumulators, quantised from there in blocks of 32 along I
    like the activations along H."""
    return lambda h: fake_quant(round_f32(h), fmt)
