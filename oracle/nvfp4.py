"""NVFP4 codec of the oracle -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
legs may import this package.  The product path (the CUDA library and its
Python binding) never does.

The format is the one the pages name for expert weights and dispatched
activations ("Driving vLLM WideEP ... on Blackwell (Part I)", sections "NVFP4
GEMM for MoE and O-proj" and "NVFP4 MoE dispatch"; "CuTeDSL at Perplexity",
section on Blackwell support: abs-max over 16 elements for NVFP4):

  * element  : E2M1, 4 bits, sign bit 3, magnitudes by code 0..7 =
               {0, 0.5, 1, 1.5, 2, 3, 4, 6}
  * block    : 16 consecutive elements along the reduction dimension share
               one E4M3 scale byte (bias 7, 3 mantissa bits, max 448,
               no infinities, 0x7f/0xff are NaN)
  * tensor   : one fp32 global scale g

Decoded value = e2m1(q) * e4m3(s) * g.

The pages leave the rounding recipe open.  The reading taken is, in IEEE
fp32 arithmetic with round-to-nearest-even:

    amax = max |x|                  over the tensor (or one group of it)
    g    = amax / 2688              (2688 = 6 * 448); g = 1 when amax == 0
    a_b  = max |x_i|                over a block of 16
    s_b  = E4M3_RNE_satfinite(a_b / (6 * g))
    q_i  = E2M1_RNE_satfinite(x_i / (dec(s_b) * g)),  magnitude 0 when dec(s_b) == 0

The sign bit of q always carries the sign of x (so -0.0 and tiny negatives
encode as 0x8).  Two codes pack into one byte: element 2j in the low nibble,
element 2j+1 in the high nibble.  Scales are raw E4M3 bytes, row-major.

Everything here is written from those definitions: the E4M3 encoder finds the
nearest representable value by comparing distances in fp64 (exact for fp32
inputs); the E2M1 encoder compares against the midpoints of its 8-value grid;
both break ties towards the even code.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32

# E2M1 magnitudes by code 0..7 (the code's low three bits).
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)

FP4_MAX = 6.0
E4M3_MAX = 448.0
GLOBAL_DIVISOR = F32(2688.0)  # 6 * 448
BLOCK = 16


def _e4m3_table() -> np.ndarray:
    """Values of the non-negative finite E4M3 codes 0x00..0x7e, in code order.

    Code = (e << 3) | m.  e == 0: subnormal m/8 * 2^-6.  e >= 1: (1 + m/8) * 2^(e-7).
    Code 0x7f (e=15, m=7) is NaN and is excluded.  The values are strictly
    increasing with the code.
    """
    vals = []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        if e == 0:
            vals.append((m / 8.0) * 2.0 ** -6)
        else:
            vals.append((1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, dtype=np.float64)


E4M3_VALUES = _e4m3_table()


def e4m3_decode(b: np.ndarray) -> np.ndarray:
    """E4M3 byte(s) -> fp32 value(s).  NaN codes are not produced by the encoder."""
    b = np.asarray(b, dtype=np.uint8)
    mag = E4M3_VALUES[np.minimum(b & 0x7F, 0x7E)]
    sign = np.where(b & 0x80, -1.0, 1.0)
    return (sign * mag).astype(F32)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """fp32 -> E4M3 byte, round to nearest, ties to the even code, saturating
    to +-448 (no NaN/Inf out).  Inputs must be finite."""
    v = np.asarray(v, dtype=F32).astype(np.float64)
    a = np.abs(v)
    grid = E4M3_VALUES
    hi = np.searchsorted(grid, a, side="left")          # grid[hi-1] < a <= grid[hi]
    hi = np.clip(hi, 0, len(grid) - 1)
    lo = np.clip(hi - 1, 0, len(grid) - 1)
    d_lo = np.abs(a - grid[lo])
    d_hi = np.abs(a - grid[hi])
    code = np.where(d_lo < d_hi, lo, hi)
    tie = d_lo == d_hi
    code = np.where(tie, np.where(lo % 2 == 0, lo, hi), code)
    code = np.where(a >= grid[-1], len(grid) - 1, code)  # satfinite
    sign = np.signbit(v).astype(np.uint8) << 7
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def e2m1_decode(q: np.ndarray) -> np.ndarray:
    """4-bit code(s) (values 0..15, one per array element) -> fp32."""
    q = np.asarray(q, dtype=np.uint8)
    mag = E2M1_GRID[q & 7]
    return np.where(q & 8, -mag, mag).astype(F32)


# Rounding to the nearest grid magnitude, ties to the even code, written
# through the midpoints between neighbouring magnitudes: a value moves past a
# midpoint when it lies strictly above it, or exactly on it when the upper
# neighbour has the even code.  Values above the largest midpoint saturate to
# the largest magnitude.
E2M1_MIDPOINTS = ((E2M1_GRID[1:] + E2M1_GRID[:-1]) / 2).astype(np.float32)
E2M1_TIE_GOES_UP = (np.arange(1, 8) % 2) == 0


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """fp32 -> 4-bit code, round to nearest grid magnitude, ties to the even
    code, saturating to 6.  Sign bit = sign of the input (also for zeros)."""
    v = np.asarray(v, dtype=F32)
    a = np.abs(v)
    mag = np.zeros(v.shape, dtype=np.uint8)
    for mid, up in zip(E2M1_MIDPOINTS, E2M1_TIE_GOES_UP):
        mag += (a >= mid) if up else (a > mid)
    sign = np.signbit(v).astype(np.uint8) << 3
    return (mag | sign).astype(np.uint8)


def global_scale(x: np.ndarray) -> np.float32:
    """g = amax(|x|) / 2688 in fp32; 1 for an all-zero tensor."""
    amax = F32(np.max(np.abs(np.asarray(x, dtype=F32)))) if np.asarray(x).size else F32(0)
    if amax == 0:
        return F32(1.0)
    return F32(amax / GLOBAL_DIVISOR)


def quantize(x: np.ndarray, g: np.float32 | None = None):
    """Quantise an fp32 matrix [rows, cols] (cols % 16 == 0) to NVFP4.

    Returns (packed codes uint8 [rows, cols/2], scales uint8 [rows, cols/16], g).
    If g is None it is derived from the whole matrix (global_scale).
    """
    x = np.asarray(x, dtype=F32)
    rows, cols = x.shape
    assert cols % BLOCK == 0
    if g is None:
        g = global_scale(x)
    g = F32(g)
    blocks = x.reshape(rows, cols // BLOCK, BLOCK)
    a_b = np.max(np.abs(blocks), axis=2)                       # exact
    six_g = F32(F32(6.0) * g)                                  # fp32 multiply
    s = e4m3_encode((a_b / six_g).astype(F32))                 # fp32 divide
    d = e4m3_decode(s)                                         # exact
    denom = (d * g).astype(F32)                                # fp32 multiply
    safe = np.where(denom == 0, F32(1.0), denom).astype(F32)
    ratio = (blocks / safe[:, :, None]).astype(F32)            # fp32 divide
    q = e2m1_encode(ratio)
    q = np.where((denom == 0)[:, :, None], q & 8, q).astype(np.uint8)
    q = q.reshape(rows, cols)
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return packed, s.astype(np.uint8), g


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    """[rows, cols/2] packed bytes -> [rows, cols] 4-bit codes."""
    packed = np.asarray(packed, dtype=np.uint8)
    rows, half = packed.shape
    q = np.empty((rows, half * 2), dtype=np.uint8)
    q[:, 0::2] = packed & 0x0F
    q[:, 1::2] = packed >> 4
    return q


def dequantize(packed: np.ndarray, scales: np.ndarray, g) -> np.ndarray:
    """NVFP4 -> fp64 values e2m1(q) * e4m3(s) * g (exact in fp64)."""
    q = unpack_codes(packed)
    rows, cols = q.shape
    vals = e2m1_decode(q).astype(np.float64).reshape(rows, cols // BLOCK, BLOCK)
    sc = e4m3_decode(scales).astype(np.float64)[:, :, None]
    return (vals * sc * np.float64(g)).reshape(rows, cols)
