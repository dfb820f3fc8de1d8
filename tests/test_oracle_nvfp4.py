"""Pins of the oracle's NVFP4 codec against values the format fixes.

Hand-worked tables (tests/golden), a library conversion (torch's
float8_e4m3fn cast), exact round trips of representable values, and the
special blocks (all zero, subnormal scale, zero scale, saturation, outliers).
"""
import json
import os
import struct

import numpy as np
import pytest
import torch

from oracle import nvfp4

F32 = np.float32


def _parse_value(tok: str) -> np.float32:
    if tok.startswith("0x"):
        return np.frombuffer(struct.pack("<I", int(tok, 16)), dtype=np.float32)[0]
    return F32(float(tok))


def _read_table(path):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            a, b = line.split()
            rows.append((_parse_value(a), int(b, 16)))
    return rows


def test_e2m1_hand_table(golden_dir):
    rows = _read_table(os.path.join(golden_dir, "e2m1_table.txt"))
    vals = np.array([r[0] for r in rows], dtype=F32)
    want = np.array([r[1] for r in rows], dtype=np.uint8)
    got = nvfp4.e2m1_encode(vals)
    bad = [(float(v), hex(g), hex(w)) for v, g, w in zip(vals, got, want) if g != w]
    assert not bad, bad


def test_e4m3_hand_table(golden_dir):
    rows = _read_table(os.path.join(golden_dir, "e4m3_table.txt"))
    vals = np.array([r[0] for r in rows], dtype=F32)
    want = np.array([r[1] for r in rows], dtype=np.uint8)
    got = nvfp4.e4m3_encode(vals)
    bad = [(float(v), hex(g), hex(w)) for v, g, w in zip(vals, got, want) if g != w]
    assert not bad, bad


def _e2m1_brute(v):
    """Nearest grid magnitude by explicit distances in fp64, ties to the even
    code, sign from the input."""
    out = []
    for x in np.asarray(v, F32).tolist():
        a = abs(x)
        d = [abs(a - g) for g in nvfp4.E2M1_GRID]
        best = min(range(8), key=lambda c: (d[c], c % 2))
        out.append(best | (8 if np.signbit(np.float32(x)) else 0))
    return np.array(out, np.uint8)


def test_e2m1_matches_distance_brute_force():
    rng = np.random.default_rng(4)
    grid = nvfp4.E2M1_GRID
    mids = (grid[1:] + grid[:-1]) / 2
    vals = np.concatenate([rng.uniform(-8, 8, 4000), rng.standard_normal(2000), mids, -mids, grid, -grid,
                           np.nextafter(mids.astype(F32), np.float32(0)), np.nextafter(mids.astype(F32), np.float32(9))])
    vals = vals.astype(F32)
    assert np.array_equal(nvfp4.e2m1_encode(vals), _e2m1_brute(vals))


def test_e2m1_grid_round_trips():
    codes = np.arange(16, dtype=np.uint8)
    vals = nvfp4.e2m1_decode(codes)
    back = nvfp4.e2m1_encode(vals)
    assert np.array_equal(back, codes)
    assert list(vals[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e4m3_all_finite_codes_round_trip():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = nvfp4.e4m3_decode(codes)
    assert np.array_equal(nvfp4.e4m3_encode(vals), codes)


def test_e4m3_matches_torch_cast():
    """torch's float8_e4m3fn cast (round to nearest even) is an independent
    implementation; compare on in-range values including every midpoint."""
    rng = np.random.default_rng(0)
    grid = nvfp4.E4M3_VALUES
    mids = ((grid[1:] + grid[:-1]) / 2).astype(F32)
    rand = np.concatenate([rng.uniform(0, 448, 20000), np.exp(rng.uniform(-12, 6, 20000))])
    vals = np.concatenate([grid.astype(F32), mids, rand.astype(F32)])
    vals = vals[vals <= 448].astype(F32)
    vals = np.concatenate([vals, -vals])
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = nvfp4.e4m3_encode(vals)
    assert np.array_equal(got, ref), np.nonzero(got != ref)


def test_e4m3_decode_matches_torch():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    assert np.array_equal(nvfp4.e4m3_decode(codes), ref)


def test_hand_worked_blocks(golden_dir):
    with open(os.path.join(golden_dir, "nvfp4_blocks.json")) as f:
        spec = json.load(f)
    for b in spec["blocks"]:
        x = np.array(b["x"], dtype=F32)[None, :]
        g = None if b["g"] is None else F32(b["g"])
        packed, s, g_out = nvfp4.quantize(x, g)
        assert s[0, 0] == int(b["scale"], 16), b["name"]
        codes = nvfp4.unpack_codes(packed)[0]
        assert list(codes) == b["codes"], (b["name"], list(codes))
        if "packed" in b:
            assert [int(v) for v in packed[0]] == [int(p, 16) for p in b["packed"]], b["name"]
        if "expected_g" in b:
            assert g_out == F32(b["expected_g"])


def test_exact_values_round_trip():
    """Values e2m1 * e4m3 * g whose block abs-max maps to the scale exactly
    survive quantise -> dequantise unchanged."""
    rng = np.random.default_rng(1)
    g = F32(0.25)
    rows = []
    for _ in range(64):
        s = F32(nvfp4.E4M3_VALUES[rng.integers(40, 100)])  # normal E4M3 scale
        q = rng.integers(0, 16, size=16).astype(np.uint8)
        q[rng.integers(0, 16)] = 7 | (rng.integers(0, 2) << 3)  # block max = 6 * s
        rows.append(nvfp4.e2m1_decode(q).astype(np.float64) * float(s) * float(g))
    x = np.array(rows, dtype=F32)
    packed, sc, _ = nvfp4.quantize(x, g)
    back = nvfp4.dequantize(packed, sc, g)
    assert np.array_equal(back.astype(F32), x)


def test_saturation_and_outliers():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((8, 64)).astype(F32)
    x[3, 5] *= 20
    packed, sc, g = nvfp4.quantize(x)
    assert g == F32(np.max(np.abs(x)) / F32(2688))
    # the outlier's block scale is the largest; its element decodes to within
    # half a grid step of the value
    deq = nvfp4.dequantize(packed, sc, g)
    blk = 5 // 16
    scale = nvfp4.e4m3_decode(sc[3, blk]) * g
    assert abs(deq[3, 5] - x[3, 5]) <= 1.0 * scale + 1e-12
    # values beyond 6 * 448 * g saturate to the largest magnitude
    y = np.full((1, 16), 1.0, F32)
    y[0, 0] = 1e6
    p2, s2, g2 = nvfp4.quantize(y, F32(1e-3))
    assert s2[0, 0] == 0x7E and (nvfp4.unpack_codes(p2)[0, 0] & 7) == 7


def test_quantisation_error_bound():
    """Every decoded element is within half a step of the block's grid,
    i.e. |x - x^| <= 1.0 * dec(s) * g (largest step is 2 between 4 and 6)
    when the block scale is not saturated."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((32, 128)) * rng.uniform(0.01, 10, (32, 1))).astype(F32)
    packed, sc, g = nvfp4.quantize(x)
    deq = nvfp4.dequantize(packed, sc, g)
    step = np.repeat(nvfp4.e4m3_decode(sc).astype(np.float64) * float(g), 16, axis=1)
    assert np.all(np.abs(deq - x) <= step + 1e-12)
    # and the relative error of the whole tensor is that of a 4-bit format
    rel = np.linalg.norm(deq - x) / np.linalg.norm(x)
    assert 0.02 < rel < 0.2


def test_zero_tensor():
    x = np.zeros((2, 32), F32)
    packed, sc, g = nvfp4.quantize(x)
    assert g == 1.0 and not packed.any() and not sc.any()


def test_packing_order():
    x = np.zeros((1, 16), F32)
    x[0, 0] = 6.0   # code 7, low nibble of byte 0
    x[0, 1] = -1.0  # code 0xA, high nibble of byte 0
    packed, sc, g = nvfp4.quantize(x, F32(1.0))
    # block max 6 -> s = E4M3(1.0) = 0x38, dec = 1
    assert sc[0, 0] == 0x38
    assert packed[0, 0] == 0xA7
