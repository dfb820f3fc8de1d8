"""Pins of the oracle's microscaling codec (oracle/mx.py): MXFP8 and MXFP4
with one E8M0 scale per 32 elements.

Independent checks: values worked out by hand from the format definition,
exact round trips of values the formats represent, the rounding error bound
of each element type, torch's own E8M0 decode, block independence and the
nibble order.  The E8M0 codec itself is also pinned to CUDA's host
conversions in test_oracle_cuda_convert.py."""
import numpy as np
import pytest
import torch

from oracle import mx, nvfp4

F32 = np.float32


def _block(values, fill=0.0):
    row = np.full(32, fill, dtype=F32)
    row[: len(values)] = values
    return row


@pytest.mark.parametrize("fmt,amax,code,first", [
    # MXFP8: e = floor(log2 amax) - 8
    ("mxfp8", 1.0, 119, 1.0),        # 1 = 256 * 2^-8: element 256 (0x78)
    ("mxfp8", 448.0, 127, 448.0),    # largest element at scale 1
    ("mxfp8", 500.0, 127, 448.0),    # floor(log2 500) = 8: 500 saturates to 448
    ("mxfp8", 0.75, 118, 0.75),      # floor(log2 0.75) = -1: 0.75 = 384 * 2^-9
    # MXFP4: e = floor(log2 amax) - 2
    ("mxfp4", 6.0, 127, 6.0),
    ("mxfp4", 1.0, 125, 1.0),        # 1 = 4 * 2^-2
    ("mxfp4", 7.0, 127, 6.0),        # 7 saturates to 6
    ("mxfp4", 448.0, 133, 384.0),    # 448 / 2^6 = 7 -> 6 -> 384
])
def test_hand_worked_blocks(fmt, amax, code, first):
    x = _block([amax, 1e-30, -amax])[None, :]
    q, s = mx.quantize(x, fmt)
    assert int(s[0, 0]) == code
    d = mx.dequantize(q, s, fmt)[0]
    assert d[0] == first and d[2] == -first and d[1] == 0.0


def test_zero_block_takes_the_smallest_scale():
    for fmt in mx.EMAX:
        q, s = mx.quantize(np.zeros((2, 64), F32), fmt)
        assert np.all(s == 0) and np.all(q == 0)
        assert np.all(mx.dequantize(q, s, fmt) == 0.0)


def test_e8m0_decode_hand_values_and_torch():
    c = np.array([0, 1, 126, 127, 128, 254])
    assert mx.e8m0_decode(c).tolist() == [2.0**-127, 2.0**-126, 0.5, 1.0, 2.0, 2.0**127]
    assert np.isnan(mx.e8m0_decode(np.array([255]))[0])
    if hasattr(torch, "float8_e8m0fnu"):
        codes = np.arange(255, dtype=np.uint8)
        ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).double().numpy()
        assert np.array_equal(mx.e8m0_decode(codes), ref)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_representable_values_round_trip_exactly(fmt):
    """Blocks of element-grid values times 2^e whose largest magnitude lies
    in the element type's top binade come back bit for bit, with scale e."""
    rng = np.random.default_rng(7)
    if fmt == "mxfp8":
        grid = nvfp4.E4M3_VALUES.astype(np.float64)
        top = grid[(grid >= 256) & (grid <= 448)]
    else:
        grid = nvfp4.E2M1_GRID
        top = grid[grid >= 4]
    rows, nb = 16, 4
    vals = rng.choice(grid, size=(rows, nb, 32)) * rng.choice([-1.0, 1.0], size=(rows, nb, 32))
    vals[:, :, 5] = rng.choice(top, size=(rows, nb)) * rng.choice([-1.0, 1.0], size=(rows, nb))
    vals = np.minimum(np.abs(vals), np.abs(vals[:, :, 5:6])) * np.sign(vals)  # keep slot 5 the largest
    e = rng.integers(-100, 100, size=(rows, nb))
    x = np.ldexp(vals, e[:, :, None]).reshape(rows, nb * 32).astype(F32)
    q, s = mx.quantize(x, fmt)
    assert np.array_equal(s.astype(np.int64) - 127, e)
    assert np.array_equal(mx.dequantize(q, s, fmt), x.astype(np.float64))


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_rounding_error_bound(fmt):
    """Every element is within half a step of the element grid at its
    magnitude, times the block scale; saturated elements lie within the
    block's top binade, above the largest element magnitude."""
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((64, 256)) * np.exp(rng.uniform(-8, 8, (64, 1)))).astype(F32)
    x[::7, 3] *= 20  # outliers
    q, s = mx.quantize(x, fmt)
    d = mx.dequantize(q, s, fmt)
    scale = np.repeat(mx.e8m0_decode(s), 32, axis=1)
    v = np.abs(x.astype(np.float64)) / scale          # magnitude in element units
    if fmt == "mxfp8":
        vmax = 448.0
        # spacing 2^(floor(log2 v) - 3) for normals (v >= 2^-6), 2^-9 below
        step = np.where(v >= 2.0**-6, np.ldexp(1.0, np.floor(np.log2(np.maximum(v, 2.0**-6))).astype(int) - 3),
                        2.0**-9)
    else:
        vmax = 6.0
        step = np.where(v < 2, 0.5, np.where(v < 4, 1.0, 2.0))
    err = np.abs(d - x.astype(np.float64)) / scale
    inside = v <= vmax
    assert np.all(err[inside] <= step[inside] / 2 + 1e-12)
    assert np.all(v < 2 * 2.0 ** mx.EMAX[fmt])      # the floor rule keeps amax below 2^(emax+1)
    assert np.all(np.abs(d)[~inside] == vmax * scale[~inside])


def test_blocks_are_independent_and_nibbles_ordered():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 96)).astype(F32)
    q, s = mx.quantize(x, "mxfp4")
    y = x.copy()
    y[:, 32:64] *= 1000
    q2, s2 = mx.quantize(y, "mxfp4")
    assert np.array_equal(s[:, [0, 2]], s2[:, [0, 2]]) and np.array_equal(q[:, :16], q2[:, :16])
    assert np.array_equal(q[:, 32:], q2[:, 32:])
    # element 2j in the low nibble: a block whose even elements are its max
    z = np.zeros((1, 32), F32)
    z[0, 0], z[0, 1] = 6.0, 1.0
    qz, _ = mx.quantize(z, "mxfp4")
    assert qz[0, 0] == (7 | (2 << 4))


def test_unknown_format_is_rejected():
    with pytest.raises(ValueError):
        mx.quantize(np.zeros((1, 32), F32), "mxfp6")


# ------------------------------------------------ the MX layers' h step ----
def _h_probe(h_values):
    """Weights that make h = h_values for the input row e_0: gate = 50
    (silu(50) == 50 in fp64), up_i = h_i / 50, down = identity."""
    I = len(h_values)
    a = np.eye(I)[:1]
    w13 = np.zeros((2 * I, I))
    w13[:I, 0] = 50.0
    w13[I:, 0] = np.asarray(h_values, np.float64) / 50.0
    return a, w13, np.eye(I)


def test_mxfp4_h_step_hand_worked():
    """Block amax 6 -> scale 2^0: h (in fp32) is rounded to the E2M1 grid
    itself, ties to the even code (1.25 -> 1, 2.5 -> 2, 3.5 -> 4, 5 -> 4;
    1.6 -> 1.5, -5.1 -> -6)."""
    from oracle.moe import expert_mlp
    h = [6.0, 1.25, 3.5, 5.0, 0.25, 2.5, -0.8, 1.6, -4.4, 0.3, 0.0, 2.9, -5.1, 0.7, 1.9, 3.2] + [0.0] * 16
    want = [6.0, 1.0, 4.0, 4.0, 0.0, 2.0, -1.0, 1.5, -4.0, 0.5, 0.0, 3.0, -6.0, 0.5, 2.0, 3.0] + [0.0] * 16
    a, w13, w2 = _h_probe(h)
    y = expert_mlp(a, w13, w2, h_quant=mx.h_quant("mxfp4"))[0]
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-12)


def test_mxfp8_h_step_hand_worked():
    """Block amax 448 -> scale 2^0: E4M3 grid, ties to the even code (17 ->
    16, 19 -> 20, 0.0068359375 = 3.5 * 2^-9 -> 4 * 2^-9)."""
    from oracle.moe import expert_mlp
    h = [448.0, 17.0, 19.0, -240.0, 3.5 * 2.0**-9] + [1.0] * 27
    want = [448.0, 16.0, 20.0, -240.0, 4 * 2.0**-9] + [1.0] * 27
    a, w13, w2 = _h_probe(h)
    y = expert_mlp(a, w13, w2, h_quant=mx.h_quant("mxfp8"))[0]
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-12)


def test_h_step_quantises_the_fp32_value():
    """h enters the codec as fp32: 1.2500001 (fp32 1.25000012) lies above
    the E2M1 tie 1.25 and goes to 1.5, where a bf16 rounding first (to 1.25
    exactly, a tie that goes to the even code 1) would give 1.  And a value
    that fp32 rounds onto the tie, 1.25 + 2^-30, goes to the even code 1."""
    from oracle.moe import expert_mlp
    h = [6.0, 1.2500001, 1.25 + 2.0**-30] + [0.0] * 29
    a, w13, w2 = _h_probe(h)
    y = expert_mlp(a, w13, w2, h_quant=mx.h_quant("mxfp4"))[0]
    assert y[1] == 1.5
    assert y[2] == 1.0
    assert mx.fake_quant(mx.round_bf16(np.array([h])), "mxfp4")[0, 1] == 1.0


def test_forward_applies_the_h_step_to_routed_and_shared_experts():
    """forward hands h_quant to every routed expert and hs_quant to the
    shared one: zeroing h in either removes exactly that part."""
    from oracle.moe import ExpertWeights, forward
    rng = np.random.default_rng(2)
    T, H, E, k, I = 5, 32, 4, 2, 32
    experts = [ExpertWeights(rng.standard_normal((2 * I, H)) * 0.1, rng.standard_normal((H, I)) * 0.1)
               for _ in range(E)]
    shared = ExpertWeights(rng.standard_normal((2 * I, H)) * 0.1, rng.standard_normal((H, I)) * 0.1)
    x = rng.standard_normal((T, H))
    logits = rng.standard_normal((T, E)).astype(F32)
    zero = lambda h: 0.0 * h
    full, *_ = forward(x, logits, k, E, lambda e: experts[e], shared)
    routed_only, *_ = forward(x, logits, k, E, lambda e: experts[e], shared, hs_quant=zero)
    shared_only, *_ = forward(x, logits, k, E, lambda e: experts[e], shared, h_quant=zero)
    assert np.abs(shared_only).max() > 0 and np.abs(routed_only).max() > 0
    np.testing.assert_allclose(routed_only + shared_only, full, rtol=1e-12, atol=1e-12)
