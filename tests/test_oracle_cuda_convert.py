"""Pins the oracle's E4M3, E2M1 and E8M0 codecs to an independent implementation:
the fp32 -> FP8 (E4M3, saturating to the largest finite value) and fp32 ->
FP4 (E2M1, round to nearest even) conversions that CUDA's cuda_fp8.h and
cuda_fp4.h declare for host code, called from a small host program
(tests/cuda_host/fp_convert.cpp) compiled with the system C++ compiler.

The values cover every grid point, every midpoint between neighbouring grid
points (the ties), random values over the whole range including the E4M3
subnormals, values beyond the largest finite one (saturation), and their
negatives (the sign of codes that round to zero included)."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle import mx, nvfp4

F32 = np.float32
HERE = os.path.dirname(os.path.abspath(__file__))
CUDA_INC = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")


@pytest.fixture(scope="module")
def converter(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None or not os.path.exists(os.path.join(CUDA_INC, "cuda_fp4.h")):
        pytest.skip("needs a C++ compiler and CUDA's cuda_fp4.h")
    exe = str(tmp_path_factory.mktemp("fpconv") / "fp_convert")
    subprocess.run([cxx, "-O1", "-std=c++17", f"-I{CUDA_INC}", os.path.join(HERE, "cuda_host", "fp_convert.cpp"),
                    "-o", exe], check=True, capture_output=True)

    def run(vals: np.ndarray, mode: str = "fp"):
        """mode "fp": fp32 values -> (E4M3 bytes, E2M1 codes); "e8m0": fp32
        values -> E8M0 bytes rounded toward zero; "e8m0dec": E8M0 bytes ->
        bf16 bit patterns of their values."""
        if mode == "e8m0dec":
            words = np.asarray(vals, dtype=np.uint32)
        else:
            words = np.ascontiguousarray(vals, dtype=F32).view(np.uint32)
        text = "\n".join(f"{b:08x}" for b in words.tolist()) + "\n"
        out = subprocess.run([exe, mode], input=text, capture_output=True, text=True, check=True).stdout.split()
        nums = np.array([int(t, 16) for t in out], dtype=np.int64)
        if mode != "fp":
            return nums
        pairs = nums.reshape(-1, 2)
        return pairs[:, 0].astype(np.uint8), pairs[:, 1].astype(np.uint8)

    return run


def _with_negatives(v):
    v = np.asarray(v, dtype=F32)
    return np.concatenate([v, -v])


def test_e4m3_encoder_matches_cuda_host_conversion(converter):
    rng = np.random.default_rng(1)
    grid = nvfp4.E4M3_VALUES.astype(np.float64)
    mids = (grid[1:] + grid[:-1]) / 2
    rand = np.concatenate([np.exp(rng.uniform(np.log(2.0**-12), np.log(600.0), 30000)),
                           rng.uniform(0, 2.0**-6, 5000)])  # subnormal range
    big = np.array([448.0, 449.0, 464.0, 480.0, 500.0, 1e4, 3e38])
    vals = _with_negatives(np.concatenate([grid, mids, rand, big, [0.0]]).astype(F32))
    ref, _ = converter(vals)
    got = nvfp4.e4m3_encode(vals)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(vals[i]), int(got[i]), int(ref[i])) for i in bad[:10]]


def test_e2m1_encoder_matches_cuda_host_conversion(converter):
    rng = np.random.default_rng(2)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    mids = (grid[1:] + grid[:-1]) / 2  # 0.25 0.75 1.25 1.75 2.5 3.5 5
    near = np.concatenate([np.nextafter(mids.astype(F32), F32(0)), np.nextafter(mids.astype(F32), F32(10))])
    rand = np.concatenate([rng.uniform(0, 8, 30000), np.exp(rng.uniform(-20, 2, 5000))])
    big = np.array([6.0, 6.5, 7.0, 100.0, 3e38])
    vals = _with_negatives(np.concatenate([grid, mids, near, rand, big, [1e-30]]).astype(F32))
    _, ref = converter(vals)
    got = nvfp4.e2m1_encode(vals)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(vals[i]), int(got[i]), int(ref[i])) for i in bad[:10]]


def test_negative_values_that_round_to_zero_keep_the_sign(converter):
    """The reading the oracle takes for the sign of zero codes (-0 and tiny
    negatives -> code 0x8) is the conversion's own."""
    vals = np.array([-0.0, -1e-30, -0.1, -0.25, 0.0, 0.1, 0.25], dtype=F32)
    _, ref = converter(vals)
    assert ref.tolist() == [8, 8, 8, 8, 0, 0, 0]
    assert nvfp4.e2m1_encode(vals).tolist() == ref.tolist()


def test_e8m0_decode_matches_cuda_host_conversion(converter):
    """Every E8M0 byte decodes to 2^(c - 127) (255: NaN), as CUDA's
    __nv_cvt_e8m0_to_bf16raw does (bf16 holds 2^-127 .. 2^127 exactly)."""
    import torch
    codes = np.arange(256)
    bits = converter(codes, "e8m0dec")
    ref = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).double().numpy()
    got = mx.e8m0_decode(codes)
    assert np.array_equal(got[:255], ref[:255]) and np.isnan(got[255]) and np.isnan(ref[255])


def test_shared_exponent_is_cudas_round_toward_zero_e8m0(converter):
    """The scale exponent of a block is floor(log2(amax)) - emax: the E8M0
    code of amax rounded toward zero (CUDA's __nv_cvt_float_to_e8m0 with
    cudaRoundZero), minus emax, for every binade of fp32 from 2^-127 up."""
    rng = np.random.default_rng(3)
    k = rng.integers(-127, 128, 20000)
    amax = np.ldexp(rng.uniform(1.0, 2.0, k.size), k).astype(F32)
    amax = np.concatenate([amax, np.ldexp(1.0, np.arange(-127, 128)).astype(F32),
                           np.nextafter(np.ldexp(1.0, np.arange(-126, 128)).astype(F32), F32(0))])
    amax = amax[np.isfinite(amax) & (amax >= F32(2.0**-127))]
    ref = converter(amax, "e8m0")
    for fmt, emax in mx.EMAX.items():
        e = mx.shared_exponent(amax, fmt)
        assert np.array_equal(e, np.clip(ref - 127 - emax, -127, 127)), fmt
