"""MXFP8 / MXFP4 quantiser (moe_quant_mx) against the oracle's codec
(oracle/mx.py), bit for bit: codes and E8M0 scale bytes.

Inputs: normal rows with x20 outliers, all-zero blocks, blocks of tiny
values (subnormal abs-max), negative zeros, signed ties of both element
grids times powers of two, and shapes from one 32-element block to the
7168-wide deepseek-v3 rows (a partial last 256-column chunk included)."""

import numpy as np
import pytest
import torch

from oracle import mx, nvfp4
from tests.helpers import require_gpu

pytestmark = pytest.mark.gpu

DEV = "cuda"
FMTS = {"mxfp8": 2, "mxfp4": 3}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _inputs(rows, cols, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g) * torch.exp(torch.randn(rows, 1, generator=g) * 3)
    mask = torch.rand(rows, cols, generator=g) < 0.001
    x = torch.where(mask, x * 20, x)
    if cols >= 128:
        x[:, 32:64] = 0.0                                   # all-zero block
        x[:, 64:96] = torch.randn(rows, 32, generator=g) * 1e-39  # subnormal abs-max
        x[0, 96:98] = -0.0
    xb = x.to(torch.bfloat16)
    if cols >= 256 and rows >= 2:
        # ties of both grids at a block whose scale is 2^0 (MXFP8) / 2^0 (MXFP4)
        e4 = nvfp4.E4M3_VALUES[(nvfp4.E4M3_VALUES > 0) & (nvfp4.E4M3_VALUES < 448)]
        mids = ((e4[1:] + e4[:-1]) / 2)[:31]
        row = np.concatenate([[448.0], mids]).astype(np.float32)
        xb[1, 128:160] = torch.from_numpy(row).to(torch.bfloat16)
        f4 = np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0] * 4, dtype=np.float32)
        xb[1, 160:192] = torch.from_numpy(-f4).to(torch.bfloat16)
    return xb


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 96), (64, 256), (257, 7168), (40, 2048 + 160)])
def test_quant_mx_bit_exact(fmt, rows, cols):
    import mixture_experts_layer_fwd_gb300 as m
    xb = _inputs(rows, cols, seed=rows + cols)
    codes, scales = m.moe_quant_mx(xb.to(DEV), FMTS[fmt])
    assert m.moe_sync_status() == 0
    rq, rs = mx.quantize(xb.float().numpy(), fmt)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rq)


def test_quant_mx_zero_rows_is_a_noop():
    import mixture_experts_layer_fwd_gb300 as m
    codes, scales = m.moe_quant_mx(torch.empty(0, 64, dtype=torch.bfloat16, device=DEV), FMTS["mxfp8"])
    assert codes.shape == (0, 64) and scales.shape == (0, 2)
    assert m.moe_sync_status() == 0
