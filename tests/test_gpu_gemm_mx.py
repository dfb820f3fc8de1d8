"""MXFP4 x MXFP4 and MXFP8 x MXFP8 grouped GEMMs (moe_grouped_gemm with
MOE_FMT_MXFP4 / MOE_FMT_MXFP8) against the fp64 product of the oracle's
dequantised operands (oracle/mx.py): ragged and empty groups, both bf16
epilogues, a one-group one-stage case first (the smallest check of the
block-scale descriptor and byte selection)."""

import numpy as np
import pytest
import torch

import oracle
from oracle import mx
from tests.helpers import require_gpu

pytestmark = pytest.mark.gpu

DEV = "cuda"
FMT = {"mxfp8": 2, "mxfp4": 3}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _ref(A, W, offs, swiglu, N):
    out = np.zeros((A.shape[0], N))
    for g in range(len(offs) - 1):
        a = A[offs[g]:offs[g + 1]]
        if swiglu:
            gt, up = a @ W[g, :N].T, a @ W[g, N:].T
            out[offs[g]:offs[g + 1]] = gt / (1 + np.exp(-gt)) * up
        else:
            out[offs[g]:offs[g + 1]] = a @ W[g].T
    return out


@pytest.mark.parametrize("fmt,epi,N,K,counts", [
    ("mxfp4", 0, 128, 512, [128]),              # one tile, one stage
    ("mxfp4", 0, 448, 1024, [0, 1, 127, 129, 300, 0, 40]),
    ("mxfp4", 1, 256, 1536, [300, 0, 513, 257, 64, 130]),
    ("mxfp4", 1, 192, 512, [7, 0, 260]),
    ("mxfp8", 0, 128, 256, [128]),              # one tile, one stage
    ("mxfp8", 0, 448, 768, [0, 1, 127, 129, 300, 0, 40]),
    ("mxfp8", 1, 256, 1280, [300, 0, 513, 257, 64, 130]),
    ("mxfp8", 1, 192, 256, [7, 0, 260]),
    ("mxfp8", 0, 256, 512, [192, 193, 385, 31, 33, 1000]),  # token blocks of the pair kernel
    ("mxfp8", 1, 384, 512, [192, 193, 385, 31, 33, 1000]),
])
def test_grouped_gemm_mx(fmt, epi, N, K, counts):
    import mixture_experts_layer_fwd_gb300 as m
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M, G = int(offs[-1]), len(counts)
    wn = N if epi == 0 else 2 * N
    g = torch.Generator().manual_seed(N + K + epi)
    x = (torch.randn(M, K, generator=g) * torch.exp(torch.randn(M, 1, generator=g))).numpy()
    Aq, As = mx.quantize(x, fmt)
    Wq, Ws = zip(*[mx.quantize((torch.randn(wn, K, generator=g) * 0.02).numpy(), fmt) for _ in range(G)])
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    C = m.moe_grouped_gemm(FMT[fmt], FMT[fmt], epi, t(offs), N, K, t(Aq), t(np.stack(Wq)), A_sf=t(As),
                           W_sf=t(np.stack(Ws)))
    assert m.moe_sync_status() == 0
    Ad = mx.dequantize(Aq, As, fmt)
    Wd = np.stack([mx.dequantize(q, s, fmt) for q, s in zip(Wq, Ws)])
    ref = _ref(Ad, Wd, offs, epi == 1, N)
    got = C.float().cpu().numpy()
    err = oracle.rel_frobenius(got, ref)
    assert err < 5e-3, err


@pytest.mark.parametrize("fmt,N,K,counts", [
    ("mxfp4", 128, 512, [128]),
    ("mxfp4", 256, 1536, [300, 0, 513, 257, 64, 130]),
    ("mxfp8", 128, 256, [128]),
    ("mxfp8", 192, 1280, [7, 0, 260, 129]),
    ("mxfp8", 256, 512, [192, 193, 385, 31, 33, 1000]),
])
def test_grouped_gemm_mx_swiglu_mx_epilogue(fmt, N, K, counts):
    """SWIGLU_MX: the epilogue quantises the fp32 SwiGLU output to the MX
    format (blocks of 32 along N).  Compared with the oracle's h step on the
    exact product (oracle.mx.h_quant): codes that sit on a rounding boundary
    may flip between the fp32 and fp64 values, so the decoded values are
    compared by relative Frobenius error."""
    import mixture_experts_layer_fwd_gb300 as m
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M, G = int(offs[-1]), len(counts)
    g = torch.Generator().manual_seed(N + K + 7)
    x = (torch.randn(M, K, generator=g) * torch.exp(torch.randn(M, 1, generator=g))).numpy()
    Aq, As = mx.quantize(x, fmt)
    Wq, Ws = zip(*[mx.quantize((torch.randn(2 * N, K, generator=g) * 0.05).numpy(), fmt) for _ in range(G)])
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    Cq, Cs = m.moe_grouped_gemm(FMT[fmt], FMT[fmt], m.MOE_EPI_SWIGLU_MX, t(offs), N, K, t(Aq), t(np.stack(Wq)),
                                A_sf=t(As), W_sf=t(np.stack(Ws)))
    assert m.moe_sync_status() == 0
    Ad = mx.dequantize(Aq, As, fmt)
    Wd = np.stack([mx.dequantize(q, s, fmt) for q, s in zip(Wq, Ws)])
    ref = mx.h_quant(fmt)(_ref(Ad, Wd, offs, True, N))
    got = mx.dequantize(Cq.cpu().numpy(), Cs.cpu().numpy(), fmt)
    err = oracle.rel_frobenius(got, ref)
    assert err < 2e-2 if fmt == "mxfp4" else err < 5e-3, err
