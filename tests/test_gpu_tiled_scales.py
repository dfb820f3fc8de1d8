"""The NVFP4 scale factors in the MMA's tile order and the grouped GEMM that
reads them (moe_sf_tile_bases, moe_sf_retile_rows, moe_sf_retile_weights,
moe_grouped_gemm_nvf4_tiled).

The tiled layouts are compared byte for byte with their definition in
include/moe_gb300.h, written out here with numpy loops.  The GEMM is compared
with moe_grouped_gemm on the same operands: both issue the same block-scaled
MMAs in the same order, so the outputs must be bit-identical.  It is also
compared with the fp64 reference within the NVFP4 tolerance.

These kernels have not run on a GPU yet, so the module runs only when
MOE_RUN_UNVALIDATED=1 is set."""
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import nvfp4
from tests.helpers import F32, require_gpu

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(os.environ.get("MOE_RUN_UNVALIDATED") != "1",
                                 reason="tiled-scale kernels not yet run on a GPU; opt in with MOE_RUN_UNVALIDATED=1")]

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def api():
    import mixture_experts_layer_fwd_gb300 as m
    return m


def _sync():
    st = api().moe_sync_status()
    assert st == 0, f"device status {st}"


def _offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def _tile_bases(offs, M):
    c = np.clip(offs.astype(np.int64), 0, M)
    rows = np.maximum(c[1:] - c[:-1], 0)
    return np.concatenate([[0], np.cumsum((rows + 127) // 128)]).astype(np.int32)


def _tiled_rows(sf, offs, K):
    """The definition: tile tile_base[g] + i // 128 holds row offsets[g] + i at
    lane (i % 128) % 32, quadrant (i % 128) // 32 of every k-step block."""
    M, ks = sf.shape[0], K // 64
    tb = _tile_bases(offs, M)
    out = np.zeros((int(tb[-1]), ks, 32, 4, 4), np.uint8)
    for g in range(len(offs) - 1):
        for i in range(int(offs[g + 1] - offs[g])):
            m = i % 128
            out[tb[g] + i // 128, :, m % 32, m // 32, :] = sf[offs[g] + i].reshape(ks, 4)
    return tb, out.reshape(-1)


def _tiled_weights(sf, N, K, swiglu):
    G, ks = sf.shape[0], K // 64
    nb = (N + 63) // 64 if swiglu else (N + 127) // 128
    out = np.zeros((G * nb, ks, 32, 4, 4), np.uint8)
    for g in range(G):
        for n in range(nb):
            for m in range(128):
                if swiglu:
                    f = 64 * n + (m & 63)
                    if f >= N:
                        continue
                    row = f if m < 64 else N + f
                else:
                    row = 128 * n + m
                    if row >= N:
                        continue
                out[g * nb + n, :, m % 32, m // 32, :] = sf[g, row].reshape(ks, 4)
    return out.reshape(-1)


def test_tile_bases_count_whole_tiles_per_group():
    counts = [0, 1, 127, 128, 129, 0, 300, 40]
    offs = _offsets(counts)
    M = int(offs[-1])
    tb = api().moe_sf_tile_bases(torch.from_numpy(offs).to(DEV), M)
    _sync()
    assert np.array_equal(tb.cpu().numpy(), _tile_bases(offs, M))


@pytest.mark.parametrize("K", [256, 512, 1280])
def test_retile_rows_matches_the_definition(K):
    counts = [0, 1, 127, 128, 129, 0, 300, 40]
    offs = _offsets(counts)
    M = int(offs[-1])
    rng = np.random.default_rng(K)
    sf = rng.integers(0, 256, size=(M, K // 16), dtype=np.uint8)
    m = api()
    offs_d = torch.from_numpy(offs).to(DEV)
    tb = m.moe_sf_tile_bases(offs_d, M)
    got = m.moe_sf_retile_rows(torch.from_numpy(sf).to(DEV), offs_d, tb, K)
    _sync()
    tb_ref, ref = _tiled_rows(sf, offs, K)
    assert np.array_equal(tb.cpu().numpy(), tb_ref)
    assert np.array_equal(got.cpu().numpy()[: ref.size], ref)


@pytest.mark.parametrize("swiglu,N,K", [(False, 448, 512), (False, 256, 256), (True, 256, 768), (True, 352, 512)])
def test_retile_weights_matches_the_definition(swiglu, N, K):
    G = 3
    wn = 2 * N if swiglu else N
    sf = np.random.default_rng(N + K).integers(0, 256, size=(G, wn, K // 16), dtype=np.uint8)
    got = api().moe_sf_retile_weights(torch.from_numpy(sf).to(DEV), N, K, swiglu)
    _sync()
    assert np.array_equal(got.cpu().numpy(), _tiled_weights(sf, N, K, swiglu))


def _gemm_ref(A, W, offs, swiglu, N):
    out = np.zeros((A.shape[0], N))
    for g in range(len(offs) - 1):
        a = A[offs[g]:offs[g + 1]]
        if swiglu:
            gt, up = a @ W[g, :N].T, a @ W[g, N:].T
            out[offs[g]:offs[g + 1]] = gt / (1 + np.exp(-gt)) * up
        else:
            out[offs[g]:offs[g + 1]] = a @ W[g].T
    return out


@pytest.mark.parametrize("epi,N,K,counts", [
    (0, 448, 512, [300, 0, 513, 257, 64, 130]),
    (1, 256, 768, [300, 0, 513, 257, 64, 130]),
    (0, 192, 256, [0, 1, 127, 129, 300, 0, 40]),
    (1, 192, 1280, [0, 1, 127, 129, 300, 0, 40]),
    (2, 352, 512, [260, 400, 0, 330]),
])
def test_tiled_gemm_equals_the_row_major_kernel(epi, N, K, counts):
    m = api()
    offs = _offsets(counts)
    M, G = int(offs[-1]), len(counts)
    wn = N if epi == 0 else 2 * N
    g = torch.Generator().manual_seed(N + K + epi)
    Aq, As, Ag = nvfp4.quantize(torch.randn(M, K, generator=g).numpy())
    Wq = [nvfp4.quantize((torch.randn(wn, K, generator=g) * 0.02).numpy()) for _ in range(G)]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    offs_d, A, A_sf = t(offs), t(Aq), t(As)
    W, W_sf = t(np.stack([q for q, _, _ in Wq])), t(np.stack([s for _, s, _ in Wq]))
    A_g = torch.tensor([Ag], dtype=torch.float32, device=DEV)
    W_g = torch.tensor([gg for _, _, gg in Wq], dtype=torch.float32, device=DEV)
    c_g = torch.tensor([F32(8.0 / 2688)], device=DEV) if epi == 2 else None
    ref = m.moe_grouped_gemm(1, 1, epi, offs_d, N, K, A, W, A_sf=A_sf, A_g=A_g, W_sf=W_sf, W_g=W_g, c_g=c_g)
    tb = m.moe_sf_tile_bases(offs_d, M)
    A_t = m.moe_sf_retile_rows(A_sf, offs_d, tb, K)
    W_t = m.moe_sf_retile_weights(W_sf, N, K, epi != 0)
    got = m.moe_grouped_gemm_nvf4_tiled(epi, offs_d, N, K, A, A_t, A_g, W, W_t, W_g, c_g=c_g)
    _sync()
    if epi == 2:
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
        return
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    Ad = nvfp4.dequantize(Aq, As, Ag)
    Wd = np.stack([nvfp4.dequantize(q, s, gg) for q, s, gg in Wq])
    err = oracle.rel_frobenius(got.float().cpu().numpy(), _gemm_ref(Ad, Wd, offs, epi == 1, N))
    assert err < 5e-3, err
