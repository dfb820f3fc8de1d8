"""Inputs outside the documented contract that only the device sees.

Three cases: expert ids outside [0, E) given to the permutation, row indices
outside [0, T*k) given to the combine, and group offsets that decrease or
run past the rows of A given to the grouped GEMM.  Each becomes a documented
result: a left-out slot, a zero contribution, or an empty or clamped group.
Ids outside the range are also reported as an error status that the host
reads.  None of them may make a kernel touch memory outside its buffers.
Also covered: the Python binding rejects wrong shapes and sizes before any
launch."""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import require_gpu

pytestmark = pytest.mark.gpu

DEV = "cuda"
MOE_ERR_INVALID_ARG = 1


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def api():
    import mixture_experts_layer_fwd_gb300 as m
    return m


def _sync():
    st = api().moe_sync_status()
    assert st == 0, f"device status {st}"


def _stable_permutation(idx, E):
    """Brute-force stable permutation of the slots whose id lies in [0, E):
    slots in flattened (token, j) order, each expert's rows in that order."""
    T, k = idx.shape
    flat = idx.reshape(-1).astype(np.int64)
    valid = (flat >= 0) & (flat < E)
    counts = np.bincount(flat[valid], minlength=E).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    nxt = offsets[:-1].astype(np.int64)
    row_of = np.full(T * k, -1, np.int32)
    src_tok = np.full(int(offsets[-1]), -1, np.int32)
    for s in range(T * k):
        if valid[s]:
            e = flat[s]
            row_of[s] = nxt[e]
            src_tok[nxt[e]] = s // k
            nxt[e] += 1
    return counts, offsets, row_of.reshape(T, k), src_tok


def test_permute_leaves_out_ids_outside_the_expert_range():
    T, E, k, H = 300, 16, 4, 64
    g = torch.Generator().manual_seed(3)
    idx = oracle.route(torch.randn(T, E, generator=g).numpy(), k)[0].copy()
    bad = np.random.default_rng(4).choice(T * k, size=40, replace=False)
    vals = np.array([-1, E, E + 1000, -2**31, 2**31 - 1], dtype=np.int64)
    flat = idx.reshape(-1)
    flat[bad] = vals[np.arange(bad.size) % vals.size]
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    m = api()
    r = m.moe_permute(torch.from_numpy(idx).to(DEV), E, x.to(DEV))
    assert m.moe_sync_status() == MOE_ERR_INVALID_ARG
    assert m.moe_sync_status() == 0  # the record is cleared
    counts, offsets, row_of, src_tok = _stable_permutation(idx, E)
    assert offsets[-1] == T * k - bad.size
    assert np.array_equal(r["counts"].cpu().numpy(), counts)
    assert np.array_equal(r["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(r["row_of"].cpu().numpy(), row_of)
    n = int(offsets[-1])
    assert np.array_equal(r["src_tok"].cpu().numpy()[:n], src_tok)
    xp = r["xp"].cpu()[:n]
    assert torch.equal(xp.view(torch.int16), x[torch.from_numpy(src_tok).long()].view(torch.int16))


def test_permute_with_valid_ids_reports_nothing():
    T, E, k = 64, 8, 2
    idx = oracle.route(torch.randn(T, E, generator=torch.Generator().manual_seed(5)).numpy(), k)[0]
    api().moe_permute(torch.from_numpy(idx).to(DEV), E)
    _sync()


def test_combine_skips_rows_outside_the_permuted_buffer():
    T, k, H, E = 64, 4, 256, 16
    g = torch.Generator().manual_seed(7)
    idx = oracle.route(torch.randn(T, E, generator=g).numpy(), k)[0]
    row_of = oracle.permute(idx, E).row_of.copy()
    row_of[::7, 1] = -1
    row_of[3::11, 2] = T * k
    row_of[5, 0] = 2**31 - 1
    w = torch.rand(T, k, generator=g)
    Y = torch.randn(T * k, H, generator=g).to(torch.bfloat16)
    out = api().moe_combine(Y.to(DEV), torch.from_numpy(row_of).to(DEV), w.to(DEV), None, T, k, H)
    _sync()
    valid = (row_of >= 0) & (row_of < T * k)
    Yd = Y.double().numpy()
    ref = np.einsum("tj,tjh->th", w.double().numpy() * valid, Yd[np.where(valid, row_of, 0)])
    err = oracle.rel_frobenius(out.float().cpu().numpy(), ref)
    assert err < 3e-3, err


def test_grouped_gemm_clamps_offsets_outside_the_contract():
    """offsets [-5, 100, 50, 400, 300] over 256 rows read as [0, 100, 50, 256,
    256]: group 0 owns rows [0, 100), group 1 is empty (end before start),
    group 2 owns rows [50, 256), group 3 is empty.  Rows [50, 100) are
    written by two groups and are not checked."""
    m = api()
    M, N, K, G = 256, 256, 256, 4
    offs = torch.tensor([-5, 100, 50, 400, 300], dtype=torch.int32)
    g = torch.Generator().manual_seed(9)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W = (torch.randn(G, N, K, generator=g) * 0.05).to(torch.bfloat16)
    C = torch.zeros(M, N, dtype=torch.bfloat16, device=DEV)
    m.moe_grouped_gemm(0, 0, 0, offs.to(DEV), N, K, A.to(DEV), W.to(DEV), C=C)
    _sync()
    Cd = C.float().cpu().numpy()
    Ad, Wd = A.double().numpy(), W.double().numpy()
    assert oracle.rel_frobenius(Cd[:50], Ad[:50] @ Wd[0].T) < 5e-3
    assert oracle.rel_frobenius(Cd[100:], Ad[100:] @ Wd[2].T) < 5e-3


def test_binding_rejects_wrong_shapes_before_any_launch():
    m = api()
    T, k, H = 8, 2, 256
    Y = torch.zeros(T * k, H, dtype=torch.bfloat16, device=DEV)
    row_of = torch.zeros(T, k, dtype=torch.int32, device=DEV)
    w = torch.zeros(T, k, dtype=torch.float32, device=DEV)
    with pytest.raises(ValueError):
        m.moe_combine(Y[: T * k - 1], row_of, w, None, T, k, H)  # Y too small
    with pytest.raises(ValueError):
        m.moe_combine(Y, row_of, w, None, T, k, H, out=torch.zeros(T, H - 8, dtype=torch.bfloat16, device=DEV))
    with pytest.raises(TypeError):
        m.moe_route(torch.zeros(T, 8, dtype=torch.float64, device=DEV), k)
    offs = torch.tensor([0, 4, 8], dtype=torch.int32, device=DEV)
    A = torch.zeros(8, 256, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError):  # two groups of 128 x 256 weights need 2x the bytes given
        m.moe_grouped_gemm(0, 0, 0, offs, 128, 256, A, torch.zeros(1, 128, 256, dtype=torch.bfloat16, device=DEV))
    with pytest.raises(ValueError):  # w13 must be [E, 2I, H] = [4, 256, 256]
        m.MoELayer(256, 4, 2, 128, 0, torch.zeros(4, 128, 256, dtype=torch.bfloat16, device=DEV),
                   torch.zeros(4, 256, 128, dtype=torch.bfloat16, device=DEV))
    _sync()
