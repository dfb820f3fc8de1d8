"""Stage parity of the CUDA path against the oracle, through the C ABI.

Bit-exact: routing ids, counts / offsets / permutation, permuted rows, NVFP4
codes, scales and global scales.  Tolerances: routing weights 1e-6 relative;
GEMM / combine outputs by relative Frobenius error (bf16 output rounding is
2^-9 relative per element)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import nvfp4
from tests.helpers import F32, require_gpu, to_np_f32

pytestmark = pytest.mark.gpu

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


# ------------------------------------------------------------------ waits ----
def test_bounded_wait_times_out_and_context_survives():
    m = api()
    m.moe_selftest_wait_timeout(2_000_000)  # 2 ms
    assert m.moe_sync_status() == 5          # MOE_ERR_TIMEOUT
    assert m.moe_sync_status() == 0          # cleared
    # the context is still usable
    idx, w = m.moe_route(torch.randn(4, 8, device=DEV), 2)
    _sync()
    assert idx.shape == (4, 2)


def test_grid_barrier_times_out_and_context_survives():
    """The fused dispatch's grid barrier: a wait for an arrival that never
    comes gives up after its limit, records MOE_ERR_TIMEOUT, and the kernel
    returns; the context stays usable."""
    m = api()
    m.moe_selftest_grid_barrier_timeout(2_000_000)  # 2 ms
    assert m.moe_sync_status() == 5                 # MOE_ERR_TIMEOUT
    assert m.moe_sync_status() == 0
    r = m.moe_route_permute(torch.randn(16, 8, device=DEV), 2)
    _sync()
    assert int(r["offsets"][-1]) == 32


# ------------------------------------------------------------------ route ----
def _check_route(logits: torch.Tensor, k: int):
    idx, w = api().moe_route(logits.to(DEV).contiguous(), k)
    _sync()
    ridx, rw = oracle.route(logits.numpy(), k)
    gi = idx.cpu().numpy()
    assert np.array_equal(gi, ridx), np.argwhere(gi != ridx)[:5]
    np.testing.assert_allclose(w.cpu().numpy().astype(np.float64), rw, rtol=1e-6, atol=0)


@pytest.mark.parametrize("name", ["tiny", "qwen3-235b", "qwen35-397b", "deepseek-v3"])
def test_route_configs(name):
    cfg = synth.CONFIGS[name]
    for T in cfg.Ts:
        acts = synth.make_activations(cfg, T, seed=0)
        _check_route(acts.logits, cfg.k)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (5, 8, 8), (300, 33, 5), (77, 1024, 32), (1000, 256, 8),
                                   (65536, 256, 8)])
def test_route_shapes(T, E, k):
    g = torch.Generator().manual_seed(T + E)
    logits = torch.randn(T, E, generator=g)
    _check_route(logits, k)


def test_route_ties_lower_index_first():
    g = torch.Generator().manual_seed(3)
    logits = torch.round(torch.randn(513, 64, generator=g) * 2) / 2  # many exact ties
    logits[0] = 0.0
    logits[1, ::2] = -0.0
    _check_route(logits, 8)


def test_route_zero_tokens_is_noop():
    m = api()
    idx = torch.full((0, 2), -1, dtype=torch.int32, device=DEV)
    out = m.moe_route(torch.empty(0, 8, device=DEV), 2, idx=idx)
    _sync()
    assert out[0].numel() == 0


# ---------------------------------------------------------------- permute ----
def _zipf_idx(T, E, k, s, seed):
    g = torch.Generator().manual_seed(seed)
    rank = torch.randperm(E, generator=g).double() + 1
    logits = (torch.randn(T, E, generator=g, dtype=torch.float64) - s * torch.log(rank)).float()
    return oracle.route(logits.numpy(), k)[0]


@pytest.mark.parametrize("T,E,k,s", [(1, 8, 2, 1.1), (64, 8, 2, 1.1), (256, 128, 8, 1.1), (1000, 512, 10, 2.0),
                                     (8192, 128, 8, 1.1), (16384, 256, 8, 2.0), (65536, 256, 8, 0.0)])
def test_permute_bit_exact(T, E, k, s):
    idx = _zipf_idx(T, E, k, s, seed=T)
    H = 64
    g = torch.Generator().manual_seed(1)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    r = api().moe_permute(torch.from_numpy(idx).to(DEV), E, x.to(DEV))
    _sync()
    p = oracle.permute(idx, E)
    assert np.array_equal(r["counts"].cpu().numpy(), p.counts)
    assert np.array_equal(r["offsets"].cpu().numpy(), p.offsets)
    assert np.array_equal(r["row_of"].cpu().numpy(), p.row_of)
    assert np.array_equal(r["src_tok"].cpu().numpy(), p.src_tok)
    xp = r["xp"].cpu()
    ref = x[torch.from_numpy(p.src_tok).long()]
    assert torch.equal(xp.view(torch.int16), ref.view(torch.int16))
    if s == 2.0:
        assert (p.counts == 0).any()  # hot experts leave others empty


def test_permute_nvfp4_rows_and_scales():
    T, E, k, H = 3000, 64, 4, 512
    idx = _zipf_idx(T, E, k, 1.1, seed=5)
    g = torch.Generator().manual_seed(2)
    rows = torch.randint(0, 256, (T, H // 2), generator=g, dtype=torch.uint8)
    sf = torch.randint(0, 256, (T, H // 16), generator=g, dtype=torch.uint8)
    r = api().moe_permute(torch.from_numpy(idx).to(DEV), E, rows.to(DEV), sf.to(DEV))
    _sync()
    p = oracle.permute(idx, E)
    src = torch.from_numpy(p.src_tok).long()
    assert torch.equal(r["xp"].cpu(), rows[src])
    assert torch.equal(r["xp_sf"].cpu(), sf[src])


def test_permute_zero_tokens():
    r = api().moe_permute(torch.empty(0, 4, dtype=torch.int32, device=DEV), 16)
    _sync()
    assert r["counts"].cpu().tolist() == [0] * 16 and r["offsets"].cpu().tolist() == [0] * 17


# ---------------------------------------------------------- fused dispatch ----
@pytest.mark.parametrize("name,T", [("tiny", 64), ("qwen3-235b", 256), ("qwen3-235b", 16), ("qwen35-397b", 64),
                                    ("qwen35-397b", 512), ("deepseek-v3", 256), ("deepseek-v3", 16384),
                                    ("qwen3-235b", 8192), ("tiny", 1), ("tiny", 153)])
def test_route_permute_matches_oracle_and_split_calls(name, T):
    """moe_route_permute (route + permutation in one cooperative launch) at
    the workloads' decode and prefill sizes: idx bit-exact and w within 1e-6
    of the oracle's router; counts, offsets, row_of, src_tok and the
    permuted rows bit-exact with the oracle's permutation; every output
    bit-exact with moe_route followed by moe_permute."""
    m = api()
    cfg = synth.CONFIGS[name]
    acts = synth.make_activations(cfg, T, seed=T)
    lg = acts.logits.to(DEV)
    x = acts.x.to(DEV)
    r = m.moe_route_permute(lg, cfg.k, x)
    _sync()
    ridx, rw = oracle.route(acts.logits.numpy(), cfg.k)
    assert np.array_equal(r["idx"].cpu().numpy(), ridx)
    np.testing.assert_allclose(r["w"].cpu().numpy().astype(np.float64), rw, rtol=1e-6, atol=0)
    p = oracle.permute(ridx, cfg.E)
    for key, ref in (("counts", p.counts), ("offsets", p.offsets), ("row_of", p.row_of), ("src_tok", p.src_tok)):
        assert np.array_equal(r[key].cpu().numpy(), ref), key
    assert torch.equal(r["xp"].cpu().view(torch.int16), acts.x[torch.from_numpy(p.src_tok).long()].view(torch.int16))
    idx, w = m.moe_route(lg, cfg.k)
    q = m.moe_permute(idx, cfg.E, x)
    _sync()
    assert torch.equal(r["idx"], idx) and torch.equal(r["w"], w)
    for key in ("counts", "offsets", "row_of", "src_tok", "xp"):
        assert torch.equal(r[key], q[key]), key


def test_route_permute_nvfp4_rows_scales_and_variants():
    """Packed rows with scale bytes, the router without renormalisation, hot
    experts that leave others empty, E = 1024 (the router's limit) with few
    and with many slots per block (placement by one warp, and split over a
    block's warps), and blocks of more than 4096 slots (k = 32: placement in
    several staged pieces)."""
    m = api()
    for T, E, k, renorm in ((3000, 64, 4, True), (700, 1024, 8, False), (5, 16, 16, True), (8192, 1024, 8, True),
                            (20000, 64, 32, True)):
        g = torch.Generator().manual_seed(T)
        rank = torch.randperm(E, generator=g).double() + 1
        logits = (torch.randn(T, E, generator=g, dtype=torch.float64) - 2.0 * torch.log(rank)).float()
        rows = torch.randint(0, 256, (T, 256), generator=g, dtype=torch.uint8)
        sf = torch.randint(0, 256, (T, 32), generator=g, dtype=torch.uint8)
        r = m.moe_route_permute(logits.to(DEV), k, rows.to(DEV), sf.to(DEV), renorm=renorm)
        _sync()
        ridx, rw = oracle.route(logits.numpy(), k, renorm=renorm)
        assert np.array_equal(r["idx"].cpu().numpy(), ridx)
        np.testing.assert_allclose(r["w"].cpu().numpy().astype(np.float64), rw, rtol=1e-6, atol=0)
        p = oracle.permute(ridx, E)
        assert np.array_equal(r["offsets"].cpu().numpy(), p.offsets)
        assert np.array_equal(r["row_of"].cpu().numpy(), p.row_of)
        src = torch.from_numpy(p.src_tok).long()
        assert torch.equal(r["xp"].cpu(), rows[src]) and torch.equal(r["xp_sf"].cpu(), sf[src])
        if (T, E) == (3000, 64):  # hot experts leave others empty
            assert (p.counts == 0).any()


def test_route_permute_ties_and_signed_zero():
    """Exact ties (lower expert id first) and -0.0 next to +0.0 through the
    fused dispatch, with enough tokens per block to split the placement."""
    m = api()
    g = torch.Generator().manual_seed(3)
    logits = torch.round(torch.randn(40000, 64, generator=g) * 2) / 2  # many exact ties
    logits[0] = 0.0
    logits[1, ::2] = -0.0
    r = m.moe_route_permute(logits.to(DEV), 8)
    _sync()
    ridx, rw = oracle.route(logits.numpy(), 8)
    assert np.array_equal(r["idx"].cpu().numpy(), ridx)
    np.testing.assert_allclose(r["w"].cpu().numpy().astype(np.float64), rw, rtol=1e-6, atol=0)
    p = oracle.permute(ridx, 64)
    for key, ref in (("counts", p.counts), ("offsets", p.offsets), ("row_of", p.row_of), ("src_tok", p.src_tok)):
        assert np.array_equal(r[key].cpu().numpy(), ref), key


# ----------------------------------------------------------------- quant ----
def _check_quant(x_bf16: torch.Tensor, g_in=None):
    codes, sf, g = api().moe_quant_nvfp4(x_bf16.to(DEV).contiguous(),
                                         None if g_in is None else g_in.to(DEV))
    _sync()
    x3 = x_bf16 if x_bf16.dim() == 3 else x_bf16.unsqueeze(0)
    c3 = codes.cpu().reshape(x3.shape[0], x3.shape[1], -1).numpy()
    s3 = sf.cpu().reshape(x3.shape[0], x3.shape[1], -1).numpy()
    for grp in range(x3.shape[0]):
        a = to_np_f32(x3[grp])
        rq, rs, rg = nvfp4.quantize(a, None if g_in is None else F32(g_in[grp].item()))
        assert g.cpu().numpy()[grp] == rg, (grp, g.cpu().numpy()[grp], rg)
        assert np.array_equal(s3[grp], rs), np.argwhere(s3[grp] != rs)[:5]
        assert np.array_equal(c3[grp], rq), np.argwhere(c3[grp] != rq)[:5]


@pytest.mark.parametrize("T", [1, 256, 16384])
def test_quant_activations_deepseek(T):
    acts = synth.make_activations(synth.DEEPSEEK_V3, T, seed=0)  # N(0,1) with 0.1% outliers x20
    _check_quant(acts.x)


def test_quant_weight_groups():
    g = torch.Generator().manual_seed(9)
    w = (torch.randn(6, 256, 512, generator=g) * 0.02).to(torch.bfloat16)
    w[2] *= 1e-6       # tiny group: scales in the E4M3 subnormals
    w[3] = 0           # all-zero group: g = 1, every code 0
    w[4, 7, :16] = 0   # a zero block inside a normal group
    _check_quant(w)


def test_quant_given_global_scale_and_saturation():
    g = torch.Generator().manual_seed(10)
    x = torch.randn(64, 256, generator=g).to(torch.bfloat16)
    x[5, 3] = 3000.0
    _check_quant(x, g_in=torch.tensor([0.01], dtype=torch.float32))  # blocks beyond 6*448*g saturate


def test_quant_hand_worked_blocks(golden_dir):
    import json, os
    with open(os.path.join(golden_dir, "nvfp4_blocks.json")) as f:
        spec = json.load(f)
    for b in spec["blocks"]:
        x = torch.tensor([b["x"]], dtype=torch.float32)
        xb = x.to(torch.bfloat16)
        if not torch.equal(xb.float(), x):
            continue  # the GPU quantiser takes bf16 input; keep blocks exact in bf16
        g_in = None if b["g"] is None else torch.tensor([b["g"]], dtype=torch.float32)
        codes, sf, g = api().moe_quant_nvfp4(xb.to(DEV), None if g_in is None else g_in.to(DEV))
        _sync()
        assert sf.item() == int(b["scale"], 16), b["name"]
        got = nvfp4.unpack_codes(codes.cpu().numpy())[0].tolist()
        assert got == b["codes"], (b["name"], got)


# --------------------------------------------------------------- combine ----
@pytest.mark.parametrize("T,k,H,shared", [(1, 2, 256, False), (333, 8, 4096, False), (64, 10, 4096, True),
                                          (2048, 8, 7168, True)])
def test_combine(T, k, H, shared):
    E = 4 * k
    idx = _zipf_idx(T, E, k, 1.1, seed=T + k)
    p = oracle.permute(idx, E)
    g = torch.Generator().manual_seed(11)
    logits = torch.randn(T, E, generator=g)
    _, w = oracle.route(logits.numpy(), k)
    Y = torch.randn(T * k, H, generator=g).to(torch.bfloat16)
    Ys = torch.randn(T, H, generator=g).to(torch.bfloat16) if shared else None
    wt = torch.from_numpy(w.astype(np.float32))
    out = api().moe_combine(Y.to(DEV), torch.from_numpy(p.row_of).to(DEV), wt.to(DEV),
                            None if Ys is None else Ys.to(DEV), T, k, H)
    _sync()
    Yd = Y.double().numpy()
    ref = np.einsum("tj,tjh->th", wt.double().numpy(), Yd[p.row_of])
    if shared:
        ref += Ys.double().numpy()
    err = oracle.rel_frobenius(out.float().cpu().numpy(), ref)
    assert err < 3e-3, err


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (300, 33, 5), (77, 1024, 32), (500, 512, 10), (64, 4, 4)])
def test_route_without_renorm(T, E, k):
    """moe_route_ex(renorm=0): the same experts as the oracle (bit-exact), and
    weights = the full softmax over E at the picks within 1e-6."""
    g = torch.Generator().manual_seed(T + E + k)
    logits = torch.randn(T, E, generator=g) * 2
    idx, w = api().moe_route(logits.to(DEV), k, renorm=False)
    _sync()
    ridx, rw = oracle.route(logits.numpy(), k, renorm=False)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=1e-5, atol=1e-7)


@pytest.mark.parametrize("T,H", [(1, 8), (300, 4096), (77, 7168)])
def test_shared_gate(T, H):
    """moe_shared_gate: sigmoid(x . g) per token in fp32 against the oracle."""
    g0 = torch.Generator().manual_seed(T + H)
    x = torch.randn(T, H, generator=g0).to(torch.bfloat16)
    gv = (torch.randn(H, generator=g0) * 0.03).to(torch.bfloat16)
    gate = api().moe_shared_gate(x.to(DEV), gv.to(DEV))
    _sync()
    ref = oracle.shared_gate(x.double().numpy(), gv.double().numpy())
    np.testing.assert_allclose(gate.cpu().numpy(), ref, rtol=0, atol=2e-6)


def test_combine_gated():
    """moe_combine_gated: the shared row scaled by a per-token gate."""
    T, k, H = 200, 8, 1024
    E = 4 * k
    idx = _zipf_idx(T, E, k, 1.1, seed=3)
    p = oracle.permute(idx, E)
    g = torch.Generator().manual_seed(13)
    _, w = oracle.route(torch.randn(T, E, generator=g).numpy(), k)
    Y = torch.randn(T * k, H, generator=g).to(torch.bfloat16)
    Ys = torch.randn(T, H, generator=g).to(torch.bfloat16)
    gate = torch.rand(T, generator=g)
    wt = torch.from_numpy(w.astype(np.float32))
    out = api().moe_combine(Y.to(DEV), torch.from_numpy(p.row_of).to(DEV), wt.to(DEV), Ys.to(DEV), T, k, H,
                            ys_gate=gate.to(DEV))
    _sync()
    ref = np.einsum("tj,tjh->th", wt.double().numpy(), Y.double().numpy()[p.row_of])
    ref += gate.double().numpy()[:, None] * Ys.double().numpy()
    assert oracle.rel_frobenius(out.float().cpu().numpy(), ref) < 3e-3


# ---------------------------------------------------------- grouped GEMM ----
def _ragged_offsets(counts):
    return torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32)


def _gemm_ref(A, W, offs, swiglu, N):
    out = np.zeros((A.shape[0], N))
    for g in range(len(offs) - 1):
        lo, hi = offs[g], offs[g + 1]
        if hi == lo:
            continue
        y = A[lo:hi] @ W[g].T
        out[lo:hi] = oracle.silu(y[:, :N]) * y[:, N:] if swiglu else y
    return out


@pytest.mark.parametrize("epi,N,K", [(0, 384, 256), (1, 192, 320), (0, 256, 1536), (1, 1536, 512)])
def test_grouped_gemm_bf16(epi, N, K):
    m = api()
    counts = [0, 1, 127, 129, 300, 0, 40]
    offs = _ragged_offsets(counts)
    M = int(offs[-1])
    G = len(counts)
    Wn = N if epi == 0 else 2 * N
    g = torch.Generator().manual_seed(N + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W = (torch.randn(G, Wn, K, generator=g) * 0.05).to(torch.bfloat16)
    C = m.moe_grouped_gemm(0, 0, epi, offs.to(DEV), N, K, A.to(DEV), W.to(DEV))
    _sync()
    ref = _gemm_ref(A.double().numpy(), W.double().numpy(), offs.numpy(), epi == 1, N)
    err = oracle.rel_frobenius(C.float().cpu().numpy(), ref)
    assert err < 5e-3, err


@pytest.mark.parametrize("epi", [0, 1])
def test_grouped_gemm_bf16_token_blocks(epi):
    """Groups that span several 256-token blocks, cut into equal blocks of a
    multiple of 16 tokens (256, 257, 513, 1000 rows), next to tiny ones."""
    m = api()
    counts = [256, 257, 16, 513, 17, 1000, 2]
    offs = _ragged_offsets(counts)
    M, G, N, K = int(offs[-1]), len(counts), 256, 448
    Wn = N if epi == 0 else 2 * N
    g = torch.Generator().manual_seed(77 + epi)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W = (torch.randn(G, Wn, K, generator=g) * 0.05).to(torch.bfloat16)
    C = m.moe_grouped_gemm(0, 0, epi, offs.to(DEV), N, K, A.to(DEV), W.to(DEV))
    _sync()
    ref = _gemm_ref(A.double().numpy(), W.double().numpy(), offs.numpy(), epi == 1, N)
    err = oracle.rel_frobenius(C.float().cpu().numpy(), ref)
    assert err < 5e-3, err
    # every row is written: no row of C keeps the allocation's contents
    row_err = np.abs(C.float().cpu().numpy() - ref).max(axis=1) / (np.abs(ref).max() + 1e-30)
    assert row_err.max() < 2e-2, int(row_err.argmax())


W4A16_COUNTS = {
    "few": [1, 2, 0, 20, 3, 2, 1, 0, 5, 1],        # <= 4 rows per group on average: 16-token tiles
    "mid": [3, 40, 0, 70, 9, 17, 1, 30],           # 5..48 rows per group: 64-token tiles
    "many": [3, 200, 0, 64, 129, 17],              # > 48 rows per group: 128-token tiles
    "huge": [300, 0, 129, 250, 64],                # 128-token tiles, groups of two and three blocks
}


@pytest.mark.parametrize("epi,N,K,rows", [(1, 256, 512, "many"), (0, 384, 768, "many"), (1, 192, 320, "many"),
                                          (0, 128, 576, "many"), (1, 256, 1024, "few"), (0, 512, 256, "few"),
                                          (1, 384, 512, "mid"), (0, 256, 768, "mid"),
                                          (1, 256, 512, "huge"), (0, 384, 768, "huge")])
def test_grouped_gemm_nvfp4_weights(epi, N, K, rows):
    """bf16 A x NVFP4 W (codes + E4M3 scales + per-group fp32 scale): K a
    multiple of 256 (weights expanded into tensor memory, fp16 MMA, in each
    of the three token-tile shapes, chosen by the rows per group) and not
    (converter kernel, bf16 MMA); ragged groups past a tile and empty ones."""
    m = api()
    counts = W4A16_COUNTS[rows]
    offs = _ragged_offsets(counts)
    M, G = int(offs[-1]), len(counts)
    Wn = 2 * N if epi == 1 else N
    g = torch.Generator().manual_seed(21 + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    Wb = (torch.randn(G, Wn, K, generator=g) * 0.02).to(torch.bfloat16)
    Wq = [nvfp4.quantize(to_np_f32(Wb[i])) for i in range(G)]  # oracle's encoding of the weights
    codes = torch.from_numpy(np.stack([q for q, _, _ in Wq]))
    sf = torch.from_numpy(np.stack([s for _, s, _ in Wq]))
    gw = torch.tensor([gg for _, _, gg in Wq], dtype=torch.float32)
    C = m.moe_grouped_gemm(0, 1, epi, offs.to(DEV), N, K, A.to(DEV), codes.to(DEV), W_sf=sf.to(DEV),
                           W_g=gw.to(DEV))
    _sync()
    Wd = np.stack([nvfp4.dequantize(q, s, gg) for q, s, gg in Wq])
    ref = _gemm_ref(A.double().numpy(), Wd, offs.numpy(), epi == 1, N)
    err = oracle.rel_frobenius(C.float().cpu().numpy(), ref)
    assert err < 5e-3, err


@pytest.mark.parametrize("epi,N,K", [(0, 384, 320), (1, 192, 576), (0, 256, 1024), (1, 128, 256)])
def test_grouped_gemm_nvfp4_both_block_scaled(epi, N, K):
    """NVFP4 A x NVFP4 W on the block-scaled FP4 MMA, bf16 outputs; K tails
    that are not multiples of the 256-element stage; ragged and empty groups."""
    m = api()
    counts = [0, 1, 127, 129, 300, 0, 40]
    offs = _ragged_offsets(counts)
    M, G = int(offs[-1]), len(counts)
    Wn = N if epi == 0 else 2 * N
    g = torch.Generator().manual_seed(N + K + epi)
    Aq, As, Ag = nvfp4.quantize(torch.randn(M, K, generator=g).numpy())
    Wq = [nvfp4.quantize((torch.randn(Wn, K, generator=g) * 0.02).numpy()) for _ in range(G)]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    C = m.moe_grouped_gemm(1, 1, epi, offs.to(DEV), N, K, t(Aq), t(np.stack([q for q, _, _ in Wq])), A_sf=t(As),
                           A_g=torch.tensor([Ag], device=DEV), W_sf=t(np.stack([s for _, s, _ in Wq])),
                           W_g=torch.tensor([gg for _, _, gg in Wq], dtype=torch.float32, device=DEV))
    _sync()
    Ad = nvfp4.dequantize(Aq, As, Ag)
    Wd = np.stack([nvfp4.dequantize(q, s, gg) for q, s, gg in Wq])
    ref = _gemm_ref(Ad, Wd, offs.numpy(), epi == 1, N)
    err = oracle.rel_frobenius(C.float().cpu().numpy(), ref)
    assert err < 5e-3, err


@pytest.mark.parametrize("epi,N,K", [(0, 448, 512), (1, 256, 768), (0, 192, 256), (1, 192, 1280)])
def test_grouped_gemm_nvfp4_both_large_groups(epi, N, K):
    """NVFP4 A x NVFP4 W with prefill-sized groups (>= 192 rows per group on
    average): groups past one and two 256-row blocks, a ragged last weight
    tile (N = 448, SwiGLU N = 256), empty groups and a group of 64 rows."""
    m = api()
    counts = [300, 0, 513, 257, 64, 130]
    offs = _ragged_offsets(counts)
    M, G = int(offs[-1]), len(counts)
    assert M >= 192 * G
    Wn = N if epi == 0 else 2 * N
    g = torch.Generator().manual_seed(N + K + 3 * epi)
    Aq, As, Ag = nvfp4.quantize(torch.randn(M, K, generator=g).numpy())
    Wq = [nvfp4.quantize((torch.randn(Wn, K, generator=g) * 0.02).numpy()) for _ in range(G)]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    C = m.moe_grouped_gemm(1, 1, epi, offs.to(DEV), N, K, t(Aq), t(np.stack([q for q, _, _ in Wq])), A_sf=t(As),
                           A_g=torch.tensor([Ag], device=DEV), W_sf=t(np.stack([s for _, s, _ in Wq])),
                           W_g=torch.tensor([gg for _, _, gg in Wq], dtype=torch.float32, device=DEV))
    _sync()
    Ad = nvfp4.dequantize(Aq, As, Ag)
    Wd = np.stack([nvfp4.dequantize(q, s, gg) for q, s, gg in Wq])
    ref = _gemm_ref(Ad, Wd, offs.numpy(), epi == 1, N)
    got = C.float().cpu().numpy()
    err = oracle.rel_frobenius(got, ref)
    assert err < 5e-3, err
    # every row is written: no row keeps the allocation's contents
    row_err = np.abs(got - ref).max(axis=1) / (np.abs(ref).max() + 1e-30)
    assert row_err.max() < 2e-2, int(row_err.argmax())


def test_grouped_gemm_nvfp4_both_large_groups_nvfp4_output():
    """Prefill-sized groups with the SwiGLU output quantised to NVFP4 (N =
    352 features: a last 64-column weight tile that is half empty)."""
    m = api()
    counts = [260, 400, 0, 330]
    offs = _ragged_offsets(counts)
    M, G, N, K = int(offs[-1]), len(counts), 352, 512
    assert M >= 192 * G
    g = torch.Generator().manual_seed(23)
    Aq, As, Ag = nvfp4.quantize(torch.randn(M, K, generator=g).numpy())
    Wq = [nvfp4.quantize((torch.randn(2 * N, K, generator=g) * 0.02).numpy()) for _ in range(G)]
    gh = F32(8.0 / 2688)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    C, C_sf = m.moe_grouped_gemm(
        1, 1, 2, offs.to(DEV), N, K, t(Aq), t(np.stack([q for q, _, _ in Wq])), A_sf=t(As),
        A_g=torch.tensor([Ag], device=DEV), W_sf=t(np.stack([s for _, s, _ in Wq])),
        W_g=torch.tensor([gg for _, _, gg in Wq], dtype=torch.float32, device=DEV),
        c_g=torch.tensor([gh], device=DEV))
    _sync()
    Ad = nvfp4.dequantize(Aq, As, Ag)
    Wd = np.stack([nvfp4.dequantize(q, s, gg) for q, s, gg in Wq])
    h = _gemm_ref(Ad, Wd, offs.numpy(), True, N)
    rq, rs, _ = nvfp4.quantize(h.astype(F32), gh)
    got_q, got_s = C.cpu().numpy(), C_sf.cpu().numpy()
    assert np.mean(got_s != rs) < 1e-3
    assert np.mean(nvfp4.unpack_codes(got_q) != nvfp4.unpack_codes(rq)) < 2e-3
    err = oracle.rel_frobenius(nvfp4.dequantize(got_q, got_s, gh), nvfp4.dequantize(rq, rs, gh))
    assert err < 1e-2, err


def test_grouped_gemm_nvfp4_both_with_nvfp4_output():
    """NVFP4 A x NVFP4 W, SwiGLU output quantised to NVFP4 with a given scale."""
    m = api()
    counts = [130, 0, 7, 260]
    offs = _ragged_offsets(counts)
    M, G, N, K = int(offs[-1]), len(counts), 256, 768
    g = torch.Generator().manual_seed(22)
    A = torch.randn(M, K, generator=g)
    Aq, As, Ag = nvfp4.quantize(A.numpy())
    Wb = (torch.randn(G, 2 * N, K, generator=g) * 0.02)
    Wq = [nvfp4.quantize(Wb[i].numpy()) for i in range(G)]
    gh = F32(8.0 / 2688)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    C, C_sf = m.moe_grouped_gemm(
        1, 1, 2, offs.to(DEV), N, K, t(Aq), t(np.stack([q for q, _, _ in Wq])), A_sf=t(As),
        A_g=torch.tensor([Ag], device=DEV), W_sf=t(np.stack([s for _, s, _ in Wq])),
        W_g=torch.tensor([gg for _, _, gg in Wq], dtype=torch.float32, device=DEV),
        c_g=torch.tensor([gh], device=DEV))
    _sync()
    Ad = nvfp4.dequantize(Aq, As, Ag)
    Wd = np.stack([nvfp4.dequantize(q, s, gg) for q, s, gg in Wq])
    h = _gemm_ref(Ad, Wd, offs.numpy(), True, N)
    rq, rs, _ = nvfp4.quantize(h.astype(F32), gh)
    got_q, got_s = C.cpu().numpy(), C_sf.cpu().numpy()
    # codes come from fp32 values that differ in the last bits between the
    # tensor-core sums and the fp64 oracle: almost every code and scale agree
    assert np.mean(got_s != rs) < 1e-3
    assert np.mean(nvfp4.unpack_codes(got_q) != nvfp4.unpack_codes(rq)) < 2e-3
    err = oracle.rel_frobenius(nvfp4.dequantize(got_q, got_s, gh), nvfp4.dequantize(rq, rs, gh))
    assert err < 1e-2, err


@pytest.mark.parametrize("epi", [0, 1, 2])
def test_grouped_gemm_nvfp4_both_many_row_blocks(epi):
    """NVFP4 x NVFP4 with groups that span several row tiles (161, 320, 321,
    1000 rows), tiles far from full (1, 17, 31, 33 rows), 159/160-row groups
    and an empty one; every epilogue, weight tiles past N (N = 448 STORE,
    320 features SwiGLU), K = 1536."""
    m = api()
    counts = [161, 320, 1, 17, 0, 321, 31, 1000, 33, 159, 160]
    offs = _ragged_offsets(counts)
    M, G, K = int(offs[-1]), len(counts), 1536
    N = 448 if epi == 0 else 320
    Wn = N if epi == 0 else 2 * N
    g = torch.Generator().manual_seed(40 + epi)
    Aq, As, Ag = nvfp4.quantize(torch.randn(M, K, generator=g).numpy())
    Wq = [nvfp4.quantize((torch.randn(Wn, K, generator=g) * 0.02).numpy()) for _ in range(G)]
    gh = F32(8.0 / 2688)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    out = m.moe_grouped_gemm(1, 1, epi, offs.to(DEV), N, K, t(Aq), t(np.stack([q for q, _, _ in Wq])), A_sf=t(As),
                             A_g=torch.tensor([Ag], device=DEV), W_sf=t(np.stack([s for _, s, _ in Wq])),
                             W_g=torch.tensor([gg for _, _, gg in Wq], dtype=torch.float32, device=DEV),
                             c_g=torch.tensor([gh], device=DEV) if epi == 2 else None)
    _sync()
    Ad = nvfp4.dequantize(Aq, As, Ag)
    Wd = np.stack([nvfp4.dequantize(q, s, gg) for q, s, gg in Wq])
    ref = _gemm_ref(Ad, Wd, offs.numpy(), epi != 0, N)
    if epi == 2:
        C, C_sf = out
        rq, rs, _ = nvfp4.quantize(ref.astype(F32), gh)
        got_q, got_s = C.cpu().numpy(), C_sf.cpu().numpy()
        assert np.mean(got_s != rs) < 1e-3
        assert np.mean(nvfp4.unpack_codes(got_q) != nvfp4.unpack_codes(rq)) < 2e-3
        got = nvfp4.dequantize(got_q, got_s, gh)
        ref = nvfp4.dequantize(rq, rs, gh)
        tol = 1e-2
    else:
        got = out.float().cpu().numpy()
        tol = 5e-3
    err = oracle.rel_frobenius(got, ref)
    assert err < tol, err
    # every row is written: no row keeps the allocation's contents
    row_err = np.abs(got - ref).max(axis=1) / (np.abs(ref).max() + 1e-30)
    assert row_err.max() < 5e-2, int(row_err.argmax())
