"""Pins of the oracle's route / permute / expert / layer functions against
brute force, invariants, closed forms and library routines (torch fp64)."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import ExpertWeights, forward, gather_rows, nvfp4, permute, rel_frobenius, route, unpermute
from oracle.moe import expert_mlp

F32 = np.float32


# ---------------------------------------------------------------- route ----
def _route_brute(logits, k):
    """Python sorted() over (value desc, index asc), weights by full softmax
    over E renormalised over the selected experts (math.exp)."""
    idx, w = [], []
    for row in logits.tolist():
        order = sorted(range(len(row)), key=lambda e: (-row[e], e))[:k]
        m = max(row)
        full = [math.exp(v - m) for v in row]
        z = sum(full)
        p = [full[e] / z for e in order]
        s = sum(p)
        idx.append(order)
        w.append([v / s for v in p])
    return np.array(idx, np.int32), np.array(w)


@pytest.mark.parametrize("T,E,k", [(7, 8, 2), (5, 16, 5), (9, 33, 10), (4, 6, 6), (3, 1, 1)])
def test_route_matches_brute_force(T, E, k):
    rng = np.random.default_rng(T * 100 + E)
    logits = (rng.standard_normal((T, E)) * 2).astype(F32)
    idx, w = route(logits, k)
    bi, bw = _route_brute(logits, k)
    assert np.array_equal(idx, bi)
    np.testing.assert_allclose(w, bw, rtol=1e-12, atol=0)


def test_route_weights_sum_to_one():
    rng = np.random.default_rng(5)
    logits = (rng.standard_normal((200, 64)) * 3).astype(F32)
    _, w = route(logits, 8)
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-12)
    assert np.all(np.diff(w, axis=1) <= 0)  # descending with the logits


def test_route_ties_go_to_lower_index():
    logits = np.array([[1.0, 3.0, 3.0, 0.5, 3.0, -0.0, 0.0]], F32)
    idx, w = route(logits, 4)
    assert idx.tolist() == [[1, 2, 4, 0]]
    np.testing.assert_allclose(w[0, :3], w[0, 0])
    idx, _ = route(np.array([[0.0, -0.0, 0.0]], F32), 3)
    assert idx.tolist() == [[0, 1, 2]]


def test_route_k_equals_E_and_single_expert():
    rng = np.random.default_rng(6)
    logits = rng.standard_normal((3, 8)).astype(F32)
    idx, w = route(logits, 8)
    for t in range(3):
        assert sorted(idx[t].tolist()) == list(range(8))
        full = np.exp(logits[t].astype(np.float64) - logits[t].max())
        np.testing.assert_allclose(w[t], (full / full.sum())[idx[t]], rtol=1e-12)
    idx, w = route(np.array([[0.3], [-2.0]], F32), 1)
    assert idx.tolist() == [[0], [0]] and np.all(w == 1.0)


# -------------------------------------------------------------- permute ----
def _permute_brute(idx, E):
    T, k = idx.shape
    rows = []
    for e in range(E):
        for t in range(T):
            for j in range(k):
                if idx[t, j] == e:
                    rows.append((t, j))
    row_of = np.zeros((T, k), np.int32)
    for r, (t, j) in enumerate(rows):
        row_of[t, j] = r
    counts = np.array([sum(1 for t in range(T) for j in range(k) if idx[t, j] == e) for e in range(E)])
    return counts, row_of, np.array([t for t, _ in rows], np.int32)


def _random_idx(rng, T, E, k):
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k", [(1, 4, 2), (13, 8, 2), (40, 16, 4), (9, 10, 10)])
def test_permute_matches_brute_force(T, E, k):
    rng = np.random.default_rng(T + E)
    idx = _random_idx(rng, T, E, k)
    p = permute(idx, E)
    c, ro, st = _permute_brute(idx, E)
    assert np.array_equal(p.counts, c)
    assert np.array_equal(p.row_of, ro)
    assert np.array_equal(p.src_tok, st)


def test_permute_invariants_with_empty_experts():
    rng = np.random.default_rng(7)
    T, E, k = 300, 64, 4
    idx = np.stack([rng.choice(16, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    p = permute(idx, E)
    assert p.counts.sum() == T * k and p.offsets[-1] == T * k and p.offsets[0] == 0
    assert np.all(np.diff(p.offsets) == p.counts)
    assert np.all(p.counts[16:] == 0)
    for e in range(E):
        seg = p.src_tok[p.offsets[e]:p.offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)           # ascending token id
        assert all(e in idx[t] for t in seg)
    # every slot lands on a row holding its own token; rows are a bijection
    assert np.array_equal(np.sort(p.row_of.reshape(-1)), np.arange(T * k))
    assert np.all(p.src_tok[p.row_of] == np.arange(T)[:, None])


def test_unpermute_inverts_permute():
    rng = np.random.default_rng(8)
    T, E, k, H = 50, 12, 3, 5
    idx = _random_idx(rng, T, E, k)
    x = rng.standard_normal((T, H))
    p = permute(idx, E)
    xp = gather_rows(x, p)
    back = unpermute(xp, p)                     # [T, k, H]
    assert np.array_equal(back, np.repeat(x[:, None, :], k, axis=1))


def test_permute_empty():
    p = permute(np.zeros((0, 3), np.int32), 5)
    assert p.counts.tolist() == [0] * 5 and p.offsets.tolist() == [0] * 6 and p.src_tok.size == 0


# --------------------------------------------------------------- expert ----
def _rand_expert(rng, H, I, scale=0.1):
    return ExpertWeights(rng.standard_normal((2 * I, H)) * scale, rng.standard_normal((H, I)) * scale)


def test_expert_mlp_matches_torch_swiglu():
    """A SwiGLU MLP written with torch's silu and matmul (library routines)."""
    rng = np.random.default_rng(9)
    H, I, n = 48, 32, 11
    W = _rand_expert(rng, H, I)
    a = rng.standard_normal((n, H))
    got = expert_mlp(a, W.w13, W.w2)
    at, w13, w2 = (torch.from_numpy(v) for v in (a, W.w13, W.w2))
    ref = torch.nn.functional.linear(
        torch.nn.functional.silu(torch.nn.functional.linear(at, w13[:I])) *
        torch.nn.functional.linear(at, w13[I:]), w2)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_expert_mlp_brute_force_scalar():
    rng = np.random.default_rng(10)
    H, I = 6, 4
    W = _rand_expert(rng, H, I, 0.5)
    a = rng.standard_normal((2, H))
    got = expert_mlp(a, W.w13, W.w2)
    for r in range(2):
        h = []
        for i in range(I):
            g = sum(W.w13[i, c] * a[r, c] for c in range(H))
            u = sum(W.w13[I + i, c] * a[r, c] for c in range(H))
            h.append(g / (1 + math.exp(-g)) * u)
        y = [sum(W.w2[o, i] * h[i] for i in range(I)) for o in range(H)]
        np.testing.assert_allclose(got[r], y, rtol=1e-12, atol=1e-14)


def _h_probe(h_values):
    """Weights that make h = h_values exactly for the input row e_0: gate = 50
    (silu(50) == 50 in fp64), up_i = h_i / 50, down = identity."""
    I = len(h_values)
    H = I
    a = np.eye(H)[:1]
    w13 = np.zeros((2 * I, H))
    w13[:I, 0] = 50.0
    w13[I:, 0] = np.asarray(h_values, np.float64) / 50.0
    w2 = np.eye(H)[:, :I]
    return a, w13, w2


def test_expert_mlp_h_quant_is_identity_on_grid():
    """h exactly on the NVFP4 grid of g_h passes the h quantisation unchanged."""
    rng = np.random.default_rng(11)
    target = nvfp4.e2m1_decode(np.array([7] + list(rng.integers(0, 16, 15)), np.uint8))
    h = target.astype(np.float64) * 448.0          # block amax 2688 -> scale 448 for g = 1
    a, w13, w2 = _h_probe(h)
    np.testing.assert_allclose(expert_mlp(a, w13, w2, h_quant_g=F32(1.0))[0], h, rtol=1e-12)


def test_expert_mlp_h_quant_hand_worked():
    """g_h = 1, block amax 6 -> scale E4M3(1.0), so h is rounded to the E2M1
    grid itself: ties go to the even code (1.25 -> 1, 3.5 -> 4, 5 -> 4,
    0.25 -> 0, 2.5 -> 2), others to the nearest value."""
    h = [6.0, 1.25, 3.5, 5.0, 0.25, 2.5, -0.8, 1.6, -4.4, 0.3, 0.0, 2.9, -5.1, 0.7, 1.9, 3.2]
    want = [6.0, 1.0, 4.0, 4.0, 0.0, 2.0, -1.0, 1.5, -4.0, 0.5, 0.0, 3.0, -6.0, 0.5, 2.0, 3.0]
    a, w13, w2 = _h_probe(h)
    y = expert_mlp(a, w13, w2, h_quant_g=F32(1.0))[0]
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- layer ----
def _tiny_layer(rng, T, H, E, k, I, I_s):
    experts = [_rand_expert(rng, H, I) for _ in range(E)]
    shared = _rand_expert(rng, H, I_s) if I_s else None
    x = rng.standard_normal((T, H))
    logits = rng.standard_normal((T, E)).astype(F32)
    return experts, shared, x, logits


def test_top1_single_expert_is_dense_mlp():
    """E = 1, k = 1, no shared expert: the layer is a dense SwiGLU MLP
    (torch silu / linear)."""
    rng = np.random.default_rng(12)
    experts, _, x, logits = _tiny_layer(rng, 9, 24, 1, 1, 16, 0)
    out, idx, w, _ = forward(x, logits, 1, 1, lambda e: experts[e])
    W = experts[0]
    xt = torch.from_numpy(x)
    ref = torch.nn.functional.linear(
        torch.nn.functional.silu(torch.nn.functional.linear(xt, torch.from_numpy(W.w13[:16]))) *
        torch.nn.functional.linear(xt, torch.from_numpy(W.w13[16:])), torch.from_numpy(W.w2))
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_layer_matches_per_token_brute_force():
    rng = np.random.default_rng(13)
    T, H, E, k, I, I_s = 12, 16, 6, 3, 8, 8
    experts, shared, x, logits = _tiny_layer(rng, T, H, E, k, I, I_s)
    out, idx, w, _ = forward(x, logits, k, E, lambda e: experts[e], shared)
    for t in range(T):
        y = expert_mlp(x[t:t + 1], shared.w13, shared.w2)[0].copy()
        for j in range(k):
            W = experts[idx[t, j]]
            y += w[t, j] * expert_mlp(x[t:t + 1], W.w13, W.w2)[0]
        np.testing.assert_allclose(out[t], y, rtol=1e-12, atol=1e-13)


def test_identical_experts_make_routing_irrelevant():
    """All routed experts equal: out = E(x) + S(x) whatever the routing,
    because the renormalised weights sum to one."""
    rng = np.random.default_rng(14)
    T, H, E, k, I = 10, 16, 8, 3, 8
    W = _rand_expert(rng, H, I)
    S = _rand_expert(rng, H, I)
    x = rng.standard_normal((T, H))
    logits = rng.standard_normal((T, E)).astype(F32)
    out, *_ = forward(x, logits, k, E, lambda e: W, S)
    ref = expert_mlp(x, W.w13, W.w2) + expert_mlp(x, S.w13, S.w2)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_token_subsample_equals_full_rows():
    rng = np.random.default_rng(15)
    T, H, E, k, I, I_s = 40, 16, 8, 2, 8, 8
    experts, shared, x, logits = _tiny_layer(rng, T, H, E, k, I, I_s)
    full, *_ = forward(x, logits, k, E, lambda e: experts[e], shared)
    toks = [0, 3, 17, 39]
    sub, *_ = forward(x, logits, k, E, lambda e: experts[e], shared, tokens=toks)
    # equal up to the fp64 rounding of BLAS calls on different batch sizes
    np.testing.assert_allclose(sub, full[toks], rtol=1e-12, atol=1e-15)


def test_nvfp4_weights_on_grid_equal_bf16_path():
    """Weights drawn exactly on the NVFP4 grid: quantise -> dequantise returns
    them unchanged, so the NVFP4-weight layer equals the plain-weight layer."""
    rng = np.random.default_rng(16)
    T, H, E, k, I = 6, 32, 4, 2, 16

    def grid_matrix(rows, cols):
        g = F32(2.0 ** -10)
        s = nvfp4.E4M3_VALUES[rng.integers(48, 90, size=(rows, cols // 16))]
        s[0, 0] = 448.0  # matrix amax = 6 * 448 * g, so the derived g equals g
        q = rng.integers(0, 16, size=(rows, cols)).astype(np.uint8)
        q[:, ::16] = 7  # block max = 6 * s
        v = nvfp4.e2m1_decode(q).astype(np.float64) * np.repeat(s, 16, axis=1) * float(g)
        return v.astype(F32)

    experts = []
    for _ in range(E):
        w13, w2 = grid_matrix(2 * I, H), grid_matrix(H, I)
        experts.append((w13, w2))

    def deq(m):
        p, s, g = nvfp4.quantize(m)
        return nvfp4.dequantize(p, s, g)

    x = rng.standard_normal((T, H))
    logits = rng.standard_normal((T, E)).astype(F32)
    plain, *_ = forward(x, logits, k, E, lambda e: ExpertWeights(experts[e][0].astype(np.float64),
                                                                 experts[e][1].astype(np.float64)))
    quant, *_ = forward(x, logits, k, E, lambda e: ExpertWeights(deq(experts[e][0]), deq(experts[e][1])))
    np.testing.assert_array_equal(plain, quant)


def test_zero_expert_as_none_equals_explicit_zero_weights():
    """get_expert returning None (an expert whose weights are all zero) gives
    the same layer as passing that expert's zero weights explicitly, also on
    the NVFP4 h path: the NVFP4 and MX codecs take an all-zero matrix to
    exactly zero."""
    from oracle import mx
    rng = np.random.default_rng(21)
    T, H, E, k, I, I_s = 30, 32, 6, 2, 32, 32
    experts, shared, x, logits = _tiny_layer(rng, T, H, E, k, I, I_s)
    zero = {1, 4}
    z = ExpertWeights(np.zeros((2 * I, H)), np.zeros((H, I)))
    explicit, *_ = forward(x, logits, k, E, lambda e: z if e in zero else experts[e], shared,
                           h_quant_g=F32(0.01))
    skipped, *_ = forward(x, logits, k, E, lambda e: None if e in zero else experts[e], shared,
                          h_quant_g=F32(0.01))
    np.testing.assert_array_equal(explicit, skipped)
    # the zero experts were routed to, so the test skipped real work
    _, idx, *_ = forward(x, logits, k, E, lambda e: experts[e])
    assert zero & set(idx.reshape(-1).tolist())
    # all-zero weights quantise and decode to exact zeros in every format
    zm = np.zeros((2 * I, H), np.float32)
    p, sc, g = nvfp4.quantize(zm)
    assert not nvfp4.dequantize(p, sc, g).any()
    for fmt in ("mxfp8", "mxfp4"):
        assert not mx.fake_quant(zm, fmt).any()


def test_dropped_shared_or_weight_is_detected():
    """Plausible mistakes (shared expert dropped, weights not applied) move
    the output far beyond any tolerance used by the parity tests."""
    rng = np.random.default_rng(17)
    T, H, E, k, I, I_s = 16, 16, 8, 2, 8, 8
    experts, shared, x, logits = _tiny_layer(rng, T, H, E, k, I, I_s)
    out, idx, w, _ = forward(x, logits, k, E, lambda e: experts[e], shared)
    no_shared, *_ = forward(x, logits, k, E, lambda e: experts[e], None)
    assert rel_frobenius(no_shared, out) > 0.05
    unweighted = expert_mlp(x, shared.w13, shared.w2)
    for t in range(T):
        for j in range(k):
            W = experts[idx[t, j]]
            unweighted[t] += expert_mlp(x[t:t + 1], W.w13, W.w2)[0]
    assert rel_frobenius(unweighted, out) > 0.05


def test_synth_inputs_are_seeded_and_shaped():
    cfg = synth.TINY
    a1 = synth.make_activations(cfg, 64, seed=0)
    a2 = synth.make_activations(cfg, 64, seed=0)
    assert torch.equal(a1.x, a2.x) and torch.equal(a1.logits, a2.logits)
    assert a1.x.dtype == torch.bfloat16 and a1.x.shape == (64, 256)
    assert a1.logits.dtype == torch.float32 and a1.logits.shape == (64, 8)
    w = synth.make_weights(cfg, 0, "cpu")
    assert w.w13.shape == (8, 1024, 256) and w.w2.shape == (8, 256, 512) and w.ws13 is None
    assert abs(w.w13.float().std().item() - 0.02) < 1e-3


def test_deepseek_h_scale_rarely_saturates():
    """The static h scale of the NVFP4-activation workload (amax bound 128)
    leaves almost every block unsaturated on its synthetic inputs (small
    oracle sample with CPU-drawn weights of the same distribution)."""
    cfg = synth.DEEPSEEK_V3
    rng = np.random.default_rng(18)
    acts = synth.make_activations(cfg, 8, seed=3)
    x = acts.x.to(torch.float64).numpy()
    w13 = (rng.standard_normal((2 * cfg.I, cfg.H)) * 0.02).astype(F32).astype(np.float64)
    I = cfg.I
    h = (lambda g, u: g / (1 + np.exp(-g)) * u)(x @ w13[:I].T, x @ w13[I:].T)
    frac = np.mean(np.abs(h) > 6 * 448 * cfg.g_h)
    assert frac < 1e-4 and np.abs(h).max() > 1.0


# ------------------------------------------- router / shared-gate variants ----
@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (50, 128, 8), (20, 512, 10), (7, 5, 5)])
def test_route_without_renorm_is_full_softmax_at_the_picks(T, E, k):
    """renorm=False: the same experts, weights = the full softmax over E
    (torch's softmax in fp64, a library routine) taken at the picks."""
    rng = np.random.default_rng(T * E + k)
    logits = (rng.standard_normal((T, E)) * 3).astype(F32)
    idx, w = route(logits, k, renorm=False)
    idx_r, w_r = route(logits, k)
    assert np.array_equal(idx, idx_r)
    p = torch.softmax(torch.from_numpy(logits.astype(np.float64)), dim=1).numpy()
    np.testing.assert_allclose(w, np.take_along_axis(p, idx, axis=1), rtol=1e-13, atol=0)
    # the renormalised weights are these weights over their sum; the sum is
    # the probability mass of the picks (1 when k == E)
    s = w.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(w / s, w_r, rtol=1e-13)
    assert np.all(s <= 1 + 1e-12)
    if k == E:
        np.testing.assert_allclose(s, 1.0, rtol=1e-13)


def test_route_without_renorm_uniform_logits():
    """Equal logits: every pick weighs exactly 1/E (ties to the lower ids)."""
    T, E, k = 3, 16, 4
    idx, w = route(np.zeros((T, E), F32), k, renorm=False)
    assert np.array_equal(idx, np.tile(np.arange(k, dtype=np.int32), (T, 1)))
    np.testing.assert_allclose(w, 1.0 / E, rtol=1e-15)


def test_shared_gate_zero_vector_halves_the_shared_expert():
    """g = 0: sigma(0) = 1/2 exactly, so the gated layer is the routed part
    plus half the shared expert."""
    rng = np.random.default_rng(11)
    T, H, E, k, I, I_s = 6, 16, 4, 2, 8, 12
    experts, shared, x, logits = _tiny_layer(rng, T, H, E, k, I, I_s)
    get = lambda e: experts[e]
    full, *_ = forward(x, logits, k, E, get, shared)
    routed, *_ = forward(x, logits, k, E, get, None)
    gated, *_ = forward(x, logits, k, E, get, shared, shared_g=np.zeros(H))
    np.testing.assert_allclose(gated, routed + 0.5 * (full - routed), rtol=1e-13, atol=1e-15)


def test_shared_gate_brute_force_scalars():
    """Gate of every token by a scalar loop (dot product, then 1/(1+e^-z)),
    and the gated layer against the ungated one row by row."""
    rng = np.random.default_rng(12)
    T, H, E, k, I, I_s = 5, 8, 3, 1, 4, 6
    experts, shared, x, logits = _tiny_layer(rng, T, H, E, k, I, I_s)
    g = rng.standard_normal(H)
    get = lambda e: experts[e]
    full, *_ = forward(x, logits, k, E, get, shared)
    routed, *_ = forward(x, logits, k, E, get, None)
    gated, *_ = forward(x, logits, k, E, get, shared, shared_g=g)
    for t in range(T):
        z = 0.0
        for h in range(H):
            z += x[t, h] * g[h]
        gate = 1.0 / (1.0 + math.exp(-z))
        np.testing.assert_allclose(gated[t], routed[t] + gate * (full[t] - routed[t]), rtol=1e-12, atol=1e-14)
    # a very large positive / negative gate input passes / blocks the shared expert
    big, *_ = forward(x, logits, k, E, get, shared, shared_g=np.full(H, 1e3), x_gate=np.ones((T, H)))
    np.testing.assert_allclose(big, full, rtol=1e-12)
    small, *_ = forward(x, logits, k, E, get, shared, shared_g=np.full(H, -1e3), x_gate=np.ones((T, H)))
    np.testing.assert_allclose(small, routed, rtol=1e-12, atol=1e-14)
