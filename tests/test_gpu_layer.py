"""Layer parity: moe_forward (through the C ABI) against the fp64 oracle.

Tolerance (relative Frobenius error of the bf16 output): 5e-3 on the bf16
weight path, 1e-2 on the NVFP4 paths.  Small shapes are compared on every
token.  The full-size workloads are compared on token subsets (each output
row depends only on its own token and the global activation scale, so the
oracle evaluates those rows exactly): a seeded sample with real weights on
every expert, and every row of a few chosen experts with the other experts'
weights set to zero."""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import nvfp4
from tests.helpers import OracleWeights, oracle_layer, require_gpu, to_np_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _tol(cfg):
    return 5e-3 if cfg.w_fmt == "bf16" else 1e-2  # NVFP4 and MX layers: 1e-2


def _run(cfg, T, seed=0, tokens=None, weights=None, cache=True):
    from mixture_experts_layer_fwd_gb300 import MoELayer, moe_sync_status
    acts = synth.make_activations(cfg, T, seed=seed)
    w = weights or synth.make_weights(cfg, seed=seed, device=DEV)
    layer = MoELayer.from_config(cfg, w)
    out = layer(acts.x.to(DEV), acts.logits.to(DEV))
    assert moe_sync_status() == 0
    got = to_np_f32(out)
    assert np.isfinite(got).all()
    ref, *_ = oracle_layer(cfg, acts, OracleWeights(cfg, w, cache=cache), tokens=tokens)
    sel = got if tokens is None else got[tokens]
    return oracle.rel_frobenius(sel, ref), layer, w


SMALL = {
    "qwen3-235b": synth.small_variant(synth.QWEN3_235B, H=512, E=16, k=4, I=256),
    "qwen35-397b": synth.small_variant(synth.QWEN35_397B, H=512, E=32, k=5, I=128, I_s=192),
    "deepseek-v3": synth.small_variant(synth.DEEPSEEK_V3, H=768, E=16, k=4, I=256, I_s=320),
}


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_layer_all_tokens(seed):
    cfg = synth.TINY
    err, *_ = _run(cfg, 64, seed=seed)
    assert err <= _tol(cfg), err


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("T", [1, 37, 300])
def test_small_layers_all_tokens(name, T):
    cfg = SMALL[name]
    err, *_ = _run(cfg, T, seed=T)
    assert err <= _tol(cfg), err


def test_zero_tokens_is_noop():
    from mixture_experts_layer_fwd_gb300 import MoELayer, moe_sync_status
    cfg = synth.TINY
    layer = MoELayer.from_config(cfg, synth.make_weights(cfg, 0, DEV))
    out = torch.full((0, cfg.H), 7, dtype=torch.bfloat16, device=DEV)
    layer(torch.empty(0, cfg.H, dtype=torch.bfloat16, device=DEV), torch.empty(0, cfg.E, device=DEV), out=out)
    assert moe_sync_status() == 0


def test_k_equals_E_and_single_expert():
    for cfg in (synth.small_variant(synth.TINY, H=256, E=4, k=4, I=128),
                synth.small_variant(synth.TINY, H=256, E=1, k=1, I=192)):
        err, *_ = _run(cfg, 50, seed=4)
        assert err <= 5e-3, (cfg, err)


def test_hot_experts_leave_others_empty():
    cfg = synth.small_variant(synth.DEEPSEEK_V3, H=512, E=64, k=4, I=128, I_s=128)
    from dataclasses import replace
    cfg = replace(cfg, zipf=2.0)
    err, *_ = _run(cfg, 200, seed=6)
    assert err <= 1e-2, err


def test_decode_one_token_per_expert():
    """All experts active with a single token each ("Hosting Qwen on
    Blackwell", section "MoE GEMM" microbenchmarks), on small shapes."""
    from mixture_experts_layer_fwd_gb300 import MoELayer, moe_sync_status
    cfg = SMALL["qwen3-235b"]
    T, logits = synth.forced_one_token_per_expert_logits(cfg)
    acts = synth.make_activations(cfg, T, seed=1)
    acts = synth.Activations(acts.x, logits)
    w = synth.make_weights(cfg, 1, DEV)
    out = MoELayer.from_config(cfg, w)(acts.x.to(DEV), acts.logits.to(DEV))
    assert moe_sync_status() == 0
    ref, idx, *_ = oracle_layer(cfg, acts, OracleWeights(cfg, w))
    assert sorted(idx.reshape(-1).tolist()) == list(range(cfg.E))
    assert oracle.rel_frobenius(to_np_f32(out), ref) <= 5e-3


def test_nvfp4_weight_codes_match_oracle():
    """The layer's NVFP4 weight preparation (library quantiser) is bit-exact
    with the oracle's encoding of the same bf16 master weights."""
    from mixture_experts_layer_fwd_gb300 import MoELayer
    cfg = SMALL["qwen35-397b"]
    w = synth.make_weights(cfg, 0, DEV)
    layer = MoELayer.from_config(cfg, w)
    ow = OracleWeights(cfg, w)
    for e in (0, 7, cfg.E - 1):
        (q13, s13, g13), (q2, s2, g2) = ow.expert_codes(e)
        assert np.array_equal(layer.w13.codes[e].cpu().numpy(), q13)
        assert np.array_equal(layer.w13.sf[e].cpu().numpy(), s13)
        assert layer.w13.g[e].item() == g13
        assert np.array_equal(layer.w2.codes[e].cpu().numpy(), q2)
        assert np.array_equal(layer.w2.sf[e].cpu().numpy(), s2)


# ------------------------------------------------------- full-size workloads
# Real weights on every expert, compared on a seeded token sample.  The
# bf16 workload decodes its weights cheaply, so it compares 512 tokens (all
# of them at T = 256); the NVFP4 workloads re-encode every expert they touch
# with the oracle's own quantiser (seconds per expert), so they compare a
# few tokens here and every row of chosen experts in the tests below.
FULL = [("qwen3-235b", 256, 256), ("qwen3-235b", 8192, 512), ("qwen35-397b", 64, 8), ("qwen35-397b", 512, 6),
        ("qwen35-397b", 4096, 6), ("deepseek-v3", 256, 3), ("deepseek-v3", 16384, 3)]


@pytest.mark.parametrize("name,T,n", FULL)
def test_full_size_sampled_tokens(name, T, n):
    cfg = synth.CONFIGS[name]
    toks = synth.sample_tokens(T, n, seed=T)
    err, *_ = _run(cfg, T, seed=0, tokens=toks, cache=False)
    assert err <= _tol(cfg), err


def _chosen_experts(counts, seed, max_rows):
    """Experts whose every routed row is compared: the hottest (at most
    max_rows rows: a group split into many token blocks), one whose row count
    is above 256 and not a multiple of 128 (several blocks and a partial
    last tile), the one with the fewest rows (fewer than 16 where routing
    leaves such an expert), and one more drawn at random."""
    counts = np.asarray(counts)
    rng = np.random.default_rng(seed)
    live = np.nonzero(counts)[0]
    fit = live[counts[live] <= max_rows]
    chosen = [int(fit[np.argmax(counts[fit])])]
    ragged = [e for e in fit if counts[e] > 256 and counts[e] % 128 and e not in chosen]
    if ragged:
        chosen.append(int(rng.choice(ragged)))
    small = [e for e in live if e not in chosen]
    chosen.append(int(min(small, key=lambda e: (counts[e], e))))
    rest = [e for e in fit if e not in chosen]
    if rest:
        chosen.append(int(rng.choice(rest)))
    return chosen


def _run_chosen_experts(cfg, T, seed=0, max_rows=8192, extra_tokens=512):
    """The whole layer at full size through moe_forward, with the master
    weights of every expert outside a chosen few set to zero.  Routing,
    permutation, every tile of the grouped GEMMs (zero experts included) and
    the combine run as usual; a zero expert contributes exactly zero (in the
    oracle it is skipped), so each token's output holds its chosen experts'
    rows and the shared expert.  Compared: every token routed to a chosen
    expert, plus a seeded sample of others."""
    from mixture_experts_layer_fwd_gb300 import MoELayer, moe_sync_status
    acts = synth.make_activations(cfg, T, seed=seed)
    idx, _ = oracle.route(acts.logits.numpy(), cfg.k)
    counts = np.bincount(idx.reshape(-1), minlength=cfg.E)
    chosen = _chosen_experts(counts, seed + T, max_rows)
    zero = np.setdiff1d(np.arange(cfg.E), chosen)
    w = synth.make_weights(cfg, seed=seed, device=DEV)
    zi = torch.from_numpy(zero).to(DEV)
    w.w13[zi] = 0
    w.w2[zi] = 0
    layer = MoELayer.from_config(cfg, w)
    out = layer(acts.x.to(DEV), acts.logits.to(DEV))
    assert moe_sync_status() == 0
    got = to_np_f32(out)
    assert np.isfinite(got).all()
    mine = np.nonzero(np.isin(idx, chosen).any(axis=1))[0]
    toks = np.union1d(mine, synth.sample_tokens(T, extra_tokens, seed=T + 1))
    ref, *_ = oracle_layer(cfg, acts, OracleWeights(cfg, w, cache=False, zero_experts=zero), tokens=toks)
    return oracle.rel_frobenius(got[toks], ref), counts[chosen], len(toks)


CHOSEN = [("qwen35-397b", 64), ("qwen35-397b", 512), ("qwen35-397b", 4096), ("deepseek-v3", 256),
          ("deepseek-v3", 16384), ("qwen3-235b", 8192), ("qwen3-235b-mxfp8", 256), ("qwen3-235b-mxfp8", 8192)]


@pytest.mark.parametrize("name,T", CHOSEN)
def test_full_size_every_row_of_chosen_experts(name, T):
    cfg = synth.CONFIGS[name]
    err, rows, ntok = _run_chosen_experts(cfg, T)
    assert ntok >= min(T, 512)
    assert err <= _tol(cfg), (err, rows)


@pytest.mark.parametrize("w_fmt,zipf,T", [("bf16", 2.0, 1), ("bf16", 0.0, 4096), ("nvfp4", 2.0, 65536),
                                          ("nvfp4", 0.0, 2), ("nvfp4", 1.1, 64), ("bf16", 1.1, 16384),
                                          ("nvfp4", 0.0, 8192)])
def test_sweep_points(w_fmt, zipf, T):
    """Size / imbalance sweep on the DeepSeek-V3 shapes.  Few tokens (up to
    64 with bf16 weights, 2 with NVFP4 weights, whose oracle re-encodes every
    expert it touches): real weights on every expert, every token compared.
    Otherwise every row of chosen experts plus a sample of 64 other tokens
    (all tokens at T = 64), as above."""
    cfg = synth.sweep_config(w_fmt, zipf)
    if T <= (64 if w_fmt == "bf16" else 2):
        err, *_ = _run(cfg, T, seed=0, cache=False)
    else:
        err, rows, ntok = _run_chosen_experts(cfg, T, max_rows=4096, extra_tokens=64)
        assert ntok >= 64
    assert err <= _tol(cfg), err


@pytest.mark.parametrize("name", ["qwen35-397b", "deepseek-v3"])
@pytest.mark.parametrize("renorm,gated", [(False, False), (True, True), (False, True)])
def test_layer_router_and_shared_gate_variants(name, renorm, gated):
    """The router without renormalisation and the sigmoid-gated shared expert
    (layer options no_renorm / ws_gate) against the oracle's variants."""
    from mixture_experts_layer_fwd_gb300 import MoELayer, moe_sync_status
    cfg = SMALL[name]
    T = 137
    acts = synth.make_activations(cfg, T, seed=5)
    w = synth.make_weights(cfg, seed=5, device=DEV)
    g = (torch.randn(cfg.H, generator=torch.Generator().manual_seed(6)) * 0.05).to(torch.bfloat16)
    layer = MoELayer(cfg.H, cfg.E, cfg.k, cfg.I, cfg.I_s, w.w13, w.w2, w.ws13, w.ws2, cfg.w_fmt, cfg.act_fmt,
                     cfg.g_h, renorm=renorm, shared_gate=g.to(DEV) if gated else None)
    out = layer(acts.x.to(DEV), acts.logits.to(DEV))
    assert moe_sync_status() == 0
    got = to_np_f32(out)
    ref, idx, wts, _ = oracle_layer(cfg, acts, OracleWeights(cfg, w), renorm=renorm, shared_g=g if gated else None)
    assert oracle.rel_frobenius(got, ref) <= _tol(cfg)
    if not renorm:
        assert np.all(wts.sum(axis=1) < 1.0)  # the variant's weights do not sum to one


@pytest.mark.parametrize("name", ["tiny", "deepseek-v3"])
def test_forward_graph_replays_the_layer(name):
    """moe_forward captured as a CUDA graph: a replay equals the direct
    forward bit for bit (the kernels are deterministic), also after the
    inputs' contents change in place."""
    from mixture_experts_layer_fwd_gb300 import MoELayer, moe_sync_status
    cfg = synth.TINY if name == "tiny" else SMALL[name]
    T = 64
    w = synth.make_weights(cfg, seed=3, device=DEV)
    layer = MoELayer.from_config(cfg, w)
    a0 = synth.make_activations(cfg, T, seed=3)
    a1 = synth.make_activations(cfg, T, seed=4)
    x, lg = a0.x.to(DEV).contiguous(), a0.logits.to(DEV).contiguous()
    gout = torch.empty(T, cfg.H, dtype=torch.bfloat16, device=DEV)
    graph = layer.capture(x, lg, gout)
    for a in (a0, a1):
        x.copy_(a.x.to(DEV))
        lg.copy_(a.logits.to(DEV))
        graph.launch()
        direct = layer(a.x.to(DEV), a.logits.to(DEV))
        assert moe_sync_status() == 0
        assert torch.equal(gout, direct)
    graph.close()


@pytest.mark.parametrize("name,n", [("tiny", 1), ("tiny", 5), ("deepseek-v3", 4)])
def test_forward_host_pipelined_equals_each_batch(name, n):
    """moe_forward_host_pipelined over n batches (copies overlapping the
    neighbours' compute, device buffers used alternately): every batch's
    host output equals the direct forward of that batch bit for bit."""
    from mixture_experts_layer_fwd_gb300 import MoELayer, moe_forward_host_pipelined, moe_sync_status
    cfg = synth.TINY if name == "tiny" else SMALL[name]
    T = 64
    w = synth.make_weights(cfg, seed=5, device=DEV)
    layer = MoELayer.from_config(cfg, w)
    acts = [synth.make_activations(cfg, T, seed=10 + i) for i in range(n)]
    xh = [a.x.pin_memory() for a in acts]
    lh = [a.logits.pin_memory() for a in acts]
    oh = [torch.empty(T, cfg.H, dtype=torch.bfloat16).pin_memory() for _ in range(n)]
    xd = torch.empty(2, T, cfg.H, dtype=torch.bfloat16, device=DEV)
    ld = torch.empty(2, T, cfg.E, dtype=torch.float32, device=DEV)
    od = torch.empty(2, T, cfg.H, dtype=torch.bfloat16, device=DEV)
    ws = layer.workspace(T)
    compute_stream, copy_stream = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    moe_forward_host_pipelined(layer.c, xh, lh, oh, xd, ld, od, ws, stream=compute_stream, copy_stream=copy_stream)
    assert moe_sync_status() == 0
    for i, a in enumerate(acts):
        direct = layer(a.x.to(DEV), a.logits.to(DEV)).cpu()
        assert torch.equal(oh[i], direct), i
