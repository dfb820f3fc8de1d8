"""Plain CPU oracle of the top-k routed MoE FFN layer forward -- TEST
INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
legs may import this module.  It shares no code with the CUDA library: it
does not import the product package and the product package does not import
it.  Arithmetic is fp64 over exactly-decoded operands unless a step is
defined in fp32 (the NVFP4 encoder, see oracle.nvfp4).

The layer computes, per token t (problem statement of "Hosting Qwen on
Blackwell", section "MoE Dispatch - Combine", and "CuTeDSL at Perplexity",
section on the local dispatch/combine kernel):

    y_t = sum_j w[t,j] * E_{idx[t,j]}(x_t) + S(x_t)

with the steps, in the pages' order:

  route    -- top-k experts of the router logits and their weights.  The pages
              fix only that the routing table holds indices and weights of
              shape [T, k] ("Como Servimos um Modelo MoE de 397B ...", section
              "Tres coletivas viram duas").  Reading taken: softmax over the E
              logits, keep the k largest, renormalise the kept weights to sum
              to one; order by descending logit, ties to the lower expert id.
  permute  -- "CuTeDSL at Perplexity", local dispatch: count tokens per expert,
              give each token a unique index inside its expert's list, copy
              the tokens into expert-contiguous buffers.  Reading taken: a
              stable order (ascending token id inside each expert), unpadded.
  experts  -- per expert, gate/up projection, SwiGLU, down projection
              ("Hosting Qwen on Blackwell", section "MoE GEMM").  W13 rows
              [0, I) are the gate, rows [I, 2I) the up projection.
  shared   -- an always-on shared expert with weight 1
              ("Como Servimos ...", MoE FFN description: top_k=10 plus one
              shared expert that is always active).
  combine  -- weighted accumulation of each token's k expert outputs plus the
              shared expert output ("CuTeDSL at Perplexity", combine kernel).

Every output row depends only on its own token (and the global NVFP4 scale of
the activations), so `forward` can evaluate any subset of tokens exactly.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Optional, Sequence

import numpy as np

from . import nvfp4

F32 = np.float32


# ----------------------------------------------------------------------------
# route
# ----------------------------------------------------------------------------
def route(logits: np.ndarray, k: int, renorm: bool = True):
    """Top-k routing with renormalised softmax weights.

    logits: fp32 [T, E].  Returns idx int32 [T, k] (descending logit, ties to
    the lower expert id) and w fp64 [T, k] with
        w_j = exp(l_j - l_max) / sum_{i in selected} exp(l_i - l_max),
    which equals the full softmax over E renormalised over the k selected
    experts (the full denominator cancels).

    renorm=False: the variant without renormalisation (the pages allude to
    router variants without fixing one; reading taken: the same selection,
    weights = the full softmax over all E logits at the selected experts),
        w_j = exp(l_j - l_max) / sum_{e < E} exp(l_e - l_max).
    """
    logits = np.asarray(logits, dtype=F32)
    T, E = logits.shape
    assert 1 <= k <= E
    # stable sort on the negated value keeps equal logits in ascending id order
    order = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")
    idx = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(logits, idx, axis=1).astype(np.float64)
    if T == 0:
        return idx, np.zeros((0, k), np.float64)
    z = np.exp(sel - sel[:, :1])
    if renorm:
        w = z / z.sum(axis=1, keepdims=True)
    else:
        full = np.exp(logits.astype(np.float64) - sel[:, :1]).sum(axis=1, keepdims=True)
        w = z / full
    return idx, w


# ----------------------------------------------------------------------------
# permute / unpermute
# ----------------------------------------------------------------------------
@dataclass
class Permutation:
    counts: np.ndarray   # int32 [E]      slots routed to each expert
    offsets: np.ndarray  # int32 [E+1]    exclusive prefix sum, offsets[E] = T*k
    row_of: np.ndarray   # int32 [T, k]   row of slot (t, j) in the expert-ordered buffer
    src_tok: np.ndarray  # int32 [T*k]    token held by each row


def permute(idx: np.ndarray, E: int) -> Permutation:
    """Stable counting sort of the flattened slots (t, j) by expert.

    Row r of expert e's segment holds the r-th token (in ascending t) routed
    to e.  A token never selects an expert twice, so the order is unique.
    """
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    flat = idx.reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    order = np.argsort(flat, kind="stable")          # slot ids in expert order
    row_of_flat = np.empty(T * k, dtype=np.int64)
    row_of_flat[order] = np.arange(T * k)
    src_tok = (order // k) if k else order
    return Permutation(counts.astype(np.int32), offsets.astype(np.int32),
                       row_of_flat.reshape(T, k).astype(np.int32),
                       src_tok.astype(np.int32))


def gather_rows(x: np.ndarray, perm: Permutation) -> np.ndarray:
    """Expert-contiguous copy of the token rows: Xp[r] = x[src_tok[r]]."""
    return np.asarray(x)[perm.src_tok]


def unpermute(xp: np.ndarray, perm: Permutation) -> np.ndarray:
    """Inverse of gather_rows for each slot: out[t, j] = xp[row_of[t, j]]."""
    return np.asarray(xp)[perm.row_of]


# ----------------------------------------------------------------------------
# expert MLP (SwiGLU)
# ----------------------------------------------------------------------------
def silu(z: np.ndarray) -> np.ndarray:
    """z * sigmoid(z) in fp64."""
    return z / (1.0 + np.exp(-z))


def expert_mlp(a: np.ndarray, w13: np.ndarray, w2: np.ndarray,
               h_quant_g: Optional[np.float32] = None,
               h_quant: Optional[Callable[[np.ndarray], np.ndarray]] = None) -> np.ndarray:
    """One expert on a batch of rows.

    a   : fp64 [n, H]   input rows (already dequantised)
    w13 : fp64 [2I, H]  rows [0, I) gate, rows [I, 2I) up
    w2  : fp64 [H, I]   down projection
    h_quant_g : when given (NVFP4-activation path), the SwiGLU output h is
        rounded to fp32 and passed through NVFP4 quantisation with this global
        scale (blocks of 16 along I) before the down projection.
    h_quant : when given (the MX layers, oracle.mx.h_quant), a function that
        takes h (fp64 [n, I]) to the values the down projection sees.
    Returns fp64 [n, H].
    """
    I = w13.shape[0] // 2
    gate = a @ w13[:I].T
    up = a @ w13[I:].T
    h = silu(gate) * up
    if h_quant_g is not None:
        q, s, _ = nvfp4.quantize(h.astype(F32), F32(h_quant_g))
        h = nvfp4.dequantize(q, s, F32(h_quant_g))
    if h_quant is not None:
        h = h_quant(h)
    return h @ w2.T


# ----------------------------------------------------------------------------
# the layer
# ----------------------------------------------------------------------------
@dataclass
class ExpertWeights:
    """fp64 dequantised weights of one expert: w13 [2I, H], w2 [H, I]."""
    w13: np.ndarray
    w2: np.ndarray


def sigmoid(z: np.ndarray) -> np.ndarray:
    """1 / (1 + e^-z), evaluated through e^-|z| so that it never overflows."""
    z = np.asarray(z, dtype=np.float64)
    e = np.exp(-np.abs(z))
    return np.where(z >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def shared_gate(x_gate: np.ndarray, g: np.ndarray) -> np.ndarray:
    """Per-token gate of the shared expert, sigma(x_t . g) ("Hosting Qwen on
    Blackwell" names new gate terms without fixing them; reading taken: a
    sigmoid of the token's dot product with one gate vector g [H], applied
    to the shared expert's output, computed from the bf16 activations)."""
    return sigmoid(np.asarray(x_gate, np.float64) @ np.asarray(g, np.float64))


def forward(x_deq: np.ndarray, logits: np.ndarray, k: int, E: int,
            get_expert: Callable[[int], ExpertWeights],
            shared: Optional[ExpertWeights] = None,
            tokens: Optional[Sequence[int]] = None,
            h_quant_g: Optional[np.float32] = None,
            hs_quant_g: Optional[np.float32] = None,
            renorm: bool = True,
            shared_g: Optional[np.ndarray] = None,
            x_gate: Optional[np.ndarray] = None,
            h_quant: Optional[Callable[[np.ndarray], np.ndarray]] = None,
            hs_quant: Optional[Callable[[np.ndarray], np.ndarray]] = None):
    """Layer output for the given tokens (all tokens when `tokens` is None).

    x_deq   : fp64 [T, H] the activations as the experts see them (bf16 values,
              or the NVFP4-dequantised values on the NVFP4-activation path)
    logits  : fp32 [T, E] router logits
    get_expert(e) -> ExpertWeights, called once per expert that the selected
              tokens use (lets the caller decode weights lazily); None stands
              for an expert whose weights are all zero: its gate, up, h and
              output are then exactly zero (zero also stays zero through the
              h quantisers: it encodes to code 0), so its rows add nothing
    Returns (out fp64 [len(tokens), H], idx, w, perm) where idx / w / perm
    cover the full T (routing is cheap) and out covers `tokens`.
    renorm  : False selects the router without renormalisation (see route)
    shared_g: gate vector [H] of the shared expert (None: ungated, weight 1);
              x_gate: the activations the gate sees ([T, H]; default x_deq)
    h_quant / hs_quant: the step between SwiGLU and down projection of the
              routed / shared experts on the MX layers (see expert_mlp)
    """
    x_deq = np.asarray(x_deq, dtype=np.float64)
    T, H = x_deq.shape
    idx, w = route(logits, k, renorm)
    perm = permute(idx, E)
    toks = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    out = np.zeros((len(toks), H), dtype=np.float64)
    pos = {int(t): i for i, t in enumerate(toks)}
    # visit experts in id order; each expert processes its selected rows
    # (rows of the expert's segment in stable order), scaled by the weight
    for e in range(E):
        lo, hi = int(perm.offsets[e]), int(perm.offsets[e + 1])
        rows = [r for r in range(lo, hi) if int(perm.src_tok[r]) in pos]
        if not rows:
            continue
        W = get_expert(e)
        if W is None:
            continue
        src = perm.src_tok[rows]
        y = expert_mlp(x_deq[src], W.w13, W.w2, h_quant_g, h_quant)
        for r, t, yr in zip(rows, src, y):
            j = int(np.nonzero(perm.row_of[t] == r)[0][0])
            out[pos[int(t)]] += w[t, j] * yr
    if shared is not None:
        ys = expert_mlp(x_deq[toks], shared.w13, shared.w2, hs_quant_g, hs_quant)
        if shared_g is not None:
            xg = x_deq if x_gate is None else np.asarray(x_gate, np.float64)
            ys = ys * shared_gate(xg[toks], shared_g)[:, None]
        out += ys
    return out, idx, w, perm


def rel_frobenius(a: np.ndarray, ref: np.ndarray) -> float:
    """||a - ref||_F / ||ref||_F in fp64."""
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(a - ref)
    return float(num / den) if den > 0 else float(num)
