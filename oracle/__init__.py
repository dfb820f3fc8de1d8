"""Oracle of the MoE FFN layer forward: plain, slow, fp64 CPU code.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
cpu_baseline / reference legs of bench.py may import it.  The CUDA library
and its Python binding never import it, and it never imports them.

Every function is pinned by tests under tests/ (marked "not gpu") against
brute force, closed forms, invariants, a library routine, or hand-worked
values in tests/golden/.  No function here is "parity unpinned".
"""
from . import mx, nvfp4
from .moe import (ExpertWeights, Permutation, expert_mlp, forward, gather_rows,
                  permute, rel_frobenius, route, shared_gate, sigmoid, silu, unpermute)

__all__ = ["mx", "nvfp4", "ExpertWeights", "Permutation", "expert_mlp", "forward",
           "gather_rows", "permute", "rel_frobenius", "route", "shared_gate",
           "sigmoid", "silu", "unpermute"]
