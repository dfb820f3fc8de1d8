"""moe_permute_noalloc: the token permutation for callers that cannot
allocate device memory when they dispatch (runtimes that give each library a
fixed set of buffers at start-up and forbid allocation on the per-step path,
embedders whose allocator owns all device memory, plugins that only get their
inputs and outputs).  It keeps its scratch in a fixed array that the library
defines in device memory instead of a caller workspace.

The GPU test calls it through the C ABI twice in a row (a large problem, then
a smaller one, so the second call runs on the scratch the first one left
behind) and compares every output with moe_permute's, bit for bit (the
outputs are integers and copied bytes).  This file is collected last so that a
run stopping at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import require_gpu

DEV = "cuda"


def _lib():
    import __graft_entry__ as g
    g.build()
    from mixture_experts_layer_fwd_gb300 import _lib as L
    return L.load(), L


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """Host-side limit check: ceil(T*k/1024) * E <= 131072, nothing launched."""
    lib, L = _lib()

    def call(T, k, E):
        return lib.moe_permute_noalloc(None, T, k, E, None, 0, None, 0, None, None, None, None, None, None, None)

    # 256 chunks of 1024 slots x 1024 experts = 262144 entries: over the limit
    assert call(32768, 8, 1024) == L.MOE_ERR_UNSUPPORTED
    # the largest sizes inside the limit pass the size check (then fail on the null outputs)
    assert call(16384, 8, 1024) == L.MOE_ERR_INVALID_ARG
    assert call(4096, 8, 4096) == L.MOE_ERR_INVALID_ARG
    # moe_permute's own limits hold here too: E <= 4096 (its shared-memory
    # histogram), even where the scratch would hold the problem
    for E in (4097, 8192, 16384):
        assert call(1, 1, E) == L.MOE_ERR_UNSUPPORTED, E
        assert lib.moe_permute(None, 1, 1, E, None, 0, None, 0, None, None, None, None, None, None, None, 0,
                               None) == L.MOE_ERR_UNSUPPORTED


def _routing(T, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    rank = torch.randperm(E, generator=g).double() + 1
    logits = (torch.randn(T, E, generator=g, dtype=torch.float64) - 1.1 * torch.log(rank)).float()
    return torch.from_numpy(oracle.route(logits.numpy(), k)[0])


def _call_noalloc(lib, idx, E, rows, sf):
    T, k = idx.shape
    o = dict(counts=torch.empty(E, dtype=torch.int32, device=DEV),
             offsets=torch.empty(E + 1, dtype=torch.int32, device=DEV),
             row_of=torch.empty(T, k, dtype=torch.int32, device=DEV),
             src_tok=torch.empty(T * k, dtype=torch.int32, device=DEV),
             xp=torch.empty((T * k,) + tuple(rows.shape[1:]), dtype=rows.dtype, device=DEV),
             xp_sf=torch.empty(T * k, sf.shape[1], dtype=torch.uint8, device=DEV))
    st = lib.moe_permute_noalloc(idx.data_ptr(), T, k, E, rows.data_ptr(), rows[0].numel() * rows.element_size(),
                                 sf.data_ptr(), sf.shape[1], o["counts"].data_ptr(), o["offsets"].data_ptr(),
                                 o["row_of"].data_ptr(), o["src_tok"].data_ptr(), o["xp"].data_ptr(),
                                 o["xp_sf"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, st
    return o


@pytest.mark.gpu
def test_noalloc_permute_matches_moe_permute_on_two_calls():
    require_gpu()
    lib, L = _lib()
    from mixture_experts_layer_fwd_gb300 import moe_permute
    cases = [(16384, 256, 8, 7168), (3000, 64, 4, 512)]  # large then small: reuses the scratch
    for T, E, k, H in cases:
        idx = _routing(T, E, k, seed=T).to(DEV)
        g = torch.Generator().manual_seed(E)
        rows = torch.randint(0, 256, (T, H // 2), generator=g, dtype=torch.uint8).to(DEV)
        sf = torch.randint(0, 256, (T, H // 16), generator=g, dtype=torch.uint8).to(DEV)
        got = _call_noalloc(lib, idx, E, rows, sf)
        ref = moe_permute(idx, E, rows, sf)
        assert lib.moe_sync_status(torch.cuda.current_stream().cuda_stream) == 0
        for key in ("counts", "offsets", "row_of", "src_tok", "xp", "xp_sf"):
            assert torch.equal(got[key], ref[key]), (T, E, key)
        # and the permutation is the oracle's
        p = oracle.permute(idx.cpu().numpy(), E)
        assert np.array_equal(got["src_tok"].cpu().numpy(), p.src_tok)


@pytest.mark.gpu
def test_noalloc_binding_with_all_outputs_allocates_nothing():
    """Through the Python binding with every output passed in, the call makes
    no device allocation (the caching allocator's count stays put)."""
    require_gpu()
    from mixture_experts_layer_fwd_gb300 import moe_permute, moe_permute_noalloc
    T, E, k, H = 777, 64, 4, 1024
    idx = _routing(T, E, k, seed=5).to(DEV)
    rows = torch.randint(0, 256, (T, H // 2), generator=torch.Generator().manual_seed(1),
                         dtype=torch.uint8).to(DEV)
    sf = torch.randint(0, 256, (T, H // 16), generator=torch.Generator().manual_seed(2),
                       dtype=torch.uint8).to(DEV)
    out = dict(counts=torch.empty(E, dtype=torch.int32, device=DEV),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=DEV),
               row_of=torch.empty(T, k, dtype=torch.int32, device=DEV),
               src_tok=torch.empty(T * k, dtype=torch.int32, device=DEV),
               xp=torch.empty(T * k, H // 2, dtype=torch.uint8, device=DEV),
               xp_sf=torch.empty(T * k, H // 16, dtype=torch.uint8, device=DEV))
    moe_permute_noalloc(idx, E, rows, sf, out=out)  # first call: looks up the scratch address
    torch.cuda.synchronize()
    before = torch.cuda.memory_stats()["allocation.all.allocated"]
    got = moe_permute_noalloc(idx, E, rows, sf, out=out)
    torch.cuda.synchronize()
    assert torch.cuda.memory_stats()["allocation.all.allocated"] == before
    ref = moe_permute(idx, E, rows, sf)
    for key in ("counts", "offsets", "row_of", "src_tok", "xp", "xp_sf"):
        assert got[key] is out[key]
        assert torch.equal(got[key], ref[key]), key
