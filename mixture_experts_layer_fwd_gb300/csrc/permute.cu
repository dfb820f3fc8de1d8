// Local dispatch (permutation into expert-contiguous order).
//
// "CuTeDSL at Perplexity", local MoE dispatch: count the tokens routed to
// each expert from the routing table, give every token a unique index inside
// its expert's list, then copy the tokens into the buffers that feed the MoE
// GEMM.  For prefill the page splits routing over blocks: indices are first
// assigned with per-block counters, then accumulated across blocks in global
// memory, and a separate copy kernel runs on many blocks and warps to use the
// full memory bandwidth.
//
// The page hands out slots with atomic counters, whose order depends on
// timing.  Here the order is deterministic and stable (rows of an expert in
// ascending token id), so that it is bit-exact and reproducible:
//   1. count   : per chunk of CH slots, a shared-memory histogram -> hist[c][e]
//   2. scan    : one block: counts, exclusive offsets, and per-chunk bases
//                base[c][e] = offsets[e] + sum_{c' < c} hist[c'][e]
//   3. assign  : per chunk, one warp walks the chunk's slots in order, 32 at a
//                time; __match_any_sync groups lanes with the same expert and
//                the rank inside the group orders them; a shared-memory
//                counter per expert carries the running position
//   4. gather  : one warp per permuted row copies the token row (16-byte
//                vectors) and its scale bytes
// An expert id outside [0, E) is a caller error: its slot is left out (not
// counted, row_of = -1, no permuted row), the device error word records
// kErrBadIndex, and no kernel touches memory outside its buffers.
#include "internal.h"
#include "permute.cuh"

namespace moe {


__global__ void __launch_bounds__(256) permute_count_kernel(const int32_t* __restrict__ idx, int S, int E,
                                                            int32_t* __restrict__ hist, unsigned int* err) {
  extern __shared__ int32_t sh[];
  const int c = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
  __syncthreads();
  const int lo = c * kPermChunk;
  const int hi = min(S, lo + kPermChunk);
  for (int s = lo + threadIdx.x; s < hi; s += blockDim.x) {
    const int e = __ldg(idx + s);
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E))
      atomicAdd(&sh[e], 1);
    else if (err != nullptr)
      atomicOr(err, kErrBadIndex);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[static_cast<size_t>(c) * E + e] = sh[e];
}

// Single block of 1024 threads.
__global__ void __launch_bounds__(1024) permute_scan_kernel(const int32_t* __restrict__ hist, int C, int E,
                                                            int32_t* __restrict__ base,
                                                            int32_t* __restrict__ counts,
                                                            int32_t* __restrict__ offsets) {
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int e0 = 0; e0 < E; e0 += blockDim.x) {
    const int e = e0 + threadIdx.x;
    // the chunk histograms are read 8 at a time so that the loads overlap
    int tot = 0;
    if (e < E)
      for (int c0 = 0; c0 < C; c0 += 8) {
        int h8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) h8[u] = (c0 + u < C) ? __ldg(hist + static_cast<size_t>(c0 + u) * E + e) : 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) tot += h8[u];
      }
    // block-wide inclusive scan of tot
    int v = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, v, off);
      if (lane >= off) v += o;
    }
    if (lane == 31) warp_tot[wid] = v;
    __syncthreads();
    if (wid == 0) {
      int wv = (lane < static_cast<int>(blockDim.x >> 5)) ? warp_tot[lane] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, wv, off);
        if (lane >= off) wv += o;
      }
      warp_tot[lane] = wv;  // inclusive over warps
    }
    __syncthreads();
    const int excl = carry + (wid ? warp_tot[wid - 1] : 0) + v - tot;
    if (e < E) {
      counts[e] = tot;
      offsets[e] = excl;
      int run = excl;
      for (int c0 = 0; c0 < C; c0 += 8) {
        int h8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) h8[u] = (c0 + u < C) ? __ldg(hist + static_cast<size_t>(c0 + u) * E + e) : 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (c0 + u < C) base[static_cast<size_t>(c0 + u) * E + e] = run;
          run += h8[u];
        }
      }
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = excl + tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) offsets[E] = carry;
}

// One warp per chunk.
__global__ void __launch_bounds__(32) permute_assign_kernel(const int32_t* __restrict__ idx, int S, int k, int E,
                                                            const int32_t* __restrict__ base,
                                                            int32_t* __restrict__ row_of,
                                                            int32_t* __restrict__ src_tok) {
  extern __shared__ int32_t ctr[];
  const int c = blockIdx.x;
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) ctr[e] = base[static_cast<size_t>(c) * E + e];
  __syncwarp();
  const int lo = c * kPermChunk;
  const int hi = min(S, lo + kPermChunk);
  // the chunk's routing ids, loaded up front (lane l holds slots lo + 32j + l)
  constexpr int J = kPermChunk / 32;
  int ev[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int s = lo + 32 * j + lane;
    ev[j] = s < hi ? __ldg(idx + s) : 0;
  }
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int s = lo + 32 * j + lane;
    if (lo + 32 * j >= hi) break;
    const int e = ev[j];
    const bool act = s < hi && static_cast<unsigned>(e) < static_cast<unsigned>(E);
    const unsigned mask = __ballot_sync(0xFFFFFFFFu, act);
    if (act) {
      const unsigned peers = __match_any_sync(mask, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int pos = ctr[e] + rank;
      __syncwarp(mask);
      if (rank == 0) ctr[e] += __popc(peers);
      row_of[s] = pos;
      src_tok[pos] = s / k;
    } else if (s < hi) {
      row_of[s] = -1;  // expert id outside [0, E): the slot is left out
    }
    __syncwarp();
  }
}

// One warp per permuted row (copy_row, permute.cuh).  Rows past offsets[E]
// exist only when slots were left out; their src_tok entries were never
// written, so a token id outside [0, T) is skipped.
template <bool TO_F16>
__global__ void __launch_bounds__(256) permute_gather_kernel(const int32_t* __restrict__ src_tok, int S, int T,
                                                             const uint8_t* __restrict__ x, int row_bytes,
                                                             const uint8_t* __restrict__ x_sf, int sf_bytes,
                                                             uint8_t* __restrict__ xp, uint8_t* __restrict__ xp_sf) {
  const int r = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= S) return;
  const int t = __ldg(src_tok + r);
  if (static_cast<unsigned>(t) >= static_cast<unsigned>(T)) return;
  copy_row<TO_F16>(x, row_bytes, x_sf, sf_bytes, t, xp, xp_sf, r, lane);
}

size_t permute_ws_bytes(int T, int k, int E) {
  const size_t S = static_cast<size_t>(T) * k;
  const size_t C = (S + kPermChunk - 1) / kPermChunk;
  return 2 * round_up(C * E * sizeof(int32_t), 256);
}

int permute_launch(const int32_t* idx, int T, int k, int E, const void* x_rows, int row_bytes, const uint8_t* x_sf,
                   int sf_row_bytes, int32_t* counts, int32_t* offsets, int32_t* row_of, int32_t* src_tok,
                   void* xp_rows, uint8_t* xp_sf, void* ws, size_t ws_bytes, cudaStream_t s, bool to_f16) {
  const int S = T * k;
  const int C = (S + kPermChunk - 1) / kPermChunk;
  Carve carve(ws, ws_bytes);
  int32_t* hist = carve.take<int32_t>(static_cast<size_t>(C) * E);
  int32_t* base = carve.take<int32_t>(static_cast<size_t>(C) * E);
  if (!carve.fits()) return MOE_ERR_WORKSPACE;
  const size_t shbytes = static_cast<size_t>(E) * sizeof(int32_t);
  unsigned int* err = device_error_word();  // NULL if the lookup failed: ids are still checked
  if (C > 0) permute_count_kernel<<<C, 256, shbytes, s>>>(idx, S, E, hist, err);
  permute_scan_kernel<<<1, 1024, 0, s>>>(hist, C, E, base, counts, offsets);
  if (C > 0) permute_assign_kernel<<<C, 32, shbytes, s>>>(idx, S, k, E, base, row_of, src_tok);
  if (xp_rows != nullptr && S > 0) {
    const int blocks = (S + 7) / 8;
    if (to_f16)
      permute_gather_kernel<true><<<blocks, 256, 0, s>>>(src_tok, S, T, static_cast<const uint8_t*>(x_rows), row_bytes,
                                                         x_sf, sf_row_bytes, static_cast<uint8_t*>(xp_rows), xp_sf);
    else
      permute_gather_kernel<false><<<blocks, 256, 0, s>>>(src_tok, S, T, static_cast<const uint8_t*>(x_rows), row_bytes,
                                                          x_sf, sf_row_bytes, static_cast<uint8_t*>(xp_rows), xp_sf);
  }
  return check_launch();
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_permute_workspace_size(int T, int k, int E) {
  if (T < 0 || k < 1 || E < 1) return 0;
  return permute_ws_bytes(T, k, E);
}

extern "C" int moe_permute(const int32_t* idx, int T, int k, int E, const void* x_rows, int row_bytes,
                           const uint8_t* x_sf, int sf_row_bytes, int32_t* counts, int32_t* offsets,
                           int32_t* row_of, int32_t* src_tok, void* xp_rows, uint8_t* xp_sf, void* ws,
                           size_t ws_bytes, void* stream) {
  if (T < 0 || k < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  if (E > kPermMaxExperts || k > E) return MOE_ERR_UNSUPPORTED;
  // the row copy runs one warp per routed row (32 * T*k threads in 32 bits)
  if (static_cast<long long>(T) * k >= (1ll << 27)) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!idx || !row_of || !src_tok)) return MOE_ERR_INVALID_ARG;
  if (xp_rows != nullptr) {
    if (!x_rows || row_bytes <= 0 || (row_bytes % 16) != 0) return MOE_ERR_INVALID_ARG;
    if (!aligned(x_rows, 16) || !aligned(xp_rows, 16)) return MOE_ERR_INVALID_ARG;
    if (x_sf != nullptr) {
      if (!xp_sf || sf_row_bytes <= 0 || (sf_row_bytes % 4) != 0) return MOE_ERR_INVALID_ARG;
      if (!aligned(x_sf, 4) || !aligned(xp_sf, 4)) return MOE_ERR_INVALID_ARG;
    }
  }
  if (ws_bytes < permute_ws_bytes(T, k, E) || (ws == nullptr && T > 0)) return MOE_ERR_WORKSPACE;
  if (ws != nullptr && !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  return permute_launch(idx, T, k, E, x_rows, row_bytes, xp_rows ? x_sf : nullptr, sf_row_bytes, counts, offsets,
                        row_of, src_tok, xp_rows, xp_sf, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}
