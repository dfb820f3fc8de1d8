// The router of one token, for one warp: softmax top-k (moe_route_ex).  Used
// by the router kernel (route.cu) and the fused dispatch (dispatch.cu).
//
// Each lane holds ceil(E/32) logits (lane-strided, so every load of the warp
// is one contiguous 128-byte segment), each also as an order-preserving
// 32-bit key (sign bit flipped for non-negative values, all bits for
// negative ones; -0 taken as +0, so that equal values have equal keys).
// k rounds of a warp-wide arg-max pick the experts in descending order,
// ties to the lower id: a lane's best key (lowest id among its equals), the
// warp's maximum key and the lowest id holding it by two integer warp
// reductions (redux.sync); the pick's key is then cleared.  Lane j keeps the
// j-th pick.  The weights are the softmax over the k picked logits, which
// equals the full softmax over E renormalised over the picks because the
// full denominator cancels.
// Without renormalisation (a router variant the pages allude to) the weights
// are the full softmax over all E logits at the picks: the warp also sums
// exp(l - l_max) over its lanes' logits.
#pragma once

#include <cfloat>

#include "common.cuh"

namespace moe {

// The logit of an order-preserving key (a -0 logit comes back as +0).
DEVINL float key_value(uint32_t key) { return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key); }

// Loads token t's logits as keys: key[j] for expert lane + 32 j, 0 past E.
template <int EPL>
DEVINL void route_load(const float* __restrict__ logits, int t, int E, int lane, uint32_t (&key)[EPL]) {
  const float* row = logits + static_cast<size_t>(t) * E;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = lane + 32 * j;
    uint32_t u = (e < E) ? __float_as_uint(__ldg(row + e)) : 0u;
    if (u == 0x80000000u) u = 0u;
    key[j] = (e < E) ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;
  }
}

// Picks token t's experts from its keys (which it clears on the way):
// writes idx[t*k + j] and w[t*k + j] for j < k.  Every lane of the warp must
// call it.
template <int EPL>
DEVINL void route_pick(uint32_t (&key)[EPL], int t, int E, int k, int renorm, int32_t* __restrict__ idx,
                       float* __restrict__ w, int lane) {
  float my_val = 0.0f;
  int my_id = 0;
  float top = 0.0f;
  float full = 0.0f;  // without renormalisation: this lane's part of the sum of exp(l - l_max) over all E
  if (!renorm) {
    uint32_t lk = 0u;
#pragma unroll
    for (int j = 0; j < EPL; ++j) lk = max(lk, key[j]);
    const uint32_t m0 = __reduce_max_sync(0xFFFFFFFFu, lk);
    const float l_max = key_value(m0);
#pragma unroll
    for (int j = 0; j < EPL; ++j)
      if (lane + 32 * j < E) full += expf(key_value(key[j]) - l_max);
  }

  for (int r = 0; r < k; ++r) {
    uint32_t bk = 0u;
    int bj = 0;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      // ascending j means ascending id, so a strict > keeps the lower id
      if (key[j] > bk) {
        bk = key[j];
        bj = j;
      }
    }
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, bk);
    const int be = static_cast<int>(
        __reduce_min_sync(0xFFFFFFFFu, bk == m ? static_cast<unsigned>(lane + 32 * bj) : 0xFFFFFFFFu));
    const bool mine = (be & 31) == lane;
#pragma unroll
    for (int j = 0; j < EPL; ++j) key[j] = (mine && j == (be >> 5)) ? 0u : key[j];
    const float bv = key_value(m);  // the picked logit
    if (r == 0) top = bv;
    if (lane == r) {
      my_val = bv;
      my_id = be;
    }
  }
  const float z = (lane < k) ? expf(my_val - top) : 0.0f;
  float sum = renorm ? z : full;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
  if (lane < k) {
    const size_t o = static_cast<size_t>(t) * k + lane;
    idx[o] = my_id;
    w[o] = __fdiv_rn(z, sum);
  }
}

// Routes token t (route_load + route_pick).
template <int EPL>
DEVINL void route_token(const float* __restrict__ logits, int t, int E, int k, int renorm, int32_t* __restrict__ idx,
                        float* __restrict__ w, int lane) {
  uint32_t key[EPL];  // 0: no expert (past E, or already picked)
  route_load<EPL>(logits, t, E, lane, key);
  route_pick<EPL>(key, t, E, k, renorm, idx, w, lane);
}

}  // namespace moe
