// The router of one token, for one warp: softmax top-k (moe_route_ex).  Used
// by the router kernel (route.cu) and the fused dispatch (dispatch.cu).
//
// Each lane holds ceil(E/32) logits (lane-strided, so every load of the warp
// is one contiguous 128-byte segment).  k rounds of a warp-wide arg-max
// (butterfly shuffles on (value, id), ties to the lower id) pick the experts
// in descending order; lane j keeps the j-th pick.  The weights are the
// softmax over the k picked logits, which equals the full softmax over E
// renormalised over the picks because the full denominator cancels.
// Without renormalisation (a router variant the pages allude to) the weights
// are the full softmax over all E logits at the picks: the warp also sums
// exp(l - l_max) over its lanes' logits.
#pragma once

#include <cfloat>

#include "common.cuh"

namespace moe {

// Routes token t: writes idx[t*k + j] and w[t*k + j] for j < k.  Every lane of
// the warp must call it.
template <int EPL>
DEVINL void route_token(const float* __restrict__ logits, int t, int E, int k, int renorm, int32_t* __restrict__ idx,
                        float* __restrict__ w, int lane) {
  const float* row = logits + static_cast<size_t>(t) * E;
  float v[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = lane + 32 * j;
    v[j] = (e < E) ? __ldg(row + e) : -FLT_MAX;
  }
  uint32_t taken = 0;
  float my_val = 0.0f;
  int my_id = 0;
  float top = 0.0f;

  for (int r = 0; r < k; ++r) {
    float bv = -FLT_MAX;
    int be = 0x7FFFFFFF;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const int e = lane + 32 * j;
      const bool ok = (e < E) && !((taken >> j) & 1u);
      // ascending j means ascending id, so a strict > keeps the lower id on ties
      if (ok && (v[j] > bv || be == 0x7FFFFFFF)) {
        bv = v[j];
        be = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
      const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, off);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (r == 0) top = bv;
    if (lane == r) {
      my_val = bv;
      my_id = be;
    }
  }
  const float z = (lane < k) ? expf(my_val - top) : 0.0f;
  float sum = z;
  if (!renorm) {
    sum = 0.0f;
#pragma unroll
    for (int j = 0; j < EPL; ++j)
      if (lane + 32 * j < E) sum += expf(v[j] - top);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
  if (lane < k) {
    const size_t o = static_cast<size_t>(t) * k + lane;
    idx[o] = my_id;
    w[o] = __fdiv_rn(z, sum);
  }
}

}  // namespace moe
