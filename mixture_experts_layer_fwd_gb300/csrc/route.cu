// Router: softmax top-k with renormalised weights, one warp per token.
//
// The routing table is expert ids and weights of shape [T, k]
// ("Como Servimos um Modelo MoE de 397B com 4.7x de Speedup em TPU v7",
// section "Tres coletivas viram duas"); the pages name top-k selection as a
// serialisation point worth fusing (same page, "Roadmap restante").
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
#include <cfloat>

#include "common.cuh"

namespace moe {

template <int EPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                    int renorm, int32_t* __restrict__ idx, float* __restrict__ w) {
  const int warp = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const float* row = logits + static_cast<size_t>(warp) * E;

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
    const size_t o = static_cast<size_t>(warp) * k + lane;
    idx[o] = my_id;
    w[o] = __fdiv_rn(z, sum);
  }
}

}  // namespace moe

using namespace moe;

extern "C" int moe_route_ex(const float* logits, int T, int E, int k, int renorm, int32_t* idx, float* w,
                            void* stream) {
  if (T < 0 || E < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (k > E || k > 32 || E > 1024) return MOE_ERR_UNSUPPORTED;
  if (T >= (1 << 27)) return MOE_ERR_UNSUPPORTED;  // one warp per token: 32 * T threads in 32 bits
  if (T == 0) return MOE_OK;
  if (!logits || !idx || !w) return MOE_ERR_INVALID_ARG;
  if (!aligned(logits, 4) || !aligned(idx, 4) || !aligned(w, 4)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int threads = 256;
  const int blocks = (T + 7) / 8;
  const int epl = (E + 31) / 32;
  if (epl <= 1)
    route_kernel<1><<<blocks, threads, 0, s>>>(logits, T, E, k, renorm ? 1 : 0, idx, w);
  else if (epl <= 2)
    route_kernel<2><<<blocks, threads, 0, s>>>(logits, T, E, k, renorm ? 1 : 0, idx, w);
  else if (epl <= 4)
    route_kernel<4><<<blocks, threads, 0, s>>>(logits, T, E, k, renorm ? 1 : 0, idx, w);
  else if (epl <= 8)
    route_kernel<8><<<blocks, threads, 0, s>>>(logits, T, E, k, renorm ? 1 : 0, idx, w);
  else if (epl <= 16)
    route_kernel<16><<<blocks, threads, 0, s>>>(logits, T, E, k, renorm ? 1 : 0, idx, w);
  else
    route_kernel<32><<<blocks, threads, 0, s>>>(logits, T, E, k, renorm ? 1 : 0, idx, w);
  return check_launch();
}

extern "C" int moe_route(const float* logits, int T, int E, int k, int32_t* idx, float* w, void* stream) {
  return moe_route_ex(logits, T, E, k, 1, idx, w, stream);
}
