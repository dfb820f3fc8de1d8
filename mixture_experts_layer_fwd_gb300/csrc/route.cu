// Router: softmax top-k with renormalised weights, one warp per token
// (route_token, route.cuh).
//
// The routing table is expert ids and weights of shape [T, k]
// ("Como Servimos um Modelo MoE de 397B com 4.7x de Speedup em TPU v7",
// section "Tres coletivas viram duas"); the pages name top-k selection as a
// serialisation point worth fusing (same page, "Roadmap restante"; fused with
// the permutation in dispatch.cu).
#include "route.cuh"

namespace moe {

template <int EPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                    int renorm, int32_t* __restrict__ idx, float* __restrict__ w) {
  const int warp = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (warp >= T) return;
  route_token<EPL>(logits, warp, E, k, renorm, idx, w, threadIdx.x & 31);
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
