// Combine / weighted unpermute ("CuTeDSL at Perplexity", combine kernel:
// vectorised accumulation in registers using the token positions computed by
// dispatch, writing the final tokens to the output buffer; "Hosting Qwen on
// Blackwell", section "MoE Dispatch - Combine": weighted accumulation after
// the MoE GEMM).
//
// One warp per token; each lane owns 8-element (16-byte) column chunks and
// accumulates, in fp32 and in the fixed order j = 0..k-1 then the shared
// expert, w[t,j] * Y[row_of[t,j]] before one round to bf16.  HBM-bound:
// reads k + 1 rows, writes one.
#include "internal.h"

namespace moe {

__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ Y, const int32_t* __restrict__ row_of,
                                                      const float* __restrict__ w, const uint16_t* __restrict__ Ys,
                                                      int T, int k, int H, uint16_t* __restrict__ out) {
  const int t = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  // lane j < k holds the j-th row / weight; broadcast by shuffles
  int my_row = 0;
  float my_w = 0.0f;
  if (lane < k) {
    my_row = __ldg(row_of + static_cast<size_t>(t) * k + lane);
    my_w = __ldg(w + static_cast<size_t>(t) * k + lane);
  }
  const int nvec = H >> 3;
  for (int c = lane; c < nvec; c += 32) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int j = 0; j < k; ++j) {
      const int r = __shfl_sync(0xFFFFFFFFu, my_row, j);
      const float wj = __shfl_sync(0xFFFFFFFFu, my_w, j);
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(Y + static_cast<size_t>(r) * H) + c);
      const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(wj, __uint_as_float(q[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = fmaf(wj, __uint_as_float(q[i] & 0xFFFF0000u), acc[2 * i + 1]);
      }
    }
    if (Ys != nullptr) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(Ys + static_cast<size_t>(t) * H) + c);
      const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] += __uint_as_float(q[i] << 16);
        acc[2 * i + 1] += __uint_as_float(q[i] & 0xFFFF0000u);
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H)[c] = o;
  }
}

int combine_launch(const uint16_t* Y, const int32_t* row_of, const float* w, const uint16_t* Ys, int T, int k, int H,
                   uint16_t* out, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  const int blocks = (T + 7) / 8;
  combine_kernel<<<blocks, 256, 0, s>>>(Y, row_of, w, Ys, T, k, H, out);
  return check_launch();
}

}  // namespace moe

using namespace moe;

extern "C" int moe_combine(const uint16_t* Y, const int32_t* row_of, const float* w, const uint16_t* Ys, int T, int k,
                           int H, uint16_t* out, void* stream) {
  if (T < 0 || k < 1 || H < 1) return MOE_ERR_INVALID_ARG;
  if (k > 32 || H % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!Y || !row_of || !w || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(Y, 16) || !aligned(out, 16) || (Ys && !aligned(Ys, 16))) return MOE_ERR_INVALID_ARG;
  return combine_launch(Y, row_of, w, Ys, T, k, H, out, static_cast<cudaStream_t>(stream));
}
