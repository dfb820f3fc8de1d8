// Combine / weighted unpermute ("CuTeDSL at Perplexity", combine kernel:
// vectorised accumulation in registers using the token positions computed by
// dispatch, writing the final tokens to the output buffer; "Hosting Qwen on
// Blackwell", section "MoE Dispatch - Combine": weighted accumulation after
// the MoE GEMM).
//
// One warp per (token, 256-column slice): lane l owns the slice's 8-element
// (16-byte) chunk l.  In fp32 and in the fixed order j = 0..k-1 then the
// shared expert, it accumulates w[t,j] * Y[row_of[t,j]] before one round to
// bf16.  HBM-bound: reads k + 1 rows, writes one.  The slice split keeps
// enough warps in flight at decode sizes (a few hundred tokens), and the k
// rows' loads are issued in batches of 8 before their FMAs.  A row index
// outside [0, T*k) (the -1 the permutation leaves for a slot whose expert id
// was out of range) contributes nothing.
#include "internal.h"

namespace moe {

constexpr int kCombineBatch = 8;

__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ Y, const int32_t* __restrict__ row_of,
                                                      const float* __restrict__ w, const uint16_t* __restrict__ Ys,
                                                      const float* __restrict__ ys_gate, int T, int k, int H,
                                                      int slices, uint16_t* __restrict__ out) {
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int t = static_cast<int>(gw / slices);
  if (t >= T) return;
  const int c = static_cast<int>(gw - static_cast<long long>(t) * slices) * 32 + lane;  // 16-byte chunk
  const bool valid = c < (H >> 3);
  const long long S = static_cast<long long>(T) * k;  // rows of Y
  // lane j < k holds the j-th row / weight; broadcast by shuffles
  int my_row = 0;
  float my_w = 0.0f;
  if (lane < k) {
    my_row = __ldg(row_of + static_cast<size_t>(t) * k + lane);
    my_w = __ldg(w + static_cast<size_t>(t) * k + lane);
  }
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  for (int j0 = 0; j0 < k; j0 += kCombineBatch) {
    uint4 v[kCombineBatch];
    float wj[kCombineBatch];
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) {
      const int j = min(j0 + u, k - 1);
      const int r = __shfl_sync(0xFFFFFFFFu, my_row, j);
      wj[u] = __shfl_sync(0xFFFFFFFFu, my_w, j);
      v[u] = (valid && j0 + u < k && r >= 0 && r < S) ? __ldg(reinterpret_cast<const uint4*>(Y + static_cast<size_t>(r) * H) + c)
                                   : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) {
      if (j0 + u >= k) break;
      const uint32_t q[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(wj[u], __uint_as_float(q[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = fmaf(wj[u], __uint_as_float(q[i] & 0xFFFF0000u), acc[2 * i + 1]);
      }
    }
  }
  if (!valid) return;
  if (Ys != nullptr) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(Ys + static_cast<size_t>(t) * H) + c);
    const uint32_t q[4] = {v.x, v.y, v.z, v.w};
    if (ys_gate != nullptr) {
      const float gt = __ldg(ys_gate + t);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(gt, __uint_as_float(q[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = fmaf(gt, __uint_as_float(q[i] & 0xFFFF0000u), acc[2 * i + 1]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] += __uint_as_float(q[i] << 16);
        acc[2 * i + 1] += __uint_as_float(q[i] & 0xFFFF0000u);
      }
    }
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H)[c] = o;
}

// Gate of the shared expert per token, sigma(x_t . g) in fp32, one warp per
// token ("Hosting Qwen on Blackwell" names new gate terms; reading: a sigmoid
// of the token's dot product with one gate vector).  HBM-bound: 2 * H bytes
// of x per token; lane l reads 16-byte chunks l, l+32, ...
__global__ void __launch_bounds__(256) shared_gate_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ g,
                                                          int T, int H, float* __restrict__ gate) {
  const int t = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
  const uint4* gr = reinterpret_cast<const uint4*>(g);
  float acc = 0.0f;
  for (int c = lane; c < (H >> 3); c += 32) {
    const uint4 a = __ldg(xr + c), b = __ldg(gr + c);
    const uint32_t qa[4] = {a.x, a.y, a.z, a.w}, qb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(__uint_as_float(qa[i] << 16), __uint_as_float(qb[i] << 16), acc);
      acc = fmaf(__uint_as_float(qa[i] & 0xFFFF0000u), __uint_as_float(qb[i] & 0xFFFF0000u), acc);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
  if (lane == 0) gate[t] = 1.0f / (1.0f + expf(-acc));
}

int shared_gate_launch(const uint16_t* x, const uint16_t* g, int T, int H, float* gate, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  shared_gate_kernel<<<(T + 7) / 8, 256, 0, s>>>(x, g, T, H, gate);
  return check_launch();
}

int combine_launch(const uint16_t* Y, const int32_t* row_of, const float* w, const uint16_t* Ys, const float* ys_gate,
                   int T, int k, int H, uint16_t* out, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  const int slices = (H / 8 + 31) / 32;
  const long long warps = static_cast<long long>(T) * slices;
  const long long blocks = (warps + 7) / 8;
  if (blocks > 0x7FFFFFFFLL) return MOE_ERR_UNSUPPORTED;
  combine_kernel<<<static_cast<unsigned int>(blocks), 256, 0, s>>>(Y, row_of, w, Ys, ys_gate, T, k, H, slices, out);
  return check_launch();
}

}  // namespace moe

using namespace moe;

extern "C" int moe_combine_gated(const uint16_t* Y, const int32_t* row_of, const float* w, const uint16_t* Ys,
                                 const float* ys_gate, int T, int k, int H, uint16_t* out, void* stream) {
  if (T < 0 || k < 1 || H < 1) return MOE_ERR_INVALID_ARG;
  if (k > 32 || H % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!Y || !row_of || !w || !out) return MOE_ERR_INVALID_ARG;
  if (ys_gate && !Ys) return MOE_ERR_INVALID_ARG;
  if (!aligned(Y, 16) || !aligned(out, 16) || (Ys && !aligned(Ys, 16)) || (ys_gate && !aligned(ys_gate, 4)))
    return MOE_ERR_INVALID_ARG;
  return combine_launch(Y, row_of, w, Ys, ys_gate, T, k, H, out, static_cast<cudaStream_t>(stream));
}

extern "C" int moe_combine(const uint16_t* Y, const int32_t* row_of, const float* w, const uint16_t* Ys, int T, int k,
                           int H, uint16_t* out, void* stream) {
  return moe_combine_gated(Y, row_of, w, Ys, nullptr, T, k, H, out, stream);
}

extern "C" int moe_shared_gate(const uint16_t* x, const uint16_t* g, int T, int H, float* gate, void* stream) {
  if (T < 0 || H < 1) return MOE_ERR_INVALID_ARG;
  if (H % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (T >= (1 << 27)) return MOE_ERR_UNSUPPORTED;  // one warp per token: 32 * T threads in 32 bits
  if (T == 0) return MOE_OK;
  if (!x || !g || !gate) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(g, 16) || !aligned(gate, 4)) return MOE_ERR_INVALID_ARG;
  return shared_gate_launch(x, g, T, H, gate, static_cast<cudaStream_t>(stream));
}
