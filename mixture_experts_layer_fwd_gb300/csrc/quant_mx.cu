// MXFP8 / MXFP4 quantisation: one E8M0 scale per 32 consecutive elements of
// a row.
//
// "Hosting Qwen on Blackwell", section "Quantização": the MoE weights are
// served in MXFP8, MXFP4 was considered; "CuTeDSL at Perplexity", Blackwell
// support: abs-max reductions over 32 elements for MXFP8 / MXFP4.  The pages
// do not define the formats; the reading is the Open Compute Project
// microscaling definition:
//   e   = floor(log2 amax32) - emax      (emax 8 for E4M3, 2 for E2M1),
//         clamped to [-127, 127]; an all-zero block gets -127
//   q_i = element_RNE_satfinite(x_i * 2^-e), the sign of x_i kept
//   scale byte = e + 127 (E8M0)
// floor(log2 amax) is the exponent field of the fp32 amax (a subnormal or
// zero amax gives e <= -127 - emax, clamped to -127), and 2^-e is a normal
// fp32, so the scaling is exact except where it underflows fp32, far below
// where every element type rounds to zero.
//
// One warp per (row, 256 columns): lane l converts elements 8l .. 8l+7 (one
// 16-byte load), four lanes share a block's amax through two shuffles, and
// the first lane of each four writes the scale byte.  HBM-bound: 2 bytes in,
// 1 (MXFP8) or 0.5 (MXFP4) + 1/32 bytes out per element.
#include "internal.h"
#include "nvfp4.cuh"

namespace moe {

namespace {

template <bool FP4>
__global__ void __launch_bounds__(256) quant_mx_kernel(const uint16_t* __restrict__ x, int rows, int cols,
                                                       uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  constexpr int EMAX = FP4 ? 2 : 8;
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int chunks = (cols + 255) / 256;
  const long long row = gw / chunks;
  if (row >= rows) return;  // warp-uniform
  const int c0 = static_cast<int>(gw - row * chunks) * 256 + lane * 8;
  const bool act = c0 < cols;  // cols % 32 == 0: a block's four lanes agree
  uint4 raw = make_uint4(0u, 0u, 0u, 0u);
  if (act) raw = __ldg(reinterpret_cast<const uint4*>(x + row * cols + c0));
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  float v[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
  a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
  a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
  const int e = max(-127, min(127, static_cast<int>((__float_as_uint(a) >> 23) & 0xFFu) - 127 - EMAX));
  const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, e <= 127 - EMAX
  if (!act) return;
  if (FP4) {
    uint32_t packed = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float s = v[i] * inv;
      const uint32_t code = e2m1_magnitude(fabsf(s)) | ((__float_as_uint(v[i]) >> 31) << 3);
      packed |= code << (4 * i);
    }
    *reinterpret_cast<uint32_t*>(codes + row * (cols / 2) + c0 / 2) = packed;
  } else {
    uint32_t lo = 0u, hi = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      lo |= e4m3_encode_satfinite(v[i] * inv) << (8 * i);
      hi |= e4m3_encode_satfinite(v[4 + i] * inv) << (8 * i);
    }
    *reinterpret_cast<uint2*>(codes + row * cols + c0) = make_uint2(lo, hi);
  }
  if ((lane & 3) == 0) scales[row * (cols / 32) + c0 / 32] = static_cast<uint8_t>(e + 127);
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" int moe_quant_mx(const uint16_t* x, int rows, int cols, int fmt, uint8_t* codes, uint8_t* scales,
                            void* stream) {
  if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
  if (fmt != MOE_FMT_MXFP8 && fmt != MOE_FMT_MXFP4) return MOE_ERR_INVALID_ARG;
  if (cols % 32 != 0) return MOE_ERR_UNSUPPORTED;
  if (rows == 0) return MOE_OK;
  if (!x || !codes || !scales) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(codes, fmt == MOE_FMT_MXFP8 ? 8 : 4)) return MOE_ERR_INVALID_ARG;
  const long long warps = static_cast<long long>(rows) * ((cols + 255) / 256);
  const long long blocks = (warps + 7) / 8;
  if (blocks > 0x7FFFFFFFLL) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (fmt == MOE_FMT_MXFP4)
    quant_mx_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, s>>>(x, rows, cols, codes, scales);
  else
    quant_mx_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, s>>>(x, rows, cols, codes, scales);
  return check_launch();
}
