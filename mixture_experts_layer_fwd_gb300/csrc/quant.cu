// NVFP4 quantiser of bf16 matrices (activations before dispatch: "Driving
// vLLM WideEP and Large-Scale Serving Toward Maturity on Blackwell (Part I)",
// section "NVFP4 MoE dispatch"; the abs-max over 16 elements: "CuTeDSL at
// Perplexity", Blackwell support).  Also used once per layer to turn bf16
// master weights into NVFP4 weights (one global scale per expert).
//
// Two passes over x, both HBM-bound:
//   amax  : grid-stride 16-byte loads, block max, atomicMax of the fp32 bit
//           pattern (valid ordering for non-negative floats) into workspace
//   quant : one thread per 16-element block: two 16-byte loads, scale byte,
//           eight code bytes (one 8-byte store), coalesced across the warp;
//           for one group (the activations) a persistent grid (as many
//           thread blocks as fit on the SMs at once) whose blocks form the
//           per-group constants and a per-scale-byte reciprocal table in
//           shared memory once, then walk the 16-element blocks with the next
//           block's two loads issued before the current one is encoded
#include <atomic>

#include "internal.h"
#include "nvfp4.cuh"

namespace moe {

// (a * r, b * r), each rounded to nearest even: two fp32 products in one
// packed instruction
DEVINL void mul_rn_f32x2(float a, float b, float r, float& ra, float& rb) {
  unsigned long long x, y, z;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a), "f"(b));
  asm("mov.b64 %0, {%1, %1};" : "=l"(y) : "f"(r));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(z) : "l"(x), "l"(y));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(ra), "=f"(rb) : "l"(z));
}

__global__ void __launch_bounds__(256) amax_kernel(const uint16_t* __restrict__ x, long long group_elems,
                                                   unsigned int* __restrict__ amax_bits) {
  const int g = blockIdx.y;
  const uint4* p = reinterpret_cast<const uint4*>(x + static_cast<size_t>(g) * group_elems);
  const long long nvec = group_elems / 8;
  float m = 0.0f;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < nvec;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint4 v = __ldg(p + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      m = fmaxf(m, fabsf(__uint_as_float(w[j] << 16)));
      m = fmaxf(m, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < static_cast<int>(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
    atomicMax(amax_bits + g, __float_as_uint(m));
  }
}

__global__ void __launch_bounds__(256) quant_kernel(const uint16_t* __restrict__ x, long long nblocks,
                                                    long long blocks_per_group, const float* __restrict__ g_in,
                                                    const unsigned int* __restrict__ amax_bits,
                                                    uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                    float* __restrict__ g_out) {
  const long long b = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (b >= nblocks) return;
  const int grp = static_cast<int>(b / blocks_per_group);
  float g;
  if (g_in != nullptr) {
    g = __ldg(g_in + grp);
  } else {
    const float amax = __uint_as_float(__ldg(amax_bits + grp));
    g = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 2688.0f);
  }
  if (b % blocks_per_group == 0) g_out[grp] = g;
  const uint4* p = reinterpret_cast<const uint4*>(x + b * 16);
  const uint4 lo = __ldg(p), hi = __ldg(p + 1);
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  float v[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    v[2 * j] = __uint_as_float(w[j] << 16);
    v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
  uint32_t c[2];
  const uint32_t s = nvfp4_quantize16(v, g, c);
  reinterpret_cast<uint2*>(codes)[b] = make_uint2(c[0], c[1]);
  sf[b] = static_cast<uint8_t>(s);
}

// One 16-element block of quant1_kernel: w holds its 16 bf16 values.
DEVINL void quant1_block(const uint32_t (&w)[8], long long b, float R, float D, const float* s_den,
                         const float* s_rcp, uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
  float v[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    v[2 * j] = __uint_as_float(w[j] << 16);
    v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  float q = __fmul_rn(amax, R);
  if (((__float_as_uint(q) + 4u) & 0x7FFFFu) <= 8u || !(q < INFINITY)) q = __fdiv_rn(amax, D);
  const uint32_t sc = e4m3_encode_satfinite(q);  // amax >= 0: a byte in [0, 0x7E]
  const float den = s_den[sc], r = s_rcp[sc];
  float qq[16];
  if (den != 0.0f && r < INFINITY) {
    // only the near-decision-point test is left per element: a product
    // that overflows is infinite, whose low mantissa bits are zero, so the
    // test sends it to the division too
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      float q0, q1;
      mul_rn_f32x2(v[i], v[i + 1], r, q0, q1);
      qq[i] = ((__float_as_uint(q0) + 8u) & 0x1FFFFFu) <= 16u ? __fdiv_rn(v[i], den) : q0;
      qq[i + 1] = ((__float_as_uint(q1) + 8u) & 0x1FFFFFu) <= 16u ? __fdiv_rn(v[i + 1], den) : q1;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) qq[i] = den != 0.0f ? e2m1_quotient(v[i], den, r) : copysignf(0.0f, v[i]);
  }
  reinterpret_cast<uint2*>(codes)[b] = make_uint2(e2m1x8_rn_satfinite(qq), e2m1x8_rn_satfinite(qq + 8));
  sf[b] = static_cast<uint8_t>(sc);
}

// Pass 2 for one group (the activations): the same codes, scales and g bit
// for bit, with the per-group work hoisted out of the 16-element blocks
// (once per thread block of a persistent grid: thread t of block c encodes
// 16-element blocks t + 256 c, t + 256 (c + grid), ...).
// Each thread block computes g, the divisor D = RN(6 g) of the scale step,
// RN(1 / D), and for every E4M3 scale byte s the decoder's denominator
// d(s) = RN(e4m3(s) * g) and RN(1 / d(s)) once, in shared memory.  A
// block's scale is then e4m3(q) with q = RN(amax * RN(1 / D)), which is
// within 2 ulp of RN(amax / D); the two can round to different E4M3 bytes
// only near a rounding boundary of E4M3 (a value of at most four
// significant bits, whose low 19 mantissa bits are zero; above 448 both
// saturate), so q is replaced by the IEEE quotient when its low 19 mantissa
// bits lie within 4 of a multiple of 2^19, or when it is not finite.
__global__ void __launch_bounds__(256) quant1_kernel(const uint16_t* __restrict__ x, long long nblocks,
                                                     const float* __restrict__ g_in,
                                                     const unsigned int* __restrict__ amax_bits,
                                                     uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                     float* __restrict__ g_out) {
  __shared__ float s_den[128], s_rcp[128];
  __shared__ float s_g;
  if (threadIdx.x == 0) {
    float g;
    if (g_in != nullptr) {
      g = __ldg(g_in);
    } else {
      const float amax = __uint_as_float(__ldg(amax_bits));
      g = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 2688.0f);
    }
    s_g = g;
    if (blockIdx.x == 0) g_out[0] = g;
  }
  __syncthreads();
  const float g = s_g;
  if (threadIdx.x < 128) {
    const float den = __fmul_rn(e4m3_decode(threadIdx.x), g);
    s_den[threadIdx.x] = den;
    s_rcp[threadIdx.x] = den != 0.0f ? __frcp_rn(den) : 0.0f;
  }
  const float D = __fmul_rn(6.0f, g);
  const float R = __frcp_rn(D);
  __syncthreads();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  long long b = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (b >= nblocks) return;
  const uint4* p = reinterpret_cast<const uint4*>(x);
  uint4 lo = __ldg(p + 2 * b), hi = __ldg(p + 2 * b + 1);
  for (; b < nblocks; b += stride) {
    uint4 next_lo = make_uint4(0u, 0u, 0u, 0u), next_hi = next_lo;
    if (b + stride < nblocks) {
      next_lo = __ldg(p + 2 * (b + stride));
      next_hi = __ldg(p + 2 * (b + stride) + 1);
    }
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    lo = next_lo;
    hi = next_hi;
    quant1_block(w, b, R, D, s_den, s_rcp, codes, sf);
  }
}

size_t quant_ws_bytes(int groups) { return round_up(static_cast<size_t>(groups) * sizeof(unsigned int), 256); }

int quant_launch(const uint16_t* x, int groups, int rows, int cols, const float* g_in, uint8_t* codes, uint8_t* sf,
                 float* g_out, void* ws, size_t ws_bytes, cudaStream_t s) {
  const long long group_elems = static_cast<long long>(rows) * cols;
  if (group_elems == 0 || groups == 0) return MOE_OK;
  unsigned int* amax = static_cast<unsigned int*>(ws);
  if (g_in == nullptr) {
    if (ws_bytes < quant_ws_bytes(groups) || ws == nullptr) return MOE_ERR_WORKSPACE;
    cudaError_t e = cudaMemsetAsync(amax, 0, static_cast<size_t>(groups) * sizeof(unsigned int), s);
    if (e != cudaSuccess) {
      set_cuda_error(e);
      return MOE_ERR_CUDA;
    }
    const long long nvec = group_elems / 8;
    int bx = static_cast<int>(std::min<long long>((nvec + 255) / 256, 4LL * num_sms() / std::max(1, groups) + 1));
    bx = std::max(bx, 1);
    dim3 grid(bx, groups);
    amax_kernel<<<grid, 256, 0, s>>>(x, group_elems, amax);
  }
  const long long nblocks = group_elems / 16 * groups;
  const long long nthreadblocks = (nblocks + 255) / 256;
  if (groups == 1) {
    // as many thread blocks as are resident at once (per device; a racing
    // first call stores the same value)
    static std::atomic<int> resident[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    int per_sm = resident[dev].load(std::memory_order_relaxed);
    if (per_sm == 0) {
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quant1_kernel, 256, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
      resident[dev].store(per_sm, std::memory_order_relaxed);
    }
    const long long grid = std::min<long long>(nthreadblocks, static_cast<long long>(per_sm) * num_sms());
    quant1_kernel<<<static_cast<unsigned int>(grid), 256, 0, s>>>(x, nblocks, g_in, amax, codes, sf, g_out);
  }
  else
    quant_kernel<<<static_cast<unsigned int>(nthreadblocks), 256, 0, s>>>(x, nblocks, group_elems / 16, g_in, amax,
                                                                           codes, sf, g_out);
  return check_launch();
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_quant_nvfp4_workspace_size(int groups) {
  if (groups < 1) return 0;
  return quant_ws_bytes(groups);
}

extern "C" int moe_quant_nvfp4(const uint16_t* x, int groups, int rows, int cols, const float* g_in, uint8_t* codes,
                               uint8_t* sf, float* g_out, void* ws, size_t ws_bytes, void* stream) {
  if (groups < 1 || rows < 0 || cols < 0) return MOE_ERR_INVALID_ARG;
  if (cols % 16 != 0) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(rows) * cols == 0) return MOE_OK;
  if (!x || !codes || !sf || !g_out) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(codes, 8) || !aligned(g_out, 4)) return MOE_ERR_INVALID_ARG;
  if (g_in == nullptr && (ws == nullptr || ws_bytes < quant_ws_bytes(groups))) return MOE_ERR_WORKSPACE;
  if (ws != nullptr && !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  return quant_launch(x, groups, rows, cols, g_in, codes, sf, g_out, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}
