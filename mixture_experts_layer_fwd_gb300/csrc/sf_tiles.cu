// NVFP4 scale factors in the order the block-scaled MMA reads them.
//
// "Driving vLLM WideEP ... (Part I)", section "NVFP4 GEMM for MoE and
// O-proj": one E4M3 scale per 16 elements, applied inside the tensor cores.
//
// One block-scaled MMA (128 rows, K = 64) reads four scale bytes per row
// from tensor memory: row m in lane m % 32 of column m / 32.  tcgen05.cp
// (32x128b, replicated into the four lane quadrants) fills those four
// columns from 512 contiguous bytes of shared memory holding row m's bytes
// at 16 * (m % 32) + 4 * (m / 32).  A tile is 128 rows of an operand; its
// scales are stored as K/64 such 512-byte blocks, one per MMA, so that a
// GEMM stage fetches the scales of all its MMAs with one contiguous copy per
// operand:
//
//   tiled[((tile * K/64 + kk) * 32 + l) * 16 + 4 * j + b] = sf[row(tile, 32 j + l)][4 kk + b]
//
// with sf the row-major [rows, K/16] scale bytes.  Rows past the end of a
// group read as zero.  Tiles are numbered:
//   rows in groups (the tokens of each expert, offsets [G+1]):
//     tile_base[g] = sum_{g' < g} ceil(rows_g' / 128); tile tile_base[g] + q
//     holds rows offsets[g] + 128 q + m
//   weights, G groups of N rows (STORE): tile g * ceil(N/128) + n holds rows
//     g * N + 128 n + m
//   weights, G groups of 2N rows (SwiGLU: gate rows [0, N), up rows [N, 2N)):
//     tile g * ceil(N/64) + n holds gate rows 64 n + m for m < 64 and up rows
//     N + 64 n + (m - 64) for m >= 64, the order of the GEMM's B tile
#include "internal.h"

namespace moe {

namespace {

constexpr int kModeRows = 0;
constexpr int kModeStore = 1;
constexpr int kModeSwiglu = 2;

DEVINL int clamp_rows(int v, int M) { return min(max(v, 0), M); }

// tile_base[0..G] from offsets[0..G], each clamped to [0, M] and empty when
// it ends before it starts (the grouped GEMM's reading).  One block of 1024
// threads; G <= 1024.
__global__ void __launch_bounds__(1024) sf_tile_base_kernel(const int32_t* __restrict__ offsets, int G, int M,
                                                            int32_t* __restrict__ tile_base) {
  __shared__ int warp_tot[32];
  const int g = threadIdx.x, lane = g & 31, wid = g >> 5;
  int n = 0;
  if (g < G) {
    const int lo = clamp_rows(__ldg(offsets + g), M);
    const int hi = clamp_rows(__ldg(offsets + g + 1), M);
    n = (max(hi - lo, 0) + 127) / 128;
  }
  int v = n;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, v, off);
    if (lane >= off) v += o;
  }
  if (lane == 31) warp_tot[wid] = v;
  __syncthreads();
  if (wid == 0) {
    int wv = warp_tot[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, wv, off);
      if (lane >= off) wv += o;
    }
    warp_tot[lane] = wv;
  }
  __syncthreads();
  if (g < G) tile_base[g + 1] = v + (wid ? warp_tot[wid - 1] : 0);
  if (g == 0) tile_base[0] = 0;
}

// One block of 128 threads per (tile, four k-steps): thread m stages row m's
// 16 scale bytes of those k-steps in shared memory, then thread u writes the
// 16 bytes of lane u % 32 for k-step u / 32.  ld = K/16 bytes per row, a
// multiple of 16.
template <int MODE>
__global__ void __launch_bounds__(128) sf_retile_kernel(const uint8_t* __restrict__ sf, int ld, int ks,
                                                        const int32_t* __restrict__ offsets,
                                                        const int32_t* __restrict__ tile_base, int G, int M, int N,
                                                        uint8_t* __restrict__ out) {
  __shared__ uint32_t s[128][5];  // one pad word: the lane-strided reads below hit distinct banks
  const int tile = blockIdx.x;
  const int c = blockIdx.y;  // k-steps 4c .. 4c+3
  const int m = threadIdx.x;
  long long row = 0;
  bool valid = false;
  if (MODE == kModeRows) {
    if (tile >= __ldg(tile_base + G)) return;  // past the last tile (the grid is an upper bound)
    int lo = 0, hi = G;                         // last g with tile_base[g] <= tile
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(tile_base + mid) <= tile) lo = mid; else hi = mid;
    }
    const int r0 = clamp_rows(__ldg(offsets + lo), M);
    const int rows = max(clamp_rows(__ldg(offsets + lo + 1), M) - r0, 0);
    const int i = (tile - __ldg(tile_base + lo)) * 128 + m;
    valid = i < rows;
    row = static_cast<long long>(r0) + i;
  } else if (MODE == kModeStore) {
    const int nb = (N + 127) / 128;
    const int g = tile / nb, n = tile - g * nb;
    valid = n * 128 + m < N;
    row = static_cast<long long>(g) * N + n * 128 + m;
  } else {
    const int nb = (N + 63) / 64;
    const int g = tile / nb, n = tile - g * nb;
    const int f = n * 64 + (m & 63);  // feature
    valid = f < N;
    row = static_cast<long long>(g) * 2 * N + (m < 64 ? 0 : N) + f;
  }
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (valid) v = __ldg(reinterpret_cast<const uint4*>(sf + row * ld + 16 * c));
  s[m][0] = v.x;
  s[m][1] = v.y;
  s[m][2] = v.z;
  s[m][3] = v.w;
  __syncthreads();
  const int kk = m >> 5, l = m & 31;
  const uint4 o = make_uint4(s[l][kk], s[l + 32][kk], s[l + 64][kk], s[l + 96][kk]);
  const size_t blk = static_cast<size_t>(tile) * ks + 4 * c + kk;
  reinterpret_cast<uint4*>(out)[blk * 32 + l] = o;
}

}  // namespace

size_t sf_tiles_bytes_rows(int M, int G, int K) {
  const size_t tiles = static_cast<size_t>((M + 127) / 128) + static_cast<size_t>(G);
  return tiles * static_cast<size_t>(K) * 8;
}

int sf_tile_base_launch(const int32_t* offsets, int G, int M, int32_t* tile_base, cudaStream_t s) {
  sf_tile_base_kernel<<<1, 1024, 0, s>>>(offsets, G, M, tile_base);
  return check_launch();
}

int sf_retile_rows_launch(const uint8_t* sf, int M, int K, const int32_t* offsets, const int32_t* tile_base, int G,
                          uint8_t* tiled, cudaStream_t s) {
  const long long tiles = (M + 127) / 128 + static_cast<long long>(G);
  if (M == 0) return MOE_OK;
  if (tiles > 0x7FFFFFFFLL) return MOE_ERR_UNSUPPORTED;
  const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(K / 256));
  sf_retile_kernel<kModeRows><<<grid, 128, 0, s>>>(sf, K / 16, K / 64, offsets, tile_base, G, M, 0, tiled);
  return check_launch();
}

int sf_retile_weights_launch(const uint8_t* sf, int G, int N, int K, bool swiglu, uint8_t* tiled, cudaStream_t s) {
  const long long nb = swiglu ? (N + 63) / 64 : (N + 127) / 128;
  const long long tiles = nb * G;
  if (tiles > 0x7FFFFFFFLL) return MOE_ERR_UNSUPPORTED;
  const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(K / 256));
  if (swiglu)
    sf_retile_kernel<kModeSwiglu><<<grid, 128, 0, s>>>(sf, K / 16, K / 64, nullptr, nullptr, G, 0, N, tiled);
  else
    sf_retile_kernel<kModeStore><<<grid, 128, 0, s>>>(sf, K / 16, K / 64, nullptr, nullptr, G, 0, N, tiled);
  return check_launch();
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_sf_tiles_size(int M_total, int G, int K) {
  if (M_total < 0 || G < 1 || K <= 0 || K % 256 != 0) return 0;
  return sf_tiles_bytes_rows(M_total, G, K);
}

extern "C" size_t moe_sf_tiles_size_weights(int G, int N, int K, int swiglu) {
  if (G < 1 || N <= 0 || K <= 0 || K % 256 != 0) return 0;
  const size_t nb = swiglu ? static_cast<size_t>((N + 63) / 64) : static_cast<size_t>((N + 127) / 128);
  return static_cast<size_t>(G) * nb * static_cast<size_t>(K) * 8;
}

extern "C" int moe_sf_tile_bases(const int32_t* offsets, int G, int M_total, int32_t* tile_base, void* stream) {
  if (G < 1 || M_total < 0 || !offsets || !tile_base) return MOE_ERR_INVALID_ARG;
  if (G > 1024) return MOE_ERR_UNSUPPORTED;
  if (!aligned(offsets, 4) || !aligned(tile_base, 4)) return MOE_ERR_INVALID_ARG;
  return sf_tile_base_launch(offsets, G, M_total, tile_base, static_cast<cudaStream_t>(stream));
}

extern "C" int moe_sf_retile_rows(const uint8_t* sf, int M_total, int K, const int32_t* offsets,
                                  const int32_t* tile_base, int G, uint8_t* tiled, void* stream) {
  if (M_total < 0 || K <= 0 || G < 1) return MOE_ERR_INVALID_ARG;
  if (K % 256 != 0 || G > 1024) return MOE_ERR_UNSUPPORTED;
  if (M_total == 0) return MOE_OK;
  if (!sf || !offsets || !tile_base || !tiled) return MOE_ERR_INVALID_ARG;
  if (!aligned(sf, 16) || !aligned(tiled, 16) || !aligned(offsets, 4) || !aligned(tile_base, 4))
    return MOE_ERR_INVALID_ARG;
  return sf_retile_rows_launch(sf, M_total, K, offsets, tile_base, G, tiled, static_cast<cudaStream_t>(stream));
}

extern "C" int moe_sf_retile_weights(const uint8_t* sf, int G, int N, int K, int swiglu, uint8_t* tiled,
                                     void* stream) {
  if (G < 1 || N <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (K % 256 != 0) return MOE_ERR_UNSUPPORTED;
  if (!sf || !tiled) return MOE_ERR_INVALID_ARG;
  if (!aligned(sf, 16) || !aligned(tiled, 16)) return MOE_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(G) * (swiglu ? 2LL * N : N);
  if (rows >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  return sf_retile_weights_launch(sf, G, N, K, swiglu != 0, tiled, static_cast<cudaStream_t>(stream));
}
