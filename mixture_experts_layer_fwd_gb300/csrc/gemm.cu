// Persistent grouped GEMM for the expert projections on sm_103a.
//
// "Hosting Qwen on Blackwell", section "MoE GEMM": every expert multiplies its
// group of routed tokens by its weights; dense at prefill (hundreds of tokens
// per expert), weight-load bound at decode (section "Decodificadores").
// "Driving vLLM WideEP ... (Part I)", section "NVFP4 GEMM for MoE and
// O-proj": NVFP4 weights (packed 4-bit values + per-group FP8 scales) are
// dequantised on the fly inside the GEMM.
//
// Design (one CTA per SM, warp-specialised):
//   warp 0      TMA producer: A tile 128 rows x 64 K (bf16, 128-byte swizzle)
//               and B tile 256 rows x 64 K per pipeline stage, mbarrier
//               complete_tx; NVFP4 operands arrive as packed codes instead
//   warp 1      TMEM allocator and MMA issuer: tcgen05.mma kind::f16,
//               M=128 N=256 K=16, fp32 accumulators in tensor memory, two
//               accumulator buffers of 256 columns (epilogue of tile i
//               overlaps the main loop of tile i+1)
//   warps 2..5  epilogue: tcgen05.ld of the accumulators, SwiGLU / scaling /
//               bf16 or NVFP4 rounding, stores of the rows of the tile that
//               belong to the tile's group
//   warps 6..13 (NVFP4 operands only) converters, one operand row per thread:
//               packed E2M1 codes x E4M3 scale -> bf16 into the swizzled
//               operand tile, through a byte -> bf16x2 table replicated per
//               lane (conflict-free lookups).  e2m1 * e4m3 is exact in bf16,
//               so the bf16 MMA computes exactly the NVFP4 products; the fp32
//               global scales are applied in the epilogue
//   warp 14     (NVFP4 operands only) scale loader: cp.async of each stage's
//               E4M3 scale words into a small ring, tracked by an mbarrier
// Tiles are (group, n-block, m-block) with m fastest; group sizes are read
// on the device (offsets), so nothing is synchronised with the host.
// The SwiGLU epilogue needs gate and up of the same feature in one thread:
// the B tile holds 128 gate rows followed by the matching 128 up rows, so
// accumulator columns [0,128) are gate and [128,256) are up.
#include <cstring>

#include "gemm_common.cuh"
#include "internal.h"

namespace moe {
namespace gg {

constexpr int BN = 256;
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int TMEM_COLS = 512;
constexpr int A_TILE = BM * BK * 2;   // 16 KB bf16
constexpr int B_TILE = BN * BK * 2;   // 32 KB bf16
constexpr int A_CODES = BM * BK / 2;  // 4 KB packed E2M1
constexpr int B_CODES = BN * BK / 2;  // 8 KB packed E2M1
template <int EPI, bool A4, bool W4>
struct Cfg {
  static constexpr bool CONV = A4 || W4;
  static constexpr int STAGES = CONV ? 3 : 4;
  static constexpr int STAGE_BYTES = A_TILE + B_TILE + (A4 ? A_CODES : 0) + (W4 ? B_CODES : 0);
  static constexpr int CONV_WARPS = 8;  // converters: warps 6..13, one operand row per thread
  static constexpr int SF_WARP = 6 + CONV_WARPS;
  static constexpr int NUM_WARPS = CONV ? SF_WARP + 1 : 6;  // + scale loader
  static constexpr int THREADS = NUM_WARPS * 32;
  static constexpr int TILE_N = (EPI == MOE_EPI_STORE_BF16) ? 256 : 128;  // output columns per tile
  static constexpr uint32_t TX_BYTES = (A4 ? A_CODES : A_TILE) + (W4 ? B_CODES : B_TILE);
  static constexpr int SF_RING_WORDS = 384;  // per stage: 128 A rows + 256 B rows, one 32-bit word each
  // byte -> two bf16 table, one copy per lane (lut[byte][lane]): lookups with
  // random bytes never collide on a bank
  static constexpr int LUT_WORDS = CONV ? 256 * 32 : 0;
  static constexpr int EXTRA =
      2048 + 4 * (2 * MAX_G + 8) + 4 * LUT_WORDS + (CONV ? STAGES * SF_RING_WORDS * 4 : 0);
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + EXTRA;
  static_assert(STAGE_BYTES % 1024 == 0, "stage must keep 1024-byte alignment");
  static_assert(SMEM <= 232448, "shared memory budget");
};

// Converts one 64-element row of packed E2M1 codes (32 bytes in smem) with
// its four E4M3 block scales into bf16, written into a 128-byte swizzled row.
DEVINL void convert_row(const uint8_t* codes, uint32_t sfw, uint8_t* tile, int row, const uint32_t* lut_lane) {
  const uint4 c0 = *reinterpret_cast<const uint4*>(codes);
  const uint4 c1 = *reinterpret_cast<const uint4*>(codes + 16);
  const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    const float sc = e4m3_decode((sfw >> (8 * (ch >> 1))) & 0xFFu);
    const __nv_bfloat162 s2 = __float2bfloat162_rn(sc);
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t lv = lut_lane[((cw[ch] >> (8 * q)) & 0xFFu) * 32];
      __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&lv);
      v = __hmul2(v, s2);
      o[q] = *reinterpret_cast<uint32_t*>(&v);
    }
    *reinterpret_cast<uint4*>(tile + row * 128 + ((ch ^ (row & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

template <int EPI, bool A4, bool W4>
__global__ void __launch_bounds__(Cfg<EPI, A4, W4>::THREADS, 1) grouped_gemm_kernel(const __grid_constant__ Params p) {
  using C = Cfg<EPI, A4, W4>;
  constexpr int S = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = base;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + S * C::STAGE_BYTES);
  uint64_t* empty = full + S;
  uint64_t* conv = empty + S;
  uint64_t* sf_full = conv + S;
  uint64_t* tfull = sf_full + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_prefix = reinterpret_cast<int*>(base + S * C::STAGE_BYTES + 256);
  int* s_off = s_prefix + MAX_G + 4;
  uint32_t* lut = reinterpret_cast<uint32_t*>(s_off + MAX_G + 4);
  uint32_t* sf_ring = lut + C::LUT_WORDS;  // [S][SF_RING_WORDS] E4M3 scale words of each stage
  __shared__ int warp_sums[32];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.G;
  const int GT = G + (p.shared_rows >= 0 ? 1 : 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&conv[s], C::CONV_WARPS * 32);
      mbar_init(&sf_full[s], 32);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  if (C::CONV) {
    for (int i = threadIdx.x; i < C::LUT_WORDS; i += C::THREADS) {
      const uint32_t b = static_cast<uint32_t>(i) >> 5;
      lut[i] = e2m1_to_bf16_bits(b & 15u) | (e2m1_to_bf16_bits(b >> 4) << 16);
    }
  }
  // ---- tile schedule: prefix over per-group tile counts
  build_schedule<C::THREADS, C::NUM_WARPS>(p, s_off, s_prefix, warp_sums);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int total = s_prefix[GT];
  const unsigned long long tmo = p.timeout_ns;

  if (warp == 0) {
    // ===================================================== TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tma_a[0]);
      tma_prefetch_desc(&p.tma_w[0]);
      if (p.shared_rows >= 0) {
        tma_prefetch_desc(&p.tma_a[1]);
        tma_prefetch_desc(&p.tma_w[1]);
      }
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued[S];
#pragma unroll
      for (int s = 0; s < S; ++s) issued[s] = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const TileInfo ti = decode_tile(t, s_prefix, s_off, GT, G, p.shared_rows);
        const Prob& P = p.prob[ti.pb];
        const void* ta = &p.tma_a[ti.pb];
        const void* tw = &p.tma_w[ti.pb];
        const int a_y = ti.row0 + ti.m_blk * BM;
        const int w_y0 = ti.g * P.w_rows + ti.n_blk * C::TILE_N;
        const int w_y1 = (EPI == MOE_EPI_STORE_BF16) ? w_y0 + 128 : w_y0 + P.n_out;
        const int nk = P.K / BK;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, tmo, p.err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sb = stages + stage * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], C::TX_BYTES);
          if (A4)
            tma_load_2d(ta, &full[stage], sb + A_TILE + B_TILE, kb * (BK / 2), a_y);
          else
            tma_load_2d(ta, &full[stage], sb, kb * BK, a_y);
          if (W4) {
            uint8_t* wc = sb + A_TILE + B_TILE + (A4 ? A_CODES : 0);
            tma_load_2d(tw, &full[stage], wc, kb * (BK / 2), w_y0);
            tma_load_2d(tw, &full[stage], wc + B_CODES / 2, kb * (BK / 2), w_y1);
          } else {
            tma_load_2d(tw, &full[stage], sb + A_TILE, kb * BK, w_y0);
            tma_load_2d(tw, &full[stage], sb + A_TILE + B_TILE / 2, kb * BK, w_y1);
          }
          issued[stage] += 1;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // let every copy already in flight land before the block exits
        for (int s = 0; s < S; ++s)
          if (issued[s]) mbar_wait_bounded(&full[s], (issued[s] - 1u) & 1u, 1000000000ull, p.err, nullptr);
      }
    }
  } else if (warp == 1) {
    // ===================================================== MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
        const TileInfo ti = decode_tile(t, s_prefix, s_off, GT, G, p.shared_rows);
        const int nk = p.prob[ti.pb].K / BK;
        const int buf = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        if (!mbar_wait_bounded(&tempty[buf], (use & 1u) ^ 1u, tmo, p.err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(C::CONV ? &conv[stage] : &full[stage], phase, tmo, p.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stages + stage * C::STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_TILE;
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            umma_f16(d, smem_desc_kmajor_sw128(a_addr + kk * 32), smem_desc_kmajor_sw128(b_addr + kk * 32), IDESC,
                     (kb | kk) ? 1u : 0u);
          }
          umma_commit(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit(&tfull[buf]);
      }
      if (!ok) {
        umma_commit(drain);
        mbar_wait_bounded(drain, 0, 1000000000ull, p.err, nullptr);
      }
    }
  } else if (warp < 6) {
    // ===================================================== epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int r_in_tile = q * 32 + lane;
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      const TileInfo ti = decode_tile(t, s_prefix, s_off, GT, G, p.shared_rows);
      const Prob& P = p.prob[ti.pb];
      const int buf = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      if (!mbar_wait_warp(&tfull[buf], use & 1u, tmo, p.err, abort_flag)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * BN);
      float scale = 1.0f;
      if (A4) scale *= __ldg(P.a_g);
      if (W4) scale *= __ldg(P.w_g + ti.g);
      epilogue_tile<EPI, BN>(P, ti, taddr, r_in_tile, scale);
      tc_fence_before();
      mbar_arrive(&tempty[buf]);
    }
  } else if (C::CONV && warp < C::SF_WARP) {
    // ===================================================== NVFP4 -> bf16 converters
    const int ct = threadIdx.x - 6 * 32;  // 0..255: one B row (and, below 128, one A row)
    const uint32_t* lut_lane = lut + lane;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const TileInfo ti = decode_tile(t, s_prefix, s_off, GT, G, p.shared_rows);
      const int nk = p.prob[ti.pb].K / BK;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait_warp(&full[stage], phase, tmo, p.err, abort_flag) ||
            !mbar_wait_warp(&sf_full[stage], phase, tmo, p.err, abort_flag)) {
          ok = false;
          break;
        }
        uint8_t* sb = stages + stage * C::STAGE_BYTES;
        const uint32_t* sfw = sf_ring + stage * C::SF_RING_WORDS;
        if (A4 && ct < BM) convert_row(sb + A_TILE + B_TILE + ct * 32, sfw[ct], sb, ct, lut_lane);
        if (W4) {
          const uint8_t* wc = sb + A_TILE + B_TILE + (A4 ? A_CODES : 0);
          convert_row(wc + ct * 32, sfw[128 + ct], sb + A_TILE, ct, lut_lane);
        }
        fence_proxy_async_smem();
        mbar_arrive(&conv[stage]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (C::CONV) {
    // ===================================================== scale loader (warp SF_WARP)
    // Asynchronous 4-byte copies of each stage's E4M3 scale words (one word =
    // the 4 block scales of a row over the stage's 64 elements) into the
    // stage's ring slot; each lane's copies arrive on sf_full when they land,
    // so several stages of scales are in flight while the converters work.
    int stage = 0;
    uint32_t phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const TileInfo ti = decode_tile(t, s_prefix, s_off, GT, G, p.shared_rows);
      const Prob& P = p.prob[ti.pb];
      const int a_y = ti.row0 + ti.m_blk * BM;
      const int w_y0 = ti.g * P.w_rows + ti.n_blk * C::TILE_N;
      const int w_y1 = (EPI == MOE_EPI_STORE_BF16) ? w_y0 + 128 : w_y0 + P.n_out;
      const int nk = P.K / BK;
      const int sf_ld = P.K / 16;
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait_warp(&empty[stage], phase ^ 1u, tmo, p.err, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t ring = smem_u32(sf_ring + stage * C::SF_RING_WORDS);
        if (A4) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = lane + 32 * i;
            const int grow = a_y + r;
            const bool v = grow < P.a_rows;
            cp_async_4(ring + 4 * r, v ? P.a_sf + static_cast<size_t>(grow) * sf_ld + kb * 4 : P.a_sf, v);
          }
        }
        if (W4) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = lane + 32 * i;
            const int grow = (r < 128) ? w_y0 + r : w_y1 + (r - 128);
            const bool v = grow < P.w_rows_total;
            cp_async_4(ring + 4 * (128 + r), v ? P.w_sf + static_cast<size_t>(grow) * sf_ld + kb * 4 : P.w_sf, v);
          }
        }
        cp_async_mbar_arrive(&sf_full[stage]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
    }
    cp_async_wait_group<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host
// 2-D tensor map over a row-major [rows, inner] matrix: bf16 with the
// 128-byte swizzle, or packed E2M1 bytes without swizzle (converter path).
static int make_map(CUtensorMap* m, const void* ptr, bool bf16, uint64_t inner, uint64_t rows, uint32_t box_inner,
                    uint32_t box_rows) {
  return encode_tmap_2d(m, ptr, bf16 ? 2 : 1, inner, rows, box_inner, box_rows, bf16);
}

}  // namespace gg

template <int EPI, bool A4, bool W4>
static int launch_impl(const gg::Params& prm, cudaStream_t s) {
  using C = gg::Cfg<EPI, A4, W4>;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gg::grouped_gemm_kernel<EPI, A4, W4>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) {
      set_cuda_error(e);
      return MOE_ERR_CUDA;
    }
    attr_done[dev] = true;
  }
  gg::grouped_gemm_kernel<EPI, A4, W4><<<num_sms(), C::THREADS, C::SMEM, s>>>(prm);
  return check_launch();
}

static int fill_prob(gg::Params& prm, int slot, int epi, bool a4, bool w4, const GemmProblem& P) {
  gg::Prob& q = prm.prob[slot];
  const int tile_n = (epi == MOE_EPI_STORE_BF16) ? 256 : 128;
  q.n_out = P.N;
  q.K = P.K;
  q.w_rows = (epi == MOE_EPI_STORE_BF16) ? P.N : 2 * P.N;
  q.n_tiles = (P.N + tile_n - 1) / tile_n;
  q.a_rows = P.a_rows;
  q.w_rows_total = P.groups * q.w_rows;
  q.c = P.C;
  q.c_sf = P.C_sf;
  q.a_g = P.A_g;
  q.w_g = P.W_g;
  q.c_g = P.c_g;
  q.a_sf = P.A_sf;
  q.w_sf = P.W_sf;
  MOE_TRY(gg::make_map(&prm.tma_a[slot], P.A, !a4, a4 ? P.K / 2 : P.K, static_cast<uint64_t>(P.a_rows),
                       a4 ? gg::BK / 2 : gg::BK, gg::BM));
  MOE_TRY(gg::make_map(&prm.tma_w[slot], P.W, !w4, w4 ? P.K / 2 : P.K, static_cast<uint64_t>(q.w_rows_total),
                       w4 ? gg::BK / 2 : gg::BK, 128));
  return MOE_OK;
}

static int check_problem(int epi, bool a4, bool w4, const GemmProblem& P) {
  if (P.N <= 0 || P.K <= 0 || P.a_rows < 0 || P.groups < 1) return MOE_ERR_INVALID_ARG;
  if (P.K % 64 != 0 || P.N % 32 != 0) return MOE_ERR_UNSUPPORTED;
  if (!P.A || !P.W || !P.C) return MOE_ERR_INVALID_ARG;
  if (!aligned(P.A, 16) || !aligned(P.W, 16) || !aligned(P.C, 16)) return MOE_ERR_INVALID_ARG;
  if (a4 && (!P.A_sf || !P.A_g || !aligned(P.A_sf, 4))) return MOE_ERR_INVALID_ARG;
  if (w4 && (!P.W_sf || !P.W_g || !aligned(P.W_sf, 4))) return MOE_ERR_INVALID_ARG;
  if (epi == MOE_EPI_SWIGLU_NVFP4 && (!P.C_sf || !P.c_g || !aligned(P.C_sf, 2))) return MOE_ERR_INVALID_ARG;
  if (P.a_f16 && (a4 || !w4)) return MOE_ERR_UNSUPPORTED;
  const long long w_rows = static_cast<long long>(P.groups) * ((epi == MOE_EPI_STORE_BF16) ? P.N : 2 * P.N);
  if (w_rows >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// Launches one persistent grouped GEMM over the routed problem (G groups,
// device offsets) plus, when `sh` is non-null, the shared-expert problem as
// one more group of `shared_rows` rows.
// MX operands: E2M1 codes (MXFP4) or E4M3 bytes (MXFP8) with one E8M0 scale
// per 32 elements, no global scales.  The MXFP4 kernel stages 16 scale bytes
// per row by TMA (K % 512, 16-byte aligned scales); the MXFP8 kernel loads 8
// per row directly (K % 256, 8-byte aligned scales).
static int check_problem_mx(const GemmProblem& P, bool fp8, bool mx_out) {
  if (P.N <= 0 || P.K <= 0 || P.a_rows < 0 || P.groups < 1) return MOE_ERR_INVALID_ARG;
  if (P.K % (fp8 ? 256 : 512) != 0 || P.N % 32 != 0) return MOE_ERR_UNSUPPORTED;
  if (!P.A || !P.W || !P.C || !P.A_sf || !P.W_sf) return MOE_ERR_INVALID_ARG;
  if (mx_out && !P.C_sf) return MOE_ERR_INVALID_ARG;
  const int sfa = fp8 ? 8 : 16;
  if (!aligned(P.A, 16) || !aligned(P.W, 16) || !aligned(P.C, 16) || !aligned(P.A_sf, sfa) || !aligned(P.W_sf, sfa))
    return MOE_ERR_INVALID_ARG;
  if (static_cast<long long>(P.groups) * 2 * P.N >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int grouped_gemm_launch(int epi, int a_fmt, int w_fmt, const GemmProblem& routed, const int32_t* offsets, int G,
                        const GemmProblem* sh, int shared_rows, cudaStream_t s) {
  const bool a4 = a_fmt == MOE_FMT_NVFP4, w4 = w_fmt == MOE_FMT_NVFP4;
  if (G < 1 || G > gg::MAX_G - 1 || !offsets) return MOE_ERR_INVALID_ARG;
  const bool mx8 = a_fmt == MOE_FMT_MXFP8 || w_fmt == MOE_FMT_MXFP8;
  if (mx8 || a_fmt == MOE_FMT_MXFP4 || w_fmt == MOE_FMT_MXFP4) {
    if (a_fmt != w_fmt) return MOE_ERR_UNSUPPORTED;
    if (epi != MOE_EPI_STORE_BF16 && epi != MOE_EPI_SWIGLU_BF16 && epi != MOE_EPI_SWIGLU_MX)
      return MOE_ERR_UNSUPPORTED;
    MOE_TRY(check_problem_mx(routed, mx8, epi == MOE_EPI_SWIGLU_MX));
    if (sh) MOE_TRY(check_problem_mx(*sh, mx8, epi == MOE_EPI_SWIGLU_MX));
    if (routed.a_rows == 0) return MOE_OK;
    if (mx8) return grouped_gemm_launch_mxf8_pair(epi, routed, offsets, G, sh, shared_rows, s);
    return grouped_gemm_launch_mxf4(epi, routed, offsets, G, sh, shared_rows, s);
  }
  if (epi == MOE_EPI_SWIGLU_MX) return MOE_ERR_UNSUPPORTED;  // MX operands only
  if ((epi < MOE_EPI_STORE_BF16 || epi > MOE_EPI_SWIGLU_NVFP4) && epi != kEpiSwigluF16) return MOE_ERR_INVALID_ARG;
  if (a4 && !w4) return MOE_ERR_UNSUPPORTED;
  if (epi == kEpiSwigluF16 && (a4 || !w4)) return MOE_ERR_UNSUPPORTED;
  if (epi == MOE_EPI_SWIGLU_NVFP4 && !(a4 && w4)) return MOE_ERR_UNSUPPORTED;
  MOE_TRY(check_problem(epi, a4, w4, routed));
  if (sh) MOE_TRY(check_problem(epi, a4, w4, *sh));
  // routed rows are T*k >= T shared rows, so an empty routed problem means
  // there is nothing to do
  if (routed.a_rows == 0) return MOE_OK;
  if (a4 && w4) return grouped_gemm_launch_nvf4(epi, routed, offsets, G, sh, shared_rows, s);
  if (!a4 && !w4) return grouped_gemm_launch_pair(epi, routed, offsets, G, sh, shared_rows, s);
  const bool have_shared = sh != nullptr && shared_rows > 0;
  // bf16 x NVFP4 weights: the tensor-memory kernel when the weight scale rows
  // are whole 16-byte slices per 256-element stage; fp16 inputs and the fp16
  // epilogue exist only there
  if (routed.K % 256 == 0 && aligned(routed.W_sf, 16) &&
      (!have_shared || (sh->K % 256 == 0 && aligned(sh->W_sf, 16))))
    return grouped_gemm_launch_w4a16(epi, routed, offsets, G, sh, shared_rows, s);
  if (epi == kEpiSwigluF16 || routed.a_f16 || (have_shared && sh->a_f16)) return MOE_ERR_UNSUPPORTED;
  gg::Params prm;
  memset(&prm, 0, sizeof(prm));
  MOE_TRY(fill_prob(prm, 0, epi, a4, w4, routed));
  prm.offsets = offsets;
  prm.G = G;
  prm.shared_rows = -1;
  if (have_shared) {
    MOE_TRY(fill_prob(prm, 1, epi, a4, w4, *sh));
    prm.shared_rows = shared_rows;
  }
  prm.err = device_error_word();
  if (!prm.err) return MOE_ERR_CUDA;
  prm.timeout_ns = wait_timeout_ns();
  // bf16 x bf16 went to the CTA-pair kernel and NVFP4 x NVFP4 to the
  // block-scaled kernel above; this kernel serves NVFP4 weights with bf16
  // activations (converted to bf16 in shared memory)
  if (!a4 && w4) {
    if (epi == MOE_EPI_STORE_BF16) return launch_impl<MOE_EPI_STORE_BF16, false, true>(prm, s);
    if (epi == MOE_EPI_SWIGLU_BF16) return launch_impl<MOE_EPI_SWIGLU_BF16, false, true>(prm, s);
  }
  return MOE_ERR_UNSUPPORTED;
}

}  // namespace moe

using namespace moe;

extern "C" int moe_grouped_gemm(int a_fmt, int w_fmt, int epilogue, int G, const int32_t* offsets, int M_total, int N,
                                int K, const void* A, const uint8_t* A_sf, const float* A_g, const void* W,
                                const uint8_t* W_sf, const float* W_g, void* C, uint8_t* C_sf, const float* c_g,
                                void* stream) {
  if (M_total < 0) return MOE_ERR_INVALID_ARG;
  if (epilogue < MOE_EPI_STORE_BF16 || epilogue > MOE_EPI_SWIGLU_MX) return MOE_ERR_INVALID_ARG;
  if (M_total == 0) return MOE_OK;
  GemmProblem P{A, A_sf, A_g, M_total, W, W_sf, W_g, G, C, C_sf, c_g, N, K};
  return grouped_gemm_launch(epilogue, a_fmt, w_fmt, P, offsets, G, nullptr, 0, static_cast<cudaStream_t>(stream));
}
