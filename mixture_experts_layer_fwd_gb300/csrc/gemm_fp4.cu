// Grouped GEMM with both operands in NVFP4, on the block-scaled FP4 tensor
// cores of sm_103a (tcgen05.mma kind::mxf4nvf4, block_scale, scale_vec::4X).
//
// "Driving vLLM WideEP ... (Part I)", section "NVFP4 GEMM for MoE and
// O-proj": the weights are packed 4-bit values with per-group FP8 scales,
// dequantised inside the tensor cores; section "NVFP4 MoE dispatch": the
// activations are quantised to FP4 before dispatch, so both GEMM operands
// arrive in NVFP4.
//
// This kernel serves the shapes the 512-element-stage kernel (gemm_fp4w.cu)
// cannot: K % 256 != 0 or scale arrays not 16-byte aligned, where the scale
// rows are not whole 16-byte slices and cannot travel by TMA.
//
// Design (one CTA per SM, warp-specialised), per pipeline stage of K = 256:
//   warp 0      TMA: A tile 128 rows x 128 bytes (256 E2M1), B tile 128 rows x
//               128 bytes, both with the 128-byte swizzle
//   warp 6      scale loader: 4-byte asynchronous copies (cp.async) of the
//               E4M3 scale words of the stage's A and B rows straight into
//               four 512-byte blocks per operand, one per MMA of K = 64: row
//               r's 4 scales go to byte 16*(r % 32) + 4*(r / 32)
//   warp 1      MMA issuer: tcgen05.cp (32x128b, replicated to the four lane
//               quadrants) moves each scale block into tensor memory, then 4
//               block-scaled MMAs M=128 N=128 K=64 accumulate in fp32 in
//               tensor memory (two 128-column accumulator buffers, a scale
//               ring of 32 columns per stage after them)
//   warps 2..5  epilogue (shared with the bf16 kernel): global scales
//               g_a * g_w[e], SwiGLU, bf16 or NVFP4 output
// For SwiGLU the B tile holds 64 gate rows and the matching 64 up rows.
#include <cstring>

#include "gemm_common.cuh"
#include "internal.h"

namespace moe {
namespace gg4 {

using gg::BM;
using gg::MAX_G;
using gg::Params;
using gg::Prob;
using gg::TileInfo;

constexpr int BN = 128;                // MMA N = accumulator columns per tile
constexpr int ROW_BYTES = 128;         // packed E2M1 bytes per row per stage (256 elements)
constexpr int KE = 2 * ROW_BYTES;      // elements per stage
constexpr int A_TILE = BM * ROW_BYTES; // 16 KB
constexpr int B_TILE = BN * ROW_BYTES; // 16 KB
constexpr int SF_TILE = 4 * 512;       // 4 scale blocks of 32 x 16 bytes
constexpr int STAGES = 5;
// per stage: A codes | B codes | A scale blocks | B scale blocks
constexpr int STAGE_BYTES = A_TILE + B_TILE + 2 * SF_TILE;
constexpr int OFF_SFA = A_TILE + B_TILE;
constexpr int OFF_SFB = OFF_SFA + SF_TILE;
constexpr int NUM_WARPS = 7;
constexpr int THREADS = NUM_WARPS * 32;
constexpr int TMEM_COLS = 512;
constexpr int ACC_COLS = 2 * BN;
constexpr int SF_COLS = 32;            // per stage: 16 (A) + 16 (B)
constexpr uint32_t TX_BYTES = A_TILE + B_TILE;
constexpr int EXTRA = 2048 + 4 * (2 * MAX_G + 8);
constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + EXTRA;
static_assert(STAGE_BYTES % 1024 == 0, "stage must keep 1024-byte alignment");
static_assert(ACC_COLS + STAGES * SF_COLS <= TMEM_COLS, "tensor memory budget");
static_assert(SMEM <= 232448, "shared memory budget");

template <int EPI>
struct Tile {
  static constexpr int N_OUT = (EPI == MOE_EPI_STORE_BF16) ? BN : BN / 2;  // output columns per tile
};

// Scale stages in flight before the loader signals the oldest one.
constexpr int SF_LAG = 3;
static_assert(SF_LAG < STAGES, "the loader must signal a stage before it needs that stage back");

// Issues the asynchronous copies of the 32-bit scale words (4 E4M3 bytes =
// one K = 64 MMA) of rows lane + 32 j, j = 0..3, for stage kb, straight into
// the scale-block layout: word (row r, MMA kk) -> byte kk*512 + 16*(r % 32) +
// 4*(r / 32).  Words past the end of K or rows outside the matrix are zero.
DEVINL void load_scale_rows_async(const uint8_t* sf, int sf_ld, int kb, const int (&rows)[4],
                                  const bool (&valid)[4], uint32_t dst, int lane) {
  const int words = sf_ld >> 2;  // scale words per row
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const int wi = kb * 4 + kk;
      const bool ok = valid[j] && wi < words;
      const uint8_t* src = ok ? sf + static_cast<size_t>(rows[j]) * sf_ld + 4 * wi : sf;
      cp_async_4(dst + kk * 512 + lane * 16 + j * 4, src, ok);
    }
  }
}

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1) grouped_gemm_nvf4_kernel(const __grid_constant__ Params p) {
  constexpr int S = STAGES;
  constexpr int TN = Tile<EPI>::N_OUT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = base;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + S * STAGE_BYTES);
  uint64_t* sf_full = full + S;
  uint64_t* empty = sf_full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_prefix = reinterpret_cast<int*>(base + S * STAGE_BYTES + 256);
  int* s_off = s_prefix + MAX_G + 4;
  __shared__ int warp_sums[32];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.G;
  const int GT = G + (p.shared_rows >= 0 ? 1 : 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&sf_full[s], 32);
      mbar_init(&empty[s], 1);
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
  gg::build_schedule<THREADS, NUM_WARPS>(p, s_off, s_prefix, warp_sums);
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
        const TileInfo ti = gg::decode_tile(t, s_prefix, s_off, GT, G, p.shared_rows);
        const Prob& P = p.prob[ti.pb];
        const void* ta = &p.tma_a[ti.pb];
        const void* tw = &p.tma_w[ti.pb];
        const int a_y = ti.row0 + ti.m_blk * BM;
        const int w_y0 = ti.g * P.w_rows + ti.n_blk * TN;
        const int w_y1 = (EPI == MOE_EPI_STORE_BF16) ? w_y0 + BN / 2 : w_y0 + P.n_out;
        const int nk = (P.K + KE - 1) / KE;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, tmo, p.err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sb = stages + stage * STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], TX_BYTES);
          tma_load_2d(ta, &full[stage], sb, kb * ROW_BYTES, a_y);
          tma_load_2d(tw, &full[stage], sb + A_TILE, kb * ROW_BYTES, w_y0);
          tma_load_2d(tw, &full[stage], sb + A_TILE + B_TILE / 2, kb * ROW_BYTES, w_y1);
          issued[stage] += 1;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < S; ++s)
          if (issued[s]) mbar_wait_bounded(&full[s], (issued[s] - 1u) & 1u, 1000000000ull, p.err, nullptr);
      }
    }
  } else if (warp == 6) {
    // ===================================================== scale loader
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    // Scale rows not 16-byte aligned (K % 256 != 0): per-word asynchronous
    // copies; a stage is signalled SF_LAG stages after its copies were issued
    // (after they completed and were fenced for the tensor cores' async
    // proxy), so several stages load concurrently.
    int issued = 0;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const TileInfo ti = gg::decode_tile(t, s_prefix, s_off, GT, G, p.shared_rows);
      const Prob& P = p.prob[ti.pb];
      const int a_y = ti.row0 + ti.m_blk * BM;
      const int w_y0 = ti.g * P.w_rows + ti.n_blk * TN;
      const int w_y1 = (EPI == MOE_EPI_STORE_BF16) ? w_y0 + BN / 2 : w_y0 + P.n_out;
      const int nk = (P.K + KE - 1) / KE;
      const int sf_ld = P.K / 16;
      int arow[4], brow[4];
      bool aval[4], bval[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = lane + 32 * j;  // row of the tile
        arow[j] = a_y + r;
        aval[j] = arow[j] < P.a_rows;
        brow[j] = (r < BN / 2) ? w_y0 + r : w_y1 + (r - BN / 2);
        bval[j] = brow[j] < P.w_rows_total;
      }
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait_warp(&empty[stage], phase ^ 1u, tmo, p.err, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t sb = smem_u32(stages + stage * STAGE_BYTES);
        load_scale_rows_async(P.a_sf, sf_ld, kb, arow, aval, sb + OFF_SFA, lane);
        load_scale_rows_async(P.w_sf, sf_ld, kb, brow, bval, sb + OFF_SFB, lane);
        cp_async_commit();
        cp_async_wait_group<SF_LAG>();  // every group but the SF_LAG newest has landed
        if (issued >= SF_LAG) {
          fence_proxy_async_smem();
          mbar_arrive(&sf_full[(issued - SF_LAG) % S]);
        }
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // signal the stages still outstanding, oldest first
    cp_async_wait_group<0>();
    fence_proxy_async_smem();
    for (int i = (issued > SF_LAG ? issued - SF_LAG : 0); i < issued; ++i) mbar_arrive(&sf_full[i % S]);
  } else if (warp == 1) {
    // ===================================================== MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_nvf4_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
        const TileInfo ti = gg::decode_tile(t, s_prefix, s_off, GT, G, p.shared_rows);
        const int nk = (p.prob[ti.pb].K + KE - 1) / KE;
        const int buf = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        if (!mbar_wait_bounded(&tempty[buf], (use & 1u) ^ 1u, tmo, p.err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, tmo, p.err, abort_flag) ||
              !mbar_wait_bounded(&sf_full[stage], phase, tmo, p.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stages + stage * STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_TILE;
          const uint32_t sfa_addr = b_addr + B_TILE;
          const uint32_t sfb_addr = sfa_addr + SF_TILE;
          const uint32_t sf_t = tmem_base + static_cast<uint32_t>(ACC_COLS + stage * SF_COLS);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            tmem_cp_32x128b_warpx4(sf_t + 4 * kk, smem_desc_kmajor_noswizzle_16B_rows(sfa_addr + 512 * kk));
            tmem_cp_32x128b_warpx4(sf_t + 16 + 4 * kk, smem_desc_kmajor_noswizzle_16B_rows(sfb_addr + 512 * kk));
          }
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            umma_nvf4(d, smem_desc_kmajor_sw128(a_addr + kk * 32), smem_desc_kmajor_sw128(b_addr + kk * 32), IDESC,
                      sf_t + 4 * kk, sf_t + 16 + 4 * kk, (kb | kk) ? 1u : 0u);
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
  } else {
    // ===================================================== epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int r_in_tile = q * 32 + lane;
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      const TileInfo ti = gg::decode_tile(t, s_prefix, s_off, GT, G, p.shared_rows);
      const Prob& P = p.prob[ti.pb];
      const int buf = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      if (!mbar_wait_warp(&tfull[buf], use & 1u, tmo, p.err, abort_flag)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * BN);
      const float scale = __ldg(P.a_g) * __ldg(P.w_g + ti.g);
      gg::epilogue_tile<EPI, BN>(P, ti, taddr, r_in_tile, scale);
      tc_fence_before();
      mbar_arrive(&tempty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int EPI>
static int launch(const Params& prm, cudaStream_t s) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(grouped_gemm_nvf4_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) {
      set_cuda_error(e);
      return MOE_ERR_CUDA;
    }
    attr_done[dev] = true;
  }
  grouped_gemm_nvf4_kernel<EPI><<<num_sms(), THREADS, SMEM, s>>>(prm);
  return check_launch();
}

static int fill(Params& prm, int slot, int epi, const GemmProblem& P) {
  Prob& q = prm.prob[slot];
  const int tn = (epi == MOE_EPI_STORE_BF16) ? BN : BN / 2;
  q.n_out = P.N;
  q.K = P.K;
  q.w_rows = (epi == MOE_EPI_STORE_BF16) ? P.N : 2 * P.N;
  q.n_tiles = (P.N + tn - 1) / tn;
  q.a_rows = P.a_rows;
  q.w_rows_total = P.groups * q.w_rows;
  q.c = P.C;
  q.c_sf = P.C_sf;
  q.a_g = P.A_g;
  q.w_g = P.W_g;
  q.c_g = P.c_g;
  q.a_sf = P.A_sf;
  q.w_sf = P.W_sf;
  MOE_TRY(encode_tmap_2d(&prm.tma_a[slot], P.A, 1, P.K / 2, static_cast<uint64_t>(P.a_rows), ROW_BYTES, BM, true));
  MOE_TRY(encode_tmap_2d(&prm.tma_w[slot], P.W, 1, P.K / 2, static_cast<uint64_t>(q.w_rows_total), ROW_BYTES,
                         BN / 2, true));
  return MOE_OK;
}

}  // namespace gg4

// Both operands NVFP4: the block-scaled FP4 tensor-core kernel.  Arguments
// were checked by grouped_gemm_launch.
// average routed rows per group from which the down projection takes the
// CTA-pair kernel
constexpr int kNvf4PairMinRows = 64;

int grouped_gemm_launch_nvf4(int epi, const GemmProblem& routed, const int32_t* offsets, int G,
                             const GemmProblem* sh, int shared_rows, cudaStream_t s) {
  gg::Params prm;
  memset(&prm, 0, sizeof(prm));
  const bool have_shared = sh != nullptr && shared_rows > 0;
  // scale rows can be fetched by TMA when every row is a whole number of
  // 16-byte stage slices (K % 256 == 0) and the scale arrays are 16-byte aligned
  const bool sf_tma = routed.K % 256 == 0 && aligned(routed.A_sf, 16) && aligned(routed.W_sf, 16) &&
                      (!have_shared || (sh->K % 256 == 0 && aligned(sh->A_sf, 16) && aligned(sh->W_sf, 16)));
  // The CTA-pair kernel (weights on M, tokens on N; whole 512-element
  // stages) for the down projection of prefill-sized groups, where it
  // measured faster (deepseek-v3 shapes, T = 16384: 1.88 against 2.16 ms);
  // the 1-SM kernel for the SwiGLU projection (2.73 against 3.15 ms) and for
  // decode-sized groups.
  const bool prefill = routed.a_rows >= kNvf4PairMinRows * G;
  if (sf_tma && epi == MOE_EPI_STORE_BF16 && prefill && routed.K % 512 == 0 && (!have_shared || sh->K % 512 == 0))
    return grouped_gemm_launch_nvf4_pair(routed, offsets, G, sh, shared_rows, s);
  if (sf_tma) return grouped_gemm_launch_nvf4_wide(epi, routed, offsets, G, sh, shared_rows, s);
  MOE_TRY(gg4::fill(prm, 0, epi, routed));
  prm.offsets = offsets;
  prm.G = G;
  prm.shared_rows = -1;
  if (have_shared) {
    MOE_TRY(gg4::fill(prm, 1, epi, *sh));
    prm.shared_rows = shared_rows;
  }
  prm.err = device_error_word();
  if (!prm.err) return MOE_ERR_CUDA;
  prm.timeout_ns = wait_timeout_ns();
  if (epi == MOE_EPI_STORE_BF16) return gg4::launch<MOE_EPI_STORE_BF16>(prm, s);
  if (epi == MOE_EPI_SWIGLU_BF16) return gg4::launch<MOE_EPI_SWIGLU_BF16>(prm, s);
  return gg4::launch<MOE_EPI_SWIGLU_NVFP4>(prm, s);
}

}  // namespace moe
