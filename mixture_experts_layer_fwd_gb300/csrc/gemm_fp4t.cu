// Grouped GEMM with both operands in NVFP4 whose scale factors are stored in
// the MMA's tile order (sf_tiles.cu): block-scaled FP4 tensor cores
// (tcgen05.mma kind::mxf4nvf4, block_scale, scale_vec::4X), 512-element k
// stages.
//
// "Driving vLLM WideEP ... (Part I)", section "NVFP4 GEMM for MoE and
// O-proj": packed 4-bit operands with one FP8 scale per 16 elements,
// dequantised inside the tensor cores.
//
// The kernel of gemm_fp4w.cu receives the scales as row-major slices and
// needs four scale warps to regroup them for tensor memory each stage.
// Here the scales of a stage's eight MMAs arrive already in the order that
// tcgen05.cp reads (8 blocks of 32 rows x 16 bytes per operand, contiguous
// in global memory), so one bulk copy per operand brings them to shared
// memory and the MMA issuer moves each block into tensor memory with
// tcgen05.cp (32x128b, replicated into the four lane quadrants) right
// before the MMAs: no warp touches the scales.
//
// Roles (one CTA per SM):
//   warp 0      TMA producer of the codes: A 128 rows x 2 x 128 bytes, B
//               likewise (SwiGLU: 64 gate rows then the 64 up rows of the
//               same features), the stage's two 256-element k-blocks as the
//               outer box dimension, 128-byte swizzle
//   warp 6      producer of the scales: two bulk copies per stage (A tile,
//               B tile), 512 bytes per MMA each
//               (both producers arrive on the stage's full barrier, which
//               completes when codes and scales have landed)
//   warp 1      TMEM allocation; MMA issuer: waits full, copies the stage's
//               scale blocks into tensor memory, issues up to 8 block-scaled
//               MMAs M=128 N=128 K=64 into one of two 128-column fp32
//               accumulators, commits the stage free
//   warps 2..5  epilogue (shared with the other kernels): global scales
//               g_a * g_w[e], SwiGLU, bf16 or NVFP4 output (row-major scales)
// Requires K % 256 == 0 and 16-byte aligned tiled scale buffers.
#include <cstring>

#include "gemm_common.cuh"
#include "internal.h"

namespace moe {
namespace gf4t {

using gg::BM;
using gg::MAX_G;
using gg::Params;
using gg::Prob;
using gg::TileInfo;

constexpr int BN = 128;                   // MMA N = accumulator columns per tile
constexpr int KB_BYTES = 128;             // packed bytes of one 256-element k-block row
constexpr int KBLK = 2;                   // k-blocks per stage
constexpr int KE = KBLK * 256;            // elements per stage
constexpr int MMAS = KE / 64;             // block-scaled MMAs per stage
constexpr int A_TILE = BM * KB_BYTES;     // 16 KB per k-block
constexpr int B_TILE = BN * KB_BYTES;     // 16 KB per k-block
constexpr int SF_BLOCK = 512;             // scales of one MMA: 32 rows x 16 bytes
constexpr int OFF_B = KBLK * A_TILE;
constexpr int OFF_SFA = OFF_B + KBLK * B_TILE;
constexpr int OFF_SFB = OFF_SFA + MMAS * SF_BLOCK;
constexpr int STAGE_BYTES = OFF_SFB + MMAS * SF_BLOCK;  // 72 KB
constexpr int STAGES = 3;
constexpr uint32_t TX_CODES = OFF_SFA;   // code boxes land whole (zero fill past K)
constexpr int SF_PROD_WARP = 6;
constexpr int NUM_WARPS = 7;
constexpr int THREADS = NUM_WARPS * 32;
constexpr int TMEM_COLS = 512;
constexpr int ACC_COLS = 2 * BN;
constexpr int SF_COLS = 2 * MMAS * 4;    // per stage: 8 MMAs x 4 columns, A then B
constexpr int EXTRA = 256 + 4 * 2 * (MAX_G + 4);
constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + EXTRA;
static_assert(STAGE_BYTES % 1024 == 0, "stage must keep 1024-byte alignment");
static_assert(ACC_COLS + STAGES * SF_COLS <= TMEM_COLS, "tensor memory budget");
static_assert(SMEM <= 232448, "shared memory budget");

template <int EPI>
struct Tile {
  static constexpr int N_OUT = (EPI == MOE_EPI_STORE_BF16) ? BN : BN / 2;  // output columns per tile
};

// Tile of the A scale buffer that holds row block m_blk of tile ti: routed
// groups are numbered by the prefix of their row blocks (the schedule's tile
// prefix divided by the column blocks per group), the shared problem is one
// group.  Clamped to the buffer's capacity, so that offsets outside the
// contract cannot send the copy past its end.
DEVINL int a_scale_tile(const Params& p, const TileInfo& ti, const int* s_prefix) {
  const int t = (ti.pb == 0) ? s_prefix[ti.g] / p.prob[0].n_tiles + ti.m_blk : ti.m_blk;
  return min(t, p.prob[ti.pb].a_sf_tiles - 1);
}

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1) grouped_gemm_nvf4t_kernel(const __grid_constant__ Params p) {
  constexpr int S = STAGES;
  constexpr int TN = Tile<EPI>::N_OUT;
  constexpr bool SWIGLU = EPI != MOE_EPI_STORE_BF16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = base;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + S * STAGE_BYTES);
  uint64_t* empty = full + S;
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
      mbar_init(&full[s], 2);  // one arrive (with its transaction bytes) per producer
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

  if (warp == 0 || warp == SF_PROD_WARP) {
    // ===================================================== producers
    if (lane == 0) {
      const bool codes = warp == 0;
      if (codes)
        for (int pb = 0; pb < (p.shared_rows >= 0 ? 2 : 1); ++pb) {
          tma_prefetch_desc(&p.tma_a[pb]);
          tma_prefetch_desc(&p.tma_w[pb]);
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
        const int a_y = ti.row0 + ti.m_blk * BM;
        // SwiGLU: features [n_blk*64, +64) of group g (gate and up halves);
        // STORE: weight rows [g*N + n_blk*128, +128)
        const int f0 = ti.n_blk * TN;
        const int w_y = ti.g * P.w_rows + ti.n_blk * TN;
        const int ks = P.K / 64;  // MMAs (512-byte scale blocks) per row of tiles
        const uint8_t* sfa = P.a_sf + static_cast<size_t>(a_scale_tile(p, ti, s_prefix)) * ks * SF_BLOCK;
        const uint8_t* sfb = P.w_sf + (static_cast<size_t>(ti.g) * P.n_tiles + ti.n_blk) * ks * SF_BLOCK;
        const int nk = (P.K + KE - 1) / KE;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, tmo, p.err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sb = stages + stage * STAGE_BYTES;
          if (codes) {
            const int kblk = kb * KBLK;
            mbar_arrive_expect_tx(&full[stage], TX_CODES);
            tma_load_3d(&p.tma_a[ti.pb], &full[stage], sb, 0, a_y, kblk);
            if (SWIGLU)
              tma_load_4d(&p.tma_w[ti.pb], &full[stage], sb + OFF_B, 0, f0, 2 * ti.g, kblk);
            else
              tma_load_3d(&p.tma_w[ti.pb], &full[stage], sb + OFF_B, 0, w_y, kblk);
          } else {
            // K % 256 == 0: the stage holds 4 or 8 MMAs' scale blocks
            const uint32_t bytes = static_cast<uint32_t>(min(MMAS, ks - kb * MMAS)) * SF_BLOCK;
            const size_t off = static_cast<size_t>(kb) * MMAS * SF_BLOCK;
            mbar_arrive_expect_tx(&full[stage], 2 * bytes);
            bulk_load(sb + OFF_SFA, sfa + off, bytes, &full[stage]);
            bulk_load(sb + OFF_SFB, sfb + off, bytes, &full[stage]);
          }
          issued[stage] += 1;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // let copies already issued land before the block can exit (the
        // other producer's arrival completes the phase; bounded either way)
        for (int s = 0; s < S; ++s)
          if (issued[s]) mbar_wait_bounded(&full[s], (issued[s] - 1u) & 1u, 1000000000ull, p.err, nullptr);
      }
    }
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
        const int K = p.prob[ti.pb].K;
        const int nk = (K + KE - 1) / KE;
        const int buf = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        if (!mbar_wait_bounded(&tempty[buf], (use & 1u) ^ 1u, tmo, p.err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, tmo, p.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sb = smem_u32(stages + stage * STAGE_BYTES);
          const uint32_t sf_t = tmem_base + static_cast<uint32_t>(ACC_COLS + stage * SF_COLS);
          // K % 256 == 0: a stage holds one or two whole k-blocks
          const int nmma = 4 * min(KBLK, (K - kb * KE) / 256);
          // scale blocks into tensor memory; the tensor pipe runs a thread's
          // copies and MMAs in issue order
          for (int m = 0; m < nmma; ++m) {
            tmem_cp_32x128b_warpx4(sf_t + 4 * m, smem_desc_kmajor_noswizzle_16B_rows(sb + OFF_SFA + m * SF_BLOCK));
            tmem_cp_32x128b_warpx4(sf_t + SF_COLS / 2 + 4 * m,
                                   smem_desc_kmajor_noswizzle_16B_rows(sb + OFF_SFB + m * SF_BLOCK));
          }
          for (int m = 0; m < nmma; ++m) {
            const int j = m >> 2, kk = m & 3;
            umma_nvf4(d, smem_desc_kmajor_sw128(sb + j * A_TILE + kk * 32),
                      smem_desc_kmajor_sw128(sb + OFF_B + j * B_TILE + kk * 32), IDESC, sf_t + 4 * m,
                      sf_t + SF_COLS / 2 + 4 * m, (kb | m) ? 1u : 0u);
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
  if (*abort_flag) {
    // a wait ran out: give copies and MMAs already in flight time to land
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) {
    }
  }
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
        cudaFuncSetAttribute(grouped_gemm_nvf4t_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) {
      set_cuda_error(e);
      return MOE_ERR_CUDA;
    }
    attr_done[dev] = true;
  }
  grouped_gemm_nvf4t_kernel<EPI><<<num_sms(), THREADS, SMEM, s>>>(prm);
  return check_launch();
}

// A_sf / W_sf of P are the tiled scale buffers; a_sf_tiles is the capacity
// of the A buffer in tiles.
static int fill(Params& prm, int slot, int epi, const GemmProblem& P, int a_sf_tiles) {
  Prob& q = prm.prob[slot];
  const bool swiglu = epi != MOE_EPI_STORE_BF16;
  const int tn = swiglu ? BN / 2 : BN;
  q.n_out = P.N;
  q.K = P.K;
  q.w_rows = swiglu ? 2 * P.N : P.N;
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
  q.a_sf_tiles = a_sf_tiles;
  const uint64_t K = static_cast<uint64_t>(P.K), nkb = K / 256;
  const uint64_t code_ld = K / 2;  // bytes per row
  {
    // A codes [a_rows, K/2] as (byte in k-block, row, k-block)
    const uint64_t dims[3] = {KB_BYTES, static_cast<uint64_t>(P.a_rows), nkb};
    const uint64_t str[2] = {code_ld, KB_BYTES};
    const uint32_t box[3] = {KB_BYTES, BM, KBLK};
    MOE_TRY(encode_tmap_nd(&prm.tma_a[slot], P.A, false, 3, dims, str, box, true));
  }
  if (swiglu) {
    // W [groups][gate N | up N][K/2] as (byte, row, gate/up + 2*group, k-block)
    const uint64_t N = static_cast<uint64_t>(P.N), g2 = 2 * static_cast<uint64_t>(P.groups);
    const uint64_t dims[4] = {KB_BYTES, N, g2, nkb};
    const uint64_t str[3] = {code_ld, N * code_ld, KB_BYTES};
    const uint32_t box[4] = {KB_BYTES, BN / 2, 2, KBLK};
    MOE_TRY(encode_tmap_nd(&prm.tma_w[slot], P.W, false, 4, dims, str, box, true));
  } else {
    const uint64_t rows = static_cast<uint64_t>(q.w_rows_total);
    const uint64_t dims[3] = {KB_BYTES, rows, nkb};
    const uint64_t str[2] = {code_ld, KB_BYTES};
    const uint32_t box[3] = {KB_BYTES, BN, KBLK};
    MOE_TRY(encode_tmap_nd(&prm.tma_w[slot], P.W, false, 3, dims, str, box, true));
  }
  return MOE_OK;
}

}  // namespace gf4t

// NVFP4 x NVFP4 with tiled scales; arguments checked by the caller.
// routed.A_sf holds the rows' scales tiled by group (tile_base order) with
// capacity sf_tiles_bytes_rows(M, G, K); the shared problem's A_sf holds its
// T rows as one group.
int grouped_gemm_launch_nvf4_tiled(int epi, const GemmProblem& routed, const int32_t* offsets, int G,
                                   const GemmProblem* sh, int shared_rows, cudaStream_t s) {
  gg::Params prm;
  memset(&prm, 0, sizeof(prm));
  MOE_TRY(gf4t::fill(prm, 0, epi, routed, (routed.a_rows + 127) / 128 + G));
  prm.offsets = offsets;
  prm.G = G;
  prm.shared_rows = -1;
  if (sh != nullptr && shared_rows > 0) {
    MOE_TRY(gf4t::fill(prm, 1, epi, *sh, (sh->a_rows + 127) / 128 + 1));
    prm.shared_rows = shared_rows;
  }
  prm.err = device_error_word();
  if (!prm.err) return MOE_ERR_CUDA;
  prm.timeout_ns = wait_timeout_ns();
  if (epi == MOE_EPI_STORE_BF16) return gf4t::launch<MOE_EPI_STORE_BF16>(prm, s);
  if (epi == MOE_EPI_SWIGLU_BF16) return gf4t::launch<MOE_EPI_SWIGLU_BF16>(prm, s);
  return gf4t::launch<MOE_EPI_SWIGLU_NVFP4>(prm, s);
}

}  // namespace moe
