// Grouped GEMM with both operands in NVFP4 on the block-scaled FP4 tensor
// cores (tcgen05.mma kind::mxf4nvf4, block_scale, scale_vec::4X), with
// 512-element k stages.
//
// "Driving vLLM WideEP ... (Part I)", section "NVFP4 GEMM for MoE and
// O-proj": packed 4-bit weights with per-group FP8 scales, dequantised inside
// the tensor cores; section "NVFP4 MoE dispatch": the activations arrive in
// NVFP4 too.
//
// Why 512-element stages: every pipeline stage costs the producer and the
// MMA issuer a fixed time in barrier operations and copy issue, and one
// M=128 x N=128 x K=64 FP4 MMA is short (64 tensor cycles), so a stage has to
// carry eight of them, and the MMA issuer does nothing but wait once and
// issue them.
//
// Scale factors: one MMA reads its 128 rows' four E4M3 scales from four
// tensor-memory columns, row r in lane r % 32 (all four lane quadrants) and
// column r / 32.  The scales arrive by TMA as row slices ([rows, K/16]
// bytes: 32 contiguous bytes = eight MMAs per row per stage).  Four scale
// warps, one per lane quadrant, gather for their lane l the words of rows
// l, l+32, l+64, l+96 from the slices and write the stage's 8 MMAs x 4
// columns with one tcgen05.st per operand (a copy instruction per MMA and
// operand would cost the stage more issue time than its MMAs).
//
// Roles (one CTA per SM):
//   warps 0, 10 TMA producers (warp 0 the codes, warp 10 the scales), four
//               copies per stage, each with the stage's
//               two 256-element k-blocks as the outer box dimension:
//               A codes 128 rows x 2 x 128 bytes (128-byte swizzle), B codes
//               likewise (SwiGLU: 64 gate rows then the 64 up rows of the
//               same features, per k-block), A scales 128 rows x 32 bytes,
//               B scales likewise
//   warps 6..9  scale warps (above): sf_full -> shared-memory gather ->
//               tcgen05.st -> arrive on the stage's full barrier (the scale
//               copies are issued first and complete on their own barrier;
//               the full barrier then covers codes and scales, so the MMA
//               issuer waits once per stage)
//   warp 1      TMEM allocation; MMA issuer: waits full, issues up to 8
//               block-scaled MMAs M=128 N=128 K=64 into one of two
//               128-column fp32 accumulators, commits the stage free
//   warps 2..5  epilogue (shared with the other kernels): global scales
//               g_a * g_w[e], SwiGLU, bf16 or NVFP4 output
// Requires K % 256 == 0 (scale rows of whole 16-byte slices) and 16-byte
// aligned scale arrays; other shapes take the kernel of gemm_fp4.cu.
#include <cstring>

#include "gemm_common.cuh"
#include "internal.h"

namespace moe {
namespace gf4 {

using gg::BM;
using gg::MAX_G;
using gg::Params;
using gg::Prob;
using gg::TileInfo;

constexpr int BN = 128;                   // MMA N = accumulator columns per tile
constexpr int KB_BYTES = 128;             // packed bytes of one 256-element k-block row
constexpr int KBLK = 2;                   // k-blocks per stage
constexpr int KE = KBLK * 256;            // elements per stage
constexpr int A_TILE = BM * KB_BYTES;     // 16 KB per k-block
constexpr int B_TILE = BN * KB_BYTES;     // 16 KB per k-block
constexpr int SF_TILE = 128 * 16;         // 2 KB of scale bytes per k-block: 16 per row
constexpr int OFF_B = KBLK * A_TILE;
constexpr int OFF_SFA = OFF_B + KBLK * B_TILE;
constexpr int OFF_SFB = OFF_SFA + KBLK * SF_TILE;
constexpr int STAGE_BYTES = OFF_SFB + KBLK * SF_TILE;  // 72 KB
constexpr int STAGES = 3;
// every copy lands whole (zero fill past K); codes and scales complete on
// separate barriers so that the scale warps start before the codes land
constexpr uint32_t TX_CODES = OFF_SFA;
constexpr uint32_t TX_SF = STAGE_BYTES - OFF_SFA;
constexpr int SF_PROD_WARP = 10;           // producer of the scale copies
constexpr int NUM_WARPS = 11;
constexpr int THREADS = NUM_WARPS * 32;
constexpr int TMEM_COLS = 512;
constexpr int ACC_COLS = 2 * BN;
constexpr int SF_COLS = 2 * KBLK * 4 * 4; // per stage: 8 MMAs x 4 columns, A and B
constexpr int EXTRA = 256 + 4 * 2 * (MAX_G + 4);
constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + EXTRA;
static_assert(STAGE_BYTES % 1024 == 0, "stage must keep 1024-byte alignment");
static_assert(ACC_COLS + STAGES * SF_COLS <= TMEM_COLS, "tensor memory budget");
static_assert(SMEM <= 232448, "shared memory budget");

template <int EPI>
struct Tile {
  static constexpr int N_OUT = (EPI == MOE_EPI_STORE_BF16) ? BN : BN / 2;  // output columns per tile
};

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1) grouped_gemm_nvf4w_kernel(const __grid_constant__ Params p) {
  constexpr int S = STAGES;
  constexpr int TN = Tile<EPI>::N_OUT;
  constexpr bool SWIGLU = EPI != MOE_EPI_STORE_BF16;
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
      mbar_init(&full[s], 1 + 4);  // the producer's arm + one arrival per scale warp
      mbar_init(&sf_full[s], 1);
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
    // ===================================================== TMA producers
    // warp 0 issues the code copies, SF_PROD_WARP the scale copies (a thread's
    // barrier operations queue behind its own outstanding copies, so two
    // issuing threads shorten each stage's issue)
    if (lane == 0) {
      const bool codes = warp == 0;
      for (int pb = 0; pb < (p.shared_rows >= 0 ? 2 : 1); ++pb) {
        if (codes) {
          tma_prefetch_desc(&p.tma_a[pb]);
          tma_prefetch_desc(&p.tma_w[pb]);
        } else {
          tma_prefetch_desc(&p.tma_asf[pb]);
          tma_prefetch_desc(&p.tma_wsf[pb]);
        }
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
        const int nk = (P.K + KE - 1) / KE;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, tmo, p.err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sb = stages + stage * STAGE_BYTES;
          const int kblk = kb * KBLK;
          if (!codes) {
            mbar_arrive_expect_tx(&sf_full[stage], TX_SF);
            tma_load_2d(&p.tma_asf[ti.pb], &sf_full[stage], sb + OFF_SFA, kb * 32, a_y);
            if (SWIGLU)
              tma_load_3d(&p.tma_wsf[ti.pb], &sf_full[stage], sb + OFF_SFB, kb * 32, f0, 2 * ti.g);
            else
              tma_load_2d(&p.tma_wsf[ti.pb], &sf_full[stage], sb + OFF_SFB, kb * 32, w_y);
          } else {
            mbar_arrive_expect_tx(&full[stage], TX_CODES);
            tma_load_3d(&p.tma_a[ti.pb], &full[stage], sb, 0, a_y, kblk);
            if (SWIGLU)
              tma_load_4d(&p.tma_w[ti.pb], &full[stage], sb + OFF_B, 0, f0, 2 * ti.g, kblk);
            else
              tma_load_3d(&p.tma_w[ti.pb], &full[stage], sb + OFF_B, 0, w_y, kblk);
          }
          issued[stage] += 1;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // let copies already issued land before the block can exit
        for (int s = 0; s < S; ++s)
          if (issued[s])
            mbar_wait_bounded(codes ? &full[s] : &sf_full[s], (issued[s] - 1u) & 1u, 1000000000ull, p.err, nullptr);
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
          // codes landed and the scale warps' tensor-memory stores are done
          if (!mbar_wait_bounded(&full[stage], phase, tmo, p.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sb = smem_u32(stages + stage * STAGE_BYTES);
          const uint32_t sf_t = tmem_base + static_cast<uint32_t>(ACC_COLS + stage * SF_COLS);
          // K % 256 == 0: a stage holds one or two whole k-blocks
          const int nblk = min(KBLK, (K - kb * KE) / 256);
          for (int j = 0; j < nblk; ++j) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_nvf4(d, smem_desc_kmajor_sw128(sb + j * A_TILE + kk * 32),
                        smem_desc_kmajor_sw128(sb + OFF_B + j * B_TILE + kk * 32), IDESC,
                        sf_t + 4 * (4 * j + kk), sf_t + SF_COLS / 2 + 4 * (4 * j + kk), (kb | j | kk) ? 1u : 0u);
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
  } else if (warp >= 6 && warp < 10) {
    // ===================================================== scale warps
    const int q = warp & 3;  // lane quadrant this warp writes
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const TileInfo ti = gg::decode_tile(t, s_prefix, s_off, GT, G, p.shared_rows);
      const int nk = (p.prob[ti.pb].K + KE - 1) / KE;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait_warp(&sf_full[stage], phase, tmo, p.err, abort_flag)) {
          ok = false;
          break;
        }
        const uint8_t* sb = stages + stage * STAGE_BYTES;
        const uint32_t sf_t = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                              static_cast<uint32_t>(ACC_COLS + stage * SF_COLS);
#pragma unroll
        for (int op = 0; op < 2; ++op) {
          // v[j][c]: the 16 scale bytes (4 MMAs) of row lane + 32c in k-block j
          uint4 v[KBLK][4];
#pragma unroll
          for (int j = 0; j < KBLK; ++j)
#pragma unroll
            for (int c = 0; c < 4; ++c)
              v[j][c] = *reinterpret_cast<const uint4*>(sb + (op ? OFF_SFB : OFF_SFA) + j * 16 +
                                                        (lane + 32 * c) * 32);
          // column 4m + c of this lane = MMA m's word of row lane + 32c
          uint32_t r[32];
#pragma unroll
          for (int m = 0; m < 4 * KBLK; ++m)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint4 w = v[m >> 2][c];
              r[4 * m + c] = (m & 3) == 0 ? w.x : (m & 3) == 1 ? w.y : (m & 3) == 2 ? w.z : w.w;
            }
          tmem_st_32x32b_x32(sf_t + (op ? SF_COLS / 2 : 0), r);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[stage]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
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
        cudaFuncSetAttribute(grouped_gemm_nvf4w_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) {
      set_cuda_error(e);
      return MOE_ERR_CUDA;
    }
    attr_done[dev] = true;
  }
  grouped_gemm_nvf4w_kernel<EPI><<<num_sms(), THREADS, SMEM, s>>>(prm);
  return check_launch();
}

static int fill(Params& prm, int slot, int epi, const GemmProblem& P) {
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
  const uint64_t K = static_cast<uint64_t>(P.K), nkb = K / 256;
  const uint64_t code_ld = K / 2, sf_ld = K / 16;  // bytes per row
  // A codes [a_rows, K/2]: (byte in k-block, row, k-block); A scales
  // [a_rows, K/16]: (byte in 16-byte slice, row, slice)
  {
    const uint64_t dims[3] = {KB_BYTES, static_cast<uint64_t>(P.a_rows), nkb};
    const uint64_t str[2] = {code_ld, KB_BYTES};
    const uint32_t box[3] = {KB_BYTES, BM, KBLK};
    MOE_TRY(encode_tmap_nd(&prm.tma_a[slot], P.A, false, 3, dims, str, box, true));
    MOE_TRY(encode_tmap_2d(&prm.tma_asf[slot], P.A_sf, 1, sf_ld, static_cast<uint64_t>(P.a_rows), 32, BM, false));
  }
  if (swiglu) {
    // W [groups][gate N | up N][K/2] as (byte, row, gate/up + 2*group, k-block)
    const uint64_t N = static_cast<uint64_t>(P.N), g2 = 2 * static_cast<uint64_t>(P.groups);
    const uint64_t dims[4] = {KB_BYTES, N, g2, nkb};
    const uint64_t str[3] = {code_ld, N * code_ld, KB_BYTES};
    const uint32_t box[4] = {KB_BYTES, BN / 2, 2, KBLK};
    MOE_TRY(encode_tmap_nd(&prm.tma_w[slot], P.W, false, 4, dims, str, box, true));
    const uint64_t sdims[3] = {sf_ld, N, g2};
    const uint64_t sstr[2] = {sf_ld, N * sf_ld};
    const uint32_t sbox[3] = {32, BN / 2, 2};
    MOE_TRY(encode_tmap_nd(&prm.tma_wsf[slot], P.W_sf, false, 3, sdims, sstr, sbox, false));
  } else {
    const uint64_t rows = static_cast<uint64_t>(q.w_rows_total);
    const uint64_t dims[3] = {KB_BYTES, rows, nkb};
    const uint64_t str[2] = {code_ld, KB_BYTES};
    const uint32_t box[3] = {KB_BYTES, BN, KBLK};
    MOE_TRY(encode_tmap_nd(&prm.tma_w[slot], P.W, false, 3, dims, str, box, true));
    MOE_TRY(encode_tmap_2d(&prm.tma_wsf[slot], P.W_sf, 1, sf_ld, rows, 32, BN, false));
  }
  return MOE_OK;
}

}  // namespace gf4

// NVFP4 x NVFP4 with K % 256 == 0 and 16-byte aligned scales (checked by the
// caller, grouped_gemm_launch_nvf4).
int grouped_gemm_launch_nvf4_wide(int epi, const GemmProblem& routed, const int32_t* offsets, int G,
                                  const GemmProblem* sh, int shared_rows, cudaStream_t s) {
  gg::Params prm;
  memset(&prm, 0, sizeof(prm));
  MOE_TRY(gf4::fill(prm, 0, epi, routed));
  prm.offsets = offsets;
  prm.G = G;
  prm.shared_rows = -1;
  if (sh != nullptr && shared_rows > 0) {
    MOE_TRY(gf4::fill(prm, 1, epi, *sh));
    prm.shared_rows = shared_rows;
  }
  prm.err = device_error_word();
  if (!prm.err) return MOE_ERR_CUDA;
  prm.timeout_ns = wait_timeout_ns();
  if (epi == MOE_EPI_STORE_BF16) return gf4::launch<MOE_EPI_STORE_BF16>(prm, s);
  if (epi == MOE_EPI_SWIGLU_BF16) return gf4::launch<MOE_EPI_SWIGLU_BF16>(prm, s);
  return gf4::launch<MOE_EPI_SWIGLU_NVFP4>(prm, s);
}

}  // namespace moe
