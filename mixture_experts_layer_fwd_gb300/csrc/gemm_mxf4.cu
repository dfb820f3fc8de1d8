// Grouped GEMM with both operands in MXFP4: E2M1 codes with one E8M0 scale
// per 32 elements along K, on the block-scaled FP4 tensor cores
// (tcgen05.mma kind::mxf4nvf4, block_scale, scale_vec::2X), 512-element k
// stages.
//
// "Hosting Qwen on Blackwell", section "Quantização": Blackwell runs the
// microscaled formats natively, Qwen3-235B is served in MXFP8 and MXFP4 was
// considered; "CuTeDSL at Perplexity", Blackwell support: MXFP8 / MXFP4 scale
// 32 elements.  Format reading: see quant_mx.cu.
//
// The structure is that of the NVFP4 kernel (gemm_fp4w.cu): TMA producers of
// the codes and of the scale rows, four scale warps that regroup the scales
// for tensor memory, one MMA issuer, four epilogue warps.  What changes:
//   * an MMA of K = 64 reads two E8M0 bytes per row (scale_vec::2X), so one
//     32-bit tensor-memory cell serves two MMAs: MMA m of a stage reads
//     cell m / 2 and picks its byte pair with scale-factor id 2 * (m % 2)
//     (instruction-descriptor bits 29-30 for A, 4-5 for B; bit 23 selects
//     E8M0 scales);
//   * a stage's scales are 16 bytes per row (two 256-element k-blocks), one
//     16-byte TMA box per operand, which needs K % 512 == 0;
//   * there are no global scales: the epilogue multiplies by 1.
// Epilogues: STORE_BF16 and SWIGLU_BF16.
#include <cstring>

#include "gemm_common.cuh"
#include "internal.h"

namespace moe {
namespace gmx {

using gg::BM;
using gg::MAX_G;
using gg::Params;
using gg::Prob;
using gg::TileInfo;

constexpr int BN = 128;                   // MMA N = accumulator columns per tile
constexpr int KB_BYTES = 128;             // packed bytes of one 256-element k-block row
constexpr int KBLK = 2;                   // k-blocks per stage
constexpr int KE = KBLK * 256;            // elements per stage
constexpr int MMAS = KE / 64;             // MMAs per stage
constexpr int SF_ROW = KE / 32;           // scale bytes per row per stage (16)
constexpr int A_TILE = BM * KB_BYTES;     // 16 KB per k-block
constexpr int B_TILE = BN * KB_BYTES;     // 16 KB per k-block
constexpr int OFF_B = KBLK * A_TILE;
constexpr int OFF_SFA = OFF_B + KBLK * B_TILE;
constexpr int OFF_SFB = OFF_SFA + BM * SF_ROW;
constexpr int STAGE_BYTES = OFF_SFB + BN * SF_ROW;  // 68 KB
constexpr int STAGES = 3;
constexpr uint32_t TX_CODES = OFF_SFA;
constexpr uint32_t TX_SF = STAGE_BYTES - OFF_SFA;
constexpr int SF_PROD_WARP = 10;
constexpr int NUM_WARPS = 11;
constexpr int THREADS = NUM_WARPS * 32;
constexpr int TMEM_COLS = 512;
constexpr int ACC_COLS = 2 * BN;
constexpr int SF_CELLS = MMAS / 2;        // 32-bit cells per row per stage
constexpr int SF_COLS = 2 * SF_CELLS * 4; // per stage: A then B, 4 columns (row groups) per cell
constexpr int EXTRA = 256 + 4 * 2 * (MAX_G + 4);
constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + EXTRA;
static_assert(STAGE_BYTES % 1024 == 0, "stage must keep 1024-byte alignment");
static_assert(SF_COLS == 32, "one 32-column tcgen05.st per stage carries both operands' scales");
static_assert(ACC_COLS + STAGES * SF_COLS <= TMEM_COLS, "tensor memory budget");
static_assert(SMEM <= 232448, "shared memory budget");

// Instruction descriptor, kind::mxf4nvf4 with E8M0 scales: E2M1 x E2M1 ->
// fp32, both K-major, scale-factor ids for A (bits 29-30) and B (bits 4-5).
__host__ __device__ constexpr uint32_t idesc_mxf4_f32(int M, int N, uint32_t sf_id) {
  return (sf_id << 4)                               // B scale-factor id
         | (1u << 7)                                // A format E2M1
         | (1u << 10)                               // B format E2M1
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (1u << 23)                               // scale format E8M0
         | (static_cast<uint32_t>(M >> 4) << 24)    // M / 16
         | (sf_id << 29);                           // A scale-factor id
}

DEVINL void umma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa_tmem,
                      uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

template <int EPI>
struct Tile {
  static constexpr int N_OUT = (EPI == MOE_EPI_STORE_BF16) ? BN : BN / 2;  // output columns per tile
};

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1) grouped_gemm_mxf4_kernel(const __grid_constant__ Params p) {
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
      mbar_init(&full[s], 1 + 4);  // the codes producer's arm + one arrival per scale warp
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
        const int f0 = ti.n_blk * TN;
        const int w_y = ti.g * P.w_rows + ti.n_blk * TN;
        const int nk = P.K / KE;  // K % 512 == 0
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, tmo, p.err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sb = stages + stage * STAGE_BYTES;
          if (!codes) {
            mbar_arrive_expect_tx(&sf_full[stage], TX_SF);
            tma_load_2d(&p.tma_asf[ti.pb], &sf_full[stage], sb + OFF_SFA, kb * SF_ROW, a_y);
            if (SWIGLU)
              tma_load_3d(&p.tma_wsf[ti.pb], &sf_full[stage], sb + OFF_SFB, kb * SF_ROW, f0, 2 * ti.g);
            else
              tma_load_2d(&p.tma_wsf[ti.pb], &sf_full[stage], sb + OFF_SFB, kb * SF_ROW, w_y);
          } else {
            const int kblk = kb * KBLK;
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
      constexpr uint32_t IDESC0 = idesc_mxf4_f32(BM, BN, 0u);
      constexpr uint32_t IDESC2 = idesc_mxf4_f32(BM, BN, 2u);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
        const TileInfo ti = gg::decode_tile(t, s_prefix, s_off, GT, G, p.shared_rows);
        const int nk = p.prob[ti.pb].K / KE;
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
#pragma unroll
          for (int m = 0; m < MMAS; ++m) {
            const int j = m >> 2, kk = m & 3, cell = m >> 1;
            umma_mxf4(d, smem_desc_kmajor_sw128(sb + j * A_TILE + kk * 32),
                      smem_desc_kmajor_sw128(sb + OFF_B + j * B_TILE + kk * 32), (m & 1) ? IDESC2 : IDESC0,
                      sf_t + 4 * cell, sf_t + SF_COLS / 2 + 4 * cell, (kb | m) ? 1u : 0u);
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
    // lane l of the warp for lane quadrant q writes, for rows r = l + 32c of
    // the tile (c = 0..3), word w of the row's 16 stage bytes (MMAs 2w and
    // 2w+1) into column 4w + c: A in columns 0..15, B in 16..31
    const int q = warp & 3;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const TileInfo ti = gg::decode_tile(t, s_prefix, s_off, GT, G, p.shared_rows);
      const int nk = p.prob[ti.pb].K / KE;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait_warp(&sf_full[stage], phase, tmo, p.err, abort_flag)) {
          ok = false;
          break;
        }
        const uint8_t* sb = stages + stage * STAGE_BYTES;
        const uint32_t sf_t = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                              static_cast<uint32_t>(ACC_COLS + stage * SF_COLS);
        uint32_t r[32];
#pragma unroll
        for (int op = 0; op < 2; ++op)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(sb + (op ? OFF_SFB : OFF_SFA) + (lane + 32 * c) * SF_ROW);
            r[16 * op + 0 + c] = v.x;
            r[16 * op + 4 + c] = v.y;
            r[16 * op + 8 + c] = v.z;
            r[16 * op + 12 + c] = v.w;
          }
        tmem_st_32x32b_x32(sf_t, r);
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
      gg::epilogue_tile<EPI, BN, true>(P, ti, taddr, r_in_tile, 1.0f);
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
        cudaFuncSetAttribute(grouped_gemm_mxf4_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) {
      set_cuda_error(e);
      return MOE_ERR_CUDA;
    }
    attr_done[dev] = true;
  }
  grouped_gemm_mxf4_kernel<EPI><<<num_sms(), THREADS, SMEM, s>>>(prm);
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
  q.c_sf = P.C_sf;  // MX codes of h (SWIGLU_MX)
  q.a_g = q.w_g = q.c_g = nullptr;
  q.a_sf = P.A_sf;
  q.w_sf = P.W_sf;
  const uint64_t K = static_cast<uint64_t>(P.K), nkb = K / 256;
  const uint64_t code_ld = K / 2, sf_ld = K / 32;  // bytes per row
  {
    // A codes [a_rows, K/2] as (byte in k-block, row, k-block); A scales
    // [a_rows, K/32] as 16-byte row slices
    const uint64_t dims[3] = {KB_BYTES, static_cast<uint64_t>(P.a_rows), nkb};
    const uint64_t str[2] = {code_ld, KB_BYTES};
    const uint32_t box[3] = {KB_BYTES, BM, KBLK};
    MOE_TRY(encode_tmap_nd(&prm.tma_a[slot], P.A, false, 3, dims, str, box, true));
    MOE_TRY(encode_tmap_2d(&prm.tma_asf[slot], P.A_sf, 1, sf_ld, static_cast<uint64_t>(P.a_rows), SF_ROW, BM,
                           false));
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
    const uint32_t sbox[3] = {SF_ROW, BN / 2, 2};
    MOE_TRY(encode_tmap_nd(&prm.tma_wsf[slot], P.W_sf, false, 3, sdims, sstr, sbox, false));
  } else {
    const uint64_t rows = static_cast<uint64_t>(q.w_rows_total);
    const uint64_t dims[3] = {KB_BYTES, rows, nkb};
    const uint64_t str[2] = {code_ld, KB_BYTES};
    const uint32_t box[3] = {KB_BYTES, BN, KBLK};
    MOE_TRY(encode_tmap_nd(&prm.tma_w[slot], P.W, false, 3, dims, str, box, true));
    MOE_TRY(encode_tmap_2d(&prm.tma_wsf[slot], P.W_sf, 1, sf_ld, rows, SF_ROW, BN, false));
  }
  return MOE_OK;
}

}  // namespace gmx

// MXFP4 x MXFP4, K % 512 == 0, 16-byte aligned scale arrays, bf16 and MX SwiGLU epilogues
// (checked by the caller, grouped_gemm_launch).
int grouped_gemm_launch_mxf4(int epi, const GemmProblem& routed, const int32_t* offsets, int G,
                             const GemmProblem* sh, int shared_rows, cudaStream_t s) {
  gg::Params prm;
  memset(&prm, 0, sizeof(prm));
  MOE_TRY(gmx::fill(prm, 0, epi, routed));
  prm.offsets = offsets;
  prm.G = G;
  prm.shared_rows = -1;
  if (sh != nullptr && shared_rows > 0) {
    MOE_TRY(gmx::fill(prm, 1, epi, *sh));
    prm.shared_rows = shared_rows;
  }
  prm.err = device_error_word();
  if (!prm.err) return MOE_ERR_CUDA;
  prm.timeout_ns = wait_timeout_ns();
  if (epi == MOE_EPI_STORE_BF16) return gmx::launch<MOE_EPI_STORE_BF16>(prm, s);
  if (epi == MOE_EPI_SWIGLU_MX) return gmx::launch<MOE_EPI_SWIGLU_MX>(prm, s);
  return gmx::launch<MOE_EPI_SWIGLU_BF16>(prm, s);
}

}  // namespace moe
