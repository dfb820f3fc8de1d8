// Grouped GEMM with both operands in MXFP8: E4M3 bytes with one E8M0 scale
// per 32 elements along K, on the block-scaled tensor cores (tcgen05.mma
// kind::mxf8f6f4, block_scale, scale_vec::1X).
//
// "Hosting Qwen on Blackwell", section "Quantização": Qwen3-235B is served
// with its weights converted to MXFP8 once after fine-tuning, which ran much
// faster than block scaling in the MoE GEMM microbenchmarks; "CuTeDSL at
// Perplexity", Blackwell support: MXFP8 scales 32 elements.  Format reading:
// see quant_mx.cu.
//
// Per pipeline stage of 256 elements: two 128-byte k-blocks of each operand
// by TMA (128-byte swizzle, the same bytes per stage as the FP4 kernels), 8
// MMAs of K = 32.  Each MMA reads one E8M0 byte per row; one 32-bit tensor-
// memory cell holds the bytes of four consecutive MMAs, picked by the
// instruction descriptor's scale-factor id m % 4 (bits 29-30 for A, 4-5 for
// B; bit 23 selects E8M0).  A stage's scales are 8 bytes per row, below the
// 16-byte minimum of a TMA box, so the four scale warps read them straight
// from global memory (one 8-byte load per row; rows outside the operand
// read as zero) and write both operands' 16 columns with one tcgen05.st.
// Roles (one CTA per SM):
//   warp 0      TMA producer of the codes
//   warp 1      TMEM allocation; MMA issuer
//   warps 2..5  epilogue (no global scales), STORE_BF16 / SWIGLU_BF16
//   warps 6..9  scale warps: wait until the stage's previous MMAs are done
//               (its empty barrier), load, tcgen05.st, arrive on full
// Requires K % 256 == 0 and 8-byte aligned scale arrays.
#include <cstring>

#include "gemm_common.cuh"
#include "internal.h"

namespace moe {
namespace gmx8 {

using gg::BM;
using gg::MAX_G;
using gg::Params;
using gg::Prob;
using gg::TileInfo;

constexpr int BN = 128;                   // MMA N = accumulator columns per tile
constexpr int KB_BYTES = 128;             // bytes (elements) of one k-block row
constexpr int KBLK = 2;                   // k-blocks per stage
constexpr int KE = KBLK * KB_BYTES;       // elements per stage
constexpr int MMAS = KE / 32;             // MMAs per stage
constexpr int SF_ROW = KE / 32;           // scale bytes per row per stage (8)
constexpr int A_TILE = BM * KB_BYTES;     // 16 KB per k-block
constexpr int B_TILE = BN * KB_BYTES;     // 16 KB per k-block
constexpr int OFF_B = KBLK * A_TILE;
constexpr int STAGE_BYTES = OFF_B + KBLK * B_TILE;  // 64 KB
constexpr int STAGES = 3;
constexpr uint32_t TX_CODES = STAGE_BYTES;
constexpr int NUM_WARPS = 10;
constexpr int THREADS = NUM_WARPS * 32;
constexpr int TMEM_COLS = 512;
constexpr int ACC_COLS = 2 * BN;
constexpr int SF_CELLS = SF_ROW / 4;      // 32-bit cells per row per stage
constexpr int SF_COLS = 2 * SF_CELLS * 4; // per stage: A then B, 4 columns (row groups) per cell
constexpr int EXTRA = 256 + 4 * 2 * (MAX_G + 4);
constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + EXTRA;
static_assert(STAGE_BYTES % 1024 == 0, "stage must keep 1024-byte alignment");
static_assert(SF_COLS == 16, "one 16-column tcgen05.st per stage carries both operands' scales");
static_assert(ACC_COLS + STAGES * SF_COLS <= TMEM_COLS, "tensor memory budget");
static_assert(SMEM <= 232448, "shared memory budget");

// Instruction descriptor, kind::mxf8f6f4 with E8M0 scales: E4M3 x E4M3 ->
// fp32 (format code 0 for both), both K-major, scale-factor ids for A (bits
// 29-30) and B (bits 4-5).
__host__ __device__ constexpr uint32_t idesc_mxf8_f32(int M, int N, uint32_t sf_id) {
  return (sf_id << 4)                               // B scale-factor id
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (1u << 23)                               // scale format E8M0
         | (static_cast<uint32_t>(M >> 4) << 24)    // M / 16
         | (sf_id << 29);                           // A scale-factor id
}

DEVINL void umma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa_tmem,
                      uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// 32 lanes x 16 columns of 32 bits into tensor memory (this warp's quadrant).
DEVINL void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

template <int EPI>
struct Tile {
  static constexpr int N_OUT = (EPI == MOE_EPI_STORE_BF16) ? BN : BN / 2;  // output columns per tile
};

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1) grouped_gemm_mxf8_kernel(const __grid_constant__ Params p) {
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
      mbar_init(&full[s], 1 + 4);  // the codes producer's arm + one arrival per scale warp
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
    // ===================================================== TMA producer (codes)
    if (lane == 0) {
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
        const int f0 = ti.n_blk * TN;
        const int w_y = ti.g * P.w_rows + ti.n_blk * TN;
        const int nk = P.K / KE;  // K % 256 == 0
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, tmo, p.err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sb = stages + stage * STAGE_BYTES;
          const int kblk = kb * KBLK;
          mbar_arrive_expect_tx(&full[stage], TX_CODES);
          tma_load_3d(&p.tma_a[ti.pb], &full[stage], sb, 0, a_y, kblk);
          if (SWIGLU)
            tma_load_4d(&p.tma_w[ti.pb], &full[stage], sb + OFF_B, 0, f0, 2 * ti.g, kblk);
          else
            tma_load_3d(&p.tma_w[ti.pb], &full[stage], sb + OFF_B, 0, w_y, kblk);
          issued[stage] += 1;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // let copies already issued land before the block can exit (the
        // phase also needs the scale warps: bounded either way)
        for (int s = 0; s < S; ++s)
          if (issued[s]) mbar_wait_bounded(&full[s], (issued[s] - 1u) & 1u, 1000000000ull, p.err, nullptr);
      }
    }
  } else if (warp == 1) {
    // ===================================================== MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC[4] = {idesc_mxf8_f32(BM, BN, 0u), idesc_mxf8_f32(BM, BN, 1u),
                                     idesc_mxf8_f32(BM, BN, 2u), idesc_mxf8_f32(BM, BN, 3u)};
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
            const int j = m >> 2, kk = m & 3;
            umma_mxf8(d, smem_desc_kmajor_sw128(sb + j * A_TILE + kk * 32),
                      smem_desc_kmajor_sw128(sb + OFF_B + j * B_TILE + kk * 32), IDESC[m & 3], sf_t + 4 * (m >> 2),
                      sf_t + SF_COLS / 2 + 4 * (m >> 2), (kb | m) ? 1u : 0u);
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
  } else if (warp >= 6) {
    // ===================================================== scale warps (6..9)
    // lane l of the warp for lane quadrant q writes, for rows r = l + 32c of
    // the tile (c = 0..3), word w of the row's 8 stage bytes (MMAs 4w..4w+3)
    // into column 4w + c: A in columns 0..7, B in 8..15
    const int q = warp & 3;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const TileInfo ti = gg::decode_tile(t, s_prefix, s_off, GT, G, p.shared_rows);
      const Prob& P = p.prob[ti.pb];
      const int ld = P.K / 32;  // scale bytes per row
      const int a_y = ti.row0 + ti.m_blk * BM;
      const int f0 = ti.n_blk * TN;
      const uint2* arow[4];
      const uint2* brow[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int m = lane + 32 * c;  // row of the tile
        const int ar = a_y + m;
        arow[c] = ar < P.a_rows ? reinterpret_cast<const uint2*>(P.a_sf + static_cast<size_t>(ar) * ld) : nullptr;
        int br;
        bool bv;
        if (SWIGLU) {
          const int f = f0 + (m & 63);
          bv = f < P.n_out;
          br = ti.g * P.w_rows + (m < 64 ? 0 : P.n_out) + f;
        } else {
          bv = f0 + m < P.n_out;
          br = ti.g * P.w_rows + f0 + m;
        }
        brow[c] = bv ? reinterpret_cast<const uint2*>(P.w_sf + static_cast<size_t>(br) * ld) : nullptr;
      }
      const int nk = P.K / KE;
      for (int kb = 0; kb < nk; ++kb) {
        uint32_t r[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint2 a = arow[c] ? __ldg(arow[c] + kb) : make_uint2(0u, 0u);
          const uint2 b = brow[c] ? __ldg(brow[c] + kb) : make_uint2(0u, 0u);
          r[c] = a.x;
          r[4 + c] = a.y;
          r[8 + c] = b.x;
          r[12 + c] = b.y;
        }
        // the stage's tensor-memory scale columns are free once its previous
        // MMAs have completed
        if (!mbar_wait_warp(&empty[stage], phase ^ 1u, tmo, p.err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sf_t = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                              static_cast<uint32_t>(ACC_COLS + stage * SF_COLS);
        tmem_st_32x32b_x16(sf_t, r);
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
      gg::epilogue_tile<EPI, BN, false>(P, ti, taddr, r_in_tile, 1.0f);
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
        cudaFuncSetAttribute(grouped_gemm_mxf8_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) {
      set_cuda_error(e);
      return MOE_ERR_CUDA;
    }
    attr_done[dev] = true;
  }
  grouped_gemm_mxf8_kernel<EPI><<<num_sms(), THREADS, SMEM, s>>>(prm);
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
  const uint64_t K = static_cast<uint64_t>(P.K), nkb = K / KB_BYTES;
  {
    // A [a_rows, K] bytes as (byte in k-block, row, k-block)
    const uint64_t dims[3] = {KB_BYTES, static_cast<uint64_t>(P.a_rows), nkb};
    const uint64_t str[2] = {K, KB_BYTES};
    const uint32_t box[3] = {KB_BYTES, BM, KBLK};
    MOE_TRY(encode_tmap_nd(&prm.tma_a[slot], P.A, false, 3, dims, str, box, true));
  }
  if (swiglu) {
    // W [groups][gate N | up N][K] as (byte, row, gate/up + 2*group, k-block)
    const uint64_t N = static_cast<uint64_t>(P.N), g2 = 2 * static_cast<uint64_t>(P.groups);
    const uint64_t dims[4] = {KB_BYTES, N, g2, nkb};
    const uint64_t str[3] = {K, N * K, KB_BYTES};
    const uint32_t box[4] = {KB_BYTES, BN / 2, 2, KBLK};
    MOE_TRY(encode_tmap_nd(&prm.tma_w[slot], P.W, false, 4, dims, str, box, true));
  } else {
    const uint64_t rows = static_cast<uint64_t>(q.w_rows_total);
    const uint64_t dims[3] = {KB_BYTES, rows, nkb};
    const uint64_t str[2] = {K, KB_BYTES};
    const uint32_t box[3] = {KB_BYTES, BN, KBLK};
    MOE_TRY(encode_tmap_nd(&prm.tma_w[slot], P.W, false, 3, dims, str, box, true));
  }
  return MOE_OK;
}

}  // namespace gmx8

// MXFP8 x MXFP8, K % 256 == 0, 8-byte aligned scale arrays, bf16 and MX SwiGLU epilogues
// (checked by the caller, grouped_gemm_launch).
int grouped_gemm_launch_mxf8(int epi, const GemmProblem& routed, const int32_t* offsets, int G,
                             const GemmProblem* sh, int shared_rows, cudaStream_t s) {
  gg::Params prm;
  memset(&prm, 0, sizeof(prm));
  MOE_TRY(gmx8::fill(prm, 0, epi, routed));
  prm.offsets = offsets;
  prm.G = G;
  prm.shared_rows = -1;
  if (sh != nullptr && shared_rows > 0) {
    MOE_TRY(gmx8::fill(prm, 1, epi, *sh));
    prm.shared_rows = shared_rows;
  }
  prm.err = device_error_word();
  if (!prm.err) return MOE_ERR_CUDA;
  prm.timeout_ns = wait_timeout_ns();
  if (epi == MOE_EPI_STORE_BF16) return gmx8::launch<MOE_EPI_STORE_BF16>(prm, s);
  if (epi == MOE_EPI_SWIGLU_MX) return gmx8::launch<MOE_EPI_SWIGLU_MX>(prm, s);
  return gmx8::launch<MOE_EPI_SWIGLU_BF16>(prm, s);
}

}  // namespace moe
