// Grouped GEMM for bf16 operands on CTA pairs: one tcgen05 MMA spans the two
// SMs of a cluster (cta_group::2), M = 256 rows x N = 256 columns per tile.
//
// Why pairs: a single SM that stages a 128 x 64 A tile and a 256 x 64 B tile
// (48 KB) per k-step fits 4 stages in shared memory, and the time a stage
// takes to come back (issue -> TMA from L2/HBM -> MMA -> free) is longer than
// 4 stages of MMA work, so the tensor core waits.  With the pair each SM
// stages its own 128 A rows and only half of B (32 KB per k-step) for the same
// MMA work per SM, so 6 stages fit and the pipeline covers the round trip.
//
// Roles (both CTAs of the pair run the same tile sequence):
//   warp 0      TMA producer of this CTA: A rows [tile_row + 128*rank, +128),
//               B rows of this CTA's half of N; both loads complete on the
//               leader CTA's full barrier (the leader arms it for both)
//   warp 1      TMEM allocation of the pair; in the leader only, the MMA
//               issuer: 4 x tcgen05.mma.cta_group::2 (M=256, N=256, K=16) per
//               stage, commits multicast to both CTAs' empty / tfull barriers
//   warps 2..5  epilogue: each CTA reads its own 128 accumulator rows from its
//               tensor memory; SwiGLU / bf16 stores as the 1-SM kernel; then
//               releases the accumulator on the leader's tempty barrier
// For SwiGLU the leader stages the 128 gate rows of the tile and the peer the
// matching 128 up rows, so accumulator columns [0,128) are gate, [128,256) up.
// Tiles are (group, column block, 256-row block); a group's last row block
// may extend past the group (rows of the next group or past the end): those
// rows are computed and not stored.
#include <cstring>

#include "gemm_common.cuh"
#include "internal.h"

namespace moe {
namespace gp {

using gg::BM;
using gg::MAX_G;
using gg::Params;
using gg::Prob;
using gg::TileInfo;

constexpr int TM = 2 * BM;            // rows per pair tile
constexpr int BN = 256;               // accumulator columns (N of the MMA)
constexpr int BK = 64;                // bf16 elements per k-step (128-byte rows)
constexpr int A_TILE = BM * BK * 2;   // 16 KB: this CTA's 128 A rows
constexpr int B_TILE = 128 * BK * 2;  // 16 KB: this CTA's half of B
constexpr int STAGES = 6;
constexpr int STAGE_BYTES = A_TILE + B_TILE;
constexpr int NUM_WARPS = 6;
constexpr int THREADS = NUM_WARPS * 32;
constexpr int TMEM_COLS = 512;
constexpr uint32_t TX_BYTES_PAIR = 2 * STAGE_BYTES;  // both CTAs' loads, counted on the leader
constexpr int EXTRA = 2048 + 4 * (2 * MAX_G + 8);
constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + EXTRA;
static_assert(STAGE_BYTES % 1024 == 0, "stage must keep 1024-byte alignment");
static_assert(SMEM <= 232448, "shared memory budget");

template <int EPI>
struct Tile {
  static constexpr int N_OUT = (EPI == MOE_EPI_STORE_BF16) ? BN : BN / 2;  // output columns per tile
};

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1) grouped_gemm_pair_kernel(const __grid_constant__ Params p) {
  constexpr int S = STAGES;
  constexpr int TN = Tile<EPI>::N_OUT;
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
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int G = p.G;
  const int GT = G + (p.shared_rows >= 0 ? 1 : 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 8);  // 4 epilogue warps of each CTA
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, TMEM_COLS);
    tmem_relinquish_pair();
  }
  gg::build_schedule<THREADS, NUM_WARPS, TM>(p, s_off, s_prefix, warp_sums);
  tc_fence_before();
  // both CTAs' barriers exist before either signals the other
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int total = s_prefix[GT];
  const int cluster_id = blockIdx.x >> 1;
  const int n_clusters = gridDim.x >> 1;
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
      bool ok = true;
      for (int t = cluster_id; t < total && ok; t += n_clusters) {
        const TileInfo ti = gg::decode_tile<TM>(t, s_prefix, s_off, GT, G, p.shared_rows);
        const Prob& P = p.prob[ti.pb];
        const void* ta = &p.tma_a[ti.pb];
        const void* tw = &p.tma_w[ti.pb];
        const int a_y = ti.row0 + ti.m_blk * TM + static_cast<int>(rank) * BM;
        const int w_base = ti.g * P.w_rows + ti.n_blk * TN;
        // this CTA's half of B: STORE -> rows [128*rank, +128) of the 256-row
        // block; SwiGLU -> the 128 gate rows (leader) or the 128 up rows (peer)
        const int w_y = (EPI == MOE_EPI_STORE_BF16) ? w_base + static_cast<int>(rank) * 128
                                                    : w_base + (leader ? 0 : P.n_out);
        const int nk = P.K / BK;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, tmo, p.err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sb = stages + stage * STAGE_BYTES;
          const uint32_t fbar = mapa_shared(smem_u32(&full[stage]), 0);
          if (leader) mbar_arrive_expect_tx(&full[stage], TX_BYTES_PAIR);
          tma_load_2d_pair(ta, fbar, sb, kb * BK, a_y);
          tma_load_2d_pair(tw, fbar, sb + A_TILE, kb * BK, w_y);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ===================================================== MMA issuer (leader)
    if (lane == 0 && leader) {
      constexpr uint32_t IDESC = idesc_bf16_f32(TM, BN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int t = cluster_id; t < total && ok; t += n_clusters, ++it) {
        const TileInfo ti = gg::decode_tile<TM>(t, s_prefix, s_off, GT, G, p.shared_rows);
        const int nk = p.prob[ti.pb].K / BK;
        const int buf = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        // both CTAs' epilogues must have drained this accumulator buffer
        {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait_cluster(&tempty[buf], (use & 1u) ^ 1u)) {
            if (*abort_flag || globaltimer_ns() - t0 > tmo) {
              atomicOr(p.err, kErrTimeout);
              *abort_flag = 1;
              ok = false;
              break;
            }
          }
          if (!ok) break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, tmo, p.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stages + stage * STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_TILE;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_f16_pair(d, smem_desc_kmajor_sw128(a_addr + kk * 32), smem_desc_kmajor_sw128(b_addr + kk * 32),
                          IDESC, (kb | kk) ? 1u : 0u);
          umma_commit_pair_multicast(&empty[stage], 0x3);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit_pair_multicast(&tfull[buf], 0x3);
      }
      if (!ok) {
        umma_commit_pair_multicast(drain, 0x1);
        mbar_wait_bounded(drain, 0, 1000000000ull, p.err, nullptr);
      }
    }
  } else {
    // ===================================================== epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int r_in_tile = q * 32 + lane;
    const uint32_t tempty_leader = mapa_shared(smem_u32(&tempty[0]), 0);
    int it = 0;
    for (int t = cluster_id; t < total; t += n_clusters, ++it) {
      TileInfo ti = gg::decode_tile<TM>(t, s_prefix, s_off, GT, G, p.shared_rows);
      const Prob& P = p.prob[ti.pb];
      const int buf = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      if (!mbar_wait_warp(&tfull[buf], use & 1u, tmo, p.err, abort_flag)) break;
      tc_fence_after();
      // this CTA holds rows [128*rank, +128) of the 256-row tile
      ti.m_blk = 2 * ti.m_blk + static_cast<int>(rank);
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * BN);
      gg::epilogue_tile<EPI, BN>(P, ti, taddr, r_in_tile, 1.0f);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(&tempty[buf]);
        else
          mbar_arrive_remote(tempty_leader + static_cast<uint32_t>(buf) * 8u);
      }
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
  // the leader's MMAs read this CTA's shared memory and write its tensor
  // memory: neither CTA leaves or frees tensor memory before both are done
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

template <int EPI>
static int launch(const Params& prm, cudaStream_t s) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(grouped_gemm_pair_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) {
      set_cuda_error(e);
      return MOE_ERR_CUDA;
    }
    attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms() & ~1), 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<EPI>, prm);
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
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
  q.c_sf = nullptr;
  q.a_g = q.w_g = q.c_g = nullptr;
  q.a_sf = q.w_sf = nullptr;
  MOE_TRY(encode_tmap_2d(&prm.tma_a[slot], P.A, 2, P.K, static_cast<uint64_t>(P.a_rows), BK, BM, true));
  MOE_TRY(encode_tmap_2d(&prm.tma_w[slot], P.W, 2, P.K, static_cast<uint64_t>(q.w_rows_total), BK, 128, true));
  return MOE_OK;
}

}  // namespace gp

// bf16 x bf16 problems on CTA pairs.  Arguments were checked by
// grouped_gemm_launch.
int grouped_gemm_launch_pair(int epi, const GemmProblem& routed, const int32_t* offsets, int G,
                             const GemmProblem* sh, int shared_rows, cudaStream_t s) {
  gg::Params prm;
  memset(&prm, 0, sizeof(prm));
  MOE_TRY(gp::fill(prm, 0, epi, routed));
  prm.offsets = offsets;
  prm.G = G;
  prm.shared_rows = -1;
  if (sh != nullptr && shared_rows > 0) {
    MOE_TRY(gp::fill(prm, 1, epi, *sh));
    prm.shared_rows = shared_rows;
  }
  prm.err = device_error_word();
  if (!prm.err) return MOE_ERR_CUDA;
  prm.timeout_ns = wait_timeout_ns();
  if (epi == MOE_EPI_STORE_BF16) return gp::launch<MOE_EPI_STORE_BF16>(prm, s);
  return gp::launch<MOE_EPI_SWIGLU_BF16>(prm, s);
}

}  // namespace moe
