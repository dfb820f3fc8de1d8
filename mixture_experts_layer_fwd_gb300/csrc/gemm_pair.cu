// Grouped GEMM for bf16 operands on CTA pairs: one tcgen05 MMA spans the two
// SMs of a cluster (cta_group::2).  The weights are the MMA's M side (256
// weight rows per pair tile, 128 per SM) and the tokens its N side (up to 256
// tokens per tile, any multiple of 16), so the accumulator holds C^T.
//
// Why pairs: each SM stages its own 128 weight rows and only half of the
// tile's tokens, so a 128-wide k step costs 64 KB of shared memory per SM for
// an M=256 x N=256 MMA, and three such stages fit.
//
// Why weights on M: a group of r routed rows is cut into ceil(r/256) token
// blocks of equal size rounded up to 16 (the MMA's N granularity), so a
// group wastes at most 15 rows of MMA work per block instead of up to 255
// rows of a 256-row M tile.
//
// Why 128-wide k stages with one copy per operand: every stage costs the
// producer and the MMA issuer a fixed amount of barrier traffic (wait, arm,
// commit) and every copy instruction adds issue time; two 64-wide k-blocks
// per stage, each operand moved by one 3-D/4-D box (k-block as the outer
// box dimension), halve that cost per MMA compared with 64-wide stages of two
// 2-D copies.  Small-N tiles remain bound by that per-stage cost.
//
// Roles (both CTAs of the pair run the same tile sequence):
//   warp 0      TMA producer of this CTA: one box of its 128 weight rows x
//               2 k-blocks and one box of h token rows (from its half of
//               the tile's tokens on; h = N/2 rounded up to 16, one tensor
//               map per height) x 2 k-blocks; both copies complete on the
//               leader CTA's full barrier, which the leader arms for both
//   warp 1      TMEM allocation of the pair; in the leader only, the MMA
//               issuer: 8 x tcgen05.mma.cta_group::2 (M=256, N=tile tokens,
//               K=16) per stage from precomputed descriptors, commits
//               multicast to both CTAs' empty / tfull barriers
//   warps 2..5  epilogue: each CTA reads its 128 accumulator lanes (weight
//               rows) x tokens from its tensor memory and stores C[token, col]
//               with 4-byte stores (two columns, exchanged between lanes);
//               then releases the accumulator on the leader's tempty barrier
// SwiGLU: each CTA stages the 64 gate rows of features [f0, f0+64) followed
// by the 64 up rows of the same features (one 4-D TMA box), so accumulator
// lanes 0..63 hold gate and 64..127 up.  The warp of gate lanes 32q and the
// warp of up lanes 32q+64 swap half of their 32-token chunks through shared
// memory (named barrier per warp pair) and each computes silu(gate) * up for
// the chunks it stores.
#include <cstring>

#include "gemm_common.cuh"
#include "internal.h"

namespace moe {
namespace gp {

using gg::MAX_G;
using gg::Params;
using gg::Prob;

constexpr int TM = 256;               // most tokens per tile (N of the MMA)
constexpr int WM = 128;               // weight rows per CTA (M of the MMA is 2 x WM)
constexpr int BK = 64;                // bf16 elements per k-block (128-byte rows)
constexpr int GU_ROWS = 64;           // SwiGLU: features per CTA (64 gate + 64 up rows)
constexpr int A_TILE = WM * BK * 2;   // 16 KB: this CTA's weight rows
constexpr int B_ROWS = 128;           // most token rows staged per CTA (half of the largest N)
constexpr int B_STEP = 16;            // a tile stages ceil(N/2 / 16) * 16 token rows per CTA
constexpr int B_TILE = B_ROWS * BK * 2;
constexpr int KSUB = 2;               // k-blocks per pipeline stage (128 of K)
constexpr int STAGES = 3;
constexpr int STAGE_BYTES = KSUB * (A_TILE + B_TILE);  // [A k-block 0][A 1][B 0][B 1]
static_assert(B_ROWS / B_STEP == 8, "one token tensor map per box height");
constexpr int NUM_WARPS = 6;
constexpr int THREADS = NUM_WARPS * 32;
constexpr int TMEM_COLS = 512;
constexpr int EXTRA = (2048 + 4 * (2 * MAX_G + 8) + 15) & ~15;
constexpr int XCH_FLOATS = 32 * 32;                // one 32-lane x 32-token chunk
constexpr int XCH_BYTES = 2 * 2 * XCH_FLOATS * 4;  // 2 warp pairs x 2 directions
constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + EXTRA + XCH_BYTES + 64;
static_assert(STAGE_BYTES % 1024 == 0, "stage must keep 1024-byte alignment");
static_assert(KSUB == 2, "the MMA issuer unrolls two k-blocks per stage");
static_assert(SMEM <= 232448, "shared memory budget");

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1) grouped_gemm_pair_kernel(const __grid_constant__ Params p) {
  constexpr int S = STAGES;
  constexpr bool SWIGLU = EPI == MOE_EPI_SWIGLU_BF16;
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
  float* xch = reinterpret_cast<float*>(base + S * STAGE_BYTES + EXTRA);
  volatile int* pair_ok = reinterpret_cast<volatile int*>(xch + 4 * XCH_FLOATS);  // [2 pairs][gate, up]
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
      tma_prefetch_desc(&p.tma_w[0]);
      if (p.shared_rows >= 0) tma_prefetch_desc(&p.tma_w[1]);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = cluster_id; t < total && ok; t += n_clusters) {
        const gg::PairTile ti = gg::decode_pair_tile<TM>(t, s_prefix, s_off, GT, G, p.shared_rows);
        const Prob& P = p.prob[ti.pb];
        // this CTA's token box: the half of the tile's N it stages, rounded
        // up to 16 rows (fewer staged bytes for small token blocks)
        const int h = (((ti.n >> 1) + B_STEP - 1) / B_STEP) * B_STEP;
        const void* ta = &p.tma_b_rows[ti.pb][h / B_STEP - 1];
        const void* tw = &p.tma_w[ti.pb];
        const uint32_t tx = 2u * static_cast<uint32_t>(KSUB * (A_TILE + h * BK * 2));  // both CTAs, on the leader
        // this CTA's tokens start half of N into the tile (half <= 128)
        const int b_y = ti.row0 + static_cast<int>(rank) * (ti.n >> 1);
        // this CTA's 128 weight rows: SwiGLU -> gate and up rows of features
        // [blk*128 + 64*rank, +64); STORE -> rows [blk*256 + 128*rank, +128)
        const int f0 = ti.blk * 128 + static_cast<int>(rank) * GU_ROWS;
        const int w_y0 = ti.g * P.w_rows + ti.blk * 256 + static_cast<int>(rank) * WM;
        const int nk = P.K / BK;
        for (int kb = 0; kb < nk; kb += KSUB) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, tmo, p.err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sb = stages + stage * STAGE_BYTES;
          const uint32_t fbar = mapa_shared(smem_u32(&full[stage]), 0);
          // one copy per operand moves both k-blocks of the stage (a k-block
          // past the end of K is zero-filled and still counted)
          if (leader) mbar_arrive_expect_tx(&full[stage], tx);
          if (SWIGLU)
            tma_load_4d_pair(tw, fbar, sb, 0, f0, 2 * ti.g, kb);
          else
            tma_load_3d_pair(tw, fbar, sb, 0, w_y0, kb);
          tma_load_3d_pair(ta, fbar, sb + KSUB * A_TILE, 0, b_y, kb);
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
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      // The issuing thread's own instruction count per MMA sets the MMA
      // rate for small N, so descriptors are built once: a stage, k-block
      // and 16-wide k step only add (byte offset >> 4) to the start field.
      const uint64_t a_desc0 = smem_desc_kmajor_sw128(smem_u32(stages));
      const uint64_t b_desc0 = smem_desc_kmajor_sw128(smem_u32(stages + KSUB * A_TILE));
      for (int t = cluster_id; t < total && ok; t += n_clusters, ++it) {
        const gg::PairTile ti = gg::decode_pair_tile<TM>(t, s_prefix, s_off, GT, G, p.shared_rows);
        const int nk = p.prob[ti.pb].K / BK;
        const uint32_t idesc = idesc_bf16_f32(2 * WM, ti.n);
        // second token k-block of a stage: after the first one's h rows
        const uint64_t b_kblk = static_cast<uint64_t>(((((ti.n >> 1) + B_STEP - 1) / B_STEP) * B_STEP * BK * 2) >> 4);
        const int buf = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        // both CTAs' epilogues must have drained this accumulator buffer
        {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait_relaxed_cluster(&tempty[buf], (use & 1u) ^ 1u)) {
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
        const uint32_t d = tmem_base + static_cast<uint32_t>(buf * TM);
        for (int kb = 0; kb < nk; kb += KSUB) {
          const int nsub = min(KSUB, nk - kb);
          if (!mbar_wait_bounded(&full[stage], phase, tmo, p.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t da = a_desc0 + static_cast<uint64_t>((stage * STAGE_BYTES) >> 4);
          const uint64_t db = b_desc0 + static_cast<uint64_t>((stage * STAGE_BYTES) >> 4);
          const uint32_t acc0 = kb != 0 ? 1u : 0u;
          umma_f16_pair(d, da, db, idesc, acc0);
#pragma unroll
          for (int kk = 1; kk < BK / 16; ++kk) umma_f16_pair(d, da + 2 * kk, db + 2 * kk, idesc, 1u);
          if (nsub > 1) {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              umma_f16_pair(d, da + (A_TILE >> 4) + 2 * kk, db + b_kblk + 2 * kk, idesc, 1u);
          }
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
    const uint32_t tempty_leader = mapa_shared(smem_u32(&tempty[0]), 0);
    // SwiGLU: quadrants 0,1 hold gate rows, 2,3 the up rows of the same
    // features; warps (q, q+2) form exchange pair pi = q & 1
    const int pi = q & 1;
    const bool is_gate = q < 2;
    float* x_to_up = xch + pi * 2 * XCH_FLOATS;  // gate values the up warp consumes
    float* x_to_gate = x_to_up + XCH_FLOATS;     // up values the gate warp consumes
    int it = 0;
    for (int t = cluster_id; t < total; t += n_clusters, ++it) {
      const gg::PairTile ti = gg::decode_pair_tile<TM>(t, s_prefix, s_off, GT, G, p.shared_rows);
      const Prob& P = p.prob[ti.pb];
      const int buf = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      bool ok = mbar_wait_warp(&tfull[buf], use & 1u, tmo, p.err, abort_flag);
      if (SWIGLU) {
        // both warps of the pair leave together if either wait gave up, so
        // that neither is left alone at the exchange barriers below
        if (lane == 0) pair_ok[pi * 2 + (is_gate ? 0 : 1)] = ok ? 1 : 0;
        named_bar_sync(1 + pi, 64);
        ok = pair_ok[pi * 2] && pair_ok[pi * 2 + 1];
      }
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * TM);
      const int nch = (ti.cnt + 31) >> 5;
      if (SWIGLU) {
        const int col = ti.blk * 128 + static_cast<int>(rank) * GU_ROWS + pi * 32 + lane;  // feature
        for (int c = 0; c < nch; c += 2) {
          const bool has1 = c + 1 < nch;
          uint32_t v0[32], v1[32];
          tmem_ld_32x32b_x32(taddr + c * 32, v0);
          if (has1) tmem_ld_32x32b_x32(taddr + (c + 1) * 32, v1);
          tmem_ld_wait();
          // the gate warp finishes chunk c, the up warp chunk c+1
          if (is_gate) {
            if (has1) {
#pragma unroll
              for (int j = 0; j < 32; ++j) x_to_up[j * 32 + lane] = __uint_as_float(v1[j]);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) x_to_gate[j * 32 + lane] = __uint_as_float(v0[j]);
          }
          named_bar_sync(1 + pi, 64);
          float h[32];
          if (is_gate) {
#pragma unroll
            for (int j = 0; j < 32; ++j) h[j] = gg::silu_f(__uint_as_float(v0[j])) * x_to_gate[j * 32 + lane];
            gg::store_pairs<32>(P, h, col, ti.row0 + c * 32, ti.cnt - c * 32, lane);
          } else if (has1) {
#pragma unroll
            for (int j = 0; j < 32; ++j) h[j] = gg::silu_f(x_to_up[j * 32 + lane]) * __uint_as_float(v1[j]);
            gg::store_pairs<32>(P, h, col, ti.row0 + (c + 1) * 32, ti.cnt - (c + 1) * 32, lane);
          }
          // the slots are rewritten by the next chunk pair
          named_bar_sync(1 + pi, 64);
        }
      } else {
        const int col = ti.blk * 256 + static_cast<int>(rank) * WM + q * 32 + lane;  // output column
        for (int c = 0; c < nch; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(taddr + c * 32, v);
          tmem_ld_wait();
          float h[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) h[j] = __uint_as_float(v[j]);
          gg::store_pairs<32>(P, h, col, ti.row0 + c * 32, ti.cnt - c * 32, lane);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(&tempty[buf]);
        else
          mbar_arrive_remote_relaxed(tempty_leader + static_cast<uint32_t>(buf) * 8u);
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
  const int tn = (epi == MOE_EPI_STORE_BF16) ? 256 : 128;  // output columns per weight block
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
  for (int i = 0; i < B_ROWS / B_STEP; ++i)
    MOE_TRY(encode_tmap_kblocks(&prm.tma_b_rows[slot][i], P.A, P.K, static_cast<uint64_t>(P.a_rows),
                                static_cast<uint32_t>(B_STEP * (i + 1)), KSUB));
  if (epi == MOE_EPI_STORE_BF16)
    MOE_TRY(encode_tmap_kblocks(&prm.tma_w[slot], P.W, P.K, static_cast<uint64_t>(q.w_rows_total), WM, KSUB));
  else
    MOE_TRY(encode_tmap_gateup(&prm.tma_w[slot], P.W, P.K, P.N, P.groups, GU_ROWS, KSUB));
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
