// Down projection (bf16 output) with both operands in NVFP4 on CTA pairs:
// one block-scaled FP4 MMA (tcgen05.mma.cta_group::2 kind::mxf4nvf4,
// block_scale, scale_vec::4X) spans the two SMs of a cluster.  The weights are
// the MMA's M side (256 weight rows per pair, 128 per SM) and the tokens its N
// side (up to 160 tokens per tile, the MMA's N the tile's tokens rounded up
// to 32), so the accumulator holds C^T, as in the bf16 and MXFP8 pair
// kernels.
//
// "Driving vLLM WideEP ... (Part I)", section "NVFP4 GEMM for MoE and
// O-proj": packed 4-bit weights with per-group FP8 scales, dequantised inside
// the tensor cores; section "NVFP4 MoE dispatch": the activations arrive in
// NVFP4 too.
//
// Why pairs with tokens on N: a 1-SM 128 x 128 tile stages 256 rows of codes
// and scales per 128 x 128 outputs; here each SM stages its 128 weight rows
// and 80 token rows for 128 x 160 outputs.  On prefill-sized groups this is
// the faster kernel for the down projection (short k loops, bf16 output);
// for the SwiGLU projection, with its long k loop and NVFP4 output, the 1-SM
// kernel of gemm_fp4w.cu measured faster, and takes it.
//
// Stages: 512 elements of K (two 256-element k-blocks of 128 bytes per row):
// 16 KB of weight codes per k-block and 10 KB of token codes per SM, by TMA
// (128-byte swizzle); 8 MMAs of K = 64.  Three stages.
//
// Scales in tensor memory: an M = 256 block-scaled MMA reads, in each CTA,
// the scales of that CTA's 128 A rows and of all N B rows; row r sits in
// lane r % 32, column r / 32 (the same in the four lane quadrants), one
// 32-bit cell of four E4M3 bytes per row and MMA.  A stage's slot is 96
// columns: A in 0..31 (column 4m + c: MMA m's word of weight row lane + 32c),
// B in 32..95 (column 32 + 8m + c, c < N/32).  Tensor memory holds two fp32
// accumulators (columns 0..159 and 256..415) and two slots in the gaps
// (columns 160 and 416), so the scales of a stage are written while the
// previous stage's MMAs run, and each slot is freed by its stage's MMA
// commit.  A stage's scales are 32 bytes per row: the four scale warps of
// each CTA copy them with cp.async (16 bytes at a time) into a ring in
// shared memory, SF_DEPTH - 1 stages ahead, and write the slot with three
// tcgen05.st.
//
// Roles (both CTAs of the pair run the same tile sequence):
//   warp 0        weight codes of this CTA's 128 rows (one 3-D box: both
//                 k-blocks); the leader arms the pair's full barrier for
//                 both CTAs' code bytes
//   warp 6        token codes: 80 rows from this CTA's half of the tile on
//   warps 7..10   scale warps, one per lane quadrant: ring of copies, wait
//                 for the slot, write it, arrive on the leader's full barrier
//   warp 1        tensor-memory allocation of the pair; in the leader only,
//                 the MMA issuer, a whole converged warp: 8 x
//                 tcgen05.mma.cta_group::2 (M=256, N=tile tokens, K=64) per
//                 stage, commits multicast to both CTAs' empty / scale-slot /
//                 tfull barriers; it starts each stage on a named-barrier
//                 signal
//   warp 11       in the leader only: the MMA warp's waits (full barrier of
//                 each stage, accumulator drained at a tile's start)
//   warps 2..5,   epilogue, two warps per lane quadrant (even and odd
//   12..15        32-token chunks): each CTA reads its 128 accumulator lanes
//                 (output columns) x tokens, applies the global scales
//                 g_a * g_w[e] and stores bf16 C[token, col]
// Requires K % 512 == 0 and 16-byte aligned scale arrays.
#include <cstring>

#include "gemm_common.cuh"
#include "internal.h"

namespace moe {
namespace gf4p {

using gg::MAX_G;
using gg::Params;
using gg::Prob;

constexpr int TN = 160;                    // most tokens per tile (N of the MMA)
constexpr int NQ = 32;                     // the MMA's N is a multiple of 32
constexpr int WM = 128;                    // weight rows per CTA (M of the MMA is 2 x WM)
constexpr int KB_BYTES = 128;              // code bytes of one 256-element k-block row
constexpr int KSUB = 2;                    // k-blocks per stage
constexpr int KE = KSUB * 256;             // elements per stage
constexpr int MMAS = KE / 64;              // MMAs per stage
constexpr int B_ROWS = TN / 2;             // token rows staged per CTA (>= half of N)
constexpr int A_TILE = WM * KB_BYTES;      // 16 KB per k-block
constexpr int B_TILE = B_ROWS * KB_BYTES;  // 10 KB per k-block
constexpr int OFF_B = KSUB * A_TILE;
constexpr int STAGE_BYTES = OFF_B + KSUB * B_TILE;  // 52 KB
constexpr int STAGES = 3;
constexpr uint32_t TX_CODES_PAIR = 2u * STAGE_BYTES;  // both CTAs' copies, counted on the leader
constexpr int ACC_STRIDE = 256;            // accumulator buffers at columns 0 and 256
constexpr int SFB_OFF = 4 * MMAS;          // B scales after A's 8 MMAs x 4 columns
constexpr int SFB_STRIDE = TN <= 128 ? 4 : 8;     // B columns per MMA (N/32 used)
constexpr int SF_SLOT_COLS = SFB_OFF + SFB_STRIDE * MMAS;
constexpr int SF_GAP0 = (ACC_STRIDE - TN) / SF_SLOT_COLS;  // slots after the first accumulator
constexpr int SF_SLOTS = 2;                // scale slots in the gaps after the accumulators
constexpr int NUM_WARPS = 16;
constexpr int W_EPI1 = 12;                 // second set of epilogue warps (12..15)
constexpr int THREADS = NUM_WARPS * 32;
constexpr int TMEM_COLS = 512;
constexpr int W_PROD_B = 6, W_SCALE0 = 7, W_WAIT = 11;
constexpr int MMA_BAR = 4;                 // named barrier of the MMA warp and the wait warp
constexpr int EXTRA = (2048 + 4 * (2 * MAX_G + 8) + 15) & ~15;
constexpr int SF_DEPTH = 3;                        // scale stages in the shared-memory ring
constexpr int SF_A_ROWS = WM;                      // ring slot: 128 weight rows, then TN token rows
constexpr int SF_ROW_BYTES = KE / 16;              // 32 scale bytes per row and stage
constexpr int SF_RING_SLOT = (SF_A_ROWS + TN) * SF_ROW_BYTES;
constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + EXTRA + SF_DEPTH * SF_RING_SLOT;
static_assert(STAGE_BYTES % 1024 == 0 && B_TILE % 1024 == 0, "tiles must keep 1024-byte alignment");
static_assert(MMAS == 8 && TN % 32 == 0 && TN / 32 <= 8, "a slot holds 8 MMAs of A and B scales");
static_assert(SF_GAP0 >= 1 && ACC_STRIDE + TN + (SF_SLOTS - SF_GAP0) * SF_SLOT_COLS <= TMEM_COLS,
              "scale slots fit the gaps after the accumulators");
static_assert(TN / 32 <= SFB_STRIDE, "B scales fit their columns");
static_assert(TN >= 128 && TN <= 256, "the 128 scale threads copy one weight row and one or two token rows");
static_assert(SMEM <= 232448, "shared memory budget");

// tensor-memory column of scale slot s
DEVINL uint32_t sf_slot(uint32_t s) {
  return s < SF_GAP0 ? TN + s * SF_SLOT_COLS : ACC_STRIDE + TN + (s - SF_GAP0) * SF_SLOT_COLS;
}

DEVINL void umma_nvf4_pair_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

DEVINL void cp_async_16(uint32_t dst_smem, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst_smem), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}

DEVINL uint4 ld_shared_u4(uint32_t saddr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(saddr)
               : "memory");
  return v;
}

__global__ void __launch_bounds__(THREADS, 1) grouped_gemm_nvf4p_kernel(const __grid_constant__ Params p) {
  constexpr int S = STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = base;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + S * STAGE_BYTES);  // leader: codes + scale-warp arrivals
  uint64_t* empty = full + S;                                            // stage free (MMA commit)
  uint64_t* sf_empty = empty + S;                                        // [2] scale slot free (MMA commit)
  uint64_t* tfull = sf_empty + SF_SLOTS;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_prefix = reinterpret_cast<int*>(base + S * STAGE_BYTES + 256);
  int* s_off = s_prefix + MAX_G + 4;
  uint8_t* sf_ring = base + S * STAGE_BYTES + EXTRA;
  __shared__ int warp_sums[32];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int G = p.G;
  const int GT = G + (p.shared_rows >= 0 ? 1 : 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1 + 8);  // the leader's arm + 4 scale warps of each CTA
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < SF_SLOTS; ++b) mbar_init(&sf_empty[b], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 16);  // 8 epilogue warps of each CTA
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, TMEM_COLS);
    tmem_relinquish_pair();
  }
  gg::build_schedule<THREADS, NUM_WARPS, TN>(p, s_off, s_prefix, warp_sums);
  tc_fence_before();
  // both CTAs' barriers exist before either signals the other
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int total = s_prefix[GT];
  const int cluster_id = blockIdx.x >> 1;
  const int n_clusters = gridDim.x >> 1;
  const unsigned long long tmo = p.timeout_ns;

  if (warp == 0 || warp == W_PROD_B) {
    // ===================================================== TMA producers
    if (lane == 0) {
      const bool is_w = warp == 0;
      for (int pb = 0; pb < (p.shared_rows >= 0 ? 2 : 1); ++pb) tma_prefetch_desc(is_w ? &p.tma_w[pb] : &p.tma_a[pb]);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = cluster_id; t < total && ok; t += n_clusters) {
        const gg::PairTile ti = gg::decode_pair_tile<TN, NQ>(t, s_prefix, s_off, GT, G, p.shared_rows);
        const Prob& P = p.prob[ti.pb];
        // this CTA's tokens start half of N into the tile (half <= 80)
        const int b_y = ti.row0 + static_cast<int>(rank) * (ti.n >> 1);
        // this CTA's 128 weight rows [blk*256 + 128*rank, +128)
        const int w_y0 = ti.g * P.w_rows + ti.blk * 256 + static_cast<int>(rank) * WM;
        const int nk = P.K / KE;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, tmo, p.err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sb = stages + stage * STAGE_BYTES;
          const uint32_t fbar = mapa_shared(smem_u32(&full[stage]), 0);
          const int kblk = kb * KSUB;
          if (is_w) {
            if (leader) mbar_arrive_expect_tx(&full[stage], TX_CODES_PAIR);
            tma_load_3d_pair(&p.tma_w[ti.pb], fbar, sb, 0, w_y0, kblk);
          } else {
            tma_load_3d_pair(&p.tma_a[ti.pb], fbar, sb + OFF_B, 0, b_y, kblk);
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ===================================================== MMA issuer (leader)
    // The whole warp walks the schedule and issues; each stage starts on the
    // go signal of the wait warp, so this warp never waits on an mbarrier
    // between its MMAs.
    if (leader) {
      int stage = 0;
      uint32_t sf_use = 0;  // stages issued so far (scale slot = sf_use % SF_SLOTS)
      bool ok = true;
      int it = 0;
      const uint64_t a_desc0 = smem_desc_kmajor_sw128(smem_u32(stages));
      const uint64_t b_desc0 = smem_desc_kmajor_sw128(smem_u32(stages + OFF_B));
      for (int t = cluster_id; t < total && ok; t += n_clusters, ++it) {
        const gg::PairTile ti = gg::decode_pair_tile<TN, NQ>(t, s_prefix, s_off, GT, G, p.shared_rows);
        const int nk = p.prob[ti.pb].K / KE;
        const uint32_t idesc = idesc_nvf4_f32(2 * WM, ti.n);
        const int buf = it & 1;
        const uint32_t d = tmem_base + static_cast<uint32_t>(buf * ACC_STRIDE);
        for (int kb = 0; kb < nk; ++kb, ++sf_use) {
          if (named_bar_red_or(MMA_BAR, 64, false)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t slot = sf_use % SF_SLOTS;
          const uint32_t sf_t = tmem_base + sf_slot(slot);
          const uint64_t da = a_desc0 + static_cast<uint64_t>((stage * STAGE_BYTES) >> 4);
          const uint64_t db = b_desc0 + static_cast<uint64_t>((stage * STAGE_BYTES) >> 4);
#pragma unroll
          for (int m = 0; m < MMAS; ++m) {
            const int j = m >> 2, kk = m & 3;  // k-block, 32-byte step inside it
            umma_nvf4_pair_warp(d, da + ((j * A_TILE + kk * 32) >> 4), db + ((j * B_TILE + kk * 32) >> 4), idesc,
                                sf_t + 4 * m, sf_t + SFB_OFF + SFB_STRIDE * m, (kb | m) ? 1u : 0u);
          }
          umma_commit_pair_multicast_warp(&empty[stage], 0x3);
          umma_commit_pair_multicast_warp(&sf_empty[slot], 0x3);
          if (++stage == S) stage = 0;
        }
        if (ok) umma_commit_pair_multicast_warp(&tfull[buf], 0x3);
      }
      if (!ok && lane == 0) {
        umma_commit_pair_multicast(drain, 0x1);
        mbar_wait_bounded(drain, 0, 1000000000ull, p.err, nullptr);
      }
    }
  } else if (warp == W_WAIT) {
    // ===================================================== waits for the MMA warp (leader)
    if (leader) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = cluster_id; t < total && ok; t += n_clusters, ++it) {
        const gg::PairTile ti = gg::decode_pair_tile<TN, NQ>(t, s_prefix, s_off, GT, G, p.shared_rows);
        const int nk = p.prob[ti.pb].K / KE;
        const int buf = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        for (int kb = 0; kb < nk; ++kb) {
          // kb == 0: both CTAs' epilogues have drained this accumulator
          // buffer; every stage: codes of both CTAs landed and all 8 scale
          // warps wrote the stage's slot
          const bool good = (kb > 0 || wait_cluster_warp(&tempty[buf], (use & 1u) ^ 1u, tmo, p.err, abort_flag)) &&
                            mbar_wait_warp(&full[stage], phase, tmo, p.err, abort_flag);
          if (named_bar_red_or(MMA_BAR, 64, !good)) {
            ok = false;
            break;
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp >= W_SCALE0 && warp < W_SCALE0 + 4) {
    // ===================================================== scale warps (7..10)
    // The 128 threads copy each stage's 32 scale bytes of the CTA's 128
    // weight rows and the tile's token rows (one to three rows each, 16
    // bytes per copy) into a ring of SF_DEPTH slots in shared memory with
    // cp.async, SF_DEPTH - 1 stages ahead of the stage they write to tensor
    // memory; after a barrier of the four warps each lane reads its rows.
    const int q = warp & 3;  // lane quadrant this warp writes
    const int st = (warp - W_SCALE0) * 32 + lane;  // copying thread 0..127
    const uint32_t full_leader = mapa_shared(smem_u32(&full[0]), 0);
    const uint32_t ring = smem_u32(sf_ring);
    // prefetch cursor: tile ct, stage ckb of cnk; this thread's rows st
    // (weight row st), SF_A_ROWS + st and SF_A_ROWS + 128 + st (token rows)
    int ct = cluster_id, ckb = 0, cnk = 0;
    const uint8_t* any = nullptr;  // a valid address for the zero-filling copies
    const uint8_t* rp[3];
    auto open_tile = [&]() {
      if (ct >= total) return;
      const gg::PairTile ti = gg::decode_pair_tile<TN, NQ>(ct, s_prefix, s_off, GT, G, p.shared_rows);
      const Prob& P = p.prob[ti.pb];
      const int ld = P.K / 16;  // scale bytes per row
      cnk = P.K / KE;
      ckb = 0;
      any = P.w_sf;
      {
        const int col = ti.blk * 256 + static_cast<int>(rank) * WM + st;  // this CTA's weight row st
        rp[0] = col < P.n_out ? P.w_sf + static_cast<size_t>(ti.g * P.w_rows + col) * ld : nullptr;
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int j = st + 128 * c;  // token of the tile (MMA column)
        rp[1 + c] = (j < TN && j < ti.cnt) ? P.a_sf + static_cast<size_t>(ti.row0 + j) * ld : nullptr;
      }
    };
    auto copy_row = [&](uint32_t dst, const uint8_t* row, int off) {
      cp_async_16(dst, row ? row + off : any, row != nullptr);
      cp_async_16(dst + 16, row ? row + off + 16 : any, row != nullptr);
    };
    // copies the cursor's stage into ring slot `slot` and advances; commits
    // a (possibly empty) group either way so that group counts stay uniform
    auto issue = [&](int slot) -> bool {
      const bool has = ct < total;
      if (has) {
        const uint32_t d = ring + static_cast<uint32_t>(slot * SF_RING_SLOT + st * SF_ROW_BYTES);
        const int off = ckb * SF_ROW_BYTES;
        copy_row(d, rp[0], off);
        copy_row(d + SF_A_ROWS * SF_ROW_BYTES, rp[1], off);
        if (st + 128 < TN) copy_row(d + (SF_A_ROWS + 128) * SF_ROW_BYTES, rp[2], off);
        if (++ckb == cnk) {
          ct += n_clusters;
          open_tile();
        }
      }
      cp_async_commit();
      return has;
    };
    open_tile();
    int pending = 0;  // stages copied and not yet written to tensor memory
#pragma unroll
    for (int i = 0; i < SF_DEPTH - 1; ++i) pending += issue(i) ? 1 : 0;
    int stage = 0, rslot = 0;
    uint32_t phase = 0, sf_use = 0;
    // all four warps run every stage of the schedule (the barrier below
    // counts them); after a wait gave up a warp only stops writing
    bool ok = true;
    while (pending > 0) {
      cp_async_wait_group<SF_DEPTH - 2>();  // this thread's copies of the ring slot landed
      // everyone's copies of the ring slot are visible, and everyone has read
      // the ring slot refilled next
      named_bar_sync(3, 128);
      pending += issue(rslot == 0 ? SF_DEPTH - 1 : rslot - 1) ? 1 : 0;
      const uint32_t d = ring + static_cast<uint32_t>(rslot * SF_RING_SLOT + lane * SF_ROW_BYTES);
      --pending;
      if (++rslot == SF_DEPTH) rslot = 0;
      const uint32_t tslot = sf_use % SF_SLOTS;
      // the tensor-memory slot is free once the MMAs of the stage that used
      // it last have completed
      if (ok) ok = mbar_wait_warp(&sf_empty[tslot], ((sf_use / SF_SLOTS) & 1u) ^ 1u, tmo, p.err, abort_flag);
      if (ok) {
        tc_fence_after();
        const uint32_t sf_t = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + sf_slot(tslot);
        {
          // A: column 4m + c = MMA m's word of weight row lane + 32c
          uint32_t r[32];
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint4 v = ld_shared_u4(d + static_cast<uint32_t>(32 * c * SF_ROW_BYTES + 16 * h));
              r[4 * (4 * h + 0) + c] = v.x;
              r[4 * (4 * h + 1) + c] = v.y;
              r[4 * (4 * h + 2) + c] = v.z;
              r[4 * (4 * h + 3) + c] = v.w;
            }
          tmem_st_32x32b_x32(sf_t, r);
        }
        constexpr int MPS = 32 / SFB_STRIDE;  // MMAs per 32-column store
#pragma unroll
        for (int h = 0; h < MMAS / MPS; ++h) {
          // B: column SFB_OFF + SFB_STRIDE * m + c = MMA m's word of token
          // row lane + 32c (MMAs MPS*h.. in this store; c < N/32, the rest
          // never read)
          uint32_t r[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
#pragma unroll
          for (int c = 0; c < TN / 32; ++c)
#pragma unroll
            for (int v4 = 0; v4 < MPS / 4; ++v4) {
              // words MPS*h + 4*v4 .. +3 of the row: 16 bytes
              const uint4 v = ld_shared_u4(
                  d + static_cast<uint32_t>((SF_A_ROWS + 32 * c) * SF_ROW_BYTES + 4 * (MPS * h + 4 * v4)));
              r[SFB_STRIDE * (4 * v4 + 0) + c] = v.x;
              r[SFB_STRIDE * (4 * v4 + 1) + c] = v.y;
              r[SFB_STRIDE * (4 * v4 + 2) + c] = v.z;
              r[SFB_STRIDE * (4 * v4 + 3) + c] = v.w;
            }
          tmem_st_32x32b_x32(sf_t + SFB_OFF + 32 * h, r);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader)
            mbar_arrive(&full[stage]);
          else
            mbar_arrive_remote_relaxed(full_leader + static_cast<uint32_t>(stage) * 8u);
        }
      }
      ++sf_use;
      if (++stage == S) {
        stage = 0;
        phase ^= 1u;
      }
    }
    cp_async_wait_group<0>();  // no copy into the ring outlives the block
  } else {
    // ===================================================== epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const uint32_t tempty_leader = mapa_shared(smem_u32(&tempty[0]), 0);
    int it = 0;
    for (int t = cluster_id; t < total; t += n_clusters, ++it) {
      const gg::PairTile ti = gg::decode_pair_tile<TN, NQ>(t, s_prefix, s_off, GT, G, p.shared_rows);
      const Prob& P = p.prob[ti.pb];
      const int buf = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      if (!mbar_wait_warp(&tfull[buf], use & 1u, tmo, p.err, abort_flag)) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * ACC_STRIDE);
      const float scale = __ldg(P.a_g) * __ldg(P.w_g + ti.g);
      const int nch = (ti.cnt + 31) >> 5;
      const int col = ti.blk * 256 + static_cast<int>(rank) * WM + q * 32 + lane;  // output column
      // two warps per lane quadrant: warps 2..5 take the even 32-token
      // chunks, warps 12..15 the odd ones
      for (int c = warp >= W_EPI1 ? 1 : 0; c < nch; c += 2) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + c * 32, v);
        tmem_ld_wait();
        float h[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) h[j] = __uint_as_float(v[j]) * scale;
        gg::store_pairs<32>(P, h, col, ti.row0 + c * 32, ti.cnt - c * 32, lane);
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
  // the leader's MMAs read this CTA's shared memory and tensor memory: neither
  // CTA leaves or frees tensor memory before both are done
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

static int launch(const Params& prm, cudaStream_t s) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(grouped_gemm_nvf4p_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, grouped_gemm_nvf4p_kernel, prm);
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return check_launch();
}

static int fill(Params& prm, int slot, const GemmProblem& P) {
  Prob& q = prm.prob[slot];
  q.n_out = P.N;
  q.K = P.K;
  q.w_rows = P.N;
  q.n_tiles = (P.N + 255) / 256;  // output columns per weight block (pair)
  q.a_rows = P.a_rows;
  q.w_rows_total = P.groups * q.w_rows;
  q.c = P.C;
  q.c_sf = nullptr;
  q.a_g = P.A_g;
  q.w_g = P.W_g;
  q.c_g = nullptr;
  q.a_sf = P.A_sf;
  q.w_sf = P.W_sf;
  const uint64_t K = static_cast<uint64_t>(P.K), nkb = K / 256;
  const uint64_t code_ld = K / 2;  // bytes per row
  {
    // tokens [a_rows, K/2] bytes as (byte in k-block, row, k-block), boxes
    // of 80 rows x both k-blocks
    const uint64_t dims[3] = {KB_BYTES, static_cast<uint64_t>(P.a_rows), nkb};
    const uint64_t str[2] = {code_ld, KB_BYTES};
    const uint32_t box[3] = {KB_BYTES, B_ROWS, KSUB};
    MOE_TRY(encode_tmap_nd(&prm.tma_a[slot], P.A, false, 3, dims, str, box, true));
  }
  {
    // W [groups * N, K/2] bytes, boxes of 128 rows x both k-blocks
    const uint64_t dims[3] = {KB_BYTES, static_cast<uint64_t>(q.w_rows_total), nkb};
    const uint64_t str[2] = {code_ld, KB_BYTES};
    const uint32_t box[3] = {KB_BYTES, WM, KSUB};
    MOE_TRY(encode_tmap_nd(&prm.tma_w[slot], P.W, false, 3, dims, str, box, true));
  }
  return MOE_OK;
}

}  // namespace gf4p

// NVFP4 x NVFP4 down projection (bf16 output) on CTA pairs: K % 512 == 0 and
// 16-byte aligned scale arrays (checked by the caller, grouped_gemm_launch_nvf4).
int grouped_gemm_launch_nvf4_pair(const GemmProblem& routed, const int32_t* offsets, int G, const GemmProblem* sh,
                                  int shared_rows, cudaStream_t s) {
  gg::Params prm;
  memset(&prm, 0, sizeof(prm));
  MOE_TRY(gf4p::fill(prm, 0, routed));
  prm.offsets = offsets;
  prm.G = G;
  prm.shared_rows = -1;
  if (sh != nullptr && shared_rows > 0) {
    MOE_TRY(gf4p::fill(prm, 1, *sh));
    prm.shared_rows = shared_rows;
  }
  prm.err = device_error_word();
  if (!prm.err) return MOE_ERR_CUDA;
  prm.timeout_ns = wait_timeout_ns();
  return gf4p::launch(prm, s);
}

}  // namespace moe
