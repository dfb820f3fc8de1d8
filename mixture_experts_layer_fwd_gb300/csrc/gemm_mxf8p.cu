// Grouped GEMM with both operands in MXFP8 on CTA pairs: one block-scaled
// MMA (tcgen05.mma.cta_group::2 kind::mxf8f6f4, block_scale, scale_vec::1X)
// spans the two SMs of a cluster.  The weights are the MMA's M side (256
// weight rows per pair, 128 per SM) and the tokens its N side (up to 192
// tokens per tile, the MMA's N the tile's tokens rounded up to 32), so the
// accumulator holds C^T, as in the bf16 pair kernel.
//
// "Hosting Qwen on Blackwell", section "Quantização": Qwen3-235B is served
// with MXFP8 weights, E4M3 bytes with one E8M0 scale per 32 elements along K
// ("CuTeDSL at Perplexity", Blackwell support).  Format reading: quant_mx.cu.
//
// Why pairs with tokens on N: an MXFP8 MMA runs twice as fast as a bf16 one
// of the same shape on half the operand bytes, so a 1-SM 128 x 128 tile
// needs (128 + 128) bytes per element of K for 2 x 128 x 128 FLOPs, and the
// shared-memory fill rate, not the tensor cores, sets its pace.  Here each
// SM stages its 128 weight rows and 96 token rows: 224 bytes per element of
// K for 2 x 128 x 192 FLOPs.  Tokens on N also cut a group of r rows into
// ceil(r/192) equal blocks rounded up to 32 instead of 128-row tiles.
//
// Stages: 256 elements of K (two 128-byte k-blocks per row): 32 KB of weight
// codes and 24 KB of token codes per SM, by TMA (128-byte swizzle); 8 MMAs
// of K = 32.  Three stages.
//
// Scales in tensor memory: an M = 256 block-scaled MMA reads, in each CTA,
// the scales of that CTA's 128 A rows and of all N B rows; row r sits in
// lane r % 32, column r / 32, the same in the four lane quadrants, and one
// 32-bit cell holds the bytes of four consecutive MMAs (picked by the
// instruction descriptor's scale-factor id m % 4).  A stage's scale slot is
// 32 columns: A in 0..7 (column 4w + c: word w of row lane + 32c), B in
// 8..23 (column 8 + 8w + c, c < N/32).  Tensor memory holds two fp32
// accumulators (columns 0..191 and 256..447) and, in the gaps, the three
// stages' slots (columns 192, 224 and 448).  A stage's scales are 8 bytes per
// row, under the 16-byte minimum of a TMA box: the 128 threads of the four
// scale warps of each CTA copy each row once with cp.async into a ring in
// shared memory, SF_DEPTH - 1 stages ahead (rows outside the operand or the
// tile read as zero), and after a barrier of the four warps each warp writes
// its lane quadrant of the slot with one tcgen05.st.
//
// Roles (both CTAs of the pair run the same tile sequence):
//   warp 0        weight codes of this CTA's 128 rows (one 3-/4-D box: both
//                 k-blocks); the leader arms the pair's full barrier for
//                 both CTAs' code bytes
//   warp 6        token codes: 96 rows from this CTA's half of the tile on
//                 (rows past the half are staged and not read by the MMA)
//   warps 7..10   scale warps, one per lane quadrant: ring of copies, wait
//                 until the stage's previous MMAs are done (its empty
//                 barrier), write the slot, arrive on the leader's full
//                 barrier
//   warp 1        tensor-memory allocation of the pair; in the leader only,
//                 the MMA issuer, a whole converged warp: 8 x
//                 tcgen05.mma.cta_group::2 (M=256, N=tile tokens, K=32) per
//                 stage, commits multicast to both CTAs' empty / tfull
//                 barriers; it starts each stage on a named-barrier signal
//   warp 11       in the leader only: the MMA warp's waits (full barrier of
//                 each stage, accumulator drained at a tile's start), so
//                 that no mbarrier wait queues behind the issued MMAs
//   warps 2..5    epilogue: each CTA reads its 128 accumulator lanes (weight
//                 rows) x tokens and stores bf16 C[token, col] (STORE,
//                 SWIGLU_BF16) or MXFP8 h (SWIGLU_MX: 32 x 32 chunks
//                 transposed through shared memory so that a lane holds one
//                 token's 32 features, one E8M0 scale per lane)
// SwiGLU: each CTA stages the 64 gate rows of features [f0, f0+64) followed
// by the 64 up rows of the same features, so accumulator lanes 0..63 hold
// gate and 64..127 up; warp q (gate) and warp q+2 (up) swap half of their
// 32-token chunks through shared memory, as in the bf16 pair kernel.
// Requires K % 256 == 0 and 8-byte aligned scale arrays.
#include <cstring>

#include "gemm_common.cuh"
#include "internal.h"

namespace moe {
namespace gmx8p {

using gg::MAX_G;
using gg::Params;
using gg::Prob;

constexpr int TN = 192;                    // most tokens per tile (N of the MMA)
constexpr int NQ = 32;                     // the MMA's N is a multiple of 32
constexpr int WM = 128;                    // weight rows per CTA (M of the MMA is 2 x WM)
constexpr int KB_BYTES = 128;              // bytes (elements) of one k-block row
constexpr int KSUB = 2;                    // k-blocks per stage
constexpr int KE = KSUB * KB_BYTES;        // elements per stage
constexpr int MMAS = KE / 32;              // MMAs per stage
constexpr int GU_ROWS = 64;                // SwiGLU: features per CTA (64 gate + 64 up rows)
constexpr int B_ROWS = TN / 2;             // token rows staged per CTA (>= half of N)
constexpr int A_TILE = WM * KB_BYTES;      // 16 KB per k-block
constexpr int B_TILE = B_ROWS * KB_BYTES;  // 12 KB per k-block
constexpr int OFF_B = KSUB * A_TILE;
constexpr int STAGE_BYTES = OFF_B + KSUB * B_TILE;  // 56 KB
constexpr int STAGES = 3;
constexpr uint32_t TX_CODES_PAIR = 2u * STAGE_BYTES;  // both CTAs' copies, counted on the leader
constexpr int ACC_STRIDE = 256;            // accumulator buffers at columns 0 and 256
constexpr int SF_WORDS = KSUB;             // 32-bit scale words per row and stage (4 MMAs each)
constexpr int SFB_OFF = 4 * SF_WORDS;      // B scales after A's cells x 4 columns
constexpr int SF_SLOT_COLS = KSUB == 1 ? 16 : 32;
constexpr int SF_GAP0 = (ACC_STRIDE - TN) / SF_SLOT_COLS;  // slots after the first accumulator
constexpr int NUM_WARPS = 12;
constexpr int THREADS = NUM_WARPS * 32;
constexpr int TMEM_COLS = 512;
constexpr int W_PROD_B = 6, W_SCALE0 = 7, W_WAIT = 11;
constexpr int MMA_BAR = 4;                 // named barrier of the MMA warp and the wait warp
constexpr int EXTRA = (2048 + 4 * (2 * MAX_G + 8) + 15) & ~15;
constexpr int XCH_FLOATS = 32 * 32;                // one 32-lane x 32-token chunk
constexpr int XCH_BYTES = 2 * 2 * XCH_FLOATS * 4;  // 2 warp pairs x 2 directions
constexpr int SF_DEPTH = STAGES;                    // scale stages in the shared-memory ring
constexpr int SF_A_ROWS = WM;                       // ring slot: 128 weight rows, then TN token rows
constexpr int SF_ROW_BYTES = 4 * SF_WORDS;          // scale bytes per row and stage
constexpr int SF_SLOT_BYTES = (SF_A_ROWS + TN) * SF_ROW_BYTES;
constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + EXTRA + XCH_BYTES + 64 + SF_DEPTH * SF_SLOT_BYTES;
static_assert(STAGE_BYTES % 1024 == 0 && B_TILE % 1024 == 0, "tiles must keep 1024-byte alignment");
static_assert(KSUB == 1 || KSUB == 2, "a stage's scales are one or two 32-bit words per row");
static_assert(SFB_OFF + 8 * (SF_WORDS - 1) + TN / 32 <= SF_SLOT_COLS, "B scales fit the slot");
static_assert(ACC_STRIDE + TN + (STAGES - SF_GAP0) * SF_SLOT_COLS <= TMEM_COLS,
              "scale slots fit the gaps after the accumulators");
static_assert(TN > 128 && TN <= 256, "the 128 scale threads copy one weight row and one or two token rows");
static_assert(SMEM <= 232448, "shared memory budget");

// tensor-memory column of stage s's scale slot
DEVINL uint32_t sf_slot(int s) {
  return s < SF_GAP0 ? TN + s * SF_SLOT_COLS : ACC_STRIDE + TN + (s - SF_GAP0) * SF_SLOT_COLS;
}

// Instruction descriptor, kind::mxf8f6f4 with E8M0 scales: E4M3 x E4M3 ->
// fp32 (format code 0 for both), both K-major, scale-factor ids for A (bits
// 29-30) and B (bits 4-5).
DEVINL uint32_t idesc_mxf8(int M, int N, uint32_t sf_id) {
  return (sf_id << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(M >> 4) << 24) | (sf_id << 29);
}

// Issued by a whole converged warp: every lane computes the (warp-uniform)
// operands and elect.sync picks the one lane that issues, which costs far
// less per MMA than a single-lane branch; these MMAs are short (about 55 ns
// of tensor work at N = 192), so a single lane's issue would set the pace.
DEVINL void umma_mxf8_pair_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa_tmem,
                                uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1) grouped_gemm_mxf8p_kernel(const __grid_constant__ Params p) {
  constexpr int S = STAGES;
  constexpr bool SWIGLU = EPI != MOE_EPI_STORE_BF16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = base;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + S * STAGE_BYTES);  // leader: codes + scale-warp arrivals
  uint64_t* empty = full + S;                                            // stage free (MMA commit)
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_prefix = reinterpret_cast<int*>(base + S * STAGE_BYTES + 256);
  int* s_off = s_prefix + MAX_G + 4;
  float* xch = reinterpret_cast<float*>(base + S * STAGE_BYTES + EXTRA);
  volatile int* pair_ok = reinterpret_cast<volatile int*>(xch + 4 * XCH_FLOATS);  // [2 pairs][gate, up]
  uint8_t* sf_stage = reinterpret_cast<uint8_t*>(xch + 4 * XCH_FLOATS) + 64;       // scale ring
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
        // this CTA's tokens start half of N into the tile (half <= 96)
        const int b_y = ti.row0 + static_cast<int>(rank) * (ti.n >> 1);
        // this CTA's 128 weight rows: SwiGLU -> gate and up rows of features
        // [blk*128 + 64*rank, +64); STORE -> rows [blk*256 + 128*rank, +128)
        const int f0 = ti.blk * 128 + static_cast<int>(rank) * GU_ROWS;
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
            if (SWIGLU)
              tma_load_4d_pair(&p.tma_w[ti.pb], fbar, sb, 0, f0, 2 * ti.g, kblk);
            else
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
    // go signal of the wait warp (both CTAs' codes and scales in place and,
    // on a tile's first stage, the accumulator drained), so this warp never
    // waits on an mbarrier between its MMAs.
    if (leader) {
      int stage = 0;
      bool ok = true;
      int it = 0;
      const uint64_t a_desc0 = smem_desc_kmajor_sw128(smem_u32(stages));
      const uint64_t b_desc0 = smem_desc_kmajor_sw128(smem_u32(stages + OFF_B));
      for (int t = cluster_id; t < total && ok; t += n_clusters, ++it) {
        const gg::PairTile ti = gg::decode_pair_tile<TN, NQ>(t, s_prefix, s_off, GT, G, p.shared_rows);
        const int nk = p.prob[ti.pb].K / KE;
        uint32_t idesc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) idesc[i] = idesc_mxf8(2 * WM, ti.n, static_cast<uint32_t>(i));
        const int buf = it & 1;
        const uint32_t d = tmem_base + static_cast<uint32_t>(buf * ACC_STRIDE);
        for (int kb = 0; kb < nk; ++kb) {
          if (named_bar_red_or(MMA_BAR, 64, false)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf_t = tmem_base + sf_slot(stage);
          const uint64_t da = a_desc0 + static_cast<uint64_t>((stage * STAGE_BYTES) >> 4);
          const uint64_t db = b_desc0 + static_cast<uint64_t>((stage * STAGE_BYTES) >> 4);
#pragma unroll
          for (int m = 0; m < MMAS; ++m) {
            const int j = m >> 2, kk = m & 3;  // k-block, 32-byte step inside it
            umma_mxf8_pair_warp(d, da + ((j * A_TILE + kk * 32) >> 4), db + ((j * B_TILE + kk * 32) >> 4),
                                idesc[kk], sf_t + 4 * j, sf_t + SFB_OFF + 8 * j, (kb | m) ? 1u : 0u);
          }
          umma_commit_pair_multicast_warp(&empty[stage], 0x3);
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
          // warps wrote the slot
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
  } else if (warp >= W_SCALE0) {
    // ===================================================== scale warps (7..10)
    // The 128 threads copy each stage's scale bytes of the CTA's 128
    // weight rows and the tile's 192 token rows (one to three rows each)
    // into a ring of SF_DEPTH slots in shared memory with cp.async, SF_DEPTH
    // - 1 stages ahead of the stage they write to tensor memory; after a
    // barrier of the four warps each lane reads the words of its rows.
    const int q = warp & 3;  // lane quadrant this warp writes
    const int st = (warp - W_SCALE0) * 32 + lane;  // copying thread 0..127
    const uint32_t full_leader = mapa_shared(smem_u32(&full[0]), 0);
    const uint32_t ring = smem_u32(sf_stage);
    // prefetch cursor: tile ct, stage ckb of cnk; this thread's rows
    // st (weight row st), SF_A_ROWS + st and SF_A_ROWS + 128 + st (token rows)
    int ct = cluster_id, ckb = 0, cnk = 0;
    const uint8_t* any = nullptr;  // a valid address for the zero-filling copies
    const uint8_t* rp[3];
    auto open_tile = [&]() {
      if (ct >= total) return;
      const gg::PairTile ti = gg::decode_pair_tile<TN, NQ>(ct, s_prefix, s_off, GT, G, p.shared_rows);
      const Prob& P = p.prob[ti.pb];
      const int ld = P.K / 32;  // scale bytes per row
      cnk = P.K / KE;
      ckb = 0;
      any = P.w_sf;
      {
        const int m = st;  // this CTA's weight row
        int wr;
        bool wv;
        if (SWIGLU) {
          const int f = ti.blk * 128 + static_cast<int>(rank) * GU_ROWS + (m & 63);
          wv = f < P.n_out;
          wr = ti.g * P.w_rows + (m < 64 ? 0 : P.n_out) + f;
        } else {
          const int col = ti.blk * 256 + static_cast<int>(rank) * WM + m;
          wv = col < P.n_out;
          wr = ti.g * P.w_rows + col;
        }
        rp[0] = wv ? P.w_sf + static_cast<size_t>(wr) * ld : nullptr;
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int j = st + 128 * c;  // token of the tile (MMA column)
        rp[1 + c] = (j < TN && j < ti.cnt) ? P.a_sf + static_cast<size_t>(ti.row0 + j) * ld : nullptr;
      }
    };
    // copies the cursor's stage into ring slot `slot` and advances; commits
    // a (possibly empty) group either way so that group counts stay uniform
    auto copy_row = [&](uint32_t dst, const uint8_t* row, int off) {
      if (SF_ROW_BYTES == 8)
        cp_async_8(dst, row ? row + off : any, row != nullptr);
      else
        cp_async_4(dst, row ? row + off : any, row != nullptr);
    };
    auto issue = [&](int slot) -> bool {
      const bool has = ct < total;
      if (has) {
        const uint32_t d = ring + static_cast<uint32_t>(slot * SF_SLOT_BYTES + st * SF_ROW_BYTES);
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
    int stage = 0, slot = 0;
    uint32_t phase = 0;
    // all four warps run every stage of the schedule (the barrier below
    // counts them); after a wait gave up a warp only stops writing
    bool ok = true;
    while (pending > 0) {
      cp_async_wait_group<SF_DEPTH - 2>();  // this thread's copies of the slot landed
      // everyone's copies of the slot are visible, and everyone has read the
      // slot refilled next
      named_bar_sync(3, 128);
      pending += issue(slot == 0 ? SF_DEPTH - 1 : slot - 1) ? 1 : 0;
      // column 4w + c: word w of weight row lane + 32c; column SFB_OFF + 8w
      // + c: word w of token row lane + 32c
      uint32_t r[SF_SLOT_COLS];
#pragma unroll
      for (int i = 0; i < SF_SLOT_COLS; ++i) r[i] = 0u;
      {
        const uint32_t d = ring + static_cast<uint32_t>(slot * SF_SLOT_BYTES + lane * SF_ROW_BYTES);
#pragma unroll
        for (int c = 0; c < 4 + TN / 32; ++c) {
          const bool is_a = c < 4;
          const uint32_t a = d + static_cast<uint32_t>((is_a ? 32 * c : SF_A_ROWS + 32 * (c - 4)) * SF_ROW_BYTES);
          uint32_t w[SF_WORDS];
          if constexpr (SF_WORDS == 2) {
            const uint2 v = ld_shared_u2(a);
            w[0] = v.x;
            w[SF_WORDS - 1] = v.y;
          } else {
            w[0] = ld_shared_u32(a);
          }
#pragma unroll
          for (int i = 0; i < SF_WORDS; ++i) r[is_a ? 4 * i + c : SFB_OFF + 8 * i + (c - 4)] = w[i];
        }
      }
      --pending;
      if (++slot == SF_DEPTH) slot = 0;
      // the tensor-memory slot is free once the stage's previous MMAs have
      // completed
      if (ok) ok = mbar_wait_warp(&empty[stage], phase ^ 1u, tmo, p.err, abort_flag);
      if (ok) {
        tc_fence_after();
        tmem_st_32x32b(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + sf_slot(stage), r);
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
    // SwiGLU: quadrants 0,1 hold gate rows, 2,3 the up rows of the same
    // features; warps (q, q+2) form exchange pair pi = q & 1
    const int pi = q & 1;
    const bool is_gate = q < 2;
    float* x_to_up = xch + pi * 2 * XCH_FLOATS;  // gate values the up warp consumes
    float* x_to_gate = x_to_up + XCH_FLOATS;     // up values the gate warp consumes
    int it = 0;
    for (int t = cluster_id; t < total; t += n_clusters, ++it) {
      const gg::PairTile ti = gg::decode_pair_tile<TN, NQ>(t, s_prefix, s_off, GT, G, p.shared_rows);
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
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * ACC_STRIDE);
      const int nch = (ti.cnt + 31) >> 5;
      if (SWIGLU) {
        const int fbase = ti.blk * 128 + static_cast<int>(rank) * GU_ROWS + pi * 32;  // first feature of the pair
        for (int c = 0; c < nch; c += 2) {
          const bool has1 = c + 1 < nch;
          // the gate warp finishes chunk c, the up warp chunk c+1; each first
          // sends the other chunk's values, then loads its own (one 32-column
          // chunk live at a time)
          const bool mine = is_gate || has1;
          const int cc = is_gate ? c : c + 1;  // chunk this warp finishes
          if (is_gate ? has1 : true) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(taddr + (is_gate ? c + 1 : c) * 32, v);
            tmem_ld_wait();
            float* dst = is_gate ? x_to_up : x_to_gate;
#pragma unroll
            for (int j = 0; j < 32; ++j) dst[j * 32 + lane] = __uint_as_float(v[j]);
          }
          uint32_t v[32];
          if (mine) {
            tmem_ld_32x32b_x32(taddr + cc * 32, v);
            tmem_ld_wait();
          }
          named_bar_sync(1 + pi, 64);
          float h[32];
          if (is_gate) {
#pragma unroll
            for (int j = 0; j < 32; ++j) h[j] = gg::silu_f(__uint_as_float(v[j])) * x_to_gate[j * 32 + lane];
          } else if (has1) {
#pragma unroll
            for (int j = 0; j < 32; ++j) h[j] = gg::silu_f(x_to_up[j * 32 + lane]) * __uint_as_float(v[j]);
          }
          if (EPI == MOE_EPI_SWIGLU_BF16) {
            if (mine) gg::store_pairs<32>(P, h, fbase + lane, ti.row0 + cc * 32, ti.cnt - cc * 32, lane);
            // the slots are rewritten by the next chunk pair
            named_bar_sync(1 + pi, 64);
          } else {
            // both warps have read the exchanged values: reuse this warp's
            // half of the pair's exchange area to transpose h (feature per
            // lane -> token per lane; column index XOR row keeps banks apart)
            named_bar_sync(1 + pi, 64);
            float* tr = is_gate ? x_to_up : x_to_gate;
            if (mine) {
#pragma unroll
              for (int j = 0; j < 32; ++j) tr[j * 32 + (lane ^ j)] = h[j];
              __syncwarp();
              const int row_t = cc * 32 + lane;
              if (row_t < ti.cnt && fbase < P.n_out) {
                // lane = token: its 32 features are one MX block of h
                float b[32];
#pragma unroll
                for (int f = 0; f < 32; ++f) b[f] = tr[lane * 32 + (f ^ lane)];
                uint32_t codes[8];
                const uint32_t sc = mx_quantize32<false>(b, codes);
                const size_t row = static_cast<size_t>(ti.row0) + row_t;
                uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(P.c) + row * P.n_out + fbase);
                dst[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
                dst[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
                P.c_sf[row * (P.n_out / 32) + fbase / 32] = static_cast<uint8_t>(sc);
              }
            }
            named_bar_sync(1 + pi, 64);
          }
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
  // the leader's MMAs read this CTA's shared memory and tensor memory: neither
  // CTA leaves or frees tensor memory before both are done
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
        cudaFuncSetAttribute(grouped_gemm_mxf8p_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, grouped_gemm_mxf8p_kernel<EPI>, prm);
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return check_launch();
}

static int fill(Params& prm, int slot, int epi, const GemmProblem& P) {
  Prob& q = prm.prob[slot];
  const bool swiglu = epi != MOE_EPI_STORE_BF16;
  const int tn = swiglu ? 128 : 256;  // output columns per weight block (pair)
  q.n_out = P.N;
  q.K = P.K;
  q.w_rows = swiglu ? 2 * P.N : P.N;
  q.n_tiles = (P.N + tn - 1) / tn;
  q.a_rows = P.a_rows;
  q.w_rows_total = P.groups * q.w_rows;
  q.c = P.C;
  q.c_sf = P.C_sf;  // MX scales of h (SWIGLU_MX)
  q.a_g = q.w_g = q.c_g = nullptr;
  q.a_sf = P.A_sf;
  q.w_sf = P.W_sf;
  const uint64_t K = static_cast<uint64_t>(P.K), nkb = K / KB_BYTES;
  {
    // tokens [a_rows, K] bytes as (byte in k-block, row, k-block), boxes of
    // 96 rows x both k-blocks
    const uint64_t dims[3] = {KB_BYTES, static_cast<uint64_t>(P.a_rows), nkb};
    const uint64_t str[2] = {K, KB_BYTES};
    const uint32_t box[3] = {KB_BYTES, B_ROWS, KSUB};
    MOE_TRY(encode_tmap_nd(&prm.tma_a[slot], P.A, false, 3, dims, str, box, true));
  }
  if (swiglu) {
    // W [groups][gate N | up N][K] as (byte, row, gate/up + 2*group, k-block):
    // per k-block 64 gate rows then the same features' 64 up rows
    const uint64_t N = static_cast<uint64_t>(P.N), g2 = 2 * static_cast<uint64_t>(P.groups);
    const uint64_t dims[4] = {KB_BYTES, N, g2, nkb};
    const uint64_t str[3] = {K, N * K, KB_BYTES};
    const uint32_t box[4] = {KB_BYTES, GU_ROWS, 2, KSUB};
    MOE_TRY(encode_tmap_nd(&prm.tma_w[slot], P.W, false, 4, dims, str, box, true));
  } else {
    const uint64_t rows = static_cast<uint64_t>(q.w_rows_total);
    const uint64_t dims[3] = {KB_BYTES, rows, nkb};
    const uint64_t str[2] = {K, KB_BYTES};
    const uint32_t box[3] = {KB_BYTES, WM, KSUB};
    MOE_TRY(encode_tmap_nd(&prm.tma_w[slot], P.W, false, 3, dims, str, box, true));
  }
  return MOE_OK;
}

}  // namespace gmx8p

// MXFP8 x MXFP8 on CTA pairs: K % 256 == 0, 8-byte aligned scale arrays
// (checked by the caller, grouped_gemm_launch).
int grouped_gemm_launch_mxf8_pair(int epi, const GemmProblem& routed, const int32_t* offsets, int G,
                                  const GemmProblem* sh, int shared_rows, cudaStream_t s) {
  gg::Params prm;
  memset(&prm, 0, sizeof(prm));
  MOE_TRY(gmx8p::fill(prm, 0, epi, routed));
  prm.offsets = offsets;
  prm.G = G;
  prm.shared_rows = -1;
  if (sh != nullptr && shared_rows > 0) {
    MOE_TRY(gmx8p::fill(prm, 1, epi, *sh));
    prm.shared_rows = shared_rows;
  }
  prm.err = device_error_word();
  if (!prm.err) return MOE_ERR_CUDA;
  prm.timeout_ns = wait_timeout_ns();
  if (epi == MOE_EPI_STORE_BF16) return gmx8p::launch<MOE_EPI_STORE_BF16>(prm, s);
  if (epi == MOE_EPI_SWIGLU_MX) return gmx8p::launch<MOE_EPI_SWIGLU_MX>(prm, s);
  return gmx8p::launch<MOE_EPI_SWIGLU_BF16>(prm, s);
}

}  // namespace moe
