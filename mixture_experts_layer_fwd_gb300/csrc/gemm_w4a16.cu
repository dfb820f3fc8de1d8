// Grouped GEMM for NVFP4 weights x bf16 activations (W4A16).
//
// "Driving vLLM WideEP ... (Part I)", section "NVFP4 GEMM for MoE and
// O-proj": packed 4-bit weights with per-group FP8 scales, dequantised on
// the fly.  There is no tensor-core MMA that takes FP4 and bf16 operands
// together, so the weights are expanded to 16-bit on the SM: cvt e2m1x2 ->
// fp16x2 (one instruction per two values) times the E4M3 block scale (exact:
// e2m1 * e4m3 has at most five significant bits and lies in fp16's normal
// range), and the MMA runs kind::f16 in fp16.  Tokens given in bf16 are
// converted to fp16 in shared memory per stage (exact for |x| in [2^-14,
// 65504], saturating beyond); inside the layer forward they arrive in fp16
// already (the permutation converts x once, the gate/up epilogue stores h
// as fp16), which spares re-converting a token block for every weight tile.
//
// Why the expanded weights go to tensor memory: written to shared memory
// they would cost 2 bytes per weight on the way in and 2 on the way out to
// the MMA, which caps the weight stream near 0.6 of HBM bandwidth; the MMA
// can read its A operand from tensor memory instead (tcgen05.mma [a-tmem]).
//
// Tiles: weights on the MMA's M side (128 weight rows), tokens on N (a group
// of r routed rows is cut into ceil(r/TM) equal token blocks rounded up to
// 16; TM = 16 when the launch averages at most 4 routed rows per expert, 128
// past 48, else 64), so a weight tile is expanded once per TM tokens and a
// decode step (a few tokens per expert) streams each weight once.
//
// Two rings of shared-memory stages, one per 256-element k step each: the
// weight ring (packed codes + scales, 18 KB a stage) is deep and is freed by
// the converters as soon as they have read a stage into registers, so the
// weight stream from HBM is not held up by the conversion and the MMA; the
// token ring (the tile's tokens for the k step, mostly L2 hits) is short and
// is freed by the MMA.
//
// Roles (one CTA per SM):
//   warp 0       TMA producer of the weight ring: the tile's packed codes
//                (128 rows x 128 bytes, 128-byte swizzle; SwiGLU: 64 gate
//                rows then the 64 up rows of the same features) and their
//                scales (128 rows x 16 bytes)
//   warp 14      TMA producer of the token ring: 4 k-blocks x 16, 64 or 128
//                rows x 128 bytes, 128-byte swizzle
//   warps 6..13  converters, two per TMEM lane quadrant (one per half of
//                the stage's K): the tokens bf16 -> fp16 in place (only when
//                given in bf16), and each thread's weight row (its TMEM lane)
//                e2m1 x e4m3 -> fp16 into one of the (two or three)
//                128-column slots of tensor memory (tcgen05.st; the first
//                half of the row is stored while the second is expanded)
//   warp 1       TMEM allocation; MMA issuer: 16 x tcgen05.mma kind::f16
//                M=128 N<=128 K=16 per stage, A from the slot, B (tokens)
//                from shared memory, into one of two accumulators, issued by
//                the converged warp (elect.sync picks the lane); it starts each
//                stage on a named-barrier signal from warp 15, which does the
//                mbarrier waits (slot expanded, tokens landed, accumulator
//                drained) so that none stalls the issue of the MMAs
//   warps 2..5   epilogue: accumulator lanes (weight rows) x tokens, scaled
//                by the weights' fp32 global scale; SwiGLU pairs gate lanes
//                32q with up lanes 32q+64 through shared memory; 4-byte bf16
//                stores of C[token, col]
// Requires K % 256 == 0 and 16-byte aligned scale arrays; other shapes take
// the converter kernel of gemm.cu.
#include <cstring>

#include "gemm_common.cuh"
#include "internal.h"

namespace moe {
namespace gw4 {

using gg::MAX_G;
using gg::Params;
using gg::Prob;

constexpr int WM = 128;                   // weight rows per tile (M of the MMA)
constexpr int SMALL_N = 16;               // tiles of <= 16 tokens stage 16 token rows
constexpr int KS = 256;                   // elements per stage
constexpr int CODE_TILE = WM * KS / 2;    // 16 KB of packed E2M1
constexpr int SF_TILE = WM * KS / 16;     // 2 KB: 16 scale bytes per row
constexpr int TOK_KBLK = KS / 64;         // 64-element k-blocks of tokens per stage
constexpr int OFF_SF = CODE_TILE;
constexpr int W_STAGE = CODE_TILE + SF_TILE;  // 18 KB per weight stage
constexpr int A_COLS = KS / 2;            // fp16 pairs per row per stage = TMEM columns per slot
constexpr int MAX_ASLOTS = 3;             // expanded-weight slots in tensor memory (at most)
constexpr int TMEM_COLS = 512;
// 4 lane quadrants x KPARTS parts of the stage's K (16 warps measured slower:
// the register cap of a 704-thread block spills the epilogue)
constexpr int CONV_WARPS = 8;
constexpr int KPARTS = CONV_WARPS / 4;
constexpr int PART_COLS = A_COLS / KPARTS;       // fp16 pairs a converter thread writes per stage
constexpr int PART_CHUNKS = 8 / KPARTS;          // 16-byte code chunks (32 values) per part
constexpr int PART_SF_WORDS = 4 / KPARTS;        // 32-bit words of scale bytes per part
constexpr int CONV_THREADS = CONV_WARPS * 32;
constexpr int TOK_WARP = 6 + CONV_WARPS;         // token-ring producer
constexpr int WAIT_WARP = TOK_WARP + 1;          // waits on behalf of the MMA warp
constexpr int NUM_WARPS = WAIT_WARP + 1;
constexpr int MMA_BAR = 3;                       // named barrier: WAIT_WARP -> MMA warp
static_assert(TOK_WARP == 14 && WAIT_WARP == 15 && NUM_WARPS == 16, "role layout");
constexpr int THREADS = NUM_WARPS * 32;
constexpr int XCH_FLOATS = 32 * 32;
constexpr int XCH_BYTES = 2 * 2 * XCH_FLOATS * 4;
constexpr int EXTRA = (512 + 4 * 2 * (MAX_G + 4) + 15) & ~15;
static_assert(W_STAGE % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(PART_COLS == 64, "a converter thread stores its part as two 32-column halves");

// Three shapes of the same pipeline: TM = 16 for launches with a few tokens
// per expert, whose 8 KB token stages leave room for 9 weight stages in
// flight from HBM; TM = 64 with 3 token stages and 5 weight stages; and
// TM = 128 for launches averaging more than 48 rows per expert, so that a
// weight tile is expanded once for up to 128 tokens (two 128-column
// accumulators leave tensor memory for two expanded-weight slots).
template <int TMT>
struct Cfg {
  static constexpr int TM = TMT;                         // most tokens per tile (N of the MMA)
  static constexpr int TOK_TILE = TMT * KS * 2;
  static constexpr int SW = TMT == SMALL_N ? 9 : (TMT == 64 ? 5 : 4);   // weight stages
  static constexpr int ST = TMT == SMALL_N ? 4 : (TMT == 64 ? 3 : 2);   // token stages
  static constexpr int ASLOTS = TMT == 128 ? 2 : 3;      // expanded-weight slots
  static constexpr int A_COL0 = TMT == 128 ? 256 : 128;  // first slot column (accumulators below)
  static constexpr int OFF_TOKS = SW * W_STAGE;
  static constexpr int RING_BYTES = OFF_TOKS + ST * TOK_TILE;
  static constexpr int ACC_COLS = TMT;                   // accumulator columns per buffer
  static constexpr int SMEM = 1024 + RING_BYTES + EXTRA + XCH_BYTES + 64;
  static_assert(TOK_TILE % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(2 * ACC_COLS <= A_COL0 && A_COL0 + ASLOTS * A_COLS <= TMEM_COLS, "tensor memory budget");
  static_assert(ASLOTS <= MAX_ASLOTS, "barrier arrays");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(2 * (SW + ST) + 2 * MAX_ASLOTS + 5 <= 60, "barrier area");
};

struct Tile {
  int pb, g, row0, cnt, n, blk;
};

// As the bf16 pair kernel's schedule, with token blocks of at most TM rows.
template <int TM>
DEVINL Tile decode_tile(int t, const int* s_prefix, const int* s_off, int GT, int G, int shared_rows) {
  int lo = 0, hi = GT;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_prefix[mid] <= t) lo = mid; else hi = mid;
  }
  Tile ti;
  const bool routed = lo < G;
  ti.pb = routed ? 0 : 1;
  ti.g = routed ? lo : 0;
  const int start = routed ? s_off[lo] : 0;
  const int rows = routed ? (s_off[lo + 1] - s_off[lo]) : shared_rows;
  const int nb = (rows + TM - 1) / TM;
  const int ng = ((rows + nb - 1) / nb + 15) & ~15;
  const int local = t - s_prefix[lo];
  ti.blk = local / nb;
  const int m = local - ti.blk * nb;
  ti.row0 = start + m * ng;
  ti.cnt = min(ng, rows - m * ng);
  ti.n = (ti.cnt + 15) & ~15;
  return ti;
}

DEVINL uint32_t bf16x2_to_f16x2_sat(uint32_t v) {
  const float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xFFFF0000u);
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}


DEVINL uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

DEVINL uint32_t pack_f16x2_sat(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Stores NV tokens x one column per lane as bf16, or fp16 when F16 (see
// gemm_pair.cu).
template <int NV, bool F16>
DEVINL void store_pairs(const Prob& P, const float (&h)[NV], int col, int row_first, int valid_tokens, int lane) {
  const bool odd = lane & 1;
  const int col_even = col & ~1;
  if (col_even >= P.n_out) return;
  uint16_t* C = static_cast<uint16_t*>(P.c);
#pragma unroll
  for (int j = 0; j < NV / 2; ++j) {
    const float send = odd ? h[2 * j] : h[2 * j + 1];
    const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, 1);
    const int t = 2 * j + (odd ? 1 : 0);
    const float lo = odd ? recv : h[2 * j];
    const float hi = odd ? h[2 * j + 1] : recv;
    if (t < valid_tokens)
      *reinterpret_cast<uint32_t*>(C + static_cast<size_t>(row_first + t) * P.n_out + col_even) =
          F16 ? pack_f16x2_sat(lo, hi) : pack_bf16x2(lo, hi);
  }
}

template <int EPI, int TMT>
__global__ void __launch_bounds__(THREADS, 1) grouped_gemm_w4a16_kernel(const __grid_constant__ Params p) {
  using C = Cfg<TMT>;
  constexpr int TM = C::TM;
  constexpr int SW = C::SW;
  constexpr int ST = C::ST;
  constexpr int ACC_COLS = C::ACC_COLS;
  constexpr int ASLOTS = C::ASLOTS;
  constexpr int A_COL0 = C::A_COL0;
  constexpr bool SWIGLU = EPI != MOE_EPI_STORE_BF16;
  constexpr bool OUT_F16 = EPI == kEpiSwigluF16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* wring = base;                    // weight stages
  uint8_t* kring = base + C::OFF_TOKS;      // token stages
  uint64_t* wfull = reinterpret_cast<uint64_t*>(base + C::RING_BYTES);
  uint64_t* wempty = wfull + SW;
  uint64_t* kfull = wempty + SW;
  uint64_t* kempty = kfull + ST;
  uint64_t* afull = kempty + ST;
  uint64_t* aempty = afull + MAX_ASLOTS;
  uint64_t* tfull = aempty + MAX_ASLOTS;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_prefix = reinterpret_cast<int*>(base + C::RING_BYTES + 512);
  int* s_off = s_prefix + MAX_G + 4;
  float* xch = reinterpret_cast<float*>(base + C::RING_BYTES + EXTRA);
  volatile int* pair_ok = reinterpret_cast<volatile int*>(xch + 4 * XCH_FLOATS);
  __shared__ int warp_sums[32];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.G;
  const int GT = G + (p.shared_rows >= 0 ? 1 : 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < SW; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], CONV_WARPS);
    }
    for (int s = 0; s < ST; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
    }
    for (int a = 0; a < ASLOTS; ++a) {
      mbar_init(&afull[a], CONV_WARPS);
      mbar_init(&aempty[a], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);  // the 4 epilogue warps
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  gg::build_schedule<THREADS, NUM_WARPS, TM>(p, s_off, s_prefix, warp_sums);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int total = s_prefix[GT];
  const unsigned long long tmo = p.timeout_ns;

  if (warp == 0 || warp == TOK_WARP) {
    // ===================================================== TMA producers
    // warp 0: tma_w (packed codes) + tma_wsf (weight scales) into the weight
    // ring; TOK_WARP: tma_a / tma_asf (tokens, 64-row / 16-row boxes) into
    // the token ring
    if (lane == 0) {
      const bool wprod = warp == 0;
      const int depth = wprod ? SW : ST;
      uint64_t* fullb = wprod ? wfull : kfull;
      uint64_t* emptyb = wprod ? wempty : kempty;
      for (int pb = 0; pb < (p.shared_rows >= 0 ? 2 : 1); ++pb) {
        if (wprod) {
          tma_prefetch_desc(&p.tma_w[pb]);
          tma_prefetch_desc(&p.tma_wsf[pb]);
        } else {
          tma_prefetch_desc(&p.tma_a[pb]);
          tma_prefetch_desc(&p.tma_asf[pb]);
        }
      }
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued[SW];
#pragma unroll
      for (int s = 0; s < SW; ++s) issued[s] = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile ti = decode_tile<TM>(t, s_prefix, s_off, GT, G, p.shared_rows);
        const Prob& P = p.prob[ti.pb];
        const bool small = ti.n <= SMALL_N;
        const void* tt = small ? &p.tma_asf[ti.pb] : &p.tma_a[ti.pb];
        const uint32_t tx = wprod ? static_cast<uint32_t>(W_STAGE)
                                  : static_cast<uint32_t>(TOK_KBLK * (small ? SMALL_N : TM) * 128);
        const int f0 = ti.blk * (WM / 2);                  // SwiGLU: 64 features
        const int w_y = ti.g * P.w_rows + ti.blk * WM;     // STORE: 128 weight rows
        const int nk = P.K / KS;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(&emptyb[stage], phase ^ 1u, tmo, p.err, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&fullb[stage], tx);
          if (wprod) {
            uint8_t* sb = wring + stage * W_STAGE;
            if (SWIGLU) {
              tma_load_3d(&p.tma_w[ti.pb], &fullb[stage], sb, kb * (KS / 2), f0, 2 * ti.g);
              tma_load_3d(&p.tma_wsf[ti.pb], &fullb[stage], sb + OFF_SF, kb * (KS / 16), f0, 2 * ti.g);
            } else {
              tma_load_2d(&p.tma_w[ti.pb], &fullb[stage], sb, kb * (KS / 2), w_y);
              tma_load_2d(&p.tma_wsf[ti.pb], &fullb[stage], sb + OFF_SF, kb * (KS / 16), w_y);
            }
          } else {
            tma_load_3d(tt, &fullb[stage], kring + stage * C::TOK_TILE, 0, ti.row0, kb * TOK_KBLK);
          }
          issued[stage] += 1;
          if (++stage == depth) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < depth; ++s)
          if (issued[s]) mbar_wait_bounded(&fullb[s], (issued[s] - 1u) & 1u, 1000000000ull, p.err, nullptr);
      }
    }
  } else if (warp >= 6 && warp < 6 + CONV_WARPS) {
    // ===================================================== converters
    const int cw = warp - 6;
    const int ctid = cw * 32 + lane;
    const int q = warp & 3;          // TMEM lane quadrant
    const int kh = cw >> 2;          // part of the stage's K this warp expands
    const int row = q * 32 + lane;   // weight row of the tile = TMEM lane
    int ws = 0, ks = 0, slot = 0;
    uint32_t wphase = 0, kphase = 0, sphase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile ti = decode_tile<TM>(t, s_prefix, s_off, GT, G, p.shared_rows);
      const int nk = p.prob[ti.pb].K / KS;
      const int kstride = (ti.n <= SMALL_N ? SMALL_N : TM) * 128;
      // 16-byte chunks of the token rows the MMA reads, when given in bf16
      const int tok_chunks = p.prob[ti.pb].a_f16 ? 0 : TOK_KBLK * ti.n * 8;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait_warp(&wfull[ws], wphase, tmo, p.err, abort_flag)) {
          ok = false;
          break;
        }
        // this thread's row, elements [kh*256/KPARTS, +256/KPARTS) of the stage,
        // into registers; then the weight stage is free for the next copy
        const uint8_t* wsb = wring + ws * W_STAGE;
        const uint8_t* crow = wsb + row * 128;
        uint32_t sw[PART_SF_WORDS];
#pragma unroll
        for (int i = 0; i < PART_SF_WORDS; ++i)
          sw[i] = *reinterpret_cast<const uint32_t*>(wsb + OFF_SF + row * 16 + kh * 4 * PART_SF_WORDS + 4 * i);
        uint4 cv[PART_CHUNKS];
#pragma unroll
        for (int c4 = 0; c4 < PART_CHUNKS; ++c4) {
          const int j = PART_CHUNKS * kh + c4;  // 16-byte chunk of the row (32 elements, two scale blocks)
          cv[c4] = *reinterpret_cast<const uint4*>(crow + ((j ^ (row & 7)) << 4));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&wempty[ws]);
        if (++ws == SW) {
          ws = 0;
          wphase ^= 1u;
        }
        if (tok_chunks) {
          // tokens: bf16 -> fp16 in place (the swizzle moves whole 16-byte chunks)
          if (!mbar_wait_warp(&kfull[ks], kphase, tmo, p.err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* ksb = kring + ks * C::TOK_TILE;
          for (int c = ctid; c < tok_chunks; c += CONV_THREADS) {
            const int kblk = c / (ti.n * 8);
            const int rem = c - kblk * ti.n * 8;
            uint4* ptr = reinterpret_cast<uint4*>(ksb + kblk * kstride + rem * 16);
            uint4 v = *ptr;
            v.x = bf16x2_to_f16x2_sat(v.x);
            v.y = bf16x2_to_f16x2_sat(v.y);
            v.z = bf16x2_to_f16x2_sat(v.z);
            v.w = bf16x2_to_f16x2_sat(v.w);
            *ptr = v;
          }
        }
        if (++ks == ST) {
          ks = 0;
          kphase ^= 1u;
        }
        const uint32_t a_dst = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                               static_cast<uint32_t>(A_COL0 + slot * A_COLS + kh * PART_COLS);
        auto conv = [&](int c4, uint32_t* rr) {
          const uint32_t sbytes = (sw[c4 >> 1] >> (16 * (c4 & 1))) & 0xFFFFu;
          const uint32_t s2 = e4m3x2_to_f16x2(sbytes);
          const uint32_t s_lo = __byte_perm(s2, 0, 0x1010), s_hi = __byte_perm(s2, 0, 0x3232);
          const uint32_t words[4] = {cv[c4].x, cv[c4].y, cv[c4].z, cv[c4].w};
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            const uint32_t sc = wi < 2 ? s_lo : s_hi;
            uint32_t o[4];
            asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
                "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
                "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
                : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
                : "r"(words[wi]));
#pragma unroll
            for (int bi = 0; bi < 4; ++bi) rr[wi * 4 + bi] = hmul2_u32(o[bi], sc);
          }
        };
        // first half of the row: expand, wait for the slot, store; the
        // second half is expanded while the first store is in flight
        {
          uint32_t r[PART_COLS / 2];
#pragma unroll
          for (int c4 = 0; c4 < PART_CHUNKS / 2; ++c4) conv(c4, r + c4 * 16);
          if (!mbar_wait_warp(&aempty[slot], sphase ^ 1u, tmo, p.err, abort_flag)) {
            ok = false;
            break;
          }
          tmem_st_32x32b_x32(a_dst, r);
          uint32_t r2[PART_COLS / 2];
#pragma unroll
          for (int c4 = 0; c4 < PART_CHUNKS / 2; ++c4) conv(PART_CHUNKS / 2 + c4, r2 + c4 * 16);
          tmem_st_32x32b_x32(a_dst + PART_COLS / 2, r2);
          tmem_st_wait();
        }
        if (tok_chunks) fence_proxy_async_smem();  // the converted tokens are read by the MMA (async proxy)
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[slot]);
        if (++slot == ASLOTS) {
          slot = 0;
          sphase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ===================================================== MMA issuer
    // The whole warp walks the schedule and issues (elect.sync picks the
    // lane, the code stays converged).  Each stage starts on
    // the go signal of WAIT_WARP (slot expanded, token stage landed and, on
    // a tile's first stage, the accumulator drained), so this warp itself
    // never waits on an mbarrier between its MMAs.
    const uint64_t tok_desc0 = smem_desc_kmajor_sw128(smem_u32(kring));
    int ks = 0, slot = 0;
    bool ok = true;
    int it = 0;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
      const Tile ti = decode_tile<TM>(t, s_prefix, s_off, GT, G, p.shared_rows);
      const int nk = p.prob[ti.pb].K / KS;
      const uint32_t idesc = idesc_f16_f32(WM, ti.n);
      const uint32_t kstride16 = static_cast<uint32_t>((ti.n <= SMALL_N ? SMALL_N : TM) * 128) >> 4;
      const uint32_t d = tmem_base + static_cast<uint32_t>((it & 1) * ACC_COLS);
      for (int kb = 0; kb < nk; ++kb) {
        if (named_bar_red_or(MMA_BAR, 64, false)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t db = tok_desc0 + static_cast<uint64_t>((ks * C::TOK_TILE) >> 4);
        const uint32_t a0 = tmem_base + static_cast<uint32_t>(A_COL0 + slot * A_COLS);
        umma_f16_ts_warp(d, a0, db, idesc, kb ? 1u : 0u);
#pragma unroll
        for (int kk = 1; kk < KS / 16; ++kk)
          umma_f16_ts_warp(d, a0 + 8 * kk, db + static_cast<uint64_t>((kk >> 2) * kstride16 + (kk & 3) * 2), idesc, 1u);
        umma_commit_warp(&kempty[ks]);
        umma_commit_warp(&aempty[slot]);
        if (++ks == ST) ks = 0;
        if (++slot == ASLOTS) slot = 0;
      }
      if (ok) umma_commit_warp(&tfull[it & 1]);
    }
    if (!ok && lane == 0) {
      umma_commit(drain);
      mbar_wait_bounded(drain, 0, 1000000000ull, p.err, nullptr);
    }
  } else if (warp == WAIT_WARP) {
    // ===================================================== waits for the MMA warp
    int ks = 0, slot = 0;
    uint32_t kphase = 0, sphase = 0;
    bool ok = true;
    int it = 0;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
      const Tile ti = decode_tile<TM>(t, s_prefix, s_off, GT, G, p.shared_rows);
      const int nk = p.prob[ti.pb].K / KS;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      for (int kb = 0; kb < nk; ++kb) {
        // afull: the slot is expanded (and, for bf16 tokens, the token stage
        // converted); kfull: the token stage has landed
        bool good = (kb > 0 || mbar_wait_warp(&tempty[it & 1], (use & 1u) ^ 1u, tmo, p.err, abort_flag)) &&
                    mbar_wait_warp(&afull[slot], sphase, tmo, p.err, abort_flag) &&
                    mbar_wait_warp(&kfull[ks], kphase, tmo, p.err, abort_flag);
        if (named_bar_red_or(MMA_BAR, 64, !good)) {
          ok = false;
          break;
        }
        if (++ks == ST) {
          ks = 0;
          kphase ^= 1u;
        }
        if (++slot == ASLOTS) {
          slot = 0;
          sphase ^= 1u;
        }
      }
    }
  } else {
    // ===================================================== epilogue (warps 2..5)
    const int q = warp & 3;
    const int pi = q & 1;
    const bool is_gate = q < 2;
    float* x_to_up = xch + pi * 2 * XCH_FLOATS;
    float* x_to_gate = x_to_up + XCH_FLOATS;
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      const Tile ti = decode_tile<TM>(t, s_prefix, s_off, GT, G, p.shared_rows);
      const Prob& P = p.prob[ti.pb];
      const int buf = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      bool ok = mbar_wait_warp(&tfull[buf], use & 1u, tmo, p.err, abort_flag);
      if (SWIGLU) {
        // both warps of the exchange pair leave together if either gave up
        if (lane == 0) pair_ok[pi * 2 + (is_gate ? 0 : 1)] = ok ? 1 : 0;
        named_bar_sync(1 + pi, 64);
        ok = pair_ok[pi * 2] && pair_ok[pi * 2 + 1];
      }
      if (!ok) break;
      tc_fence_after();
      const float scale = __ldg(P.w_g + ti.g);
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * ACC_COLS);
      const int nch = (ti.cnt + 31) >> 5;
      if (SWIGLU) {
        const int col = ti.blk * (WM / 2) + pi * 32 + lane;  // feature
        for (int c = 0; c < nch; c += 2) {
          const bool has1 = c + 1 < nch;
          uint32_t v0[32], v1[32];
          tmem_ld_32x32b_x32(taddr + c * 32, v0);
          if (has1) tmem_ld_32x32b_x32(taddr + (c + 1) * 32, v1);
          tmem_ld_wait();
          if (is_gate) {
            if (has1) {
#pragma unroll
              for (int j = 0; j < 32; ++j) x_to_up[j * 32 + lane] = __uint_as_float(v1[j]) * scale;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) x_to_gate[j * 32 + lane] = __uint_as_float(v0[j]) * scale;
          }
          named_bar_sync(1 + pi, 64);
          float h[32];
          if (is_gate) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              h[j] = gg::silu_f(__uint_as_float(v0[j]) * scale) * x_to_gate[j * 32 + lane];
            store_pairs<32, OUT_F16>(P, h, col, ti.row0 + c * 32, ti.cnt - c * 32, lane);
          } else if (has1) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              h[j] = gg::silu_f(x_to_up[j * 32 + lane]) * (__uint_as_float(v1[j]) * scale);
            store_pairs<32, OUT_F16>(P, h, col, ti.row0 + (c + 1) * 32, ti.cnt - (c + 1) * 32, lane);
          }
          named_bar_sync(1 + pi, 64);
        }
      } else {
        const int col = ti.blk * WM + q * 32 + lane;  // output column
        for (int c = 0; c < nch; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(taddr + c * 32, v);
          tmem_ld_wait();
          float h[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) h[j] = __uint_as_float(v[j]) * scale;
          store_pairs<32, false>(P, h, col, ti.row0 + c * 32, ti.cnt - c * 32, lane);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
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

template <int EPI, int TMT>
static int launch(const Params& prm, cudaStream_t s) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_w4a16_kernel<EPI, TMT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<TMT>::SMEM);
    if (e != cudaSuccess) {
      set_cuda_error(e);
      return MOE_ERR_CUDA;
    }
    attr_done[dev] = true;
  }
  grouped_gemm_w4a16_kernel<EPI, TMT><<<num_sms(), THREADS, Cfg<TMT>::SMEM, s>>>(prm);
  return check_launch();
}

template <int EPI>
static int launch_shape(const Params& prm, int tm, cudaStream_t s) {
  if (tm == SMALL_N) return launch<EPI, SMALL_N>(prm, s);
  if (tm == 64) return launch<EPI, 64>(prm, s);
  return launch<EPI, 128>(prm, s);
}

static int fill(Params& prm, int slot, int epi, const GemmProblem& P, int tm) {
  Prob& q = prm.prob[slot];
  const bool swiglu = epi != MOE_EPI_STORE_BF16;
  const int tn = swiglu ? WM / 2 : WM;  // output columns per weight tile
  q.n_out = P.N;
  q.K = P.K;
  q.w_rows = swiglu ? 2 * P.N : P.N;
  q.n_tiles = (P.N + tn - 1) / tn;
  q.a_rows = P.a_rows;
  q.w_rows_total = P.groups * q.w_rows;
  q.c = P.C;
  q.c_sf = nullptr;
  q.a_g = nullptr;
  q.w_g = P.W_g;
  q.c_g = nullptr;
  q.a_sf = nullptr;
  q.w_sf = P.W_sf;
  q.a_f16 = P.a_f16 ? 1 : 0;
  const uint64_t K = static_cast<uint64_t>(P.K);
  // tokens [a_rows, K] bf16 as (element in k-block, row, 64-element k-block)
  for (int small = 0; small < 2; ++small) {
    const uint64_t dims[3] = {64, static_cast<uint64_t>(P.a_rows), K / 64};
    const uint64_t str[2] = {K * 2, 128};
    const uint32_t box[3] = {64, static_cast<uint32_t>(small ? SMALL_N : tm), TOK_KBLK};
    MOE_TRY(encode_tmap_nd(small ? &prm.tma_asf[slot] : &prm.tma_a[slot], P.A, true, 3, dims, str, box, true));
  }
  if (swiglu) {
    // codes [groups][gate N | up N][K/2] as (byte, row, gate/up + 2*group)
    const uint64_t N = static_cast<uint64_t>(P.N), g2 = 2 * static_cast<uint64_t>(P.groups);
    const uint64_t dims[3] = {K / 2, N, g2};
    const uint64_t str[2] = {K / 2, N * (K / 2)};
    const uint32_t box[3] = {KS / 2, WM / 2, 2};
    MOE_TRY(encode_tmap_nd(&prm.tma_w[slot], P.W, false, 3, dims, str, box, true));
    const uint64_t sdims[3] = {K / 16, N, g2};
    const uint64_t sstr[2] = {K / 16, N * (K / 16)};
    const uint32_t sbox[3] = {KS / 16, WM / 2, 2};
    MOE_TRY(encode_tmap_nd(&prm.tma_wsf[slot], P.W_sf, false, 3, sdims, sstr, sbox, false));
  } else {
    MOE_TRY(encode_tmap_2d(&prm.tma_w[slot], P.W, 1, K / 2, static_cast<uint64_t>(q.w_rows_total), KS / 2, WM, true));
    MOE_TRY(encode_tmap_2d(&prm.tma_wsf[slot], P.W_sf, 1, K / 16, static_cast<uint64_t>(q.w_rows_total), KS / 16, WM,
                           false));
  }
  return MOE_OK;
}

}  // namespace gw4

// bf16 activations x NVFP4 weights with K % 256 == 0 and 16-byte aligned
// weight scales (checked by the caller, grouped_gemm_launch).
int grouped_gemm_launch_w4a16(int epi, const GemmProblem& routed, const int32_t* offsets, int G,
                              const GemmProblem* sh, int shared_rows, cudaStream_t s) {
  gg::Params prm;
  memset(&prm, 0, sizeof(prm));
  // a few routed rows per expert (decode): 16-token tiles and a deeper
  // pipeline; from ~10 rows per expert on, splitting the busier groups into
  // 16-token tiles re-expands their weights more often than it gains; past
  // 48 rows per expert on average, 128-token tiles expand each weight tile
  // once for most groups
  const long long rows = routed.a_rows;
  const int tm = rows <= 4ll * G ? gw4::SMALL_N : (rows > 48ll * G ? 128 : 64);
  MOE_TRY(gw4::fill(prm, 0, epi, routed, tm));
  prm.offsets = offsets;
  prm.G = G;
  prm.shared_rows = -1;
  if (sh != nullptr && shared_rows > 0) {
    MOE_TRY(gw4::fill(prm, 1, epi, *sh, tm));
    prm.shared_rows = shared_rows;
  }
  prm.err = device_error_word();
  if (!prm.err) return MOE_ERR_CUDA;
  prm.timeout_ns = wait_timeout_ns();
  if (epi == MOE_EPI_STORE_BF16) return gw4::launch_shape<MOE_EPI_STORE_BF16>(prm, tm, s);
  if (epi == kEpiSwigluF16) return gw4::launch_shape<kEpiSwigluF16>(prm, tm, s);
  return gw4::launch_shape<MOE_EPI_SWIGLU_BF16>(prm, tm, s);
}

}  // namespace moe
