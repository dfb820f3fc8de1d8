// Pieces shared by the grouped-GEMM kernels: problem description, the
// persistent tile schedule over ragged groups, and the epilogues that turn a
// tensor-memory accumulator tile into the layer's outputs.
#pragma once

#include "nvfp4.cuh"

namespace moe {
namespace gg {

constexpr int BM = 128;       // rows (tokens) per tile = MMA M
constexpr int MAX_G = 1025;   // routed groups + the shared expert

struct Prob {
  int n_out;         // output columns N
  int K;             // reduction length
  int w_rows;        // weight rows per group (N, or 2N for SwiGLU)
  int n_tiles;       // column blocks per group
  int a_rows;        // rows of A (bounds of the scale loads)
  int w_rows_total;  // rows of W over all groups
  void* c;
  uint8_t* c_sf;
  const float* a_g;
  const float* w_g;
  const float* c_g;
  const uint8_t* a_sf;
  const uint8_t* w_sf;
  int a_f16;         // A holds fp16 (else bf16), NVFP4-weight kernel
};

struct Params {
  CUtensorMap tma_a[2];  // [0] routed problem, [1] shared-expert problem
  CUtensorMap tma_w[2];
  CUtensorMap tma_asf[2];  // scale rows of A / W (512-element-stage FP4 kernel)
  CUtensorMap tma_wsf[2];
  // token boxes of 16, 32, ..., 128 rows (bf16 CTA-pair kernel: each CTA
  // stages the half of a tile's tokens it needs, rounded up to 16 rows)
  CUtensorMap tma_b_rows[2][8];
  Prob prob[2];
  const int32_t* offsets;  // [G+1] rows of each routed group in A
  int G;
  int shared_rows;  // rows of the shared problem; < 0: none
  unsigned int* err;
  unsigned long long timeout_ns;
};

struct TileInfo {
  int pb;     // problem: 0 routed, 1 shared
  int g;      // group inside the problem
  int row0;   // first row of the group in A / C
  int rows;   // rows of the group
  int m_blk;  // row block inside the group
  int n_blk;  // column block
};

// Tile t -> (group, column block, row block), row blocks fastest.  s_prefix
// holds the exclusive prefix of tiles per group (GT+1 entries); TM is the
// number of rows per tile (128, or 256 for the 2-SM kernel's pair tiles).
template <int TM = BM>
DEVINL TileInfo decode_tile(int t, const int* s_prefix, const int* s_off, int GT, int G, int shared_rows) {
  int lo = 0, hi = GT;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_prefix[mid] <= t) lo = mid; else hi = mid;
  }
  TileInfo ti;
  const bool routed = lo < G;
  ti.pb = routed ? 0 : 1;
  ti.g = routed ? lo : 0;
  ti.row0 = routed ? s_off[lo] : 0;
  ti.rows = routed ? (s_off[lo + 1] - s_off[lo]) : shared_rows;
  const int mt = (ti.rows + TM - 1) / TM;
  const int local = t - s_prefix[lo];
  ti.n_blk = local / mt;
  ti.m_blk = local - ti.n_blk * mt;
  return ti;
}

struct PairTile {
  int pb;    // problem: 0 routed, 1 shared
  int g;     // group inside the problem
  int row0;  // first row of the tile's tokens in A / C
  int cnt;   // tokens of the tile (1..TM)
  int n;     // MMA N: cnt rounded up to 16 (or 32)
  int blk;   // weight block: 128 features (SwiGLU) or 256 output columns
};

// Tile t -> (group, weight block, token block) of the CTA-pair kernels
// (weights on the MMA's M side, tokens on N), token blocks fastest so that
// the pairs working at the same time share a weight block through L2.  A
// group of `rows` rows has ceil(rows/TM) token blocks of ng rows each (ng =
// rows / blocks rounded up to NQ, the MMA's N granularity: 16, or 32 for the
// block-scaled MMAs); the last one takes the remainder, its N rounded up to
// NQ.  TM is a multiple of NQ.
template <int TM, int NQ = 16>
DEVINL PairTile decode_pair_tile(int t, const int* s_prefix, const int* s_off, int GT, int G, int shared_rows) {
  int lo = 0, hi = GT;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_prefix[mid] <= t) lo = mid; else hi = mid;
  }
  PairTile ti;
  const bool routed = lo < G;
  ti.pb = routed ? 0 : 1;
  ti.g = routed ? lo : 0;
  const int start = routed ? s_off[lo] : 0;
  const int rows = routed ? (s_off[lo + 1] - s_off[lo]) : shared_rows;
  const int nb = (rows + TM - 1) / TM;
  static_assert(TM % NQ == 0 && (NQ & (NQ - 1)) == 0, "token blocks are whole MMA N steps");
  const int ng = ((rows + nb - 1) / nb + NQ - 1) & ~(NQ - 1);
  const int local = t - s_prefix[lo];
  ti.blk = local / nb;
  const int m = local - ti.blk * nb;
  ti.row0 = start + m * ng;
  ti.cnt = min(ng, rows - m * ng);
  ti.n = (ti.cnt + NQ - 1) & ~(NQ - 1);
  return ti;
}

// Loads the group offsets and builds the per-group tile prefix in shared
// memory.  Called by every thread of the block (contains barriers).
// Offsets are clamped to [0, rows of A] and a group whose end lies before its
// start gets no tiles, so offsets that break the documented contract (non-
// decreasing, offsets[G] <= M_total) cannot send a tile outside A or C; the
// tile decoders only ever land on groups with at least one tile.
template <int THREADS, int NUM_WARPS, int TM = BM>
DEVINL void build_schedule(const Params& p, int* s_off, int* s_prefix, int* warp_sums) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  const int GT = G + (p.shared_rows >= 0 ? 1 : 0);
  for (int i = threadIdx.x; i <= G; i += THREADS) s_off[i] = min(max(p.offsets[i], 0), p.prob[0].a_rows);
  __syncthreads();
  const int per = (GT + THREADS - 1) / THREADS;
  const int g0 = threadIdx.x * per;
  int local = 0;
  for (int g = g0; g < min(GT, g0 + per); ++g) {
    const int rows = (g < G) ? max(s_off[g + 1] - s_off[g], 0) : p.shared_rows;
    local += ((rows + TM - 1) / TM) * p.prob[g < G ? 0 : 1].n_tiles;
  }
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = (lane < NUM_WARPS) ? warp_sums[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, v, off);
      if (lane >= off) v += o;
    }
    warp_sums[lane] = v;
  }
  __syncthreads();
  int run = incl - local + (warp ? warp_sums[warp - 1] : 0);
  for (int g = g0; g < min(GT, g0 + per); ++g) {
    s_prefix[g] = run;
    const int rows = (g < G) ? max(s_off[g + 1] - s_off[g], 0) : p.shared_rows;
    run += ((rows + TM - 1) / TM) * p.prob[g < G ? 0 : 1].n_tiles;
  }
  if (threadIdx.x == 0) s_prefix[GT] = warp_sums[NUM_WARPS - 1];
}

// silu(g) = g * sigmoid(g) with the fast exponential and division (a few ulp;
// exact zero for g below about -88, where e^-g overflows)
DEVINL float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Stores NV tokens x one column per lane as bf16: lanes 2j and 2j+1 hold
// columns col_even and col_even+1 of the same tokens; after one exchange each
// lane writes both columns of one token (even lane: tokens 2i, odd lane:
// tokens 2i+1).  Tokens from valid_tokens on are not stored.
template <int NV>
DEVINL void store_pairs(const Prob& P, const float (&h)[NV], int col, int row_first, int valid_tokens, int lane) {
  const bool odd = lane & 1;
  const int col_even = col & ~1;
  if (col_even >= P.n_out) return;  // uniform over the lanes sharing tokens: n_out % 32 == 0
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
          pack_bf16x2(lo, hi);
  }
}


// Epilogue of one tile held in tensor memory: ACC_N fp32 columns per row.
// STORE: C[row, n_blk*ACC_N + c] = bf16(scale * acc[c]).
// SWIGLU: columns [0, ACC_N/2) are gate, [ACC_N/2, ACC_N) up of the same
// features; C[row, n_blk*ACC_N/2 + c] = silu(scale*g) * (scale*u), stored as
// bf16 or quantised to NVFP4 with global scale *P.c_g.
// Every lane of the warp must call it (tcgen05.ld is warp-collective); only
// rows inside the tile's group are stored.
// SWIGLU_MX: the result is quantised to MXFP4 (MX_FP4) or MXFP8, one E8M0
// scale per 32 columns (one tensor-memory chunk of a row).
template <int EPI, int ACC_N, bool MX_FP4 = false>
DEVINL void epilogue_tile(const Prob& P, const TileInfo& ti, uint32_t taddr, int r_in_tile, float scale) {
  const int m_local = ti.m_blk * BM + r_in_tile;
  const bool valid = m_local < ti.rows;
  const size_t row = static_cast<size_t>(ti.row0) + m_local;
  if (EPI == MOE_EPI_STORE_BF16) {
#pragma unroll 1
    for (int cc = 0; cc < ACC_N / 32; ++cc) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(taddr + cc * 32, r);
      tmem_ld_wait();
      const int col = ti.n_blk * ACC_N + cc * 32;
      if (valid && col < P.n_out) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(P.c) + row * P.n_out + col);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 o;
          o.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]) * scale, __uint_as_float(r[8 * v + 1]) * scale);
          o.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]) * scale, __uint_as_float(r[8 * v + 3]) * scale);
          o.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]) * scale, __uint_as_float(r[8 * v + 5]) * scale);
          o.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]) * scale, __uint_as_float(r[8 * v + 7]) * scale);
          dst[v] = o;
        }
      }
    }
  } else {
    constexpr int HALF = ACC_N / 2;
    const float cg = (EPI == MOE_EPI_SWIGLU_NVFP4) ? __ldg(P.c_g) : 1.0f;
#pragma unroll 1
    for (int cc = 0; cc < HALF / 32; ++cc) {
      uint32_t rg[32], ru[32];
      tmem_ld_32x32b_x32(taddr + cc * 32, rg);
      tmem_ld_32x32b_x32(taddr + HALF + cc * 32, ru);
      tmem_ld_wait();
      const int col = ti.n_blk * HALF + cc * 32;
      if (valid && col < P.n_out) {
        float h[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
          h[i] = silu_f(__uint_as_float(rg[i]) * scale) * (__uint_as_float(ru[i]) * scale);
        if (EPI == MOE_EPI_SWIGLU_BF16) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(P.c) + row * P.n_out + col);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(pack_bf16x2(h[8 * v], h[8 * v + 1]), pack_bf16x2(h[8 * v + 2], h[8 * v + 3]),
                                pack_bf16x2(h[8 * v + 4], h[8 * v + 5]), pack_bf16x2(h[8 * v + 6], h[8 * v + 7]));
        } else if (EPI == MOE_EPI_SWIGLU_MX) {
          uint32_t q[MX_FP4 ? 4 : 8];
          const uint32_t sc = mx_quantize32<MX_FP4>(h, q);
          if constexpr (MX_FP4) {
            *reinterpret_cast<uint4*>(static_cast<uint8_t*>(P.c) + row * (P.n_out / 2) + col / 2) =
                make_uint4(q[0], q[1], q[2], q[3]);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(P.c) + row * P.n_out + col);
            dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
            dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
          }
          P.c_sf[row * (P.n_out / 32) + col / 32] = static_cast<uint8_t>(sc);
        } else {
          float b0[16], b1[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            b0[i] = h[i];
            b1[i] = h[16 + i];
          }
          uint32_t c0[2], c1[2];
          const uint32_t s0 = nvfp4_quantize16(b0, cg, c0);
          const uint32_t s1 = nvfp4_quantize16(b1, cg, c1);
          uint8_t* cdst = static_cast<uint8_t*>(P.c) + row * (P.n_out / 2) + col / 2;
          *reinterpret_cast<uint4*>(cdst) = make_uint4(c0[0], c0[1], c1[0], c1[1]);
          *reinterpret_cast<uint16_t*>(P.c_sf + row * (P.n_out / 16) + col / 16) =
              static_cast<uint16_t>(s0 | (s1 << 8));
        }
      }
    }
  }
}

}  // namespace gg
}  // namespace moe
