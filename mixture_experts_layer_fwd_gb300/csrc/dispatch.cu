// Fused dispatch: the router's top-k and the stable permutation in one
// cooperative launch joined by two grid barriers.
//
// "CuTeDSL at Perplexity", local MoE dispatch, decode variant: routing
// processed inside the dispatch kernel, which signals the rest of the grid
// and hands out slots from shared-memory counters instead of launching a
// second kernel; its grid-sync section prices a grid barrier at about 3 us
// against a separate launch.  "Como Servimos um Modelo MoE de 397B ...",
// section "Roadmap restante", names fusing the top-k selection.
//
// The results are those of moe_route_ex followed by moe_permute, bit for bit
// (same per-token router, same stable slot order):
//   phase A  block b routes its contiguous token chunk (one warp per token),
//            counts its slots per expert in shared memory -> hist[e][b]
//   barrier
//   phase B  one warp per expert scans the row hist[e][*] (a lane's eight
//            consecutive blocks by two 16-byte loads, then one warp scan of
//            the lane totals):
//            base[e][b] = sum of hist[e][b'] over b' < b, counts[e] = total
//   barrier
//   phase C  every block scans counts (offsets; block 0 stores them), seeds
//            its shared counters with offsets[e] + base[e][b], places its
//            slots in order to write row_of / src_tok (ranks inside a warp
//            from __match_any_sync; more than 128 slots: split over the 32
//            warps, with per-warp expert counts scanned in warp order), then
//            copies its slots' token rows
// A block's chunk is contiguous and blocks are ordered, so inside an expert
// the rows stay in ascending token order.
//
// Grid barrier: a counter in the workspace (zeroed by a memset on the same
// stream before each launch) counts block arrivals; barrier i completes at
// (i + 1) * gridDim.x arrivals.  The launch is cooperative, so every block
// is resident and every arrival comes.  Each wait is bounded in wall time
// (moe_set_wait_timeout_ns): a wait that runs out records MOE_ERR_TIMEOUT in
// the device error word and the block returns.
#include <atomic>
#include <cstring>

#include "internal.h"
#include "permute.cuh"
#include "route.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;  // 32 warps: enough row copies in flight per SM to stream at HBM speed
constexpr int kWarps = kThreads / 32;
constexpr int kScanPer = (1024 + kThreads - 1) / kThreads;  // experts per thread in the offsets scan
constexpr int kMaxBlocks = 256;  // grid of the fused dispatch: one block per SM, at most this many
constexpr int kWalk = 4096;      // slots whose expert ids the walk stages in shared memory at a time
constexpr int kMaxE = 1024;      // experts (moe_route_permute's limit)
constexpr int kSerialWalk = 128; // a block with at most this many slots places them from one warp

struct DispatchArgs {
  const float* logits;
  int T, E, k, renorm;
  int32_t* idx;
  float* w;
  const uint8_t* x;
  int row_bytes;
  const uint8_t* x_sf;
  int sf_bytes;
  int32_t* counts;
  int32_t* offsets;
  int32_t* row_of;
  int32_t* src_tok;
  uint8_t* xp;
  uint8_t* xp_sf;
  int32_t* hist;  // [E][kMaxBlocks]: per-block slot counts of each expert
  int32_t* base;  // [E][kMaxBlocks]: each block's first position inside each expert
  unsigned int* bar;
  unsigned int* err;
  unsigned long long timeout_ns;
};

// Arrive on the grid barrier and wait (bounded) until `target` blocks have
// arrived.  Called by every thread of the block; returns false in every
// thread if the wait ran out.
DEVINL bool grid_barrier(unsigned int* bar, unsigned int target, unsigned long long timeout_ns, unsigned int* err,
                         volatile int* s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // this block's global writes before its arrival
    atomicAdd(bar, 1u);
    int ok = 1;
    volatile unsigned int* v = bar;
    if (*v < target) {
      const uint64_t t0 = globaltimer_ns();
      while (*v < target) {
        if (globaltimer_ns() - t0 > timeout_ns) {
          atomicOr(err, kErrTimeout);
          ok = 0;
          break;
        }
      }
    }
    __threadfence();  // the other blocks' writes before this block's reads
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

// Places slots [w0, w1) in order, one warp: slot s goes to position
// ctr[e] + (its rank among the group's earlier slots of expert e), and
// ctr[e] advances by the group's count; writes row_of and src_tok.  The
// slots' expert ids are ids[s - id0].  Ids outside [0, E) (routing of NaN
// logits) are left out.
DEVINL void place_slots(const DispatchArgs& a, const int32_t* ids, int id0, int w0, int w1, int32_t* ctr, int lane) {
  for (int j0 = w0; j0 < w1; j0 += 32) {
    const int s = j0 + lane;
    const int e = s < w1 ? ids[s - id0] : 0;
    const bool act = s < w1 && static_cast<unsigned>(e) < static_cast<unsigned>(a.E);
    const unsigned mask = __ballot_sync(0xFFFFFFFFu, act);
    if (act) {
      const unsigned peers = __match_any_sync(mask, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int pos = ctr[e] + rank;
      __syncwarp(mask);
      if (rank == 0) ctr[e] += __popc(peers);
      a.row_of[s] = pos;
      a.src_tok[pos] = s / a.k;
    } else if (s < w1) {
      a.row_of[s] = -1;  // left out
    }
    __syncwarp();
  }
}

template <int EPL, bool TO_F16>
__global__ void __launch_bounds__(kThreads) route_permute_kernel(const DispatchArgs a) {
  extern __shared__ int32_t sh[];  // E counters, then hw: kWarps x E per-warp counts
  int32_t* hw = sh + a.E;
  __shared__ int32_t s_idx[kWalk];
  __shared__ int warp_tot[kWarps];
  __shared__ int s_ok;
  const int nb = gridDim.x, b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E, k = a.k;
  const int per = (a.T + nb - 1) / nb;
  const int t0 = min(a.T, b * per), t1 = min(a.T, t0 + per);
  const int s0 = t0 * k, s1 = t1 * k;

  // ---- phase A: route this block's tokens (a warp's next token's logits
  // loaded while it picks the current one's experts, up to 256 experts),
  // histogram of its slots
  if (EPL <= 8) {
    uint32_t cur[EPL];
    int t = t0 + warp;
    if (t < t1) route_load<EPL>(a.logits, t, E, lane, cur);
    for (; t < t1; t += kWarps) {
      uint32_t nxt[EPL];
      const bool more = t + kWarps < t1;
      if (more) route_load<EPL>(a.logits, t + kWarps, E, lane, nxt);
      route_pick<EPL>(cur, t, E, k, a.renorm, a.idx, a.w, lane);
      if (more) {
#pragma unroll
        for (int j = 0; j < EPL; ++j) cur[j] = nxt[j];
      }
    }
  } else {
    for (int t = t0 + warp; t < t1; t += kWarps) route_token<EPL>(a.logits, t, E, k, a.renorm, a.idx, a.w, lane);
  }
  for (int e = threadIdx.x; e < E; e += kThreads) sh[e] = 0;
  __syncthreads();
  // the router's ids lie in [0, E) for finite logits; anything else (NaN
  // logits) is left out of the permutation as moe_permute does
  for (int s = s0 + threadIdx.x; s < s1; s += kThreads) {
    const int e = a.idx[s];
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E))
      atomicAdd(&sh[e], 1);
    else
      atomicOr(a.err, kErrBadIndex);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kThreads) a.hist[static_cast<size_t>(e) * kMaxBlocks + b] = sh[e];
  if (!grid_barrier(a.bar, static_cast<unsigned int>(nb), a.timeout_ns, a.err, &s_ok)) return;

  // ---- phase B: per-expert scans over the blocks, one warp per expert
  // (expert b * kWarps + warp, so E / 32 blocks take part).  The counts of
  // expert e lie in row e of hist (kMaxBlocks entries, those of blocks >= nb
  // unused): lane l loads blocks 8 l .. 8 l + 7 with two 16-byte loads, one
  // warp scan of the lane totals, then each lane's running sum over its own
  // blocks, stored to row e of base the same way
  for (int e = b * kWarps + warp; e < E; e += nb * kWarps) {
    static_assert(kMaxBlocks == 32 * 8, "eight blocks per lane");
    const int4* src = reinterpret_cast<const int4*>(a.hist + static_cast<size_t>(e) * kMaxBlocks) + 2 * lane;
    const int4 q0 = __ldcg(src), q1 = __ldcg(src + 1);
    int h[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    int tot = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (8 * lane + u >= nb) h[u] = 0;
      tot += h[u];
    }
    int incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += o;
    }
    int o[8];
    int run = incl - tot;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      o[u] = run;
      run += h[u];
    }
    int4* dst = reinterpret_cast<int4*>(a.base + static_cast<size_t>(e) * kMaxBlocks) + 2 * lane;
    dst[0] = make_int4(o[0], o[1], o[2], o[3]);
    dst[1] = make_int4(o[4], o[5], o[6], o[7]);
    if (lane == 31) a.counts[e] = incl;
  }
  if (!grid_barrier(a.bar, 2u * static_cast<unsigned int>(nb), a.timeout_ns, a.err, &s_ok)) return;

  // ---- phase C: offsets (exclusive scan of counts, E <= 1024: kScanPer
  // per thread), this block's starting positions, slot assignment, row copies
  int c4[kScanPer];
  int loc = 0;
#pragma unroll
  for (int u = 0; u < kScanPer; ++u) {
    const int e = threadIdx.x * kScanPer + u;
    c4[u] = e < E ? __ldcg(a.counts + e) : 0;
    loc += c4[u];
  }
  int incl = loc;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int run = incl - loc;
  for (int i = 0; i < warp; ++i) run += warp_tot[i];
#pragma unroll
  for (int u = 0; u < kScanPer; ++u) {
    const int e = threadIdx.x * kScanPer + u;
    if (e < E) {
      sh[e] = run + __ldcg(a.base + static_cast<size_t>(e) * kMaxBlocks + b);
      if (b == 0) a.offsets[e] = run;
    }
    run += c4[u];
  }
  if (b == 0 && threadIdx.x == kThreads - 1) a.offsets[E] = run;  // the last thread's run is the total
  __syncthreads();
  if (s1 - s0 <= kSerialWalk) {
    // few slots: the block stages their expert ids, warp 0 places them
    for (int s = s0 + threadIdx.x; s < s1; s += kThreads) s_idx[s - s0] = __ldcg(a.idx + s);
    __syncthreads();
    if (warp == 0) place_slots(a, s_idx, s0, s0, s1, sh, lane);
    __syncthreads();
  } else {
    // kWalk slots at a time: warp w takes the w-th of 32 contiguous pieces
    // and counts its experts (its row of hw), each expert's warp rows are
    // scanned in order from the block's running position, and every warp
    // then places its piece's slots, all warps at once
    int32_t* hrow = hw + static_cast<size_t>(warp) * E;
    for (int c0 = s0; c0 < s1; c0 += kWalk) {
      const int c1 = min(s1, c0 + kWalk);
      const int q = (c1 - c0 + kWarps - 1) / kWarps;
      const int w0 = min(c1, c0 + warp * q), w1 = min(c1, w0 + q);
      for (int e = lane; e < E; e += 32) hrow[e] = 0;
      __syncwarp();
      for (int s = w0 + lane; s < w1; s += 32) {
        const int e = __ldcg(a.idx + s);
        s_idx[s - c0] = e;
        if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) atomicAdd(&hrow[e], 1);
      }
      __syncthreads();
      for (int e = threadIdx.x; e < E; e += kThreads) {
        int run = sh[e];
        for (int v = 0; v < kWarps; ++v) {
          const int c = hw[static_cast<size_t>(v) * E + e];
          hw[static_cast<size_t>(v) * E + e] = run;
          run += c;
        }
        sh[e] = run;
      }
      __syncthreads();
      place_slots(a, s_idx, c0, w0, w1, hrow, lane);
      __syncthreads();
    }
  }
  if (a.xp != nullptr)
    for (int s = s0 + warp; s < s1; s += kWarps) {
      const int pos = a.row_of[s];
      if (pos >= 0) copy_row<TO_F16>(a.x, a.row_bytes, a.x_sf, a.sf_bytes, s / k, a.xp, a.xp_sf, pos, lane);
    }
}

__global__ void selftest_grid_barrier_kernel(unsigned int* bar, unsigned int* err, unsigned long long timeout_ns) {
  __shared__ int s_ok;
  // one more arrival than the grid can make: the wait must give up
  grid_barrier(bar, gridDim.x + 1u, timeout_ns, err, &s_ok);
}

__device__ unsigned int g_selftest_bar;

int grid_size(int T) { return std::max(1, std::min({T, num_sms(), kMaxBlocks})); }

template <class Kern, class... Args>
int launch_cooperative(Kern kern, int grid, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return check_launch();
}

template <int EPL, bool TO_F16>
int launch_epl(const DispatchArgs& a, int grid, cudaStream_t s) {
  // E counters + kWarps x E per-warp counts (up to 132 KB at E = 1024)
  const size_t smem = static_cast<size_t>(a.E) * (1 + kWarps) * sizeof(int32_t);
  // the attribute is per device; a racing first call sets the same value
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (!attr_set[dev].load(std::memory_order_relaxed)) {
    const int max_dyn = static_cast<int>(static_cast<size_t>(kMaxE) * (1 + kWarps) * sizeof(int32_t));
    cudaError_t e = cudaFuncSetAttribute(route_permute_kernel<EPL, TO_F16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn);
    if (e != cudaSuccess) {
      set_cuda_error(e);
      return MOE_ERR_CUDA;
    }
    attr_set[dev].store(true, std::memory_order_relaxed);
  }
  return launch_cooperative(route_permute_kernel<EPL, TO_F16>, grid, smem, s, a);
}

template <bool TO_F16>
int launch_dispatch(const DispatchArgs& a, int grid, cudaStream_t s) {
  const int epl = (a.E + 31) / 32;
  if (epl <= 1) return launch_epl<1, TO_F16>(a, grid, s);
  if (epl <= 2) return launch_epl<2, TO_F16>(a, grid, s);
  if (epl <= 4) return launch_epl<4, TO_F16>(a, grid, s);
  if (epl <= 8) return launch_epl<8, TO_F16>(a, grid, s);
  if (epl <= 16) return launch_epl<16, TO_F16>(a, grid, s);
  return launch_epl<32, TO_F16>(a, grid, s);
}

}  // namespace

size_t route_permute_ws_bytes(int T, int E) {
  (void)T;
  // barrier counter, hist and base: [E][kMaxBlocks] each
  return 256 + 2 * round_up(static_cast<size_t>(kMaxBlocks) * E * sizeof(int32_t), 256);
}

int route_permute_launch(const float* logits, int T, int E, int k, int renorm, int32_t* idx, float* w,
                         const void* x_rows, int row_bytes, const uint8_t* x_sf, int sf_row_bytes, int32_t* counts,
                         int32_t* offsets, int32_t* row_of, int32_t* src_tok, void* xp_rows, uint8_t* xp_sf,
                         void* ws, size_t ws_bytes, cudaStream_t s, bool to_f16) {
  if (ws_bytes < route_permute_ws_bytes(T, E) || ws == nullptr) return MOE_ERR_WORKSPACE;
  const int grid = grid_size(T);
  Carve c(ws, ws_bytes);
  DispatchArgs a;
  a.bar = c.take<unsigned int>(1);
  a.hist = c.take<int32_t>(static_cast<size_t>(kMaxBlocks) * E);
  a.base = c.take<int32_t>(static_cast<size_t>(kMaxBlocks) * E);
  a.logits = logits;
  a.T = T;
  a.E = E;
  a.k = k;
  a.renorm = renorm ? 1 : 0;
  a.idx = idx;
  a.w = w;
  a.x = static_cast<const uint8_t*>(x_rows);
  a.row_bytes = row_bytes;
  a.x_sf = xp_rows != nullptr ? x_sf : nullptr;
  a.sf_bytes = sf_row_bytes;
  a.counts = counts;
  a.offsets = offsets;
  a.row_of = row_of;
  a.src_tok = src_tok;
  a.xp = static_cast<uint8_t*>(xp_rows);
  a.xp_sf = xp_sf;
  a.err = device_error_word();
  if (a.err == nullptr) return MOE_ERR_CUDA;
  a.timeout_ns = wait_timeout_ns();
  cudaError_t e = cudaMemsetAsync(a.bar, 0, sizeof(unsigned int), s);
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return to_f16 ? launch_dispatch<true>(a, grid, s) : launch_dispatch<false>(a, grid, s);
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_route_permute_workspace_size(int T, int k, int E) {
  if (T < 0 || k < 1 || E < 1) return 0;
  return route_permute_ws_bytes(T, E);
}

extern "C" int moe_route_permute(const float* logits, int T, int E, int k, int renorm, int32_t* idx, float* w,
                                 const void* x_rows, int row_bytes, const uint8_t* x_sf, int sf_row_bytes,
                                 int32_t* counts, int32_t* offsets, int32_t* row_of, int32_t* src_tok, void* xp_rows,
                                 uint8_t* xp_sf, void* ws, size_t ws_bytes, void* stream) {
  if (T < 0 || E < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (k > E || k > 32 || E > 1024) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(T) * k >= (1ll << 27)) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!logits || !idx || !w || !row_of || !src_tok) return MOE_ERR_INVALID_ARG;
  if (!aligned(logits, 4) || !aligned(idx, 4) || !aligned(w, 4)) return MOE_ERR_INVALID_ARG;
  if (xp_rows != nullptr) {
    if (!x_rows || row_bytes <= 0 || (row_bytes % 16) != 0) return MOE_ERR_INVALID_ARG;
    if (!aligned(x_rows, 16) || !aligned(xp_rows, 16)) return MOE_ERR_INVALID_ARG;
    if (x_sf != nullptr) {
      if (!xp_sf || sf_row_bytes <= 0 || (sf_row_bytes % 4) != 0) return MOE_ERR_INVALID_ARG;
      if (!aligned(x_sf, 4) || !aligned(xp_sf, 4)) return MOE_ERR_INVALID_ARG;
    }
  }
  if (ws != nullptr && !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  return route_permute_launch(logits, T, E, k, renorm, idx, w, x_rows, row_bytes, x_sf, sf_row_bytes, counts,
                              offsets, row_of, src_tok, xp_rows, xp_sf, ws, ws_bytes,
                              static_cast<cudaStream_t>(stream), false);
}

extern "C" int moe_selftest_grid_barrier_timeout(unsigned long long timeout_ns, void* stream) {
  unsigned int* err = device_error_word();
  if (!err) return MOE_ERR_CUDA;
  void* bar = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&bar, g_selftest_bar);
  if (e == cudaSuccess) e = cudaMemsetAsync(bar, 0, sizeof(unsigned int), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return launch_cooperative(selftest_grid_barrier_kernel, 2, 0, static_cast<cudaStream_t>(stream),
                            static_cast<unsigned int*>(bar), err, timeout_ns);
}
