// Shared helpers of the sm_103a kernels: status plumbing, inline-PTX wrappers
// for mbarriers, TMA (cp.async.bulk.tensor) and the 5th-generation tensor
// cores (tcgen05: TMEM allocation, MMA, commit, TMEM loads).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/moe_gb300.h"

namespace moe {

// ---------------------------------------------------------------- host side
void set_cuda_error(cudaError_t e);
int check_launch();                 // MOE_OK or MOE_ERR_CUDA after a launch
int num_sms();                      // SMs of the current device
unsigned long long wait_timeout_ns();
unsigned int* device_error_word();  // device address of the error word (current device)
// 2-D TMA descriptor over a row-major [rows, inner] matrix of 2-byte (bf16)
// or 1-byte elements; zero fill out of bounds; optional 128-byte swizzle.
int encode_tmap_2d(CUtensorMap* m, const void* ptr, int elem_bytes, uint64_t inner, uint64_t rows, uint32_t box_inner,
                   uint32_t box_rows, bool swizzle128);
// Tiled TMA descriptor of any rank (<= 5) over bf16 or byte elements: dims
// and box innermost first, strides in bytes for dims 1..rank-1 (they need
// not increase: an outer box dimension may step along the inner one).
int encode_tmap_nd(CUtensorMap* m, const void* ptr, bool bf16, int rank, const uint64_t* dims,
                   const uint64_t* strides, const uint32_t* box, bool swizzle128);
// bf16 [rows, K] (K % 64 == 0) as k-blocks of 64: a box at (0, r, kb)
// stages `kblocks` consecutive 64-wide k-blocks of box_rows rows, each as its
// own 128-byte-swizzled tile (zero fill past the end of K or the rows).
int encode_tmap_kblocks(CUtensorMap* m, const void* ptr, uint64_t K, uint64_t rows, uint32_t box_rows,
                        uint32_t kblocks);
// bf16 SwiGLU weights [groups][gate N | up N][K] as k-blocks: a box at
// (0, f, 2g, kb) stages, per k-block, box_rows gate rows f.. of group g
// followed by the same up rows.
int encode_tmap_gateup(CUtensorMap* m, const void* ptr, uint64_t K, uint64_t N, uint64_t groups,
                       uint32_t box_rows, uint32_t kblocks);

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Bump allocator over a caller workspace (256-byte aligned slices).
struct Carve {
  char* base;
  size_t cap;
  size_t used = 0;
  Carve(void* b, size_t c) : base(static_cast<char*>(b)), cap(c) {}
  template <class T>
  T* take(size_t count) {
    size_t bytes = round_up(count * sizeof(T), 256);
    T* p = base ? reinterpret_cast<T*>(base + used) : nullptr;
    used += bytes;
    return p;
  }
  bool fits() const { return used <= cap; }
};

#define MOE_TRY(expr)              \
  do {                             \
    int _st = (expr);              \
    if (_st != MOE_OK) return _st; \
  } while (0)

// -------------------------------------------------------------- device side
#define DEVINL __device__ __forceinline__

DEVINL uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

DEVINL uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier
DEVINL void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
DEVINL void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
DEVINL void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
DEVINL void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
DEVINL bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that lets the hardware suspend the thread until the phase
// completes or about `hint_ns` nanoseconds pass (the thread stops issuing
// while it waits).
DEVINL bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Error word bits (device side).  The host maps kErrTimeout to
// MOE_ERR_TIMEOUT and kErrBadIndex (an expert id outside [0, E) met by the
// permutation, which then leaves that slot out) to MOE_ERR_INVALID_ARG.
constexpr unsigned int kErrTimeout = 1u;
constexpr unsigned int kErrBadIndex = 2u;

// Bounded wait on an mbarrier phase.  Gives up after `timeout_ns` of wall
// time (or as soon as *abort is set by another role of the block), records
// kErrTimeout in *err and returns false.
// `suspend`: let the hardware park the thread while it waits (for warps that
// are idle anyway); otherwise poll, for the latency-critical single-thread
// roles (TMA producer, MMA issuer).
DEVINL bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, unsigned long long timeout_ns,
                              unsigned int* err, volatile int* abort, bool suspend = false) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (suspend ? mbar_try_wait_suspend(bar, parity, 100000u) : mbar_try_wait(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      atomicOr(err, kErrTimeout);
      if (abort != nullptr) *abort = 1;
      return false;
    }
  }
}

// The same wait for a whole warp: lane 0 waits (so one thread, not 32, polls
// the barrier), then every lane observes the completed phase once, which
// gives each lane the acquire ordering of the barrier.  Warp-uniform result.
DEVINL bool mbar_wait_warp(uint64_t* bar, uint32_t parity, unsigned long long timeout_ns, unsigned int* err,
                           volatile int* abort) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, timeout_ns, err, abort, true) ? 1 : 0;
  ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
  if (ok) mbar_try_wait(bar, parity);
  return ok != 0;
}

// ---- TMA
DEVINL void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}
DEVINL void tma_load_2d(const void* tmap, uint64_t* bar, void* smem_dst, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
DEVINL void tma_load_3d(const void* tmap, uint64_t* bar, void* smem_dst, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
DEVINL void tma_load_4d(const void* tmap, uint64_t* bar, void* smem_dst, int x, int y, int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], "
      "[%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}
DEVINL void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---- cp.async (4-byte asynchronous copies global -> shared)
// Copies 4 bytes, or writes 4 zero bytes when `valid` is false (nothing is
// read then; `src` must still be a valid global address).
DEVINL void cp_async_4(uint32_t dst_smem, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst_smem), "l"(src), "r"(valid ? 4 : 0)
               : "memory");
}
// The same for 8 bytes (8-byte aligned addresses).
DEVINL void cp_async_8(uint32_t dst_smem, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst_smem), "l"(src), "r"(valid ? 8 : 0)
               : "memory");
}
DEVINL void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
DEVINL uint32_t ld_shared_u32(uint32_t saddr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(saddr) : "memory");
  return v;
}
DEVINL uint2 ld_shared_u2(uint32_t saddr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(saddr) : "memory");
  return v;
}
template <int N>
DEVINL void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Arrive on `bar` once all cp.async of this thread issued so far complete
// (the barrier's expected count includes this arrival).
DEVINL void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ---- tcgen05 (5th-generation tensor cores, tensor memory)
DEVINL void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
DEVINL void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
DEVINL void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
DEVINL void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DEVINL void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Named barrier `id` (1..15) over `threads` threads (a multiple of 32).
DEVINL void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
// Named barrier over `threads` threads (whole warps) that also returns the OR
// of `pred` over them.  The MMA-issuing warps take their go signal this way
// from a helper warp that does the mbarrier waits: a memory instruction
// (mbarrier wait or shared load) in the issuing warp queues behind its
// outstanding tcgen05.mma instructions and stalls the issue for ~150 ns,
// the named barrier does not.
DEVINL bool named_bar_red_or(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate).
DEVINL void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= (A * sfA) * (B * sfB)^T with packed E2M1 operands in shared
// memory and one E4M3 scale per 16 elements along K, read from tensor memory
// (kind::mxf4nvf4, block_scale, scale_vec::4X: K = 64 per instruction).
DEVINL void umma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa_tmem,
                      uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Copy 32 rows x 128 bits from shared memory into tensor memory, replicated
// into the four 32-lane quadrants (row i -> lanes i, 32+i, 64+i, 96+i).
DEVINL void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 (A: 128 lanes = rows, K along
// columns, two 16-bit elements per 32-bit column), issued by a whole
// converged warp: every lane computes the (warp-uniform) operands and
// elect.sync picks the one lane that issues.  For short MMAs next to busy
// warps this costs far less per MMA than issuing from a single-lane branch
// (measured on GB300: ~10 ns per M=128 N=16 K=16 MMA alone and ~19 ns next
// to busy conversion warps, against ~26 and ~52 ns from a lane-0 branch);
// kernels with long MMAs measured no gain.
DEVINL void umma_f16_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// umma_commit from a whole converged warp (elect.sync picks the lane, the
// lowest active one, which is the lane that issued the warp's MMAs).
DEVINL void umma_commit_warp(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}
// Arrive on `bar` once every tcgen05 op issued so far by this thread completes.
DEVINL void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// ---- CTA pairs (cluster of 2) sharing one MMA (tcgen05 cta_group::2)
DEVINL uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
DEVINL void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
DEVINL uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Arrive on a barrier of the peer CTA without a cluster-scope release, for
// signals that publish only tensor-memory state: tensor-memory stores
// completed by tcgen05.wait::st, or an accumulator fully read
// (tcgen05.wait::ld), ordered by tcgen05.fence::before_thread_sync.  A
// release at cluster scope fences every outstanding memory operation of the
// thread (on GB300 it cost the NVFP4 pair GEMM 1.7x its time when done per
// k step).
DEVINL void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Phase test without acquire, for barriers whose arrivals publish only
// tensor-memory state or TMA data (followed by tcgen05.fence::after_thread_sync).
DEVINL bool mbar_try_wait_relaxed_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.relaxed.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait of a whole warp on a barrier whose completions publish
// tensor-memory state from both CTAs (relaxed cluster-scope test).
DEVINL bool wait_cluster_warp(uint64_t* bar, uint32_t parity, unsigned long long tmo, unsigned int* err,
                              volatile int* abort) {
  bool done = mbar_try_wait_relaxed_cluster(bar, parity);
  const uint64_t t0 = globaltimer_ns();
  while (!__all_sync(0xFFFFFFFFu, done)) {
    if (*abort) return false;
    if (globaltimer_ns() - t0 > tmo) {
      if ((threadIdx.x & 31) == 0) atomicOr(err, kErrTimeout);
      *abort = 1;
      return false;
    }
    done = done || mbar_try_wait_relaxed_cluster(bar, parity);
  }
  return true;
}
DEVINL void tma_load_3d_pair(const void* tmap, uint32_t bar_cluster_addr, void* smem_dst, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar_cluster_addr), "r"(x), "r"(y), "r"(z)
      : "memory");
}
DEVINL void tma_load_4d_pair(const void* tmap, uint32_t bar_cluster_addr, void* smem_dst, int x, int y, int z,
                             int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4, %5, %6}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar_cluster_addr), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}
DEVINL void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
DEVINL void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
DEVINL void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D[tmem of both CTAs] (+)= A * B^T over the CTA pair (M = 256: rows 0..127
// from this CTA's A tile, 128..255 from the peer's; B split along N), kind::f16.
DEVINL void umma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on the mbarrier at `bar`'s offset in every CTA of `cta_mask` once all
// tcgen05 ops issued so far by this thread complete.
DEVINL void umma_commit_pair_multicast(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// The same from a whole converged warp (elect.sync picks the lane, the
// lowest active one, which is the lane that issued the warp's MMAs).
DEVINL void umma_commit_pair_multicast_warp(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (base lane + i), columns [col, col+32).
DEVINL void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
DEVINL void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32 lanes x 32 consecutive 32-bit columns from registers: thread i of the
// warp writes lane (base lane + i), columns [col, col+32).
DEVINL void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// 32 lanes x 16 columns of 32 bits.
DEVINL void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
DEVINL void tmem_st_32x32b(uint32_t taddr, const uint32_t (&r)[16]) { tmem_st_32x32b_x16(taddr, r); }
DEVINL void tmem_st_32x32b(uint32_t taddr, const uint32_t (&r)[32]) { tmem_st_32x32b_x32(taddr, r); }
DEVINL void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Two E4M3 bytes (low byte = first) -> two fp16 (exact).
DEVINL uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  asm("{\n\t.reg .b16 h;\n\tcvt.u16.u32 h, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, h;\n\t}" : "=r"(r) : "r"(two_bytes));
  return r;
}

// Shared-memory matrix descriptor of a K-major operand tile stored with the
// 128-byte swizzle (rows of 128 bytes, 8-row groups 1024 bytes apart), as TMA
// writes it with CU_TENSOR_MAP_SWIZZLE_128B into a 1024-byte aligned buffer.
DEVINL uint64_t smem_desc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFF) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                  // leading byte offset (unused for SW128 K-major)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;          // stride byte offset: 8 rows * 128 B
  d |= static_cast<uint64_t>(1) << 46;                  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;                  // swizzle mode: 128B
  return d;
}

// Shared-memory descriptor of a K-major operand without swizzle whose rows
// are 16 bytes, stored contiguously (8-row core matrices 128 bytes apart):
// the layout of a 32 x 128-bit block of scale factors for tcgen05.cp.
DEVINL uint64_t smem_desc_kmajor_noswizzle_16B_rows(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFF) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                  // leading byte offset (one core matrix along K)
  d |= static_cast<uint64_t>(128 >> 4) << 32;           // stride byte offset: 8 rows * 16 B
  d |= static_cast<uint64_t>(1) << 46;                  // descriptor version for tcgen05
  return d;                                              // swizzle mode 0: none
}

// Instruction descriptor, kind::mxf4nvf4 with block scaling: E2M1 x E2M1 ->
// fp32, E4M3 scale factors (scale format bit 0), both operands K-major,
// scale-factor ids 0, K = 64 per instruction.
__host__ __device__ constexpr uint32_t idesc_nvf4_f32(int M, int N) {
  return (1u << 7)                                  // A format E2M1
         | (1u << 10)                               // B format E2M1
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// Instruction descriptor, kind::f16: fp16 x fp16 -> fp32, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4)                                  // D format fp32 (A, B format 0: fp16)
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// Instruction descriptor, kind::f16: bf16 x bf16 -> fp32, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                                  // D format fp32
         | (1u << 7)                                // A format bf16
         | (1u << 10)                               // B format bf16
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

DEVINL uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace moe
