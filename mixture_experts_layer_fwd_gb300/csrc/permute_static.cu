// moe_permute_noalloc: the token permutation without a caller workspace.
//
// moe_permute needs a scratch workspace (per-chunk expert histograms and
// per-chunk start positions) that the caller allocates.  Some callers cannot
// allocate device memory when they dispatch tokens: runtimes that hand every
// library a fixed set of buffers at start-up and forbid allocation on the
// per-step path (cudaMalloc can synchronise the device and its latency is
// unbounded), embedders whose own allocator owns all device memory, and
// plugins that are only given their input and output buffers.  For them this
// entry point keeps its scratch in a fixed array in device memory that the
// library itself defines, so the call needs nothing but inputs and outputs.
//
// The scratch is the file-scope array below: 2 x 131072 int32 (1 MiB), held
// on every device that loads the library until the process exits.  It limits
// the problem size to ceil(T*k / 1024) * E <= 131072 (for example T*k up to
// 131072 slots with E <= 1024, or T*k up to 32768 with E = 4096).
// Every call shares the array, so two calls that overlap on the GPU (on
// different streams, or on one stream from several host threads without
// ordering) race on it; calls ordered on one stream are safe.  Nothing in the
// array needs clearing between calls: the kernels write every entry they later
// read.
#include <atomic>

#include "internal.h"

namespace moe {
namespace {

constexpr size_t kStaticEntries = 131072;  // int32 entries per scratch array

static __device__ __align__(256) int32_t g_permute_scratch[2 * kStaticEntries];

// Device address of the scratch array on the current device, looked up once
// per device (the array's name in host code is only a stand-in).  Host
// threads may make their first calls at the same time: the entries are
// atomics, and a racing lookup stores the same address.
int32_t* static_scratch() {
  static std::atomic<int32_t*> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  int32_t* p = cache[dev].load(std::memory_order_relaxed);
  if (p == nullptr) {
    void* a = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&a, g_permute_scratch);
    if (e != cudaSuccess) {
      set_cuda_error(e);
      return nullptr;
    }
    p = static_cast<int32_t*>(a);
    cache[dev].store(p, std::memory_order_relaxed);
  }
  return p;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_permute_noalloc(const int32_t* idx, int T, int k, int E, const void* x_rows, int row_bytes,
                                   const uint8_t* x_sf, int sf_row_bytes, int32_t* counts, int32_t* offsets,
                                   int32_t* row_of, int32_t* src_tok, void* xp_rows, uint8_t* xp_sf,
                                   void* stream) {
  // the same size checks as moe_permute, then the scratch limit
  if (T < 0 || k < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  if (E > kPermMaxExperts || k > E) return MOE_ERR_UNSUPPORTED;
  const long long slots = static_cast<long long>(T) * k;
  if (slots >= (1ll << 27)) return MOE_ERR_UNSUPPORTED;
  const long long chunks = (slots + kPermChunk - 1) / kPermChunk;
  if (chunks * E > static_cast<long long>(kStaticEntries)) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!idx || !row_of || !src_tok)) return MOE_ERR_INVALID_ARG;
  if (xp_rows != nullptr) {
    if (!x_rows || row_bytes <= 0 || (row_bytes % 16) != 0) return MOE_ERR_INVALID_ARG;
    if (!aligned(x_rows, 16) || !aligned(xp_rows, 16)) return MOE_ERR_INVALID_ARG;
    if (x_sf != nullptr) {
      if (!xp_sf || sf_row_bytes <= 0 || (sf_row_bytes % 4) != 0) return MOE_ERR_INVALID_ARG;
      if (!aligned(x_sf, 4) || !aligned(xp_sf, 4)) return MOE_ERR_INVALID_ARG;
    }
  }
  int32_t* scratch = static_scratch();
  if (scratch == nullptr) return MOE_ERR_CUDA;
  return permute_launch(idx, T, k, E, x_rows, row_bytes, xp_rows ? x_sf : nullptr, sf_row_bytes, counts, offsets,
                        row_of, src_tok, xp_rows, xp_sf, scratch, 2 * kStaticEntries * sizeof(int32_t),
                        static_cast<cudaStream_t>(stream));
}
