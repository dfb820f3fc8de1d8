// Library-wide host plumbing: version, status strings, CUDA error capture,
// the device error word of the bounded waits, and the wait time-out hook.
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstring>

#include "common.cuh"

namespace moe {

static char g_last_err[256] = "no error";
static unsigned long long g_timeout_ns = 1000000000ull;

// One error word per device: bits set by bounded device waits that run out
// and by the permutation when it meets an expert id outside [0, E).
__device__ unsigned int g_err_word;

void set_cuda_error(cudaError_t e) {
  snprintf(g_last_err, sizeof(g_last_err), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
}

int check_launch() {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

unsigned long long wait_timeout_ns() { return g_timeout_ns; }

unsigned int* device_error_word() {
  static unsigned int* cache[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (cache[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_err_word);
    if (e != cudaSuccess) {
      set_cuda_error(e);
      return nullptr;
    }
    cache[dev] = static_cast<unsigned int*>(p);
  }
  return cache[dev];
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
    if (e == cudaSuccess && q == cudaDriverEntryPointSuccess) fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

int encode_tmap_2d(CUtensorMap* m, const void* ptr, int elem_bytes, uint64_t inner, uint64_t rows, uint32_t box_inner,
                   uint32_t box_rows, bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) return MOE_ERR_CUDA;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * static_cast<uint64_t>(elem_bytes)};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                  const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

// Any-rank tiled descriptor (rank <= 5): dims / box innermost first,
// strides (bytes) of dims 1.. ; zero fill out of bounds.
int encode_tmap_nd(CUtensorMap* m, const void* ptr, bool bf16, int rank, const uint64_t* dims,
                   const uint64_t* strides, const uint32_t* box, bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) return MOE_ERR_CUDA;
  if (rank < 1 || rank > 5) return MOE_ERR_INVALID_ARG;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                  static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), d, st, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

// bf16 [rows, K] viewed as [K/64 k-blocks][rows][64]: a box {64, box_rows,
// kblocks} at (0, r, kb) stages k-blocks kb.. of rows r.. as consecutive
// 128-byte-row tiles (one per k-block), 128-byte swizzle.
int encode_tmap_kblocks(CUtensorMap* m, const void* ptr, uint64_t K, uint64_t rows, uint32_t box_rows,
                        uint32_t kblocks) {
  auto fn = encode_fn();
  if (!fn) return MOE_ERR_CUDA;
  cuuint64_t dims[3] = {64, rows, K / 64};
  cuuint64_t strides[2] = {K * 2, 128};
  cuuint32_t box[3] = {64, box_rows, kblocks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

// bf16 SwiGLU weights [groups][gate N rows | up N rows][K] viewed as
// [K/64 k-blocks][2*groups][N][64]: a box {64, box_rows, 2, kblocks} at
// (0, f, 2g, kb) stages, per k-block, rows f.. of group g's gate half
// followed by the same rows of its up half.
int encode_tmap_gateup(CUtensorMap* m, const void* ptr, uint64_t K, uint64_t N, uint64_t groups,
                       uint32_t box_rows, uint32_t kblocks) {
  auto fn = encode_fn();
  if (!fn) return MOE_ERR_CUDA;
  cuuint64_t dims[4] = {64, N, 2 * groups, K / 64};
  cuuint64_t strides[3] = {K * 2, N * K * 2, 128};
  cuuint32_t box[4] = {64, box_rows, 2, kblocks};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

__global__ void selftest_wait_kernel(unsigned int* err, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // nothing ever arrives on `bar`: the bounded wait must give up and record it
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, timeout_ns, err, nullptr);
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_version(void) { return 100; }

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    default: return "MOE_ERR_UNKNOWN";
  }
}

const char* moe_last_cuda_error(void) { return g_last_err; }

int moe_set_wait_timeout_ns(unsigned long long ns) {
  g_timeout_ns = ns ? ns : 1000000000ull;
  return MOE_OK;
}

int moe_sync_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_err_word, sizeof(v));
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  if (v != 0) {
    unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_err_word, &zero, sizeof(zero));
    if (e != cudaSuccess) {
      set_cuda_error(e);
      return MOE_ERR_CUDA;
    }
    return (v & kErrTimeout) ? MOE_ERR_TIMEOUT : MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

int moe_selftest_wait_timeout(unsigned long long timeout_ns, void* stream) {
  unsigned int* err = device_error_word();
  if (!err) return MOE_ERR_CUDA;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, timeout_ns);
  return check_launch();
}

}  // extern "C"
