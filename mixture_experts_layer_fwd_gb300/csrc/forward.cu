// The whole layer: (NVFP4 / MX activation quantisation) -> router top-k and
// permutation (one cooperative launch, dispatch.cu) -> grouped GEMM gate/up +
// SwiGLU -> grouped GEMM down -> combine, all stream-ordered on the caller's
// stream with no host synchronisation.
//
// Step order follows the pages: routing table, local dispatch into expert
// buffers, MoE GEMM, weighted combine ("CuTeDSL at Perplexity", local
// dispatch / combine; "Hosting Qwen on Blackwell", sections "MoE Dispatch -
// Combine" and "MoE GEMM"); activations are quantised to NVFP4 before
// dispatch ("Driving vLLM WideEP ... (Part I)", section "NVFP4 MoE
// dispatch").  The shared expert is folded into both grouped GEMM launches
// as one more group over all T tokens.
#include "internal.h"

namespace moe {
namespace {

struct FwdBufs {
  int32_t* idx;
  float* w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* row_of;
  int32_t* src_tok;
  void* perm_ws;
  size_t perm_ws_bytes;
  uint8_t* xq;
  uint8_t* xsf;
  float* gx;
  void* qws;
  void* xp;
  uint8_t* xp_sf;
  void* h;
  uint8_t* h_sf;
  void* hs;
  uint8_t* hs_sf;
  uint16_t* Y;
  uint16_t* Ys;
  float* gate;  // shared-expert gate per token (gated layers)
};

inline bool is_mx(int fmt) { return fmt == MOE_FMT_MXFP4 || fmt == MOE_FMT_MXFP8; }

// Router top-k and permutation of the layer's rows in one cooperative launch
// (dispatch.cu; measured faster than the router + permutation kernels at
// every size of the workloads here).  x_rows: bf16 or coded rows of
// row_bytes, with optional scale bytes.
int dispatch(const float* logits, int T, int E, int k, int renorm, const FwdBufs& b, const void* x_rows,
             int row_bytes, const uint8_t* x_sf, int sf_bytes, cudaStream_t s, bool to_f16 = false) {
  return route_permute_launch(logits, T, E, k, renorm, b.idx, b.w, x_rows, row_bytes, x_sf, sf_bytes, b.counts,
                              b.offsets, b.row_of, b.src_tok, b.xp, b.xp_sf, b.perm_ws, b.perm_ws_bytes, s, to_f16);
}

// bytes of n MX-coded elements (MXFP4 packs two per byte)
inline size_t mx_code_bytes(int fmt, size_t n) { return fmt == MOE_FMT_MXFP4 ? n / 2 : n; }

// MX layers: both operands in the same MX format, E8M0 scales, no global
// scales; the reduction lengths meet the MX GEMMs' stage sizes.
int validate_mx_layer(const moe_layer* L) {
  if (L->act_fmt != L->w_fmt) return MOE_ERR_UNSUPPORTED;
  const int kq = L->w_fmt == MOE_FMT_MXFP4 ? 512 : 256;
  if (L->H % kq || L->I % kq || L->I_s % kq) return MOE_ERR_UNSUPPORTED;
  if (!L->w13 || !L->w2 || !L->w13_sf || !L->w2_sf) return MOE_ERR_INVALID_ARG;
  if (L->I_s && (!L->ws13 || !L->ws2 || !L->ws13_sf || !L->ws2_sf)) return MOE_ERR_INVALID_ARG;
  if (L->ws_gate && (!L->I_s || !aligned(L->ws_gate, 16))) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

int validate_layer(const moe_layer* L) {
  if (!L) return MOE_ERR_INVALID_ARG;
  if (L->H < 1 || L->E < 1 || L->k < 1 || L->I < 1 || L->I_s < 0) return MOE_ERR_INVALID_ARG;
  if (L->k > L->E || L->k > 32 || L->E > 1024) return MOE_ERR_UNSUPPORTED;
  if (L->H % 64 || L->I % 64 || L->I_s % 64) return MOE_ERR_UNSUPPORTED;
  if (is_mx(L->w_fmt) || is_mx(L->act_fmt)) return validate_mx_layer(L);
  const bool w4 = L->w_fmt == MOE_FMT_NVFP4, a4 = L->act_fmt == MOE_FMT_NVFP4;
  if (L->w_fmt != MOE_FMT_BF16 && !w4) return MOE_ERR_INVALID_ARG;
  if (L->act_fmt != MOE_FMT_BF16 && !a4) return MOE_ERR_INVALID_ARG;
  if (a4 && !w4) return MOE_ERR_UNSUPPORTED;
  if (!L->w13 || !L->w2) return MOE_ERR_INVALID_ARG;
  if (w4 && (!L->w13_sf || !L->w13_g || !L->w2_sf || !L->w2_g)) return MOE_ERR_INVALID_ARG;
  if (L->I_s) {
    if (!L->ws13 || !L->ws2) return MOE_ERR_INVALID_ARG;
    if (w4 && (!L->ws13_sf || !L->ws13_g || !L->ws2_sf || !L->ws2_g)) return MOE_ERR_INVALID_ARG;
  }
  if (a4 && (!L->g_h || (L->I_s && !L->g_hs))) return MOE_ERR_INVALID_ARG;
  if (L->ws_gate && (!L->I_s || !aligned(L->ws_gate, 16))) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// Lays the buffers out in the workspace (ws may be null to size it).
size_t carve(const moe_layer* L, int T, void* ws, size_t cap, FwdBufs* b) {
  const size_t Tk = static_cast<size_t>(T) * L->k;
  const bool a4 = L->act_fmt == MOE_FMT_NVFP4;
  Carve c(ws, cap);
  b->idx = c.take<int32_t>(Tk);
  b->w = c.take<float>(Tk);
  b->counts = c.take<int32_t>(L->E);
  b->offsets = c.take<int32_t>(L->E + 1);
  b->row_of = c.take<int32_t>(Tk);
  b->src_tok = c.take<int32_t>(Tk);
  b->perm_ws_bytes = route_permute_ws_bytes(T, L->E);
  b->perm_ws = c.take<uint8_t>(b->perm_ws_bytes);
  b->xq = b->xsf = nullptr;
  b->gx = nullptr;
  b->qws = nullptr;
  b->xp_sf = b->h_sf = b->hs_sf = nullptr;
  b->hs = nullptr;
  b->Ys = nullptr;
  if (is_mx(L->w_fmt)) {
    const int f = L->w_fmt;
    b->xq = c.take<uint8_t>(mx_code_bytes(f, static_cast<size_t>(T) * L->H));
    b->xsf = c.take<uint8_t>(static_cast<size_t>(T) * L->H / 32);
    b->xp = c.take<uint8_t>(mx_code_bytes(f, Tk * L->H));
    b->xp_sf = c.take<uint8_t>(Tk * L->H / 32);
    b->h = c.take<uint8_t>(mx_code_bytes(f, Tk * L->I));
    b->h_sf = c.take<uint8_t>(Tk * L->I / 32);
    if (L->I_s) {
      b->hs = c.take<uint8_t>(mx_code_bytes(f, static_cast<size_t>(T) * L->I_s));
      b->hs_sf = c.take<uint8_t>(static_cast<size_t>(T) * L->I_s / 32);
    }
  } else if (a4) {
    b->xq = c.take<uint8_t>(static_cast<size_t>(T) * L->H / 2);
    b->xsf = c.take<uint8_t>(static_cast<size_t>(T) * L->H / 16);
    b->gx = c.take<float>(1);
    b->qws = c.take<uint8_t>(quant_ws_bytes(1));
    b->xp = c.take<uint8_t>(Tk * L->H / 2);
    b->xp_sf = c.take<uint8_t>(Tk * L->H / 16);
    b->h = c.take<uint8_t>(Tk * L->I / 2);
    b->h_sf = c.take<uint8_t>(Tk * L->I / 16);
    if (L->I_s) {
      b->hs = c.take<uint8_t>(static_cast<size_t>(T) * L->I_s / 2);
      b->hs_sf = c.take<uint8_t>(static_cast<size_t>(T) * L->I_s / 16);
    }
  } else {
    b->xp = c.take<uint16_t>(Tk * L->H);
    b->h = c.take<uint16_t>(Tk * L->I);
    if (L->I_s) b->hs = c.take<uint16_t>(static_cast<size_t>(T) * L->I_s);
  }
  b->Y = c.take<uint16_t>(Tk * L->H);
  if (L->I_s) b->Ys = c.take<uint16_t>(static_cast<size_t>(T) * L->H);
  b->gate = (L->I_s && L->ws_gate) ? c.take<float>(T) : nullptr;
  return c.used;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_forward_workspace_size(const moe_layer* L, int T) {
  if (validate_layer(L) != MOE_OK || T < 0) return 0;
  if (static_cast<long long>(T) * L->k >= (1ll << 27)) return 0;  // moe_forward rejects it
  FwdBufs b;
  return carve(L, T, nullptr, 0, &b);
}

extern "C" int moe_quant_mx(const uint16_t* x, int rows, int cols, int fmt, uint8_t* codes, uint8_t* scales,
                            void* stream);

namespace {
inline int mark(void* const* events, int i, cudaStream_t s) {
  if (events == nullptr || events[i] == nullptr) return MOE_OK;
  cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s);
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
}  // namespace

extern "C" int moe_forward_profiled(const moe_layer* L, const uint16_t* x, const float* logits, int T, uint16_t* out,
                                    void* ws, size_t ws_bytes, void* const* events, void* stream);

extern "C" int moe_forward(const moe_layer* L, const uint16_t* x, const float* logits, int T, uint16_t* out, void* ws,
                           size_t ws_bytes, void* stream) {
  return moe_forward_profiled(L, x, logits, T, out, ws, ws_bytes, nullptr, stream);
}

extern "C" int moe_forward_profiled(const moe_layer* L, const uint16_t* x, const float* logits, int T, uint16_t* out,
                                    void* ws, size_t ws_bytes, void* const* events, void* stream) {
  MOE_TRY(validate_layer(L));
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !logits || !out || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(logits, 4) || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  // one warp per routed row in the permutation (32 * T*k threads in 32 bits)
  if (static_cast<long long>(T) * L->k >= (1ll << 27)) return MOE_ERR_UNSUPPORTED;
  FwdBufs b;
  if (carve(L, T, ws, ws_bytes, &b) > ws_bytes) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool a4 = L->act_fmt == MOE_FMT_NVFP4;
  const int H = L->H, E = L->E, k = L->k;
  const int Tk = T * k;

  const int renorm = L->no_renorm ? 0 : 1;
  MOE_TRY(mark(events, 0, s));
  if (b.gate) MOE_TRY(shared_gate_launch(x, L->ws_gate, T, H, b.gate, s));
  if (is_mx(L->w_fmt)) {
    // MX layers: x quantised in blocks of 32 along H; the gate/up GEMM's
    // epilogue quantises h the same way along I from its fp32 value
    const int f = L->w_fmt;
    const int I = L->I, I_s = L->I_s;
    MOE_TRY(moe_quant_mx(x, T, H, f, b.xq, b.xsf, stream));
    MOE_TRY(mark(events, 1, s));
    MOE_TRY(dispatch(logits, T, E, k, renorm, b, b.xq, static_cast<int>(mx_code_bytes(f, H)), b.xsf, H / 32, s));
    MOE_TRY(mark(events, 2, s));
    GemmProblem r1{b.xp, b.xp_sf, nullptr, Tk, L->w13, L->w13_sf, nullptr, E, b.h, b.h_sf, nullptr, I, H};
    GemmProblem s1{b.xq, b.xsf, nullptr, T, L->ws13, L->ws13_sf, nullptr, 1, b.hs, b.hs_sf, nullptr, I_s, H};
    MOE_TRY(grouped_gemm_launch(MOE_EPI_SWIGLU_MX, f, f, r1, b.offsets, E, I_s ? &s1 : nullptr, T, s));
    MOE_TRY(mark(events, 3, s));
    GemmProblem r2{b.h, b.h_sf, nullptr, Tk, L->w2, L->w2_sf, nullptr, E, b.Y, nullptr, nullptr, H, I};
    GemmProblem s2{b.hs, b.hs_sf, nullptr, T, L->ws2, L->ws2_sf, nullptr, 1, b.Ys, nullptr, nullptr, H, I_s};
    MOE_TRY(grouped_gemm_launch(MOE_EPI_STORE_BF16, f, f, r2, b.offsets, E, I_s ? &s2 : nullptr, T, s));
    MOE_TRY(mark(events, 4, s));
    MOE_TRY(combine_launch(b.Y, b.row_of, b.w, b.Ys, b.gate, T, k, H, out, s));
    return mark(events, 5, s);
  }
  if (a4) MOE_TRY(quant_launch(x, 1, T, H, nullptr, b.xq, b.xsf, b.gx, b.qws, quant_ws_bytes(1), s));
  MOE_TRY(mark(events, 1, s));
  // NVFP4 weights with bf16 activations: when the tensor-memory kernel takes
  // all four problems (every K a multiple of 256, 16-byte aligned weight
  // scales), x is permuted into fp16 once and h is kept in fp16, the inputs
  // of that kernel's fp16 MMA
  const bool w4 = L->w_fmt == MOE_FMT_NVFP4;
  const bool f16 = w4 && !a4 && H % 256 == 0 && L->I % 256 == 0 && aligned(L->w13_sf, 16) &&
                   aligned(L->w2_sf, 16) &&
                   (L->I_s == 0 || (L->I_s % 256 == 0 && aligned(L->ws13_sf, 16) && aligned(L->ws2_sf, 16)));
  if (a4)
    MOE_TRY(dispatch(logits, T, E, k, renorm, b, b.xq, H / 2, b.xsf, H / 16, s));
  else
    MOE_TRY(dispatch(logits, T, E, k, renorm, b, x, H * 2, nullptr, 0, s, f16));
  MOE_TRY(mark(events, 2, s));

  // gate/up projection + SwiGLU (routed groups + shared expert)
  const int epi1 = a4 ? MOE_EPI_SWIGLU_NVFP4 : (f16 ? kEpiSwigluF16 : MOE_EPI_SWIGLU_BF16);
  GemmProblem r1{b.xp, b.xp_sf, b.gx, Tk, L->w13, L->w13_sf, L->w13_g, E, b.h, b.h_sf, L->g_h, L->I, H, f16};
  GemmProblem s1{a4 ? static_cast<const void*>(b.xq) : static_cast<const void*>(x),
                 b.xsf, b.gx, T, L->ws13, L->ws13_sf, L->ws13_g, 1, b.hs, b.hs_sf, L->g_hs, L->I_s, H};
  MOE_TRY(grouped_gemm_launch(epi1, L->act_fmt, L->w_fmt, r1, b.offsets, E, L->I_s ? &s1 : nullptr, T, s));

  MOE_TRY(mark(events, 3, s));

  // down projection
  GemmProblem r2{b.h, b.h_sf, L->g_h, Tk, L->w2, L->w2_sf, L->w2_g, E, b.Y, nullptr, nullptr, H, L->I, f16};
  GemmProblem s2{b.hs, b.hs_sf, L->g_hs, T, L->ws2, L->ws2_sf, L->ws2_g, 1, b.Ys, nullptr, nullptr, H, L->I_s, f16};
  MOE_TRY(grouped_gemm_launch(MOE_EPI_STORE_BF16, L->act_fmt, L->w_fmt, r2, b.offsets, E, L->I_s ? &s2 : nullptr, T,
                              s));

  MOE_TRY(mark(events, 4, s));
  MOE_TRY(combine_launch(b.Y, b.row_of, b.w, b.Ys, b.gate, T, k, H, out, s));
  return mark(events, 5, s);
}

extern "C" int moe_forward_host(const moe_layer* L, const uint16_t* x_host, const float* logits_host, int T,
                                uint16_t* out_host, uint16_t* x_dev, float* logits_dev, uint16_t* out_dev, void* ws,
                                size_t ws_bytes, void* stream) {
  MOE_TRY(validate_layer(L));
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x_host || !logits_host || !out_host || !x_dev || !logits_dev || !out_dev) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t xb = static_cast<size_t>(T) * L->H * sizeof(uint16_t);
  const size_t lb = static_cast<size_t>(T) * L->E * sizeof(float);
  cudaError_t e = cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(logits_dev, logits_host, lb, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  MOE_TRY(moe_forward(L, x_dev, logits_dev, T, out_dev, ws, ws_bytes, stream));
  e = cudaMemcpyAsync(out_host, out_dev, xb, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return moe_sync_status(stream);
}

// Batches alternate between the two halves of the device buffers.  On the
// copy stream, batch i+1's inputs are enqueued after batch i-1's output copy,
// which waits for batch i-1's compute: the inputs never overwrite a half
// still being read.  Batch i's compute waits for its inputs and, from i = 2
// on, for the copy-out of batch i-2 from the same output half.
extern "C" int moe_forward_host_pipelined(const moe_layer* L, int n, const uint16_t* const* x_host,
                                          const float* const* logits_host, int T, uint16_t* const* out_host,
                                          uint16_t* x_dev, float* logits_dev, uint16_t* out_dev, void* ws,
                                          size_t ws_bytes, void* stream, void* copy_stream) {
  MOE_TRY(validate_layer(L));
  if (n < 1 || T < 0) return MOE_ERR_INVALID_ARG;
  if (!x_host || !logits_host || !out_host || !x_dev || !logits_dev || !out_dev) return MOE_ERR_INVALID_ARG;
  if (!copy_stream || stream == copy_stream) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i)
    if (!x_host[i] || !logits_host[i] || !out_host[i]) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  cudaStream_t cs = static_cast<cudaStream_t>(stream), ps = static_cast<cudaStream_t>(copy_stream);
  const size_t xe = static_cast<size_t>(T) * L->H, le = static_cast<size_t>(T) * L->E;
  const size_t xb = xe * sizeof(uint16_t), lb = le * sizeof(float);
  cudaEvent_t ev[6] = {};  // [0,1] inputs landed, [2,3] compute done, [4,5] output copied, per half
  int made = 0;
  cudaError_t e = cudaSuccess;
  for (; made < 6 && e == cudaSuccess; ++made) e = cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming);
  if (e != cudaSuccess) {
    --made;  // the failed creation made nothing
    for (int i = 0; i < made; ++i) cudaEventDestroy(ev[i]);
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  auto h2d = [&](int i) {
    const int b = i & 1;
    cudaError_t r = cudaMemcpyAsync(x_dev + b * xe, x_host[i], xb, cudaMemcpyHostToDevice, ps);
    if (r == cudaSuccess) r = cudaMemcpyAsync(logits_dev + b * le, logits_host[i], lb, cudaMemcpyHostToDevice, ps);
    if (r == cudaSuccess) r = cudaEventRecord(ev[b], ps);
    return r;
  };
  int st = MOE_OK;
  e = h2d(0);
  for (int i = 0; i < n && e == cudaSuccess && st == MOE_OK; ++i) {
    const int b = i & 1;
    e = cudaStreamWaitEvent(cs, ev[b], 0);
    if (e == cudaSuccess && i >= 2) e = cudaStreamWaitEvent(cs, ev[4 + b], 0);
    if (e != cudaSuccess) break;
    st = moe_forward(L, x_dev + b * xe, logits_dev + b * le, T, out_dev + b * xe, ws, ws_bytes, stream);
    if (st != MOE_OK) break;
    e = cudaEventRecord(ev[2 + b], cs);
    if (e == cudaSuccess && i + 1 < n) e = h2d(i + 1);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ps, ev[2 + b], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(out_host[i], out_dev + b * xe, xb, cudaMemcpyDeviceToHost, ps);
    if (e == cudaSuccess) e = cudaEventRecord(ev[4 + b], ps);
  }
  // whatever was enqueued finishes before the events go and the call returns
  cudaError_t e2 = cudaStreamSynchronize(cs);
  cudaError_t e3 = cudaStreamSynchronize(ps);
  for (int i = 0; i < 6; ++i) cudaEventDestroy(ev[i]);
  if (e == cudaSuccess) e = e2 != cudaSuccess ? e2 : e3;
  if (st != MOE_OK) return st;
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return moe_sync_status(stream);
}

extern "C" int moe_forward_graph_create(const moe_layer* L, const uint16_t* x, const float* logits, int T,
                                        uint16_t* out, void* ws, size_t ws_bytes, void* stream, void** graph) {
  if (!graph) return MOE_ERR_INVALID_ARG;
  *graph = nullptr;
  if (T < 1) return MOE_ERR_INVALID_ARG;
  // one ordinary run: argument checks, first-launch attribute setup
  MOE_TRY(moe_forward(L, x, logits, T, out, ws, ws_bytes, stream));
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  cudaStream_t cs = nullptr;
  e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  cudaGraph_t g = nullptr;
  cudaGraphExec_t exec = nullptr;
  int st = MOE_OK;
  e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  if (e == cudaSuccess) {
    st = moe_forward(L, x, logits, T, out, ws, ws_bytes, cs);
    e = cudaStreamEndCapture(cs, &g);  // ends the capture whatever moe_forward returned
    if (st == MOE_OK && e == cudaSuccess) e = cudaGraphInstantiate(&exec, g, 0);
  }
  if (g) cudaGraphDestroy(g);
  cudaStreamDestroy(cs);
  if (st != MOE_OK) return st;
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  *graph = exec;
  return MOE_OK;
}

extern "C" int moe_graph_launch(void* graph, void* stream) {
  if (!graph) return MOE_ERR_INVALID_ARG;
  cudaError_t e = cudaGraphLaunch(static_cast<cudaGraphExec_t>(graph), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

extern "C" int moe_graph_destroy(void* graph) {
  if (!graph) return MOE_OK;
  cudaError_t e = cudaGraphExecDestroy(static_cast<cudaGraphExec_t>(graph));
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
