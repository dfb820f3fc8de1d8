// Internal launchers shared between the translation units of the library.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kPermChunk = 1024;        // routed slots per chunk of the permutation
constexpr int kPermMaxExperts = 4096;   // largest E the permutation takes (E int32 of shared memory)
size_t permute_ws_bytes(int T, int k, int E);
// to_f16: the rows are bf16 and are written to xp_rows as fp16 (saturating).
int permute_launch(const int32_t* idx, int T, int k, int E, const void* x_rows, int row_bytes, const uint8_t* x_sf,
                   int sf_row_bytes, int32_t* counts, int32_t* offsets, int32_t* row_of, int32_t* src_tok,
                   void* xp_rows, uint8_t* xp_sf, void* ws, size_t ws_bytes, cudaStream_t s, bool to_f16 = false);

// Fused router + permutation in one cooperative launch (dispatch.cu); the
// same results as moe_route_ex followed by permute_launch.  E <= 1024.
size_t route_permute_ws_bytes(int T, int E);
int route_permute_launch(const float* logits, int T, int E, int k, int renorm, int32_t* idx, float* w,
                         const void* x_rows, int row_bytes, const uint8_t* x_sf, int sf_row_bytes, int32_t* counts,
                         int32_t* offsets, int32_t* row_of, int32_t* src_tok, void* xp_rows, uint8_t* xp_sf,
                         void* ws, size_t ws_bytes, cudaStream_t s, bool to_f16 = false);

size_t quant_ws_bytes(int groups);
int quant_launch(const uint16_t* x, int groups, int rows, int cols, const float* g_in, uint8_t* codes, uint8_t* sf,
                 float* g_out, void* ws, size_t ws_bytes, cudaStream_t s);

int combine_launch(const uint16_t* Y, const int32_t* row_of, const float* w, const uint16_t* Ys, const float* ys_gate,
                   int T, int k, int H, uint16_t* out, cudaStream_t s);
int shared_gate_launch(const uint16_t* x, const uint16_t* g, int T, int H, float* gate, cudaStream_t s);

// One problem set of the grouped GEMM: all routed groups (rows given by
// device offsets), or the shared expert as a single group over all tokens.
struct GemmProblem {
  const void* A;       // bf16 [a_rows, K] or packed E2M1 [a_rows, K/2]
  const uint8_t* A_sf; // [a_rows, K/16] E4M3 (NVFP4 A)
  const float* A_g;    // device scalar (NVFP4 A)
  int a_rows;
  const void* W;       // bf16 [groups * Wn, K] or packed E2M1 [groups * Wn, K/2]
  const uint8_t* W_sf; // [groups * Wn, K/16] (NVFP4 W)
  const float* W_g;    // [groups] (NVFP4 W)
  int groups;
  void* C;             // bf16 [a_rows, N] or packed E2M1 [a_rows, N/2]
  uint8_t* C_sf;       // [a_rows, N/16] (NVFP4 C)
  const float* c_g;    // device scalar (NVFP4 C)
  int N, K;
  bool a_f16 = false;  // bf16-activation problems: A already holds fp16 (layer-internal)
};

// Layer-internal epilogue of the NVFP4-weight / bf16-activation path: SwiGLU
// with h stored as fp16 for the down projection's fp16 MMA.
constexpr int kEpiSwigluF16 = 16;

int grouped_gemm_launch(int epi, int a_fmt, int w_fmt, const GemmProblem& routed, const int32_t* offsets, int G,
                        const GemmProblem* sh, int shared_rows, cudaStream_t s);

// Both operands bf16: MMA over CTA pairs (gemm_pair.cu).
int grouped_gemm_launch_pair(int epi, const GemmProblem& routed, const int32_t* offsets, int G,
                             const GemmProblem* sh, int shared_rows, cudaStream_t s);

// Both operands NVFP4: block-scaled FP4 tensor-core kernels; dispatches to
// the 512-element-stage kernel (gemm_fp4w.cu) when K % 256 == 0 and the
// scale arrays are 16-byte aligned, else to gemm_fp4.cu's kernel.
int grouped_gemm_launch_nvf4(int epi, const GemmProblem& routed, const int32_t* offsets, int G,
                             const GemmProblem* sh, int shared_rows, cudaStream_t s);
// bf16 activations x NVFP4 weights, K % 256 == 0: weights expanded into
// tensor memory, fp16 MMA (gemm_w4a16.cu).
int grouped_gemm_launch_w4a16(int epi, const GemmProblem& routed, const int32_t* offsets, int G,
                              const GemmProblem* sh, int shared_rows, cudaStream_t s);
int grouped_gemm_launch_nvf4_wide(int epi, const GemmProblem& routed, const int32_t* offsets, int G,
                                  const GemmProblem* sh, int shared_rows, cudaStream_t s);
// NVFP4 x NVFP4 down projection (bf16 output) on CTA pairs (weights on the
// MMA's M side, tokens on N), K % 512 == 0 and 16-byte aligned scale arrays
// (gemm_nvf4p.cu).
int grouped_gemm_launch_nvf4_pair(const GemmProblem& routed, const int32_t* offsets, int G, const GemmProblem* sh,
                                  int shared_rows, cudaStream_t s);
// Both operands MXFP4 (E2M1 codes, E8M0 scales per 32), K % 512 == 0, bf16
// epilogues (gemm_mxf4.cu).
int grouped_gemm_launch_mxf4(int epi, const GemmProblem& routed, const int32_t* offsets, int G,
                             const GemmProblem* sh, int shared_rows, cudaStream_t s);
// Both operands MXFP8 (E4M3 bytes, E8M0 scales per 32), K % 256 == 0, bf16
// and MX SwiGLU epilogues, on CTA pairs: weights on the MMA's M side and
// tokens on N (gemm_mxf8p.cu).
int grouped_gemm_launch_mxf8_pair(int epi, const GemmProblem& routed, const int32_t* offsets, int G,
                                  const GemmProblem* sh, int shared_rows, cudaStream_t s);

}  // namespace moe
