/*
 * moe_gb300.h -- C ABI of the GB300 (sm_103a) top-k routed MoE FFN layer
 * forward.
 *
 * The layer computes, for every token t,
 *
 *     out_t = sum_{j<k} w[t,j] * E_{idx[t,j]}(x_t) + S(x_t)
 *
 * where E_e is a SwiGLU expert (gate/up projection, silu(gate) * up, down
 * projection) and S an always-on shared expert ("Hosting Qwen on Blackwell",
 * sections "MoE Dispatch - Combine" and "MoE GEMM"; "Como Servimos um Modelo
 * MoE de 397B com 4.7x de Speedup em TPU v7", MoE FFN description; "CuTeDSL
 * at Perplexity", local dispatch / combine kernels).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every call returns an int status (MOE_OK or one of MOE_ERR_*).
 *  - All tensors are caller-owned DEVICE pointers unless a parameter says
 *    "host".  The compute calls never allocate or free memory: scratch space
 *    is a caller-supplied workspace whose size the matching
 *    *_workspace_size() call returns.  Workspaces must be 256-byte aligned.
 *    The exceptions are named where they are declared: the CUDA-graph calls
 *    (moe_forward_graph_create creates a stream and an executable graph,
 *    moe_graph_destroy frees the graph), the fixed device array of
 *    moe_permute_noalloc, and the CUDA events that
 *    moe_forward_host_pipelined creates and destroys within the call.
 *  - Every call is asynchronous on the caller's CUDA stream (`stream` is a
 *    cudaStream_t passed as void*; NULL is the legacy default stream).  The
 *    library does no host synchronisation except in moe_sync_status(),
 *    moe_forward_host() and moe_forward_host_pipelined().
 *  - Layouts are row-major with the innermost dimension contiguous.  bf16
 *    tensors are passed as uint16_t bit patterns.
 *  - NVFP4 tensors are three arrays: packed E2M1 codes (uint8, element 2j in
 *    the low nibble, 2j+1 in the high nibble), one E4M3 scale byte per 16
 *    consecutive elements along the reduction dimension (row-major
 *    [rows, cols/16]), and an fp32 global scale.  Decoded value =
 *    e2m1(q) * e4m3(s) * g ("Driving vLLM WideEP and Large-Scale Serving
 *    Toward Maturity on Blackwell (Part I)", sections "NVFP4 GEMM for MoE and
 *    O-proj" and "NVFP4 MoE dispatch").
 *  - MX tensors (MOE_FMT_MXFP8 / MOE_FMT_MXFP4) are codes (E4M3 bytes, or
 *    E2M1 packed as for NVFP4) and one E8M0 scale byte per 32 consecutive
 *    elements along the reduction dimension ([rows, cols/32]); no global
 *    scale.  Decoded value = element(q) * 2^(s - 127) (moe_quant_mx).
 *  - Argument errors are detected on the host before anything is launched:
 *    MOE_ERR_INVALID_ARG (null or misaligned pointer, negative size),
 *    MOE_ERR_UNSUPPORTED (shape outside what the kernels handle, see each
 *    call), MOE_ERR_WORKSPACE (workspace too small).  Launch failures return
 *    MOE_ERR_CUDA; moe_last_cuda_error() gives the CUDA message.
 *  - The only device-side waits are mbarrier waits inside one thread block.
 *    Each is bounded in time (moe_set_wait_timeout_ns, default 1 s); a wait
 *    that runs out records MOE_ERR_TIMEOUT in a device error word and the
 *    kernel returns.  moe_sync_status() reports (and clears) it.
 *  - What only the device reads is checked there, so that no input sends a
 *    kernel outside its buffers: expert ids outside [0, E) (left out of the
 *    permutation, reported as MOE_ERR_INVALID_ARG by moe_sync_status()),
 *    combine rows outside [0, T*k) (skipped), group offsets (clamped).
 *  - The first call on each device that launches a permutation or a grouped
 *    GEMM looks up the device error word (cudaGetSymbolAddress) and sets
 *    kernel attributes; make such a call once before capturing any of them
 *    into a CUDA graph yourself (moe_forward_graph_create does it for you).
 *  - Inputs are assumed finite; NaN / Inf inputs give unspecified results.
 *  - T = 0 (no tokens) is a valid no-op returning MOE_OK.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ status */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG 1
#define MOE_ERR_UNSUPPORTED 2
#define MOE_ERR_WORKSPACE 3
#define MOE_ERR_CUDA 4
#define MOE_ERR_TIMEOUT 5

/* ------------------------------------------------------------ data formats */
#define MOE_FMT_BF16 0
#define MOE_FMT_NVFP4 1
#define MOE_FMT_MXFP8 2   /* E4M3 elements, one E8M0 scale per 32 (moe_quant_mx) */
#define MOE_FMT_MXFP4 3   /* E2M1 elements, one E8M0 scale per 32 (moe_quant_mx) */

/* -------------------------------------------------- grouped GEMM epilogues */
#define MOE_EPI_STORE_BF16 0   /* C = A * W^T, rounded to bf16                        */
#define MOE_EPI_SWIGLU_BF16 1  /* W has 2N rows per group: gate [0,N), up [N,2N);
                                  C = silu(A W_gate^T) * (A W_up^T), rounded to bf16   */
#define MOE_EPI_SWIGLU_NVFP4 2 /* as SWIGLU_BF16, but the fp32 result is quantised to
                                  NVFP4 with a caller-given global scale              */
#define MOE_EPI_SWIGLU_MX 3    /* as SWIGLU_BF16, but the fp32 result is quantised to
                                  the operands' MX format (moe_quant_mx's recipe,
                                  blocks of 32 along N)                               */

/* Library version: major * 10000 + minor * 100 + patch. */
int moe_version(void);

/* Static string for a status code. */
const char* moe_status_string(int status);

/* Message of the last CUDA error seen by this library in this process
 * (thread-unsafe, diagnostic only). */
const char* moe_last_cuda_error(void);

/* Time limit of every device-side wait, in nanoseconds (default 1e9).
 * ns == 0 restores the default. */
int moe_set_wait_timeout_ns(unsigned long long ns);

/* Synchronises `stream`, then returns MOE_ERR_TIMEOUT if any kernel of this
 * library recorded a wait time-out since the last call, else
 * MOE_ERR_INVALID_ARG if a permutation met an expert id outside [0, E)
 * (clearing the record either way), MOE_ERR_CUDA on a CUDA error, else
 * MOE_OK. */
int moe_sync_status(void* stream);

/* Test hook for the time-out path: launches one block whose thread waits on
 * an mbarrier that nothing ever arrives on, with the library's bounded wait.
 * The wait gives up after `timeout_ns`, records MOE_ERR_TIMEOUT in the device
 * error word and the kernel returns; the context stays usable.  Read the
 * result with moe_sync_status(). */
int moe_selftest_wait_timeout(unsigned long long timeout_ns, void* stream);

/* ------------------------------------------------------------------- route
 * Router softmax and top-k with renormalised weights.
 * Pages: the routing table holds expert indices and weights of shape [T, k]
 * ("Como Servimos um Modelo MoE de 397B ...", section "Tres coletivas viram
 * duas"); the softmax / top-k / renormalisation is the layer's stated router.
 *
 *   logits : fp32 [T, E]   router logits (x W_r + bias, computed upstream)
 *   idx    : int32 [T, k]  chosen experts, by descending logit; equal logits
 *                          are ordered by ascending expert id
 *   w      : fp32 [T, k]   w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the
 *                          k chosen logits (= softmax over E renormalised)
 * One warp per token.  Supports 1 <= k <= min(E, 32), 1 <= E <= 1024,
 * T < 2^27. */
int moe_route(const float* logits, int T, int E, int k,
              int32_t* idx, float* w, void* stream);

/* moe_route with a choice of weights.  renorm != 0: as moe_route.  renorm ==
 * 0: the router without renormalisation (the pages allude to router
 * variants without fixing one; reading taken): the same experts and order,
 * w_j = exp(l_j - l_0) / sum_{e<E} exp(l_e - l_0), the full softmax over E
 * at the picks (so sum_j w_j <= 1).  Same arguments and limits. */
int moe_route_ex(const float* logits, int T, int E, int k, int renorm,
                 int32_t* idx, float* w, void* stream);

/* ----------------------------------------------------------------- permute
 * Local dispatch: count tokens per expert, give each routed slot a unique
 * position inside its expert's list, copy the token rows into an
 * expert-contiguous buffer ("CuTeDSL at Perplexity", local MoE dispatch /
 * combine kernel: counting, unique index per token, copy into the buffers
 * that feed the MoE GEMM; prefill routing split over blocks with per-block
 * counters accumulated in global memory).
 * The order is deterministic and stable: inside expert e's segment, rows are
 * in ascending token id.  Segments are unpadded.
 * Ids in idx are read on the device, so they are checked there: a slot whose
 * id lies outside [0, E) is left out (not counted, row_of = -1, offsets[E]
 * short by one per such slot, permuted rows past offsets[E] unspecified) and
 * the next moe_sync_status() returns MOE_ERR_INVALID_ARG.
 *
 *   idx      : int32 [T, k]   expert of each slot (0 <= idx < E, distinct per token)
 *   x_rows   : [T, row_bytes] token rows (bf16 row: 2H bytes; NVFP4 row: H/2
 *              bytes); may be NULL when xp_rows is NULL
 *   x_sf     : [T, sf_row_bytes] per-row scale bytes copied alongside (NVFP4
 *              rows: H/16 bytes), or NULL
 *   counts   : int32 [E]      slots routed to each expert
 *   offsets  : int32 [E+1]    exclusive prefix sum of counts; offsets[E] = T*k
 *   row_of   : int32 [T, k]   row of slot (t, j) in the permuted buffer
 *   src_tok  : int32 [T*k]    token of each permuted row
 *   xp_rows  : [T*k, row_bytes] permuted rows (NULL: metadata only)
 *   xp_sf    : [T*k, sf_row_bytes] permuted scale rows (NULL if x_sf is NULL)
 * row_bytes must be a positive multiple of 16; sf_row_bytes a positive
 * multiple of 4 (when x_sf is given); pointers 16-byte aligned.
 * E <= 4096, T*k < 2^27.  Workspace: moe_permute_workspace_size(T, k, E). */
size_t moe_permute_workspace_size(int T, int k, int E);
int moe_permute(const int32_t* idx, int T, int k, int E,
                const void* x_rows, int row_bytes,
                const uint8_t* x_sf, int sf_row_bytes,
                int32_t* counts, int32_t* offsets, int32_t* row_of, int32_t* src_tok,
                void* xp_rows, uint8_t* xp_sf,
                void* ws, size_t ws_bytes, void* stream);

/* moe_permute without a caller workspace.  The pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory at
 * dispatch time -- runtimes that hand out a fixed set of buffers at start-up
 * and forbid allocation on the per-step path (cudaMalloc may synchronise the
 * device and has unbounded latency), embedders whose own allocator owns all
 * device memory, plugins that only receive their inputs and outputs.
 * Same arguments, results and checks as moe_permute, minus ws / ws_bytes.
 * Its scratch is a 1 MiB array defined by the library in device memory
 * (held on every device that loads the library until the process exits),
 * which limits the size to ceil(T*k / 1024) * E <= 131072 (e.g. T*k <= 131072
 * with E <= 1024); larger problems return MOE_ERR_UNSUPPORTED before any
 * launch.  The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * All calls share the array: calls that overlap on the GPU race on it, calls
 * ordered on one stream do not.  No allocation of any kind is made. */
int moe_permute_noalloc(const int32_t* idx, int T, int k, int E,
                        const void* x_rows, int row_bytes,
                        const uint8_t* x_sf, int sf_row_bytes,
                        int32_t* counts, int32_t* offsets, int32_t* row_of, int32_t* src_tok,
                        void* xp_rows, uint8_t* xp_sf, void* stream);

/* ----------------------------------------------------------- route_permute
 * Fused dispatch: moe_route_ex followed by moe_permute in one cooperative
 * launch of min(T, SMs, 256) blocks of 1024 threads, joined by two grid
 * barriers
 * ("CuTeDSL at Perplexity", local dispatch, decode variant: routing inside
 * the dispatch kernel, which signals the rest of the grid and hands out
 * slots from shared-memory counters; grid-sync section: a grid barrier costs
 * about 3 us against a second launch; "Como Servimos um Modelo MoE de
 * 397B ...", section "Roadmap restante": fuse the top-k selection).
 * Results (idx, w, counts, offsets, row_of, src_tok, permuted rows and
 * scales) are those of the two calls, bit for bit; arguments as there.
 * Each grid-barrier wait is bounded in time (moe_set_wait_timeout_ns); a
 * wait that runs out records MOE_ERR_TIMEOUT (moe_sync_status) and the
 * kernel returns with the outputs unspecified.  The workspace holds the
 * per-block histograms and the barrier counter, which a memset on `stream`
 * zeroes before the launch.
 * Limits: 1 <= k <= min(E, 32), E <= 1024, T*k < 2^27.  Workspace:
 * moe_route_permute_workspace_size(T, k, E). */
size_t moe_route_permute_workspace_size(int T, int k, int E);
int moe_route_permute(const float* logits, int T, int E, int k, int renorm,
                      int32_t* idx, float* w,
                      const void* x_rows, int row_bytes,
                      const uint8_t* x_sf, int sf_row_bytes,
                      int32_t* counts, int32_t* offsets, int32_t* row_of, int32_t* src_tok,
                      void* xp_rows, uint8_t* xp_sf,
                      void* ws, size_t ws_bytes, void* stream);

/* Test hook for the grid barrier's time-out: a cooperative launch of two
 * blocks waits for a third arrival that never comes; each wait gives up
 * after `timeout_ns`, records MOE_ERR_TIMEOUT in the device error word and
 * the kernel returns; the context stays usable.  Read the result with
 * moe_sync_status(). */
int moe_selftest_grid_barrier_timeout(unsigned long long timeout_ns, void* stream);

/* ------------------------------------------------------------ quant_nvfp4
 * NVFP4 quantisation of bf16 matrices (activations before dispatch:
 * "Driving vLLM WideEP ... (Part I)", section "NVFP4 MoE dispatch"; abs-max
 * over 16 elements: "CuTeDSL at Perplexity", Blackwell support).
 * Recipe, in IEEE fp32 with round-to-nearest-even:
 *   g   = amax(|x|) / 2688 per group (1 if the group is all zero), unless g_in
 *   s_b = E4M3_satfinite(amax_b / (6 g))           per 16 elements of a row
 *   q_i = E2M1_satfinite(x_i / (e4m3(s_b) g))      magnitude 0 if e4m3(s_b) == 0
 * Ties round to the even code; the code's sign bit is the sign of x_i.
 *
 *   x      : bf16 [groups, rows, cols]
 *   g_in   : fp32 [groups] device, or NULL to derive g from each group's amax
 *   codes  : uint8 [groups, rows, cols/2]
 *   sf     : uint8 [groups, rows, cols/16] (E4M3)
 *   g_out  : fp32 [groups] device (required; receives g)
 * cols must be a multiple of 16.  Workspace:
 * moe_quant_nvfp4_workspace_size(groups). */
size_t moe_quant_nvfp4_workspace_size(int groups);
int moe_quant_nvfp4(const uint16_t* x, int groups, int rows, int cols,
                    const float* g_in, uint8_t* codes, uint8_t* sf, float* g_out,
                    void* ws, size_t ws_bytes, void* stream);

/* --------------------------------------------------------------- quant_mx
 * Microscaling quantisation of bf16 rows (the pages name MXFP8, served for
 * Qwen3-235B, and MXFP4 with abs-max over 32 elements: "Hosting Qwen on
 * Blackwell", section "Quantização"; "CuTeDSL at Perplexity", Blackwell
 * support).  Reading (Open Compute Project microscaling definition), per 32
 * consecutive elements of a row:
 *   e   = floor(log2 amax) - emax   (emax 8 for MXFP8's E4M3, 2 for MXFP4's
 *         E2M1), clamped to [-127, 127]; -127 for an all-zero block
 *   q_i = element_RNE_satfinite(x_i / 2^e), sign kept
 *   scale byte = e + 127 (E8M0)
 *   x      : bf16 [rows, cols], 16-byte aligned
 *   fmt    : MOE_FMT_MXFP8 or MOE_FMT_MXFP4
 *   codes  : MXFP8 uint8 [rows, cols] (8-byte aligned); MXFP4 packed uint8
 *            [rows, cols/2] (element 2j in the low nibble; 4-byte aligned)
 *   scales : uint8 [rows, cols/32]
 * cols must be a multiple of 32.  No workspace, no tensor-wide scale.
 * x must be finite: a block holding Inf or NaN gets an unspecified scale
 * and codes. */
int moe_quant_mx(const uint16_t* x, int rows, int cols, int fmt, uint8_t* codes, uint8_t* scales,
                 void* stream);

/* ------------------------------------------------------------ grouped GEMM
 * Expert GEMMs over expert-contiguous rows ("Hosting Qwen on Blackwell",
 * section "MoE GEMM"; NVFP4 weights dequantised inside the MMA path:
 * "Driving vLLM WideEP ... (Part I)", section "NVFP4 GEMM for MoE and
 * O-proj").  For every group g and every row r in [offsets[g], offsets[g+1]):
 *   STORE_BF16  : C[r, :N]  = bf16( a_g w_g[g] * sum_k A[r,k] W[g,n,k] )
 *   SWIGLU_*    : G = A W[g, 0:N]^T, U = A W[g, N:2N]^T (scaled likewise),
 *                 C[r, :N] = silu(G) * U  (bf16, or NVFP4 with global scale *c_g)
 * Operand formats: A bf16 [M_total, K] or NVFP4 (A = codes [M_total, K/2],
 * A_sf [M_total, K/16], *A_g); W bf16 [G, Wn, K] or NVFP4 (W_sf
 * [G, Wn, K/16], W_g [G]); Wn = N (STORE) or 2N (SWIGLU).  Scale pointers
 * (A_g, W_g, c_g) are device pointers; pass NULL for bf16 operands.
 * SWIGLU_NVFP4 writes C = codes [M_total, N/2] and C_sf [M_total, N/16].
 * MX formats (a_fmt = w_fmt), scales E8M0
 * [.., K/32] (moe_quant_mx), no global scales (A_g, W_g, c_g ignored),
 * STORE_BF16, SWIGLU_BF16 and SWIGLU_MX (the MX-only epilogue: C = codes
 * [M_total, N] (MXFP8) or [M_total, N/2] (MXFP4), C_sf = E8M0 [M_total,
 * N/32]):
 *   MOE_FMT_MXFP4: codes as NVFP4; K % 512 == 0, 16-byte aligned scales
 *   MOE_FMT_MXFP8: E4M3 bytes [.., K]; K % 256 == 0, 8-byte aligned scales
 * The kernel is persistent (one CTA per SM), reads offsets on the device,
 * stages tiles with TMA into shared memory, and runs tcgen05 MMAs with
 * fp32 accumulators in tensor memory.
 * Requirements: K % 64 == 0, N % 32 == 0, G <= 1024, M_total < 2^31,
 * offsets non-decreasing with offsets[G] <= M_total; A and W 16-byte aligned.
 * Offsets are read on the device: each is clamped to [0, M_total] and a
 * group whose end lies before its start is empty, so offsets that break the
 * contract give unspecified values but no access outside A, W or C.
 */
int moe_grouped_gemm(int a_fmt, int w_fmt, int epilogue,
                     int G, const int32_t* offsets, int M_total, int N, int K,
                     const void* A, const uint8_t* A_sf, const float* A_g,
                     const void* W, const uint8_t* W_sf, const float* W_g,
                     void* C, uint8_t* C_sf, const float* c_g,
                     void* stream);

/* ----------------------------------------------------------------- combine
 * Weighted unpermute ("CuTeDSL at Perplexity", combine kernel: vectorised
 * accumulation in registers using the token positions from dispatch):
 *   out[t, :] = bf16( sum_{j<k} w[t,j] * Y[row_of[t,j], :]  (+ Ys[t, :]) )
 * accumulated in fp32 in the order j = 0..k-1, then the shared expert row.
 * An entry of row_of outside [0, T*k) (the -1 of a left-out slot) adds
 * nothing.
 *   Y  : bf16 [T*k, H]   expert outputs in permuted order
 *   Ys : bf16 [T, H]     shared expert output, or NULL
 *   out: bf16 [T, H]
 * H must be a multiple of 8; pointers 16-byte aligned. */
int moe_combine(const uint16_t* Y, const int32_t* row_of, const float* w,
                const uint16_t* Ys, int T, int k, int H,
                uint16_t* out, void* stream);

/* moe_combine with a gated shared expert: the shared row enters as
 * ys_gate[t] * Ys[t, :] (fp32 multiply-add in the same accumulation order).
 *   ys_gate : fp32 [T] per-token gate (from moe_shared_gate), or NULL for
 *             weight 1; requires Ys when given; 4-byte aligned. */
int moe_combine_gated(const uint16_t* Y, const int32_t* row_of, const float* w,
                      const uint16_t* Ys, const float* ys_gate, int T, int k, int H,
                      uint16_t* out, void* stream);

/* Gate of the shared expert ("Hosting Qwen on Blackwell" names new gate
 * terms without fixing them; reading taken: a sigmoid of the token's dot
 * product with one gate vector):
 *   gate[t] = 1 / (1 + exp(-(x_t . g)))   dot in fp32, one warp per token
 *   x    : bf16 [T, H] activations (before any quantisation)
 *   g    : bf16 [H]    gate vector
 *   gate : fp32 [T]
 * H must be a multiple of 8, T < 2^27; x and g 16-byte aligned. */
int moe_shared_gate(const uint16_t* x, const uint16_t* g, int T, int H,
                    float* gate, void* stream);

/* ----------------------------------------------------------- whole layer
 * Weight description of one layer.  All pointers are device pointers.
 *   bf16 weights : w13 [E, 2I, H] (rows [0,I) gate, [I,2I) up), w2 [E, H, I],
 *                  ws13 [2I_s, H], ws2 [H, I_s]; *_sf and *_g NULL
 *   NVFP4 weights: w13 codes [E, 2I, H/2], w13_sf [E, 2I, H/16], w13_g [E];
 *                  w2 codes [E, H, I/2], w2_sf [E, H, I/16], w2_g [E];
 *                  shared likewise with one global scale each
 *   act_fmt NVFP4 (requires w_fmt NVFP4): x is quantised to NVFP4 (one global
 *                  scale over x) before dispatch, and the SwiGLU output h is
 *                  quantised to NVFP4 with the caller's global scales
 *                  *g_h (routed) and *g_hs (shared) before the down GEMM.
 *   NVFP4 weights with bf16 activations: when H, I and I_s are multiples
 *                  of 256 and the weight scales 16-byte aligned, the layer
 *                  runs its fp16 tensor-core path: x is converted to fp16
 *                  while it is permuted and h is kept in fp16.  bf16 -> fp16
 *                  is exact for 2^-14 <= |x| <= 65504; larger magnitudes
 *                  saturate to +-65504 and magnitudes below 2^-14 keep fewer
 *                  significant bits (fp16 subnormals), so activations or h
 *                  outside that range give results that differ from a bf16
 *                  computation.  Other shapes compute in bf16.
 *   MX layers (w_fmt = act_fmt = MOE_FMT_MXFP4 or MOE_FMT_MXFP8): codes
 *                  as moe_quant_mx writes them
 *                  (w13 [E, 2I, H or H/2], w2 [E, H, I or I/2]), scales E8M0
 *                  [.., K/32], no global scales (*_g, g_h, g_hs ignored); x
 *                  and h are quantised the same way inside the layer, h from
 *                  its fp32 value in the gate/up GEMM's epilogue.  H, I, I_s multiples of 512 (MXFP4) or 256
 *                  (MXFP8).
 * I_s = 0 means no shared expert.
 * Variants (zero-initialised fields keep the default layer):
 *   no_renorm != 0 : route without renormalisation (moe_route_ex, renorm 0)
 *   ws_gate        : bf16 [H] gate vector of the shared expert (requires
 *                    I_s > 0; 16-byte aligned): the shared output is scaled
 *                    by sigma(x_t . ws_gate) (moe_shared_gate); NULL: weight 1 */
typedef struct {
  int H, E, k, I, I_s;
  int w_fmt, act_fmt;
  const void* w13; const uint8_t* w13_sf; const float* w13_g;
  const void* w2;  const uint8_t* w2_sf;  const float* w2_g;
  const void* ws13; const uint8_t* ws13_sf; const float* ws13_g;
  const void* ws2;  const uint8_t* ws2_sf;  const float* ws2_g;
  const float* g_h;
  const float* g_hs;
  int no_renorm;
  const uint16_t* ws_gate;
} moe_layer;

/* Workspace bytes moe_forward needs for T tokens (0 on an invalid layer or
 * a T that moe_forward rejects). */
size_t moe_forward_workspace_size(const moe_layer* L, int T);

/* The whole layer: (NVFP4 / MX activation quantisation) -> router top-k and
 * permutation in one launch (as moe_route_permute) -> grouped GEMM gate/up +
 * SwiGLU -> grouped GEMM down -> combine, with the shared expert folded into
 * both grouped GEMM launches.
 *   x      : bf16 [T, H]
 *   logits : fp32 [T, E]
 *   out    : bf16 [T, H]
 * Constraints: those of each stage (H % 64 == 0, I % 64 == 0, I_s % 64 == 0,
 * k <= 32, E <= 1024, T*k < 2^27). */
int moe_forward(const moe_layer* L, const uint16_t* x, const float* logits, int T,
                uint16_t* out, void* ws, size_t ws_bytes, void* stream);

/* moe_forward that also records caller-created CUDA events (cudaEvent_t
 * passed as void*) on `stream` at the stage boundaries, for live per-stage
 * timing: events[0] before the first launch, [1] after the activation
 * quantisation and the shared-expert gate (nothing is launched there on
 * plain bf16 layers), [2] after the router top-k and the permutation (one
 * fused launch, as moe_route_permute), [3] after the gate/up grouped GEMM, [4]
 * after the down grouped GEMM, [5] after the combine.  `events` may be NULL,
 * and any entry may be NULL to skip it.  Launches exactly the kernels of
 * moe_forward. */
int moe_forward_profiled(const moe_layer* L, const uint16_t* x, const float* logits, int T,
                         uint16_t* out, void* ws, size_t ws_bytes, void* const* events,
                         void* stream);

/* moe_forward with HOST inputs and output: copies x_host (bf16 [T,H]) and
 * logits_host (fp32 [T,E]) into the caller's device buffers x_dev and
 * logits_dev, runs the layer, copies the result into out_host (bf16 [T,H])
 * through out_dev, and synchronises `stream`.  Host buffers should be pinned
 * for asynchronous copies. */
int moe_forward_host(const moe_layer* L, const uint16_t* x_host, const float* logits_host,
                     int T, uint16_t* out_host,
                     uint16_t* x_dev, float* logits_dev, uint16_t* out_dev,
                     void* ws, size_t ws_bytes, void* stream);

/* moe_forward_host over n consecutive batches of T tokens, with the copies
 * of one batch overlapping the compute of its neighbours (a serving loop:
 * batch i+1's inputs go to the device and batch i-1's output comes back
 * while batch i runs).  x_host[i], logits_host[i], out_host[i] (arrays of n
 * host pointers, bf16 [T,H], fp32 [T,E], bf16 [T,H]) are batch i's buffers,
 * pinned for asynchronous copies.  x_dev, logits_dev, out_dev are device
 * buffers of TWO batches each (bf16 [2,T,H], fp32 [2,T,E], bf16 [2,T,H]),
 * used alternately; ws is one moe_forward workspace for T tokens.  The layer
 * runs on `stream`, the copies on `copy_stream` (a different, non-NULL
 * stream; the copies overlap the compute only when neither stream
 * synchronises with the other, e.g. two streams created non-blocking).  Every out_host[i] holds batch i's result, identical to
 * moe_forward_host's, when the call returns: both streams are synchronised.
 * The call creates its CUDA events and destroys them before it returns.
 * Errors: MOE_ERR_INVALID_ARG for n < 1, a NULL pointer, a NULL
 * copy_stream, or copy_stream == stream; the moe_forward checks for the
 * rest. */
int moe_forward_host_pipelined(const moe_layer* L, int n, const uint16_t* const* x_host,
                               const float* const* logits_host, int T, uint16_t* const* out_host,
                               uint16_t* x_dev, float* logits_dev, uint16_t* out_dev,
                               void* ws, size_t ws_bytes, void* stream, void* copy_stream);

/* moe_forward as a CUDA graph, for launch-bound sizes (decode, small
 * layers): the layer's kernels are captured once on fixed buffers and
 * replayed with one launch.  moe_forward_graph_create runs moe_forward once
 * on `stream` (which sets up the kernels' launch attributes and writes
 * `out`), then captures it on a stream of its own and returns the
 * instantiated graph in *graph.  moe_graph_launch replays it on `stream`:
 * the same layer, T, and buffers (x, logits, out, ws), whose contents may
 * change between replays.  moe_graph_destroy frees it.  The moe_layer
 * struct is read only while the graph is created; the weights, scales and
 * buffers it and the call point to must outlive the graph.  The wait limit
 * (moe_set_wait_timeout_ns) in force at creation is the one the replays
 * use. */
int moe_forward_graph_create(const moe_layer* L, const uint16_t* x, const float* logits, int T,
                             uint16_t* out, void* ws, size_t ws_bytes, void* stream,
                             void** graph);
int moe_graph_launch(void* graph, void* stream);
int moe_graph_destroy(void* graph);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
