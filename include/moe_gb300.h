/*
 * moe_gb300.h -- C ABI of the GB300 (sm_103a) MoE-layer forward library.
 *
 * The library computes the forward pass of a Qwen3-MoE-style mixture-of-experts
 * layer on one GPU, as the page "基于Atlas A3、950训练/推理集群的Qwen3-MoE模型低时延
 * 推理性能优化实践" decomposes it into fused operators:
 *   router logits -> gating top-k softmax (§快速选择专家) -> init_routing and
 *   compute_expert_tokens (§高效排序和token路由) -> grouped matmul over the merged
 *   gate/up weight w13 with SwiGLU (§计算分解, §高性能专家计算) -> grouped matmul
 *   over down_proj -> finalize_routing (§高效排序和token路由).
 * Each expert is the MLP  y = down( SiLU(x . gate) * (x . up) ), w13 = [gate | up].
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - Pointers are DEVICE pointers of the current CUDA device unless stated, owned
 *    by the caller; the library never allocates or frees device memory.  Buffers
 *    named "ws" are caller-provided scratch of at least the queried size, 256-byte
 *    aligned; their contents on entry do not matter.
 *  - All calls are asynchronous on `stream` (0 = legacy default stream) and return
 *    after validating arguments and enqueueing work.  The return value reports
 *    host-side validation and launch errors only.
 *  - Problems found by kernels (an expert id outside [0,E), a wait that ran out of
 *    time) are OR-ed into a per-device status word, read with
 *    moe_get_device_status (synchronises the stream) and cleared with
 *    moe_clear_device_status.  Kernels never trap.
 *  - bf16 tensors are passed as raw 16-bit patterns (moe_bf16), row-major.
 *    Matrix pointers must be 16-byte aligned.
 *  - Shapes: 1 <= T; H % 128 == 0; I % 64 == 0; 1 <= E <= 256; 1 <= k <= min(E, 32);
 *    T*k < 2^31.  Other shapes return MOE_ERR_UNSUPPORTED_SHAPE.
 *  - The library runs only on compute capability 10.3 (GB300, sm_103a) and on
 *    device indices 0..63; other devices return MOE_ERR_UNSUPPORTED_ARCH.
 *  - Per-device facts (SM count, the status word's address, kernel attributes)
 *    are looked up on the first call on each device and kept.  They belong to the
 *    device's primary context: the library assumes that context is not destroyed
 *    (cudaDeviceReset) while it stays loaded.
 *  - Token-expert pairs are numbered token-major: pair j = t*k + s is slot s of
 *    token t.  P = T*k.
 */
#ifndef MOE_GB300_H_
#define MOE_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef struct CUstream_st* moe_stream_t; /* identical to cudaStream_t */
typedef uint16_t moe_bf16;                /* bfloat16 bit pattern */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,       /* null / misaligned pointer, negative size */
  MOE_ERR_UNSUPPORTED_SHAPE = 2, /* shape outside the supported set above */
  MOE_ERR_UNSUPPORTED_ARCH = 3,  /* current device is not sm_103, or its index is >= 64 */
  MOE_ERR_WORKSPACE = 4,         /* ws too small or misaligned */
  MOE_ERR_CUDA = 5               /* a CUDA runtime call or launch failed */
} moe_status;

/* Bits of the device status word. */
#define MOE_DEV_BAD_EXPERT_ID 0x1 /* a topk id outside [0,E): that pair was skipped */
#define MOE_DEV_WAIT_TIMEOUT 0x2  /* a bounded device wait expired; outputs invalid */

/* Version of this ABI (bumped on any signature change). */
MOE_API int moe_abi_version(void);

/* Human-readable text for a moe_status value (static storage). */
MOE_API const char* moe_status_string(int status);

/* Reads (after synchronising `stream`) the current device's status word. */
MOE_API moe_status moe_get_device_status(int32_t* status_out /* host */, moe_stream_t stream);
/* Clears the current device's status word (asynchronously on `stream`). */
MOE_API moe_status moe_clear_device_status(moe_stream_t stream);

/* ---------------------------------------------------------------- router --
 * Router scores logits[t,e] = sum_h x[t,h] * Wg[h,e], fp32 FMA accumulation.
 * The page's §融合RMSNorm Cast keeps the gate (router) computation in FP32.
 *   x       (T,H)  bf16
 *   Wg      (H,E)  fp32
 *   logits  (T,E)  fp32, written
 *   ws      >= moe_router_logits_workspace_size(T,H,E) bytes (may be 0 -> NULL ok)
 * Deterministic: the split-K partial sums are added in a fixed order.
 */
MOE_API size_t moe_router_logits_workspace_size(int T, int H, int E);
MOE_API moe_status moe_router_logits(const moe_bf16* x, const float* Wg, int T, int H, int E,
                             float* logits, void* ws, size_t ws_bytes, moe_stream_t stream);

/* ----------------------------------------------------------------- gating --
 * §快速选择专家: one fused op for "softmax over experts, top-k".  Per token:
 * experts are ranked by (fp32 logit descending, expert id ascending); the first k
 * are kept, slot s holding the s-th ranked.  With renormalize != 0 the weights are
 * softmax over the k kept logits (= full softmax, top-k, renormalised to sum 1);
 * with renormalize == 0 they are the full-softmax probabilities of the kept ones.
 *   logits   (T,E) fp32 (finite values)
 *   topk_ids (T,k) int32, written
 *   topk_w   (T,k) fp32, written
 */
MOE_API moe_status moe_gating_topk_softmax(const float* logits, int T, int E, int k, int renormalize,
                                   int32_t* topk_ids, float* topk_w, moe_stream_t stream);

/* ---------------------------------------------------------------- routing --
 * §高效排序和token路由 (init_routing): stable counting sort of the P pairs by
 * expert id.  Pair j goes to row p(j) = expert_offsets[id_j] + #{j' < j with the
 * same id}.
 *   x                (T,H) bf16; may be NULL when expanded_x is NULL
 *   topk_ids         (T,k) int32 ids in [0,E); an id outside sets
 *                    MOE_DEV_BAD_EXPERT_ID and that pair is dropped
 *                    (expanded_row_idx = -1, not counted)
 *   expanded_x       (P,H) bf16 or NULL: row p = x[sorted_row_idx[p] / k]
 *   expanded_row_idx (P)   int32 pair -> row  (j -> p(j))
 *   sorted_row_idx   (P)   int32 row  -> pair (inverse permutation)
 *   expert_offsets   (E+1) int32 exclusive prefix sum of the counts
 *   counts           (E)   int32 or NULL: pairs per expert
 *   ws               >= moe_init_routing_workspace_size(T,E,k) bytes
 */
MOE_API size_t moe_init_routing_workspace_size(int T, int E, int k);
MOE_API moe_status moe_init_routing(const moe_bf16* x, const int32_t* topk_ids, int T, int H, int E, int k,
                            moe_bf16* expanded_x, int32_t* expanded_row_idx,
                            int32_t* sorted_row_idx, int32_t* expert_offsets, int32_t* counts,
                            void* ws, size_t ws_bytes, moe_stream_t stream);

/* §高效排序和token路由 (compute_expert_tokens): tokens each expert must compute.
 *   topk_ids (P) int32;  counts (E) int32 written;  expert_offsets (E+1) or NULL. */
MOE_API moe_status moe_compute_expert_tokens(const int32_t* topk_ids, int P, int E, int32_t* counts,
                                     int32_t* expert_offsets, moe_stream_t stream);

/* ----------------------------------------------------- weight packing ----
 * Load-time, untimed.  Rewrites the logical weights into the K-major tiles the
 * grouped GEMMs stream with TMA.
 *   w13  (E,H,2I) bf16: columns [0,I) gate_proj, [I,2I) up_proj (§计算分解: the
 *        SwiGLU op chunks the merged product in two and gates the first half)
 *   down (E,I,H)  bf16
 *   w13_packed  >= moe_packed_weight_bytes(E,H,I,0) bytes: per expert 2I rows of H
 *        (row block b of 128 rows covers features 64b..64b+63; in each 32-row
 *        quarter q, rows 0-15 are gate columns 64b+16q.. and rows 16-31 the matching
 *        up columns)
 *   down_packed >= moe_packed_weight_bytes(E,H,I,1) bytes: per expert H rows of I
 * Either input may be NULL to skip it.
 */
MOE_API size_t moe_packed_weight_bytes(int E, int H, int I, int which /* 0: w13, 1: down */);
MOE_API moe_status moe_pack_weights(const moe_bf16* w13, const moe_bf16* down, int E, int H, int I,
                            void* w13_packed, void* down_packed, moe_stream_t stream);

/* --------------------------------------------------------- grouped GEMMs --
 * §高性能专家计算 (grouped_matmul) fused with §计算分解's SwiGLU: for each expert e,
 * the rows r in [expert_offsets[e], expert_offsets[e+1]) of A:
 *   h[r, c] = SiLU(g) * u,  g = sum_k A[r,k] w13[e][k][c],  u = sum_k A[r,k] w13[e][k][I+c]
 * fp32 accumulation in tensor memory, h rounded once to bf16.
 *   A  (P,K) bf16 expert-sorted rows (K = H);  w13_packed from moe_pack_weights;
 *   expert_offsets (E+1) int32 (device), offsets[E] <= P;  h (P,N) bf16 (N = I).
 *   ws >= moe_grouped_matmul_workspace_size() bytes (NULL when 0).
 * Rows of A or h past expert_offsets[E] are not read / written.
 */
MOE_API size_t moe_grouped_matmul_workspace_size(void);
MOE_API moe_status moe_grouped_matmul_swiglu(const moe_bf16* A, const void* w13_packed,
                                     const int32_t* expert_offsets, int E, int P, int K, int N,
                                     moe_bf16* h, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Plain grouped GEMM (the down projection): y[r, n] = sum_k A[r,k] down[e][k][n]
 * for r in expert e's rows; fp32 accumulation, y rounded once to bf16.
 *   A (P,K) bf16 (K = I); w_packed = down_packed; y (P,N) bf16 (N = H). */
MOE_API moe_status moe_grouped_matmul(const moe_bf16* A, const void* w_packed,
                              const int32_t* expert_offsets, int E, int P, int K, int N,
                              moe_bf16* y, void* ws, size_t ws_bytes, moe_stream_t stream);

/* -------------------------------------------------------------- finalize --
 * §高效排序和token路由 (finalize_routing): put expert outputs back in token order
 * and add them with the router weights:
 *   out[t,:] = sum_{s<k} topk_w[t,s] * y2[expanded_row_idx[t*k+s], :]
 * summed in fp32 in slot order (deterministic), rounded once to bf16.  Pairs with
 * expanded_row_idx < 0 are skipped.
 *   y2 (P,H) bf16; topk_w (T,k) fp32; expanded_row_idx (P) int32; out (T,H) bf16.
 */
MOE_API moe_status moe_finalize_routing(const moe_bf16* y2, const float* topk_w,
                                const int32_t* expanded_row_idx, int T, int k, int H,
                                moe_bf16* out, moe_stream_t stream);

/* --------------------------------------------------------- whole layer ----
 * The full layer in one call: router -> gating (renormalised) -> init_routing ->
 * grouped GEMM + SwiGLU -> grouped GEMM -> finalize.  Both GEMMs run in one
 * persistent launch; a down-projection tile starts once every gate/up tile of its
 * expert has been written.  At decode sizes (T <= 64, router run) the router
 * launch also asks L2 to prefetch the front of w13_packed (at most 5/8 of L2) while
 * routing runs; this changes no result.
 *   x (T,H) bf16; Wg (H,E) fp32
 *   logits_override (T,E) fp32 or NULL: when given, replaces the router output
 *   w13_packed, down_packed from moe_pack_weights
 *   out (T,H) bf16
 *   topk_ids_out (T,k) int32 or NULL; topk_w_out (T,k) fp32 or NULL
 *   ws >= moe_forward_workspace_size(T,H,E,k,I) bytes
 */
MOE_API size_t moe_forward_workspace_size(int T, int H, int E, int k, int I);
MOE_API moe_status moe_forward(const moe_bf16* x, const float* Wg, const float* logits_override,
                       const void* w13_packed, const void* down_packed, int T, int H, int E, int k,
                       int I, moe_bf16* out, int32_t* topk_ids_out, float* topk_w_out, void* ws,
                       size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------ MXFP8 --
 * §融合RMSNorm MX量化: residual add, RMSNorm and MXFP8 dynamic quantisation in one
 * pass.  MX format (OCP Microscaling v1.0; the page names only "MXFP8", round mode
 * "rint" and float8_e4m3fn): blocks of 32 consecutive elements share an E8M0 scale
 * 2^X with X = floor(log2(max|v|)) - 8 clamped to [-127,127] (all-zero block:
 * X = -127); elements are e4m3(v / 2^X), nearest-even, saturating at +-448.
 * Scale byte = X + 127.
 *
 * moe_add_rmsnorm_mxquant:  s = x + r (fp32);  residual_out = bf16(s);
 *   y = s * rsqrt(mean(s^2) + eps) * w (fp32);  y32_out = y;  q, scale = MX(y) along H.
 *   x, r (T,H) bf16 (r may be NULL: no residual, the page's first-layer variant);
 *   w (H) bf16; residual_out (T,H) bf16 or NULL; y32_out (T,H) fp32 or NULL;
 *   q (T,H) e4m3 bytes; scale (T,H/32) bytes.  H % 256 == 0.
 */
MOE_API moe_status moe_add_rmsnorm_mxquant(const moe_bf16* x, const moe_bf16* r, const moe_bf16* w,
                                           float eps, int T, int H, moe_bf16* residual_out,
                                           float* y32_out, uint8_t* q, uint8_t* scale,
                                           moe_stream_t stream);

/* Dynamic MX quantisation of an fp32 (rows, n) matrix along its rows (the page's
 * npu_dynamic_mx_quant, §计算分解 AllGather方案).  n % 32 == 0; q (rows,n) bytes;
 * scale (rows, n/32) bytes.  y 16-byte aligned. */
MOE_API moe_status moe_mx_quantize(const float* y, int rows, int n, uint8_t* q, uint8_t* scale,
                                   moe_stream_t stream);

/* MX pre-quantisation of the expert weights along their reduction axis (H for w13,
 * I for down), load-time.  Codes are K-major in the same row order as
 * moe_pack_weights; scales are stored as 512-byte atoms per (expert, 128-row
 * block, 128-element K step): byte (r%32)*16 + (r/32)*4 + b holds the scale of row r,
 * K block b.  Requires H % 128 == 0 and I % 128 == 0.
 *   which: 0 w13 codes (E*2I*H bytes), 1 w13 scales (E*2I*H/32), 2 down codes
 *   (E*H*I), 3 down scales (E*H*I/32). */
MOE_API size_t moe_packed_weight_bytes_mx(int E, int H, int I, int which);
MOE_API moe_status moe_pack_weights_mx(const moe_bf16* w13, const moe_bf16* down, int E, int H,
                                       int I, void* w13_q, void* w13_sf, void* down_q,
                                       void* down_sf, moe_stream_t stream);

/* The MXFP8 layer in one call: add+RMSNorm+MX quant -> router on the fp32 normalised
 * activations (§融合RMSNorm Cast) -> gating -> init_routing -> block-scaled grouped
 * GEMM over w13 + SwiGLU, h MX-quantised along I -> block-scaled grouped GEMM over
 * down -> finalize.  Arguments as moe_forward plus r, norm_w, eps and residual_out
 * (T,H bf16 or NULL), with the packed MX weights.  H % 256 == 0, I % 128 == 0.
 * As in moe_forward, decode sizes also ask L2 to prefetch the front of the w13 codes.
 *   ws >= moe_forward_mx_workspace_size(T,H,E,k,I) bytes. */
MOE_API size_t moe_forward_mx_workspace_size(int T, int H, int E, int k, int I);
MOE_API moe_status moe_forward_mx(const moe_bf16* x, const moe_bf16* r, const moe_bf16* norm_w,
                                  float eps, const float* Wg, const float* logits_override,
                                  const void* w13_q, const void* w13_sf, const void* down_q,
                                  const void* down_sf, int T, int H, int E, int k, int I,
                                  moe_bf16* out, moe_bf16* residual_out, int32_t* topk_ids_out,
                                  float* topk_w_out, void* ws, size_t ws_bytes,
                                  moe_stream_t stream);

/* Standalone block-scaled grouped GEMMs (§高性能专家计算 grouped_matmul on MXFP8
 * operands; SwiGLU from §计算分解; h MX-quantised as in moe_forward_mx).
 *   A_q (P,K) e4m3 codes of expert-sorted rows (expert e owns rows
 *   [expert_offsets[e], expert_offsets[e+1])), A_scale (P,K/32) E8M0 bytes, row-major
 *   (the layout moe_mx_quantize and moe_add_rmsnorm_mxquant produce);
 *   weights from moe_pack_weights_mx (weight_format 0, e4m3) or moe_pack_weights_mx4
 *   (weight_format 1, e2m1; code buffer 32-byte aligned); expert_offsets (E+1) int32
 *   on the device, offsets[E] <= P.
 * moe_grouped_matmul_swiglu_mx: g = A.w13[e][:, :N], u = A.w13[e][:, N:] (fp32
 *   accumulation), h = SiLU(g) * u, MX-quantised along N: h_q (P,N) e4m3 and
 *   h_scale (P,N/32) E8M0, row-major.  N = I.
 * moe_grouped_matmul_mx: y = A.w[e] (fp32 accumulation) rounded once to bf16, y (P,N).
 * Rows at or past expert_offsets[E] are neither read nor written.  K % 128 == 0,
 * N % 128 == 0, E <= 256.  ws >= moe_grouped_matmul_mx_workspace_size(E,P,K,N,swiglu)
 * bytes, 256-byte aligned (the rows are re-laid out there with each expert padded for
 * the block-scaled tensor-core tiles). */
MOE_API size_t moe_grouped_matmul_mx_workspace_size(int E, int P, int K, int N, int swiglu);
MOE_API moe_status moe_grouped_matmul_swiglu_mx(const uint8_t* A_q, const uint8_t* A_scale,
                                                const void* w13_q, const void* w13_sf,
                                                int weight_format, const int32_t* expert_offsets,
                                                int E, int P, int K, int N, uint8_t* h_q,
                                                uint8_t* h_scale, void* ws, size_t ws_bytes,
                                                moe_stream_t stream);
MOE_API moe_status moe_grouped_matmul_mx(const uint8_t* A_q, const uint8_t* A_scale,
                                         const void* w_q, const void* w_sf, int weight_format,
                                         const int32_t* expert_offsets, int E, int P, int K, int N,
                                         moe_bf16* y, void* ws, size_t ws_bytes,
                                         moe_stream_t stream);

/* ------------------------------------------------------------------ W4A8 --
 * The MXFP8 layer with MXFP4 expert weights (W4A8: 4-bit weights, 8-bit
 * activations).  Page "基于Atlas A3、950训练/推理集群的Qwen3-MoE模型低时延推理性能优化实践",
 * §概述 (W4A8 mixed-precision prefill) and §计算分解 AllGather方案 (W4A8 = MXFP4
 * weights, activations through npu_dynamic_mx_quant); the page fixes no rounding or
 * scale rule, so this library takes OCP MXFP4 v1.0: blocks of 32 consecutive weights along the reduction axis
 * share an E8M0 scale 2^X, X = floor(log2(max|v|)) - 2 (2 = the exponent of e2m1's
 * largest value 6) clamped to [-127,127], all-zero block X = -127; codes are
 * e2m1(v / 2^X), nearest-even, saturating at +-6.  Activations and h stay MXFP8 as
 * in moe_forward_mx.
 *
 * moe_pack_weights_mx4: as moe_pack_weights_mx, but codes are packed two per byte
 * (element 2j of a row in the low nibble of byte j) and stored tile-major: the
 * codes of row r, K-elements [128 s, 128 s + 128) of expert e are the 64 bytes at
 * ((e * rows / 128 + r / 128) * K / 128 + s) * 8192 + (r % 128) * 64, rows = 2I for
 * w13 (K = H) and H for down (K = I).  Scale atoms are as moe_pack_weights_mx.
 *   which: 0 w13 codes (E*2I*H/2 bytes), 1 w13 scales (E*2I*H/32), 2 down codes
 *   (E*H*I/2), 3 down scales (E*H*I/32).  H % 128 == 0, I % 128 == 0.
 * moe_forward_w4a8: arguments as moe_forward_mx with the packed MXFP4 weights; code
 *   buffers 32-byte aligned (MOE_ERR_INVALID_ARG otherwise).  Workspace size as
 *   moe_forward_mx. */
MOE_API size_t moe_packed_weight_bytes_mx4(int E, int H, int I, int which);
MOE_API moe_status moe_pack_weights_mx4(const moe_bf16* w13, const moe_bf16* down, int E, int H,
                                        int I, void* w13_q, void* w13_sf, void* down_q,
                                        void* down_sf, moe_stream_t stream);
MOE_API size_t moe_forward_w4a8_workspace_size(int T, int H, int E, int k, int I);
MOE_API moe_status moe_forward_w4a8(const moe_bf16* x, const moe_bf16* r, const moe_bf16* norm_w,
                                    float eps, const float* Wg, const float* logits_override,
                                    const void* w13_q, const void* w13_sf, const void* down_q,
                                    const void* down_sf, int T, int H, int E, int k, int I,
                                    moe_bf16* out, moe_bf16* residual_out, int32_t* topk_ids_out,
                                    float* topk_w_out, void* ws, size_t ws_bytes,
                                    moe_stream_t stream);

/* ------------------------------------------------------------- next rows --
 * §融合RMSNorm Cast: residual add + RMSNorm with two outputs, FP32 for the gate
 * (router) and BF16 for the experts.  s = x + r; residual_out = bf16(s);
 * y = s * rsqrt(mean(s^2) + eps) * w; y32_out = y (fp32, may be NULL);
 * ybf16_out = bf16(y).  x, r (T,H) bf16 (r may be NULL); w (H) bf16.  H % 256 == 0.
 */
MOE_API moe_status moe_add_rmsnorm_cast(const moe_bf16* x, const moe_bf16* r, const moe_bf16* w,
                                        float eps, int T, int H, moe_bf16* residual_out,
                                        float* y32_out, moe_bf16* ybf16_out, moe_stream_t stream);

/* Expert-range routing (the page's init_routing_v2 of §计算分解 AllGather方案, which
 * keeps only this rank's experts): pairs whose id lies in [expert_begin, expert_end)
 * are sorted stably by local id (id - expert_begin), exactly as moe_init_routing;
 * pairs with another valid id in [0, E_total) (another rank's expert, or a
 * zero-computation expert) get expanded_row_idx = -1 without an error; ids outside
 * [0, E_total) also get -1 and set MOE_DEV_BAD_EXPERT_ID.  Arrays are sized for the
 * local experts: counts (E_local), expert_offsets (E_local+1); sorted_row_idx has
 * expert_offsets[E_local] valid entries.  E_local = expert_end - expert_begin <= 256. */
MOE_API size_t moe_init_routing_v2_workspace_size(int T, int E_local, int k);
MOE_API moe_status moe_init_routing_v2(const moe_bf16* x, const int32_t* topk_ids, int T, int H,
                                       int k, int E_total, int expert_begin, int expert_end,
                                       moe_bf16* expanded_x, int32_t* expanded_row_idx,
                                       int32_t* sorted_row_idx, int32_t* expert_offsets,
                                       int32_t* counts, void* ws, size_t ws_bytes,
                                       moe_stream_t stream);

/* Re-routing after an expert-parallel AlltoAll (§计算分解 Double Routing方案,
 * npu_moe_re_routing): the N received rows arrive grouped by source rank r and,
 * within a rank, by local expert e (tokens_per_expert[r][e] rows each, int32 (R,
 * E_local), device).  They are reordered expert-major, then by rank (stable).
 * x_out[perm[i]] = x_recv[i]; expert_offsets (E_local+1) of the output.  x_recv and
 * x_out may be NULL (only perm and offsets).  H % 8 == 0. */
MOE_API size_t moe_re_routing_workspace_size(int R, int E_local);
MOE_API moe_status moe_re_routing(const moe_bf16* x_recv, const int32_t* tokens_per_expert, int R,
                                  int E_local, int N, int H, moe_bf16* x_out, int32_t* perm,
                                  int32_t* expert_offsets, void* ws, size_t ws_bytes,
                                  moe_stream_t stream);

/* finalize_routing with zero-computation experts (page "基于Atlas A3集群的LongCat-
 * Flash模型推理性能优化实践", §MoE模块实现Expert Parallel: copy_expert_num,
 * MoE(ori_x) = ori_x): pair j adds w * y2[expanded_row_idx[j]] when that row is
 * >= 0, else w * x_in[t] when topk_ids[j] lies in [E, E_total) (a zero-computation
 * expert returns its input), else nothing.  topk_ids (T,k) and x_in (T,H) bf16. */
MOE_API moe_status moe_finalize_routing_v2(const moe_bf16* y2, const float* topk_w,
                                           const int32_t* expanded_row_idx,
                                           const int32_t* topk_ids, const moe_bf16* x_in, int T,
                                           int k, int H, int E, int E_total, moe_bf16* out,
                                           moe_stream_t stream);

/* The bf16 layer with the optional fused add+RMSNorm+cast in front and optional
 * zero-computation experts.  norm_w NULL: no norm (x feeds router and experts, r
 * and residual_out unused).  norm_w given: s = x + r, y = RMSNorm(s); the router
 * runs on fp32 y and the experts on bf16(y); residual_out = bf16(s) (may be NULL).
 * Wg (H, E+Z) fp32 scores E routed experts then Z zero-computation experts; top-k
 * is taken over all E+Z; zero-computation experts add w * (their input).
 * logits_override (T, E+Z) or NULL.  E + Z <= 256. */
MOE_API size_t moe_forward_v2_workspace_size(int T, int H, int E, int Z, int k, int I);
MOE_API moe_status moe_forward_v2(const moe_bf16* x, const moe_bf16* r, const moe_bf16* norm_w,
                                  float eps, const float* Wg, const float* logits_override,
                                  const void* w13_packed, const void* down_packed, int T, int H,
                                  int E, int Z, int k, int I, moe_bf16* out,
                                  moe_bf16* residual_out, int32_t* topk_ids_out,
                                  float* topk_w_out, void* ws, size_t ws_bytes,
                                  moe_stream_t stream);

/* ------------------------------------------------ allocation-free routing --
 * No counterpart in the pages: an extra entry point for callers that cannot
 * allocate device memory -- code living inside a host framework that owns all
 * device memory and offers no allocator to it, or a serving loop that must not
 * allocate once it is running.  It does what moe_init_routing does, with the
 * same arguments minus the workspace; its scratch (about 33 KB) is a fixed array
 * in the library's own device memory, present on every GPU that loads the
 * library until the process exits.
 *  - T*k must be <= MOE_NOALLOC_MAX_PAIRS, else MOE_ERR_UNSUPPORTED_SHAPE.
 *  - It calls no allocator.  Its first call on a device (with that device
 *    current) looks up the scratch address; make that first call before any
 *    stream capture on that device.
 *  - All calls on a device share the scratch: calls that may overlap on the GPU
 *    (unordered streams) race and must be serialised by the caller.
 */
#define MOE_NOALLOC_MAX_PAIRS 65536
MOE_API moe_status moe_init_routing_noalloc(const moe_bf16* x, const int32_t* topk_ids, int T, int H,
                                            int E, int k, moe_bf16* expanded_x,
                                            int32_t* expanded_row_idx, int32_t* sorted_row_idx,
                                            int32_t* expert_offsets, int32_t* counts,
                                            moe_stream_t stream);

/* -------------------------------------------------------------- profiling --
 * Measurement aid, not part of the page's operator set: when set (non-NULL), every
 * later moe_forward call made by this host thread records `ev_begin` on its stream
 * just before the grouped-GEMM launch and `ev_end` just after it, so a caller can
 * time that kernel alone with cudaEventElapsedTime.  Both are cudaEvent_t handles
 * owned by the caller; pass NULL, NULL to stop.
 */
MOE_API moe_status moe_set_gemm_events(void* ev_begin, void* ev_end);

/* ------------------------------------------------------------- test hook --
 * Test aid, not part of the page's operator set: makes the bounded device waits of
 * the one-CTA grouped GEMM (the decode-size tiles) run out on purpose, so that the
 * timeout path can be checked without a fault.  With stage >= 0, every later launch
 * of that kernel (from any host thread) bounds each of its waits by `wait_ns`
 * (1 us .. 2 s, else MOE_ERR_INVALID_ARG), and in every CTA the TMA producer stops
 * before its stage-th pipeline stage: it issues no copy for that stage or any later
 * one.  The MMA thread's wait for that stage then runs out, the CTA's roles unwind
 * (MMAs and copies already issued complete first, TMEM is freed), the launch
 * returns, and MOE_DEV_WAIT_TIMEOUT is set in the status word; the layer's outputs
 * of that call are invalid.  stage < 0 switches the hook off and restores the
 * library-wide limit (2 s).  The CTA-pair and block-scaled GEMMs ignore it.
 */
MOE_API moe_status moe_debug_set_gemm_stall(int stage, long long wait_ns);

/* Test aid: the CTA-pair grouped GEMM (prefill-size bf16 tiles) runs the experts
 * with at most 32 rows on a second, light pipeline when, by its per-stage cost
 * estimates, their weight streaming hides under the other experts' tensor work;
 * else every expert runs on the one pipeline.  The choice is made on the device from
 * the expert counts.  mode 0 restores that choice (the default), 1 uses the light
 * pipeline whenever such experts exist, 2 never uses it.  It affects every later
 * pair launch from any host thread; results agree in every mode.  Other modes:
 * MOE_ERR_INVALID_ARG.
 */
MOE_API moe_status moe_debug_set_pair_light(int mode);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H_ */
