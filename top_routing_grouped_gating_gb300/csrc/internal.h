// Internal launchers shared between the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// ---- router / gating (router_gating.cu)
struct RouterPlan {
  bool small;      // decode-size tiles (32 tokens x 32 experts x 128 rows of H)
  bool tc = false; // tensor-core path (bf16x3 split, router_tc.cu)
  int splits;      // split-K factor (partials part[splits][T][E] when > 1)
  int t_tiles;     // ceil(T / 32)
  int e_tiles;     // expert tiles
  int nseg = 0;    // tc: K segments (3: bf16 activations, 6: fp32 activations)
  size_t extra_bytes = 0;  // tc: packed weights, offsets, split activations
};
RouterPlan router_plan(int T, int H, int E);  // CUDA-core plans only
// The plan moe_forward uses: the tensor-core path for prefill-size T.
RouterPlan router_plan_ex(int T, int H, int E, bool f32in);
// Workspace of a router launch under router_plan_ex: partials + extra.
size_t router_ws_bytes(int T, int H, int E, bool f32in);
// Tensor-core router: x is (T,H) bf16, or fp32 when f32in.  Writes partial
// sums part[plan.splits][T][E]; extra holds plan.extra_bytes of scratch.  With
// f32in and presplit, x is unused: the launch before wrote the exact three-piece
// bf16 split of the fp32 activations, (T, 3H) = [y1 | y2 | y3], at
// router_split_rows(extra, plan, H, E).
cudaError_t launch_router_tc(const void* x, bool f32in, bool presplit, const float* Wg, int T,
                             int H, int E, const RouterPlan& plan, float* partial, void* extra,
                             int* zero_word, int* status, cudaStream_t s);
uint16_t* router_split_rows(void* extra, const RouterPlan& plan, int H, int E);
// partial[s][T][E] when splits > 1, else writes out directly.  zero_word (may be
// null) is set to 0 by the launch (the fused gating/routing counter).  With a
// decode-size plan, the launch also asks L2 to prefetch [l2_hint, l2_hint +
// l2_hint_bytes) (16-byte aligned, inside one allocation; bytes rounded down to
// whole 32 KB chunks), for data that later kernels of the stream read.
cudaError_t launch_router(const uint16_t* x, const float* Wg, int T, int H, int E,
                          const RouterPlan& plan, float* partial_or_out, int* zero_word,
                          cudaStream_t s, const void* l2_hint = nullptr,
                          size_t l2_hint_bytes = 0);
// Same with fp32 activations (the MXFP8 path routes on the fp32 normalised input).
cudaError_t launch_router_f32(const float* x, const float* Wg, int T, int H, int E,
                              const RouterPlan& plan, float* partial_or_out, int* zero_word,
                              cudaStream_t s, const void* l2_hint = nullptr,
                              size_t l2_hint_bytes = 0);
cudaError_t launch_router_reduce(const float* partial, int splits, int T, int E, float* logits,
                                 cudaStream_t s);
// Optional init_routing fused into the gating launch (one-CTA routing, P <= 4096):
// the last gating CTA routes all pairs.  counter must be 0 at launch.
struct GatingRouting {
  int* counter;
  int32_t* counts;
  int32_t* offsets;
  int32_t* eri;
  int32_t* sri;
  int* done;     // E + 1 ints cleared for the grouped GEMM (per-expert dependency
                 // counters, then its unit counter)
  int E_routed;  // experts [0, E_routed) are routed; ids >= E_routed (zero-computation
                 // experts) are skipped.  0: all E gating columns are routed experts.
};
// Gating reads sum_{s<splits} src[s*T*E + t*E + e] (splits == 1: plain logits).
cudaError_t launch_gating(const float* src, int splits, int T, int E, int k, int renormalize,
                          int32_t* ids, float* w, const GatingRouting* fuse, int* status,
                          cudaStream_t s);

// ---- routing (routing.cu)
struct RoutingPlan {
  bool single_cta;
  int chunks;        // multi-CTA path: number of pair chunks
  int chunk_pairs;   // pairs per chunk
};
RoutingPlan routing_plan(int P, int E);
size_t routing_ws_bytes(int P, int E);
// ids (P); writes counts (may be null), offsets (E+1), eri (P), sri (P).
// zero_counter (E + 1 ints, may be null) is cleared for the fused GEMM: the
// per-expert dependency counters and its unit counter.
cudaError_t launch_routing(const int32_t* ids, int P, int E, int32_t* counts, int32_t* offsets,
                           int32_t* eri, int32_t* sri, void* ws, int* zero_counter, int* status,
                           cudaStream_t s);
// Routing of the local experts [e_begin, e_begin + E) out of ids [0, E_total).
cudaError_t launch_routing_range(const int32_t* ids, int P, int e_begin, int E, int E_total,
                                 int32_t* counts, int32_t* offsets, int32_t* eri, int32_t* sri,
                                 void* ws, int* zero_counter, int* status, cudaStream_t s);
// expanded_x = the token rows in expert order, from the routing's eri (k slots per
// token, -1 for a pair routed elsewhere) and sri: at T >= kScatterMinTokens each
// token row is read once and written to its slots, below by a gather per sorted row.
constexpr int kScatterMinTokens = 256;
cudaError_t launch_expand_rows(const uint16_t* x, const int32_t* eri, const int32_t* sri,
                               const int32_t* offsets, int E, int T, int H, int k, uint16_t* xe,
                               cudaStream_t s);
cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* sri, const int32_t* offsets,
                               int E, int P, int H, int k, uint16_t* expanded_x, cudaStream_t s);
cudaError_t launch_expert_tokens(const int32_t* ids, int P, int E, int32_t* counts,
                                 int32_t* offsets, int* status, cudaStream_t s);
cudaError_t launch_finalize(const uint16_t* y2, const float* w, const int32_t* eri, int T, int k,
                            int H, uint16_t* out, cudaStream_t s);

// ---- grouped GEMM (gmm.cu)
struct GemmPhase {
  const void* A_weights;   // packed weights, rows = E * MW, cols = K
  const uint16_t* B_act;   // activations (P, b_inner or K)
  uint16_t* out;           // (P, n_out) bf16, epi 0 and 1
  int K;                   // reduction length
  int MW;                  // weight rows per expert (2I for gate/up, H for down)
  int n_out;               // output columns (I for gate/up, H for down); row stride of out_f32
  int epi;                 // 0: SwiGLU on interleaved gate/up rows, 1: plain, 2: fp32 partials
  int ksplit = 1;          // split of K into units (epi 2)
  int b_inner = 0;         // B's row length when it differs from K
  int bseg = 0;            // see GemmArgs::bseg
  uint32_t bmap = 0;
  float* out_f32 = nullptr;// epi 2: part[ksplit][rows_total][n_out]
  int mvalid = 0;
  int rows_total = 0;
};
// phases[0] and/or phases[1] (null A_weights = phase absent).  When both are
// present they run in one persistent launch with a per-expert dependency on
// done_counter (E + 1 ints, zeroed beforehand; the last one counts drawn units).
cudaError_t launch_grouped_gemm(const GemmPhase* ph0, const GemmPhase* ph1,
                                const int32_t* offsets, int E, int P, int max_rows_hint,
                                int* done_counter, int* status, cudaStream_t s);
// Test hook of the one-CTA grouped GEMM (moe_debug_set_gemm_stall); stage < 0: off.
void set_gemm_stall(int stage, unsigned long long wait_ns);
// Test hook of the CTA-pair grouped GEMM (moe_debug_set_pair_light): 0 automatic,
// 1 light pipeline whenever experts of at most 32 rows exist, 2 never.
void set_pair_light(int mode);
cudaError_t launch_pack_w13(const uint16_t* w13, int E, int H, int I, uint16_t* out,
                            cudaStream_t s);
cudaError_t launch_pack_down(const uint16_t* down, int E, int H, int I, uint16_t* out,
                             cudaStream_t s);

// ---- MXFP8 (mx.cu, gmm_mx.cu)
// ys_out (may be null): the exact three-piece bf16 split of y, (T, 3H) = [y1 | y2 | y3],
// the tensor-core router's activations.
cudaError_t launch_add_rmsnorm_mxquant(const uint16_t* x, const uint16_t* r, const uint16_t* w,
                                       float eps, int T, int H, uint16_t* residual_out,
                                       float* y32_out, uint16_t* ys_out, uint8_t* q,
                                       uint8_t* scale, cudaStream_t s);
cudaError_t launch_mx_quantize(const float* y, int rows, int n, uint8_t* q, uint8_t* scale,
                               cudaStream_t s);
cudaError_t launch_pack_mx(const uint16_t* w13, const uint16_t* down, int E, int H, int I,
                           uint8_t* w13q, uint8_t* w13sf, uint8_t* downq, uint8_t* downsf,
                           cudaStream_t s);
cudaError_t launch_pack_mx4(const uint16_t* w13, const uint16_t* down, int E, int H, int I,
                            uint8_t* w13q, uint8_t* w13sf, uint8_t* downq, uint8_t* downsf,
                            cudaStream_t s);
// Expert-sorted MX rows <-> the padded GEMM layout (standalone block-scaled GEMMs).
cudaError_t launch_mx_pad_sorted(const uint8_t* q, const uint8_t* sc, const int32_t* offsets,
                                 int E, int P, int K, int pad, uint8_t* out_q, uint8_t* out_sf,
                                 int32_t* row_map, cudaStream_t s);
cudaError_t launch_mx_unpad(const uint8_t* pq, const uint8_t* psf, const uint16_t* pbf,
                            const int32_t* row_map, const int32_t* offsets_end, int P, int N,
                            int pad, uint8_t* q, uint8_t* sc, uint16_t* y, cudaStream_t s);
// Row padding of the expert-sorted MX activations, and with it the block-scaled
// GEMM's tile shape: 32 (narrow tiles, one scale atom per 32 rows) when the layer
// has at most 16 token-expert pairs per expert on average, else 128.
inline int mx_pad_rows(long long P, int E) { return P <= 16LL * E ? 32 : 128; }
cudaError_t launch_mx_expand(const uint8_t* xq, const uint8_t* xs, const int32_t* ids,
                             const int32_t* eri, const int32_t* offsets, int E, int P, int H,
                             int k, int pad, uint8_t* xe, uint8_t* xe_sf, int32_t* eri_pad,
                             cudaStream_t s);
struct GemmPhaseMx {
  const void* A_q;          // packed e4m3 weights, rows = E * MW, K bytes each
  const uint8_t* A_sf;      // weight scale atoms
  const uint8_t* B_q;       // padded expert-sorted activation codes (rows, K)
  const uint8_t* B_sf;      // their scale atoms
  uint8_t* out_q;           // phase 0: h codes (rows, n_out)
  uint8_t* out_sf;          // phase 0: h scale atoms
  uint16_t* out_bf16;       // phase 1: y (rows, n_out)
  int K, MW, n_out;
  bool a_fp4 = false;       // weights are packed e2m1 (two per byte) instead of e4m3
};
// pad = mx_pad_rows(P, E) of the activation layout (selects the tile shape);
// P_pad_rows = rows of that padded layout.  With both phases, done holds E + 1
// zeroed ints: the per-expert dependency counters, then a unit counter from which
// the CTA-pair kernel's pairs draw their units.
cudaError_t launch_grouped_gemm_mx(const GemmPhaseMx* ph0, const GemmPhaseMx* ph1,
                                   const int32_t* offsets, int E, int pad, int P_pad_rows,
                                   int* done, int* status, cudaStream_t s);

// ---- next rows (norm_route2.cu)
cudaError_t launch_add_rmsnorm_cast(const uint16_t* x, const uint16_t* r, const uint16_t* w,
                                    float eps, int T, int H, uint16_t* residual_out,
                                    float* y32_out, uint16_t* ybf_out, cudaStream_t s);
cudaError_t launch_finalize_v2(const uint16_t* y2, const float* w, const int32_t* eri,
                               const int32_t* ids, const uint16_t* xin, int T, int k, int H, int E,
                               int E_total, uint16_t* out, cudaStream_t s);
size_t reroute_ws_bytes(int R, int El);
cudaError_t launch_re_routing(const uint16_t* xin, const int32_t* cnt, int R, int El, int N, int H,
                              uint16_t* xout, int32_t* perm, int32_t* offsets, void* ws,
                              cudaStream_t s);

// ---- profiling switch (api.cu)
// True when the environment variable MOE_GB300_PAIR_NONCOOPERATIVE is set to 1 (read
// once): the CTA-pair grouped GEMMs are then launched as plain cluster launches
// instead of cooperative ones, because profilers refuse cooperative cluster launches.
// The grid is one CTA per SM either way; co-residency of the two projections' CTAs is
// then expected rather than guaranteed (on an otherwise idle GPU every CTA is
// resident), and a phase-1 wait that could not end runs out its bounded limit and
// sets MOE_DEV_WAIT_TIMEOUT.  Off by default; for profiling only.
bool pair_launch_noncooperative();

// ---- device facts (api.cu)
int device_sm_count();
int* device_status_ptr();  // the current device's status word, or null
bool encode_tmap_2d(CUtensorMap* tm, CUtensorMapDataType dtype, uint32_t elem_bytes,
                    const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                    uint32_t box_rows);
bool encode_tmap_2d_bf16(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t rows,
                         uint32_t box_inner, uint32_t box_rows);
// Explicit row pitch (bytes), for packed sub-byte element types.
bool encode_tmap_2d_strided(CUtensorMap* tm, CUtensorMapDataType dtype, const void* base,
                            uint64_t inner, uint64_t rows, uint64_t row_bytes, uint32_t box_inner,
                            uint32_t box_rows);

}  // namespace moe
