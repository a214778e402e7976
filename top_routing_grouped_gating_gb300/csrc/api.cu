// C-ABI entry points of the MoE-layer library: argument validation, per-device
// facts (architecture, SM count, status word address), TMA descriptor encoding,
// workspace layouts, and the sequence of launches for each operator.  The
// operators follow the page "基于Atlas A3、950训练/推理集群的Qwen3-MoE模型低时延
// 推理性能优化实践": gating top-k softmax (§快速选择专家), init_routing /
// compute_expert_tokens / finalize_routing (§高效排序和token路由), grouped matmul
// (§高性能专家计算) with SwiGLU (§计算分解).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "../../include/moe_gb300.h"
#include "internal.h"

namespace {

constexpr int kAbiVersion = 1;

// The device status word; each device holds its own copy.  Host code must not
// use its name as an address: the device address comes from
// cudaGetSymbolAddress, taken once per device.
__device__ int g_device_status;

struct DeviceFacts {
  bool probed = false;
  bool arch_ok = false;
  int sm_count = 0;
  size_t l2_bytes = 0;
  int* status = nullptr;
};
std::mutex g_mu;
DeviceFacts g_dev[64];

// Decode forward: while the router, gating and routing run, HBM is idle, so the
// router launch asks L2 for the front of packed w13 (w13_bytes in all, row_bytes
// per weight row of K = H).  This is the weight prefetch of the page
// "基于Atlas A3集群的LongCat-Flash模型推理性能优化实践" (§权重预取): weights of a
// memory-bound operator are pulled from HBM into L2 while an operator that needs
// little bandwidth runs, at most bandwidth x the time available, and less if the
// overlapped operator slows down.  The grouped GEMM's first wave is one 128-row w13
// block per CTA of the lowest active experts; 5/8 of that wave, and at most 5/8 of
// L2, is requested (bf16 on a GB300: about 50 MB at H = 2048 and 80 MB at H = 4096,
// the sizes that shortened the step most in a sweep; more delays the routing
// kernels by more than the GEMM gains).
size_t decode_l2_hint_bytes(const DeviceFacts& d, size_t w13_bytes, size_t row_bytes) {
  const size_t wave = static_cast<size_t>(d.sm_count) * 128 * row_bytes;
  return std::min({w13_bytes, wave * 5 / 8, d.l2_bytes * 5 / 8});
}

moe_status current_device(DeviceFacts** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED_ARCH;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceFacts& d = g_dev[dev];
  if (!d.probed) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    int l2 = 0;
    if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    d.arch_ok = (major == 10 && minor == 3);
    d.sm_count = sms;
    d.l2_bytes = static_cast<size_t>(l2);
    if (d.arch_ok) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return MOE_ERR_CUDA;
      d.status = static_cast<int*>(p);
    }
    d.probed = true;
  }
  if (!d.arch_ok) return MOE_ERR_UNSUPPORTED_ARCH;
  *out = &d;
  return MOE_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

moe_status check_layer_shape(int T, int H, int E, int k, int I) {
  if (T < 1 || H < 1 || E < 1 || k < 1 || I < 1) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (H % 128 != 0 || I % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (E > 256 || k > E || k > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((long long)T * k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                      \
  do {                                     \
    const moe_status st_ = (expr);         \
    if (st_ != MOE_OK) return st_;         \
  } while (0)
#define MOE_CUDA(expr) MOE_TRY(cuda_status(expr))

// Workspace of moe_forward, in call order.
struct ForwardLayout {
  size_t router, ids, w, routing, counts, offsets, eri, sri, done, counter, xe, h, y2, total;
};

ForwardLayout forward_layout(int T, int H, int E, int k, int I) {
  ForwardLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align256(bytes);
    return at;
  };
  const size_t P = (size_t)T * k;
  L.router = take(moe::router_ws_bytes(T, H, E, false));
  L.ids = take(P * sizeof(int32_t));
  L.w = take(P * sizeof(float));
  L.routing = take(moe::routing_ws_bytes((int)P, E));
  L.counts = take((size_t)E * sizeof(int32_t));
  L.offsets = take((size_t)(E + 1) * sizeof(int32_t));
  L.eri = take(P * sizeof(int32_t));
  L.sri = take(P * sizeof(int32_t));
  L.done = take((size_t)(E + 1) * sizeof(int32_t));   // + the GEMM's unit counter
  L.counter = take(sizeof(int32_t));
  L.xe = take(P * H * 2);
  L.h = take(P * I * 2);
  L.y2 = take(P * H * 2);
  L.total = o;
  return L;
}

thread_local cudaEvent_t t_gemm_ev_begin = nullptr;
thread_local cudaEvent_t t_gemm_ev_end = nullptr;

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

}  // namespace

namespace moe {

bool pair_launch_noncooperative() {
  static const bool on = [] {
    const char* v = std::getenv("MOE_GB300_PAIR_NONCOOPERATIVE");
    return v != nullptr && v[0] == '1' && v[1] == '\0';
  }();
  return on;
}

int device_sm_count() {
  DeviceFacts* d = nullptr;
  if (current_device(&d) != MOE_OK) return 1;
  return d->sm_count;
}

int* device_status_ptr() {
  DeviceFacts* d = nullptr;
  if (current_device(&d) != MOE_OK) return nullptr;
  return d->status;
}

bool encode_tmap_2d(CUtensorMap* tm, CUtensorMapDataType dtype, uint32_t elem_bytes,
                    const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                    uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * elem_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(tm, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_2d_strided(CUtensorMap* tm, CUtensorMapDataType dtype, const void* base,
                            uint64_t inner, uint64_t rows, uint64_t row_bytes, uint32_t box_inner,
                            uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(tm, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_2d_bf16(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t rows,
                         uint32_t box_inner, uint32_t box_rows) {
  return encode_tmap_2d(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, rows, box_inner,
                        box_rows);
}

}  // namespace moe

extern "C" {

int moe_abi_version(void) { return kAbiVersion; }

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad size)";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_UNSUPPORTED_ARCH:
      return "unsupported device: compute capability 10.3 and a device index below 64 required";
    case MOE_ERR_WORKSPACE: return "workspace too small or misaligned";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}

moe_status moe_get_device_status(int32_t* status_out, moe_stream_t stream) {
  if (status_out == nullptr) return MOE_ERR_INVALID_ARG;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  int v = 0;
  MOE_CUDA(cudaMemcpyAsync(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost, stream));
  MOE_CUDA(cudaStreamSynchronize(stream));
  *status_out = v;
  return MOE_OK;
}

moe_status moe_clear_device_status(moe_stream_t stream) {
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  MOE_CUDA(cudaMemsetAsync(d->status, 0, sizeof(int), stream));
  return MOE_OK;
}

// ------------------------------------------------------------------ router --
size_t moe_router_logits_workspace_size(int T, int H, int E) {
  if (T < 1 || H < 1 || E < 1) return 0;
  const moe::RouterPlan rp = moe::router_plan_ex(T, H, E, false);
  return (rp.splits > 1 || rp.tc) ? moe::router_ws_bytes(T, H, E, false) : 0;
}

moe_status moe_router_logits(const moe_bf16* x, const float* Wg, int T, int H, int E,
                             float* logits, void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!x || !Wg || !logits || !aligned16(x)) return MOE_ERR_INVALID_ARG;
  if (T < 1 || E < 1 || E > 256 || H < 32 || H % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  const moe::RouterPlan rp = moe::router_plan_ex(T, H, E, false);
  if (rp.splits > 1 || rp.tc) {
    if (ws == nullptr || ws_bytes < moe_router_logits_workspace_size(T, H, E) ||
        (reinterpret_cast<uintptr_t>(ws) & 255u))
      return MOE_ERR_WORKSPACE;
    float* partial = static_cast<float*>(ws);
    if (rp.tc) {
      void* extra = at<uint8_t>(ws, align256((size_t)rp.splits * T * E * sizeof(float)));
      MOE_CUDA(moe::launch_router_tc(x, false, false, Wg, T, H, E, rp, partial, extra, nullptr,
                                     d->status, stream));
    } else {
      MOE_CUDA(moe::launch_router(x, Wg, T, H, E, rp, partial, nullptr, stream));
    }
    MOE_CUDA(moe::launch_router_reduce(partial, rp.splits, T, E, logits, stream));
  } else {
    MOE_CUDA(moe::launch_router(x, Wg, T, H, E, rp, logits, nullptr, stream));
  }
  return MOE_OK;
}

// ------------------------------------------------------------------ gating --
moe_status moe_gating_topk_softmax(const float* logits, int T, int E, int k, int renormalize,
                                   int32_t* topk_ids, float* topk_w, moe_stream_t stream) {
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (T < 1 || E < 1 || E > 256 || k < 1 || k > E || k > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  MOE_CUDA(moe::launch_gating(logits, 1, T, E, k, renormalize, topk_ids, topk_w, nullptr,
                              d->status, stream));
  return MOE_OK;
}

// ----------------------------------------------------------------- routing --
size_t moe_init_routing_workspace_size(int T, int E, int k) {
  if (T < 1 || E < 1 || k < 1) return 0;
  const int P = T * k;
  return align256(moe::routing_ws_bytes(P, E)) + align256((size_t)E * sizeof(int32_t));
}

moe_status moe_init_routing(const moe_bf16* x, const int32_t* topk_ids, int T, int H, int E, int k,
                            moe_bf16* expanded_x, int32_t* expanded_row_idx,
                            int32_t* sorted_row_idx, int32_t* expert_offsets, int32_t* counts,
                            void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!topk_ids || !expanded_row_idx || !sorted_row_idx || !expert_offsets)
    return MOE_ERR_INVALID_ARG;
  if (expanded_x && (!x || !aligned16(x) || !aligned16(expanded_x))) return MOE_ERR_INVALID_ARG;
  if (T < 1 || E < 1 || E > 256 || k < 1 || k > 32 || (long long)T * k >= (1LL << 31))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (expanded_x && (H < 8 || H % 8 != 0)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (ws == nullptr || ws_bytes < moe_init_routing_workspace_size(T, E, k) ||
      (reinterpret_cast<uintptr_t>(ws) & 255u))
    return MOE_ERR_WORKSPACE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  const int P = T * k;
  int32_t* cnt = counts ? counts : at<int32_t>(ws, align256(moe::routing_ws_bytes(P, E)));
  MOE_CUDA(moe::launch_routing(topk_ids, P, E, cnt, expert_offsets, expanded_row_idx,
                               sorted_row_idx, ws, nullptr, d->status, stream));
  if (expanded_x)
    MOE_CUDA(moe::launch_expand_rows(x, expanded_row_idx, sorted_row_idx, expert_offsets, E, T, H,
                                     k, expanded_x, stream));
  return MOE_OK;
}

moe_status moe_compute_expert_tokens(const int32_t* topk_ids, int P, int E, int32_t* counts,
                                     int32_t* expert_offsets, moe_stream_t stream) {
  if (!topk_ids || !counts) return MOE_ERR_INVALID_ARG;
  if (P < 1 || E < 1 || E > 256) return MOE_ERR_UNSUPPORTED_SHAPE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  MOE_CUDA(moe::launch_expert_tokens(topk_ids, P, E, counts, expert_offsets, d->status, stream));
  return MOE_OK;
}

// ---------------------------------------------------------- weight packing --
size_t moe_packed_weight_bytes(int E, int H, int I, int which) {
  if (E < 1 || H < 1 || I < 1) return 0;
  return (size_t)E * H * I * 2 * (which == 0 ? 2 : 1);
}

moe_status moe_pack_weights(const moe_bf16* w13, const moe_bf16* down, int E, int H, int I,
                            void* w13_packed, void* down_packed, moe_stream_t stream) {
  if ((w13 && !w13_packed) || (down && !down_packed)) return MOE_ERR_INVALID_ARG;
  if (E < 1 || E > 256 || H % 128 != 0 || I % 64 != 0 || H < 128 || I < 64)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  if (w13) MOE_CUDA(moe::launch_pack_w13(w13, E, H, I, static_cast<uint16_t*>(w13_packed), stream));
  if (down)
    MOE_CUDA(moe::launch_pack_down(down, E, H, I, static_cast<uint16_t*>(down_packed), stream));
  return MOE_OK;
}

// ----------------------------------------------------------- grouped GEMMs --
size_t moe_grouped_matmul_workspace_size(void) { return 0; }

static moe_status grouped_common(const moe_bf16* A, const void* w, const int32_t* offsets, int E,
                                 int P, int K, int N, moe_bf16* out, bool swiglu,
                                 moe_stream_t stream) {
  if (!A || !w || !offsets || !out || !aligned16(A) || !aligned16(w) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  if (E < 1 || E > 256 || P < 1 || K < 64 || K % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (swiglu ? (N < 64 || N % 64 != 0) : (N < 128 || N % 128 != 0))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  moe::GemmPhase ph{};
  ph.A_weights = w;
  ph.B_act = A;
  ph.out = out;
  ph.K = K;
  ph.MW = swiglu ? 2 * N : N;
  ph.n_out = N;
  ph.epi = swiglu ? 0 : 1;
  MOE_CUDA(moe::launch_grouped_gemm(swiglu ? &ph : nullptr, swiglu ? nullptr : &ph, offsets, E, P,
                                    P, nullptr, d->status, stream));
  return MOE_OK;
}

moe_status moe_grouped_matmul_swiglu(const moe_bf16* A, const void* w13_packed,
                                     const int32_t* expert_offsets, int E, int P, int K, int N,
                                     moe_bf16* h, void* ws, size_t ws_bytes, moe_stream_t stream) {
  (void)ws;
  (void)ws_bytes;
  return grouped_common(A, w13_packed, expert_offsets, E, P, K, N, h, true, stream);
}

moe_status moe_grouped_matmul(const moe_bf16* A, const void* w_packed,
                              const int32_t* expert_offsets, int E, int P, int K, int N,
                              moe_bf16* y, void* ws, size_t ws_bytes, moe_stream_t stream) {
  (void)ws;
  (void)ws_bytes;
  return grouped_common(A, w_packed, expert_offsets, E, P, K, N, y, false, stream);
}

// ---------------------------------------------------------------- finalize --
moe_status moe_finalize_routing(const moe_bf16* y2, const float* topk_w,
                                const int32_t* expanded_row_idx, int T, int k, int H,
                                moe_bf16* out, moe_stream_t stream) {
  if (!y2 || !topk_w || !expanded_row_idx || !out || !aligned16(y2) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  if (T < 1 || k < 1 || k > 32 || H < 8 || H % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  MOE_CUDA(moe::launch_finalize(y2, topk_w, expanded_row_idx, T, k, H, out, stream));
  return MOE_OK;
}

// ------------------------------------------------------------- whole layer --
size_t moe_forward_workspace_size(int T, int H, int E, int k, int I) {
  if (check_layer_shape(T, H, E, k, I) != MOE_OK) return 0;
  return forward_layout(T, H, E, k, I).total;
}

moe_status moe_forward(const moe_bf16* x, const float* Wg, const float* logits_override,
                       const void* w13_packed, const void* down_packed, int T, int H, int E, int k,
                       int I, moe_bf16* out, int32_t* topk_ids_out, float* topk_w_out, void* ws,
                       size_t ws_bytes, moe_stream_t stream) {
  if (!x || !w13_packed || !down_packed || !out) return MOE_ERR_INVALID_ARG;
  if (!logits_override && !Wg) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w13_packed) || !aligned16(down_packed) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_layer_shape(T, H, E, k, I));
  const ForwardLayout L = forward_layout(T, H, E, k, I);
  if (ws == nullptr || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return MOE_ERR_WORKSPACE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  const int P = T * k;
  int32_t* ids = topk_ids_out ? topk_ids_out : at<int32_t>(ws, L.ids);
  float* w = topk_w_out ? topk_w_out : at<float>(ws, L.w);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* eri = at<int32_t>(ws, L.eri);
  int32_t* sri = at<int32_t>(ws, L.sri);
  int* done = at<int>(ws, L.done);
  uint16_t* xe = at<uint16_t>(ws, L.xe);
  uint16_t* h = at<uint16_t>(ws, L.h);
  uint16_t* y2 = at<uint16_t>(ws, L.y2);

  // Small P: init_routing runs inside the gating launch (its last CTA routes all
  // pairs); the counter it uses is zeroed by the router launch, or here.
  const bool fused_routing = moe::routing_plan(P, E).single_cta;
  moe::GatingRouting fr{};
  fr.counter = at<int>(ws, L.counter);
  fr.counts = at<int32_t>(ws, L.counts);
  fr.offsets = offsets;
  fr.eri = eri;
  fr.sri = sri;
  fr.done = done;
  const moe::GatingRouting* fuse = fused_routing ? &fr : nullptr;
  if (logits_override) {
    if (fused_routing) MOE_CUDA(cudaMemsetAsync(fr.counter, 0, sizeof(int), stream));
    MOE_CUDA(moe::launch_gating(logits_override, 1, T, E, k, 1, ids, w, fuse, d->status, stream));
  } else {
    const moe::RouterPlan rp = moe::router_plan_ex(T, H, E, false);
    float* part = at<float>(ws, L.router);
    int* zw = fused_routing ? fr.counter : nullptr;
    if (rp.tc) {
      void* extra = at<uint8_t>(ws, L.router + align256((size_t)rp.splits * T * E * sizeof(float)));
      MOE_CUDA(moe::launch_router_tc(x, false, false, Wg, T, H, E, rp, part, extra, zw, d->status,
                                     stream));
    } else {
      const size_t hint = decode_l2_hint_bytes(*d, moe_packed_weight_bytes(E, H, I, 0), 2u * H);
      MOE_CUDA(moe::launch_router(x, Wg, T, H, E, rp, part, zw, stream, w13_packed, hint));
    }
    MOE_CUDA(moe::launch_gating(part, rp.splits, T, E, k, 1, ids, w, fuse, d->status, stream));
  }
  if (!fused_routing)
    MOE_CUDA(moe::launch_routing(ids, P, E, fr.counts, offsets, eri, sri,
                                 at<void>(ws, L.routing), done, d->status, stream));
  MOE_CUDA(moe::launch_expand_rows(x, eri, sri, offsets, E, T, H, k, xe, stream));
  moe::GemmPhase g1{}, g2{};
  g1.A_weights = w13_packed;
  g1.B_act = xe;
  g1.out = h;
  g1.K = H;
  g1.MW = 2 * I;
  g1.n_out = I;
  g1.epi = 0;
  g2.A_weights = down_packed;
  g2.B_act = h;
  g2.out = y2;
  g2.K = I;
  g2.MW = H;
  g2.n_out = H;
  g2.epi = 1;
  if (t_gemm_ev_begin) MOE_CUDA(cudaEventRecord(t_gemm_ev_begin, stream));
  MOE_CUDA(moe::launch_grouped_gemm(&g1, &g2, offsets, E, P, T, done, d->status, stream));
  if (t_gemm_ev_end) MOE_CUDA(cudaEventRecord(t_gemm_ev_end, stream));
  MOE_CUDA(moe::launch_finalize(y2, w, eri, T, k, H, out, stream));
  return MOE_OK;
}

// ------------------------------------------------------------------- MXFP8 --
moe_status moe_add_rmsnorm_mxquant(const moe_bf16* x, const moe_bf16* r, const moe_bf16* w,
                                   float eps, int T, int H, moe_bf16* residual_out,
                                   float* y32_out, uint8_t* q, uint8_t* scale,
                                   moe_stream_t stream) {
  if (!x || !w || !q || !scale) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || (r && !aligned16(r)) || !aligned16(w) ||
      (residual_out && !aligned16(residual_out)) || (y32_out && !aligned16(y32_out)) ||
      (reinterpret_cast<uintptr_t>(q) & 7u))
    return MOE_ERR_INVALID_ARG;
  if (T < 1 || H < 256 || H % 256 != 0 || H > 32768) return MOE_ERR_UNSUPPORTED_SHAPE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  MOE_CUDA(moe::launch_add_rmsnorm_mxquant(x, r, w, eps, T, H, residual_out, y32_out, nullptr, q, scale,
                                           stream));
  return MOE_OK;
}

moe_status moe_mx_quantize(const float* y, int rows, int n, uint8_t* q, uint8_t* scale,
                           moe_stream_t stream) {
  if (!y || !q || !scale || !aligned16(y) || (reinterpret_cast<uintptr_t>(q) & 3u))
    return MOE_ERR_INVALID_ARG;
  if (rows < 1 || n < 32 || n % 32 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  MOE_CUDA(moe::launch_mx_quantize(y, rows, n, q, scale, stream));
  return MOE_OK;
}

size_t moe_packed_weight_bytes_mx(int E, int H, int I, int which) {
  if (E < 1 || H < 1 || I < 1) return 0;
  const size_t w = (size_t)E * H * I;
  switch (which) {
    case 0: return 2 * w;
    case 1: return 2 * w / 32;
    case 2: return w;
    case 3: return w / 32;
    default: return 0;
  }
}

moe_status moe_pack_weights_mx(const moe_bf16* w13, const moe_bf16* down, int E, int H, int I,
                               void* w13_q, void* w13_sf, void* down_q, void* down_sf,
                               moe_stream_t stream) {
  if ((w13 && (!w13_q || !w13_sf)) || (down && (!down_q || !down_sf))) return MOE_ERR_INVALID_ARG;
  if (E < 1 || E > 256 || H < 128 || I < 128 || H % 128 != 0 || I % 128 != 0)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  MOE_CUDA(moe::launch_pack_mx(w13, down, E, H, I, static_cast<uint8_t*>(w13_q),
                               static_cast<uint8_t*>(w13_sf), static_cast<uint8_t*>(down_q),
                               static_cast<uint8_t*>(down_sf), stream));
  return MOE_OK;
}

namespace {

struct ForwardMxLayout {
  size_t y32, xq, xs, router, ids, w, routing, counts, offsets, eri, sri, done, counter, xe,
      xe_sf, eri_pad, hq, h_sf, y2, total;
  int pad_rows;
  int pad;  // row padding of each expert block (one scale atom per pad rows and K step)
};

ForwardMxLayout forward_mx_layout(int T, int H, int E, int k, int I) {
  ForwardMxLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align256(bytes);
    return at;
  };
  const size_t P = (size_t)T * k;
  // an upper bound on the padded rows for either padding (a multiple of 128)
  const size_t R = ((P + 127) / 128) * 128 + 128 * (size_t)E;
  L.pad_rows = (int)R;
  L.pad = moe::mx_pad_rows((long long)P, E);
  L.y32 = take((size_t)T * H * 4);
  L.xq = take((size_t)T * H);
  L.xs = take((size_t)T * H / 32);
  L.router = take(moe::router_ws_bytes(T, H, E, true));
  L.ids = take(P * 4);
  L.w = take(P * 4);
  L.routing = take(moe::routing_ws_bytes((int)P, E));
  L.counts = take((size_t)E * 4);
  L.offsets = take((size_t)(E + 1) * 4);
  L.eri = take(P * 4);
  L.sri = take(P * 4);
  L.done = take((size_t)(E + 1) * 4);   // + the GEMM's unit counter
  L.counter = take(4);
  L.xe = take(R * H);
  L.xe_sf = take(R / L.pad * (H / 128) * 512);
  L.eri_pad = take(P * 4);
  L.hq = take(R * I);
  L.h_sf = take(R / L.pad * (I / 128) * 512);
  L.y2 = take(R * H * 2);
  L.total = o;
  return L;
}

moe_status check_mx_shape(int T, int H, int E, int k, int I) {
  MOE_TRY(check_layer_shape(T, H, E, k, I));
  if (H % 256 != 0 || I % 128 != 0 || H > 32768) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((long long)T * k + 128LL * E + 128 >= (1LL << 31) / 4) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

}  // namespace

size_t moe_forward_mx_workspace_size(int T, int H, int E, int k, int I) {
  if (check_mx_shape(T, H, E, k, I) != MOE_OK) return 0;
  return forward_mx_layout(T, H, E, k, I).total;
}

namespace {

// The block-scaled layer; w4 selects MXFP4 (packed e2m1) expert weights.
moe_status forward_mx_impl(const moe_bf16* x, const moe_bf16* r, const moe_bf16* norm_w, float eps,
                           const float* Wg, const float* logits_override, const void* w13_q,
                           const void* w13_sf, const void* down_q, const void* down_sf, int T,
                           int H, int E, int k, int I, moe_bf16* out, moe_bf16* residual_out,
                           int32_t* topk_ids_out, float* topk_w_out, void* ws, size_t ws_bytes,
                           bool w4, cudaStream_t stream) {
  if (!x || !norm_w || !w13_q || !w13_sf || !down_q || !down_sf || !out)
    return MOE_ERR_INVALID_ARG;
  // packed e2m1 rows are read by TMA from 32-byte aligned addresses
  if (w4 && ((reinterpret_cast<uintptr_t>(w13_q) | reinterpret_cast<uintptr_t>(down_q)) & 31u))
    return MOE_ERR_INVALID_ARG;
  if (!logits_override && !Wg) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || (r && !aligned16(r)) || !aligned16(norm_w) || !aligned16(w13_q) ||
      !aligned16(w13_sf) || !aligned16(down_q) || !aligned16(down_sf) || !aligned16(out) ||
      (residual_out && !aligned16(residual_out)))
    return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_mx_shape(T, H, E, k, I));
  const ForwardMxLayout L = forward_mx_layout(T, H, E, k, I);
  if (ws == nullptr || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return MOE_ERR_WORKSPACE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  const int P = T * k;
  float* y32 = at<float>(ws, L.y32);
  uint8_t* xq = at<uint8_t>(ws, L.xq);
  uint8_t* xs = at<uint8_t>(ws, L.xs);
  int32_t* ids = topk_ids_out ? topk_ids_out : at<int32_t>(ws, L.ids);
  float* w = topk_w_out ? topk_w_out : at<float>(ws, L.w);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* eri = at<int32_t>(ws, L.eri);
  int32_t* sri = at<int32_t>(ws, L.sri);
  int* done = at<int>(ws, L.done);
  // The router reads the fp32 RMSNorm output: the tensor-core router as its exact
  // bf16 split, which the norm kernel writes straight into the router's scratch;
  // with given logits nothing reads it.
  const moe::RouterPlan rp = moe::router_plan_ex(T, H, E, true);
  void* router_extra = at<uint8_t>(ws, L.router + align256((size_t)rp.splits * T * E * sizeof(float)));
  const bool presplit = !logits_override && rp.tc;
  uint16_t* ys = presplit ? moe::router_split_rows(router_extra, rp, H, E) : nullptr;
  float* y32_used = (logits_override || presplit) ? nullptr : y32;
  MOE_CUDA(moe::launch_add_rmsnorm_mxquant(x, r, norm_w, eps, T, H, residual_out, y32_used, ys,
                                           xq, xs, stream));
  const bool fused_routing = moe::routing_plan(P, E).single_cta;
  moe::GatingRouting fr{};
  fr.counter = at<int>(ws, L.counter);
  fr.counts = at<int32_t>(ws, L.counts);
  fr.offsets = offsets;
  fr.eri = eri;
  fr.sri = sri;
  fr.done = done;
  const moe::GatingRouting* fuse = fused_routing ? &fr : nullptr;
  if (logits_override) {
    if (fused_routing) MOE_CUDA(cudaMemsetAsync(fr.counter, 0, sizeof(int), stream));
    MOE_CUDA(moe::launch_gating(logits_override, 1, T, E, k, 1, ids, w, fuse, d->status, stream));
  } else {
    float* part = at<float>(ws, L.router);
    int* zw = fused_routing ? fr.counter : nullptr;
    if (rp.tc) {
      MOE_CUDA(moe::launch_router_tc(nullptr, true, true, Wg, T, H, E, rp, part, router_extra, zw,
                                     d->status, stream));
    } else {
      // e4m3 rows are H bytes, packed e2m1 rows H / 2
      const size_t row = w4 ? (size_t)H / 2 : (size_t)H;
      MOE_CUDA(moe::launch_router_f32(y32, Wg, T, H, E, rp, part, zw, stream, w13_q,
                                      decode_l2_hint_bytes(*d, row * 2 * I * E, row)));
    }
    MOE_CUDA(moe::launch_gating(part, rp.splits, T, E, k, 1, ids, w, fuse, d->status, stream));
  }
  if (!fused_routing)
    MOE_CUDA(moe::launch_routing(ids, P, E, fr.counts, offsets, eri, sri,
                                 at<void>(ws, L.routing), done, d->status, stream));
  uint8_t* xe = at<uint8_t>(ws, L.xe);
  uint8_t* xe_sf = at<uint8_t>(ws, L.xe_sf);
  int32_t* eri_pad = at<int32_t>(ws, L.eri_pad);
  MOE_CUDA(moe::launch_mx_expand(xq, xs, ids, eri, offsets, E, P, H, k, L.pad, xe, xe_sf, eri_pad,
                                 stream));
  uint8_t* hq = at<uint8_t>(ws, L.hq);
  uint8_t* h_sf = at<uint8_t>(ws, L.h_sf);
  uint16_t* y2 = at<uint16_t>(ws, L.y2);
  moe::GemmPhaseMx g1{}, g2{};
  g1.A_q = w13_q;
  g1.A_sf = static_cast<const uint8_t*>(w13_sf);
  g1.B_q = xe;
  g1.B_sf = xe_sf;
  g1.out_q = hq;
  g1.out_sf = h_sf;
  g1.K = H;
  g1.MW = 2 * I;
  g1.n_out = I;
  g2.A_q = down_q;
  g2.A_sf = static_cast<const uint8_t*>(down_sf);
  g2.B_q = hq;
  g2.B_sf = h_sf;
  g2.out_bf16 = y2;
  g2.K = I;
  g2.MW = H;
  g2.n_out = H;
  g1.a_fp4 = g2.a_fp4 = w4;
  if (t_gemm_ev_begin) MOE_CUDA(cudaEventRecord(t_gemm_ev_begin, stream));
  MOE_CUDA(moe::launch_grouped_gemm_mx(&g1, &g2, offsets, E, L.pad, L.pad_rows, done, d->status,
                                         stream));
  if (t_gemm_ev_end) MOE_CUDA(cudaEventRecord(t_gemm_ev_end, stream));
  MOE_CUDA(moe::launch_finalize(y2, w, eri_pad, T, k, H, out, stream));
  return MOE_OK;
}

}  // namespace

moe_status moe_forward_mx(const moe_bf16* x, const moe_bf16* r, const moe_bf16* norm_w, float eps,
                          const float* Wg, const float* logits_override, const void* w13_q,
                          const void* w13_sf, const void* down_q, const void* down_sf, int T,
                          int H, int E, int k, int I, moe_bf16* out, moe_bf16* residual_out,
                          int32_t* topk_ids_out, float* topk_w_out, void* ws, size_t ws_bytes,
                          moe_stream_t stream) {
  return forward_mx_impl(x, r, norm_w, eps, Wg, logits_override, w13_q, w13_sf, down_q, down_sf, T,
                         H, E, k, I, out, residual_out, topk_ids_out, topk_w_out, ws, ws_bytes,
                         false, stream);
}

// ------------------------------------------------------------------ W4A8 --
size_t moe_packed_weight_bytes_mx4(int E, int H, int I, int which) {
  if (E < 1 || H < 1 || I < 1) return 0;
  const size_t w = (size_t)E * H * I;
  switch (which) {
    case 0: return w;           // 2I x H e2m1 codes per expert, two per byte
    case 1: return 2 * w / 32;
    case 2: return w / 2;
    case 3: return w / 32;
    default: return 0;
  }
}

moe_status moe_pack_weights_mx4(const moe_bf16* w13, const moe_bf16* down, int E, int H, int I,
                                void* w13_q, void* w13_sf, void* down_q, void* down_sf,
                                moe_stream_t stream) {
  if ((w13 && (!w13_q || !w13_sf)) || (down && (!down_q || !down_sf))) return MOE_ERR_INVALID_ARG;
  if (E < 1 || E > 256 || H < 128 || I < 128 || H % 128 != 0 || I % 128 != 0)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  MOE_CUDA(moe::launch_pack_mx4(w13, down, E, H, I, static_cast<uint8_t*>(w13_q),
                                static_cast<uint8_t*>(w13_sf), static_cast<uint8_t*>(down_q),
                                static_cast<uint8_t*>(down_sf), stream));
  return MOE_OK;
}

// ------------------------------------------- standalone block-scaled GEMMs --
namespace {

struct GemmMxLayout {
  size_t xq, xsf, row_map, oq, osf, obf, total;
  int pad, rows;
};

GemmMxLayout gemm_mx_layout(int E, int P, int K, int N, bool swiglu) {
  GemmMxLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align256(bytes);
    return at;
  };
  const size_t R = (((size_t)P + 127) / 128) * 128 + 128 * (size_t)E;
  L.rows = (int)R;
  L.pad = moe::mx_pad_rows((long long)P, E);
  L.xq = take(R * K);
  L.xsf = take(R / L.pad * (K / 128) * 512);
  L.row_map = take((size_t)P * 4);
  if (swiglu) {
    L.oq = take(R * N);
    L.osf = take(R / L.pad * (N / 128) * 512);
  } else {
    L.obf = take(R * N * 2);
  }
  L.total = o;
  return L;
}

moe_status check_gemm_mx_shape(int E, int P, int K, int N) {
  if (E < 1 || E > 256 || P < 1 || K < 128 || N < 128 || K % 128 != 0 || N % 128 != 0)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((long long)P + 128LL * E + 128 >= (1LL << 31) / 4 || K > 32768 || N > 32768)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

moe_status gemm_mx_common(const uint8_t* A_q, const uint8_t* A_scale, const void* w_q,
                          const void* w_sf, int weight_format, const int32_t* offsets, int E,
                          int P, int K, int N, bool swiglu, uint8_t* h_q, uint8_t* h_scale,
                          moe_bf16* y, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!A_q || !A_scale || !w_q || !w_sf || !offsets) return MOE_ERR_INVALID_ARG;
  if (swiglu ? (!h_q || !h_scale) : !y) return MOE_ERR_INVALID_ARG;
  if (weight_format != 0 && weight_format != 1) return MOE_ERR_INVALID_ARG;
  if (!aligned16(A_q) || !aligned16(w_q) || !aligned16(w_sf) ||
      (swiglu ? !aligned16(h_q) : !aligned16(y)))
    return MOE_ERR_INVALID_ARG;
  if (weight_format == 1 && (reinterpret_cast<uintptr_t>(w_q) & 31u)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_gemm_mx_shape(E, P, K, N));
  const GemmMxLayout L = gemm_mx_layout(E, P, K, N, swiglu);
  if (ws == nullptr || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return MOE_ERR_WORKSPACE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  uint8_t* xq = at<uint8_t>(ws, L.xq);
  uint8_t* xsf = at<uint8_t>(ws, L.xsf);
  int32_t* row_map = at<int32_t>(ws, L.row_map);
  MOE_CUDA(moe::launch_mx_pad_sorted(A_q, A_scale, offsets, E, P, K, L.pad, xq, xsf, row_map,
                                     stream));
  moe::GemmPhaseMx g{};
  g.A_q = w_q;
  g.A_sf = static_cast<const uint8_t*>(w_sf);
  g.B_q = xq;
  g.B_sf = xsf;
  g.K = K;
  g.n_out = N;
  g.a_fp4 = weight_format == 1;
  if (swiglu) {
    g.MW = 2 * N;
    g.out_q = at<uint8_t>(ws, L.oq);
    g.out_sf = at<uint8_t>(ws, L.osf);
    MOE_CUDA(moe::launch_grouped_gemm_mx(&g, nullptr, offsets, E, L.pad, L.rows, nullptr,
                                         d->status, stream));
    MOE_CUDA(moe::launch_mx_unpad(g.out_q, g.out_sf, nullptr, row_map, offsets + E, P, N, L.pad,
                                  h_q, h_scale, nullptr, stream));
  } else {
    g.MW = N;
    g.out_bf16 = at<uint16_t>(ws, L.obf);
    MOE_CUDA(moe::launch_grouped_gemm_mx(nullptr, &g, offsets, E, L.pad, L.rows, nullptr,
                                         d->status, stream));
    MOE_CUDA(moe::launch_mx_unpad(nullptr, nullptr, g.out_bf16, row_map, offsets + E, P, N, L.pad,
                                  nullptr, nullptr, y, stream));
  }
  return MOE_OK;
}

}  // namespace

size_t moe_grouped_matmul_mx_workspace_size(int E, int P, int K, int N, int swiglu) {
  if (check_gemm_mx_shape(E, P, K, N) != MOE_OK) return 0;
  return gemm_mx_layout(E, P, K, N, swiglu != 0).total;
}

moe_status moe_grouped_matmul_swiglu_mx(const uint8_t* A_q, const uint8_t* A_scale,
                                        const void* w13_q, const void* w13_sf, int weight_format,
                                        const int32_t* expert_offsets, int E, int P, int K, int N,
                                        uint8_t* h_q, uint8_t* h_scale, void* ws, size_t ws_bytes,
                                        moe_stream_t stream) {
  return gemm_mx_common(A_q, A_scale, w13_q, w13_sf, weight_format, expert_offsets, E, P, K, N,
                        true, h_q, h_scale, nullptr, ws, ws_bytes, stream);
}

moe_status moe_grouped_matmul_mx(const uint8_t* A_q, const uint8_t* A_scale, const void* w_q,
                                 const void* w_sf, int weight_format,
                                 const int32_t* expert_offsets, int E, int P, int K, int N,
                                 moe_bf16* y, void* ws, size_t ws_bytes, moe_stream_t stream) {
  return gemm_mx_common(A_q, A_scale, w_q, w_sf, weight_format, expert_offsets, E, P, K, N, false,
                        nullptr, nullptr, y, ws, ws_bytes, stream);
}

size_t moe_forward_w4a8_workspace_size(int T, int H, int E, int k, int I) {
  return moe_forward_mx_workspace_size(T, H, E, k, I);
}

moe_status moe_forward_w4a8(const moe_bf16* x, const moe_bf16* r, const moe_bf16* norm_w,
                            float eps, const float* Wg, const float* logits_override,
                            const void* w13_q, const void* w13_sf, const void* down_q,
                            const void* down_sf, int T, int H, int E, int k, int I, moe_bf16* out,
                            moe_bf16* residual_out, int32_t* topk_ids_out, float* topk_w_out,
                            void* ws, size_t ws_bytes, moe_stream_t stream) {
  return forward_mx_impl(x, r, norm_w, eps, Wg, logits_override, w13_q, w13_sf, down_q, down_sf, T,
                         H, E, k, I, out, residual_out, topk_ids_out, topk_w_out, ws, ws_bytes,
                         true, stream);
}

// --------------------------------------------------------------- next rows --
moe_status moe_add_rmsnorm_cast(const moe_bf16* x, const moe_bf16* r, const moe_bf16* w,
                                float eps, int T, int H, moe_bf16* residual_out, float* y32_out,
                                moe_bf16* ybf16_out, moe_stream_t stream) {
  if (!x || !w || !ybf16_out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || (r && !aligned16(r)) || !aligned16(w) || !aligned16(ybf16_out) ||
      (residual_out && !aligned16(residual_out)) || (y32_out && !aligned16(y32_out)))
    return MOE_ERR_INVALID_ARG;
  if (T < 1 || H < 256 || H % 256 != 0 || H > 32768) return MOE_ERR_UNSUPPORTED_SHAPE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  MOE_CUDA(moe::launch_add_rmsnorm_cast(x, r, w, eps, T, H, residual_out, y32_out, ybf16_out,
                                        stream));
  return MOE_OK;
}

size_t moe_init_routing_v2_workspace_size(int T, int E_local, int k) {
  if (T < 1 || E_local < 1 || k < 1) return 0;
  return align256(moe::routing_ws_bytes(T * k, E_local)) + align256((size_t)E_local * 4);
}

moe_status moe_init_routing_v2(const moe_bf16* x, const int32_t* topk_ids, int T, int H, int k,
                               int E_total, int expert_begin, int expert_end, moe_bf16* expanded_x,
                               int32_t* expanded_row_idx, int32_t* sorted_row_idx,
                               int32_t* expert_offsets, int32_t* counts, void* ws,
                               size_t ws_bytes, moe_stream_t stream) {
  if (!topk_ids || !expanded_row_idx || !sorted_row_idx || !expert_offsets)
    return MOE_ERR_INVALID_ARG;
  if (expanded_x && (!x || !aligned16(x) || !aligned16(expanded_x))) return MOE_ERR_INVALID_ARG;
  const int El = expert_end - expert_begin;
  if (T < 1 || k < 1 || k > 32 || El < 1 || El > 256 || expert_begin < 0 ||
      expert_end > E_total || (long long)T * k >= (1LL << 31))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (expanded_x && (H < 8 || H % 8 != 0)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (ws == nullptr || ws_bytes < moe_init_routing_v2_workspace_size(T, El, k) ||
      (reinterpret_cast<uintptr_t>(ws) & 255u))
    return MOE_ERR_WORKSPACE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  const int P = T * k;
  int32_t* cnt = counts ? counts : at<int32_t>(ws, align256(moe::routing_ws_bytes(P, El)));
  MOE_CUDA(moe::launch_routing_range(topk_ids, P, expert_begin, El, E_total, cnt, expert_offsets,
                                     expanded_row_idx, sorted_row_idx, ws, nullptr, d->status,
                                     stream));
  if (expanded_x)
    MOE_CUDA(moe::launch_expand_rows(x, expanded_row_idx, sorted_row_idx, expert_offsets, El, T,
                                     H, k, expanded_x, stream));
  return MOE_OK;
}

size_t moe_re_routing_workspace_size(int R, int E_local) {
  if (R < 1 || E_local < 1) return 0;
  return align256(moe::reroute_ws_bytes(R, E_local));
}

moe_status moe_re_routing(const moe_bf16* x_recv, const int32_t* tokens_per_expert, int R,
                          int E_local, int N, int H, moe_bf16* x_out, int32_t* perm,
                          int32_t* expert_offsets, void* ws, size_t ws_bytes,
                          moe_stream_t stream) {
  if (!tokens_per_expert || !perm || !expert_offsets) return MOE_ERR_INVALID_ARG;
  if ((x_recv == nullptr) != (x_out == nullptr)) return MOE_ERR_INVALID_ARG;
  if (x_recv && (!aligned16(x_recv) || !aligned16(x_out))) return MOE_ERR_INVALID_ARG;
  if (R < 1 || E_local < 1 || (long long)R * E_local > (1 << 20) || N < 0 ||
      (x_recv && (H < 8 || H % 8 != 0)))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (ws == nullptr || ws_bytes < moe_re_routing_workspace_size(R, E_local) ||
      (reinterpret_cast<uintptr_t>(ws) & 255u))
    return MOE_ERR_WORKSPACE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  MOE_CUDA(moe::launch_re_routing(x_recv, tokens_per_expert, R, E_local, N, H, x_out, perm,
                                  expert_offsets, ws, stream));
  return MOE_OK;
}

moe_status moe_finalize_routing_v2(const moe_bf16* y2, const float* topk_w,
                                   const int32_t* expanded_row_idx, const int32_t* topk_ids,
                                   const moe_bf16* x_in, int T, int k, int H, int E, int E_total,
                                   moe_bf16* out, moe_stream_t stream) {
  if (!y2 || !topk_w || !expanded_row_idx || !topk_ids || !x_in || !out || !aligned16(y2) ||
      !aligned16(x_in) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  if (T < 1 || k < 1 || k > 32 || H < 8 || H % 8 != 0 || E < 0 || E_total < E)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  MOE_CUDA(moe::launch_finalize_v2(y2, topk_w, expanded_row_idx, topk_ids, x_in, T, k, H, E,
                                   E_total, out, stream));
  return MOE_OK;
}

namespace {

struct ForwardV2Layout {
  ForwardLayout base;
  size_t y32, ybf, total;
};

ForwardV2Layout forward_v2_layout(int T, int H, int E, int Z, int k, int I) {
  ForwardV2Layout L{};
  L.base = forward_layout(T, H, E, k, I);
  size_t o = L.base.total;
  // the router region of the base layout is sized for E gating columns, bf16 input;
  // append one sized for E+Z columns and either input kind
  const int Eg = E + Z;
  const size_t rbytes = std::max(moe::router_ws_bytes(T, H, Eg, false),
                                 moe::router_ws_bytes(T, H, Eg, true));
  L.base.router = o;
  o += align256(rbytes);
  L.y32 = o;
  o += align256((size_t)T * H * 4);
  L.ybf = o;
  o += align256((size_t)T * H * 2);
  L.total = o;
  return L;
}

}  // namespace

size_t moe_forward_v2_workspace_size(int T, int H, int E, int Z, int k, int I) {
  if (Z < 0 || E + Z > 256 || check_layer_shape(T, H, E + Z, k, I) != MOE_OK ||
      check_layer_shape(T, H, E, 1, I) != MOE_OK)
    return 0;
  return forward_v2_layout(T, H, E, Z, k, I).total;
}

moe_status moe_forward_v2(const moe_bf16* x, const moe_bf16* r, const moe_bf16* norm_w, float eps,
                          const float* Wg, const float* logits_override, const void* w13_packed,
                          const void* down_packed, int T, int H, int E, int Z, int k, int I,
                          moe_bf16* out, moe_bf16* residual_out, int32_t* topk_ids_out,
                          float* topk_w_out, void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!x || !w13_packed || !down_packed || !out) return MOE_ERR_INVALID_ARG;
  if (!logits_override && !Wg) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || (r && !aligned16(r)) || (norm_w && !aligned16(norm_w)) ||
      !aligned16(w13_packed) || !aligned16(down_packed) || !aligned16(out) ||
      (residual_out && !aligned16(residual_out)))
    return MOE_ERR_INVALID_ARG;
  if (Z < 0 || E + Z > 256) return MOE_ERR_UNSUPPORTED_SHAPE;
  MOE_TRY(check_layer_shape(T, H, E + Z, k, I));
  MOE_TRY(check_layer_shape(T, H, E, 1, I));
  if (norm_w && (H % 256 != 0 || H > 32768)) return MOE_ERR_UNSUPPORTED_SHAPE;
  const ForwardV2Layout LV = forward_v2_layout(T, H, E, Z, k, I);
  const ForwardLayout& L = LV.base;
  if (ws == nullptr || ws_bytes < LV.total || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return MOE_ERR_WORKSPACE;
  DeviceFacts* d = nullptr;
  MOE_TRY(current_device(&d));
  const int P = T * k;
  const int Eg = E + Z;
  int32_t* ids = topk_ids_out ? topk_ids_out : at<int32_t>(ws, L.ids);
  float* w = topk_w_out ? topk_w_out : at<float>(ws, L.w);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* eri = at<int32_t>(ws, L.eri);
  int32_t* sri = at<int32_t>(ws, L.sri);
  int* done = at<int>(ws, L.done);
  const moe_bf16* expert_in = x;
  const float* y32 = nullptr;
  if (norm_w) {
    float* y = at<float>(ws, LV.y32);
    uint16_t* ybf = at<uint16_t>(ws, LV.ybf);
    MOE_CUDA(moe::launch_add_rmsnorm_cast(x, r, norm_w, eps, T, H, residual_out, y, ybf, stream));
    y32 = y;
    expert_in = ybf;
  }
  const bool fused_routing = moe::routing_plan(P, E).single_cta;
  moe::GatingRouting fr{};
  fr.counter = at<int>(ws, L.counter);
  fr.counts = at<int32_t>(ws, L.counts);
  fr.offsets = offsets;
  fr.eri = eri;
  fr.sri = sri;
  fr.done = done;
  fr.E_routed = E;
  const moe::GatingRouting* fuse = fused_routing ? &fr : nullptr;
  if (logits_override) {
    if (fused_routing) MOE_CUDA(cudaMemsetAsync(fr.counter, 0, sizeof(int), stream));
    MOE_CUDA(moe::launch_gating(logits_override, 1, T, Eg, k, 1, ids, w, fuse, d->status, stream));
  } else {
    const bool f32in = y32 != nullptr;
    const moe::RouterPlan rp = moe::router_plan_ex(T, H, Eg, f32in);
    const size_t hint = decode_l2_hint_bytes(*d, moe_packed_weight_bytes(E, H, I, 0), 2u * H);
    float* part = at<float>(ws, L.router);
    int* zw = fused_routing ? fr.counter : nullptr;
    if (rp.tc) {
      void* extra = at<uint8_t>(ws, L.router + align256((size_t)rp.splits * T * Eg * 4));
      MOE_CUDA(moe::launch_router_tc(f32in ? static_cast<const void*>(y32) : x, f32in, false, Wg, T, H,
                                     Eg, rp, part, extra, zw, d->status, stream));
    } else if (f32in) {
      MOE_CUDA(moe::launch_router_f32(y32, Wg, T, H, Eg, rp, part, zw, stream, w13_packed,
                                      hint));
    } else {
      MOE_CUDA(moe::launch_router(x, Wg, T, H, Eg, rp, part, zw, stream, w13_packed, hint));
    }
    MOE_CUDA(moe::launch_gating(part, rp.splits, T, Eg, k, 1, ids, w, fuse, d->status, stream));
  }
  if (!fused_routing)
    MOE_CUDA(moe::launch_routing_range(ids, P, 0, E, Eg, fr.counts, offsets, eri, sri,
                                       at<void>(ws, L.routing), done, d->status, stream));
  uint16_t* xe = at<uint16_t>(ws, L.xe);
  uint16_t* h = at<uint16_t>(ws, L.h);
  uint16_t* y2 = at<uint16_t>(ws, L.y2);
  MOE_CUDA(moe::launch_expand_rows(expert_in, eri, sri, offsets, E, T, H, k, xe, stream));
  moe::GemmPhase g1{}, g2{};
  g1.A_weights = w13_packed;
  g1.B_act = xe;
  g1.out = h;
  g1.K = H;
  g1.MW = 2 * I;
  g1.n_out = I;
  g1.epi = 0;
  g2.A_weights = down_packed;
  g2.B_act = h;
  g2.out = y2;
  g2.K = I;
  g2.MW = H;
  g2.n_out = H;
  g2.epi = 1;
  if (t_gemm_ev_begin) MOE_CUDA(cudaEventRecord(t_gemm_ev_begin, stream));
  MOE_CUDA(moe::launch_grouped_gemm(&g1, &g2, offsets, E, P, T, done, d->status, stream));
  if (t_gemm_ev_end) MOE_CUDA(cudaEventRecord(t_gemm_ev_end, stream));
  MOE_CUDA(moe::launch_finalize_v2(y2, w, eri, ids, expert_in, T, k, H, E, Eg, out, stream));
  return MOE_OK;
}

moe_status moe_debug_set_pair_light(int mode) {
  if (mode < 0 || mode > 2) return MOE_ERR_INVALID_ARG;
  moe::set_pair_light(mode);
  return MOE_OK;
}

moe_status moe_debug_set_gemm_stall(int stage, long long wait_ns) {
  if (stage >= 0 && (wait_ns < 1000 || wait_ns > 2000000000LL)) return MOE_ERR_INVALID_ARG;
  moe::set_gemm_stall(stage, static_cast<unsigned long long>(wait_ns));
  return MOE_OK;
}

moe_status moe_set_gemm_events(void* ev_begin, void* ev_end) {
  if ((ev_begin == nullptr) != (ev_end == nullptr)) return MOE_ERR_INVALID_ARG;
  t_gemm_ev_begin = static_cast<cudaEvent_t>(ev_begin);
  t_gemm_ev_end = static_cast<cudaEvent_t>(ev_end);
  return MOE_OK;
}

}  // extern "C"
