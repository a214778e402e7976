// Router scores and top-k softmax gating.
//
// Router: logits = x (T,H bf16) . Wg (H,E fp32) on CUDA cores in fp32 FMA -- the
// page "基于Atlas A3、950训练/推理集群的Qwen3-MoE模型低时延推理性能优化实践"
// (§融合RMSNorm Cast) keeps the gate computation in FP32.  Tiles of 32 tokens x
// 128 experts; the H axis is split across CTAs when there are few tiles (decode),
// and the partial sums are added later in a fixed order, so results are
// bit-reproducible.
//
// Gating (§快速选择专家): one warp per token.  Lane l holds experts l, l+32, ...;
// k rounds of a warp-wide arg-max under (logit desc, expert id asc) pick the
// slots; weights are softmax over the chosen logits (renormalised) or the
// full-softmax probabilities.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "routing_dev.cuh"

namespace moe {

namespace {

constexpr int kRT = 32;    // tokens per router tile
constexpr int kRE = 128;   // experts per router tile
constexpr int kRK = 32;    // H rows per smem step

template <typename XT>
__global__ void __launch_bounds__(256) router_kernel(const XT* __restrict__ x,
                                                     const float* __restrict__ Wg, int T, int H,
                                                     int E, int h_per_split,
                                                     float* __restrict__ out, int* zero_word) {
  __shared__ float xs[kRT][kRK + 1];
  pdl_wait();
  pdl_trigger();
  if (zero_word != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 &&
      threadIdx.x == 0)
    *zero_word = 0;
  __shared__ float ws[kRK][kRE];
  const int tid = threadIdx.x;
  const int tx = tid & 31;          // experts e0 + tx + 32*i
  const int ty = tid >> 5;          // tokens t0 + 4*ty + j
  const int t0 = blockIdx.x * kRT;
  const int e0 = blockIdx.y * kRE;
  const int split = blockIdx.z;
  const int hb = split * h_per_split;
  float acc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;

  for (int h0 = hb; h0 < hb + h_per_split; h0 += kRK) {
    {  // x tile: 32 tokens x 32 h (bf16 -> fp32); 4 elements per thread
      const int tt = tid >> 3, hh = (tid & 7) * 4;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (t0 + tt < T) {
        if constexpr (sizeof(XT) == 4) {
          const float4 f = *reinterpret_cast<const float4*>(x + (size_t)(t0 + tt) * H + h0 + hh);
          v[0] = f.x;
          v[1] = f.y;
          v[2] = f.z;
          v[3] = f.w;
        } else {
          const uint2 raw = *reinterpret_cast<const uint2*>(x + (size_t)(t0 + tt) * H + h0 + hh);
          v[0] = bf16_lo(raw.x);
          v[1] = bf16_hi(raw.x);
          v[2] = bf16_lo(raw.y);
          v[3] = bf16_hi(raw.y);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) xs[tt][hh + q] = v[q];
    }
#pragma unroll
    for (int r = 0; r < (kRK * kRE) / 256; ++r) {  // Wg tile: 32 h x 128 experts
      const int idx = tid + 256 * r;
      const int hh = idx / kRE, ee = idx % kRE;
      ws[hh][ee] = (e0 + ee < E) ? Wg[(size_t)(h0 + hh) * E + e0 + ee] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kRK; ++kk) {
      float xv[4], wv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) xv[j] = xs[4 * ty + j][kk];
#pragma unroll
      for (int i = 0; i < 4; ++i) wv[i] = ws[kk][tx + 32 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[j][i] = fmaf(xv[j], wv[i], acc[j][i]);
    }
    __syncthreads();
  }
  float* dst = out + (size_t)split * T * E;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int t = t0 + 4 * ty + j;
    if (t >= T) continue;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = e0 + tx + 32 * i;
      if (e < E) dst[(size_t)t * E + e] = acc[j][i];
    }
  }
}

// Decode-size router: tiles of 32 tokens x 32 experts over a 128-row slice of H,
// the whole slice loaded into shared memory before any arithmetic, so each CTA
// pays one round of load latency.  Partial sums go to partial[split][T][E].
constexpr int kSmallRows = 128;
constexpr int kSmallExp = 32;
constexpr uint32_t kPrefetchChunk = 32768;

template <typename XT>
__global__ void __launch_bounds__(256) router_small_kernel(const XT* __restrict__ x,
                                                           const float* __restrict__ Wg, int T,
                                                           int H, int E,
                                                           float* __restrict__ partial,
                                                           int* zero_word, const uint8_t* l2_hint,
                                                           size_t l2_hint_chunks) {
  __shared__ float ws[kSmallRows][kSmallExp];
  pdl_wait();
  pdl_trigger();
  if (zero_word != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 &&
      threadIdx.x == 0)
    *zero_word = 0;
  __shared__ float xs[kRT][kSmallRows + 1];
  const int tid = threadIdx.x;
  const int tx = tid & 31;          // expert e0 + tx
  const int ty = tid >> 5;          // tokens t0 + 4*ty + j
  const int e0 = blockIdx.x * kSmallExp;
  const int split = blockIdx.y;
  const int t0 = blockIdx.z * kRT;
  const int hb = split * kSmallRows;
#pragma unroll
  for (int r = 0; r < (kSmallRows * kSmallExp) / 256; ++r) {
    const int idx = tid + 256 * r;
    const int hh = idx >> 5, ee = idx & 31;
    ws[hh][ee] = (e0 + ee < E) ? Wg[(size_t)(hb + hh) * E + e0 + ee] : 0.f;
  }
  if constexpr (sizeof(XT) == 4) {
#pragma unroll
    for (int r = 0; r < (kRT * kSmallRows) / (256 * 4); ++r) {
      const int idx = tid + 256 * r;
      const int tt = idx >> 5, h4 = (idx & 31) * 4;
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t0 + tt < T) f = *reinterpret_cast<const float4*>(x + (size_t)(t0 + tt) * H + hb + h4);
      xs[tt][h4] = f.x;
      xs[tt][h4 + 1] = f.y;
      xs[tt][h4 + 2] = f.z;
      xs[tt][h4 + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int r = 0; r < (kRT * kSmallRows) / (256 * 8); ++r) {
      const int idx = tid + 256 * r;
      const int tt = idx >> 4, h8 = (idx & 15) * 8;
      uint4 raw = make_uint4(0u, 0u, 0u, 0u);
      if (t0 + tt < T) raw = *reinterpret_cast<const uint4*>(x + (size_t)(t0 + tt) * H + hb + h8);
      const uint32_t u[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        xs[tt][h8 + 2 * q] = bf16_lo(u[q]);
        xs[tt][h8 + 2 * q + 1] = bf16_hi(u[q]);
      }
    }
  }
  __syncthreads();
  if (l2_hint_chunks != 0 && threadIdx.x < 32) {
    // Weight prefetch into L2 (page "基于Atlas A3集群的LongCat-Flash模型推理性能优化
    // 实践", §权重预取).  Issued after this CTA's own loads have landed, so they do
    // not queue behind the hint.  Chunk c goes to lane c / nblk of CTA c % nblk: the front of the
    // range (read first) is requested first.
    const size_t nblk = (size_t)gridDim.x * gridDim.y * gridDim.z;
    const size_t b = blockIdx.x + (size_t)gridDim.x * (blockIdx.y + (size_t)gridDim.y * blockIdx.z);
    for (size_t c = b + nblk * threadIdx.x; c < l2_hint_chunks; c += nblk * 32)
      prefetch_l2_bulk(l2_hint + c * kPrefetchChunk, kPrefetchChunk);
  }
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
  for (int h = 0; h < kSmallRows; ++h) {
    const float wv = ws[h][tx];
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = fmaf(xs[4 * ty + j][h], wv, acc[j]);
  }
  const int e = e0 + tx;
  if (e < E) {
    float* dst = partial + (size_t)split * T * E;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int t = t0 + 4 * ty + j;
      if (t < T) dst[(size_t)t * E + e] = acc[j];
    }
  }
}

__global__ void router_reduce_kernel(const float* __restrict__ partial, int splits, size_t n,
                                     float* __restrict__ out) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    float s = partial[i];
    for (int p = 1; p < splits; ++p) s += partial[(size_t)p * n + i];
    out[i] = s;
  }
}

// (a beats b) under logit descending, expert id ascending.
__device__ __forceinline__ bool beats(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__device__ __forceinline__ void gating_token(const float* __restrict__ src, int splits, int t,
                                             int T, int E, int k, int renormalize,
                                             int32_t* __restrict__ ids, float* __restrict__ w,
                                             int lane) {
  const size_t n = (size_t)T * E;
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = (lane + 32 * i < E) ? 0.f : -INFINITY;
  // sum the split-K partials in split order; independent loads kept in flight
#pragma unroll 4
  for (int p = 0; p < splits; ++p) {
    const float* row = src + (size_t)p * n + (size_t)t * E;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (lane + 32 * i < E) v[i] += __ldcg(row + lane + 32 * i);
  }
  uint32_t taken = 0;
  float my_v = -INFINITY;
  int my_i = 0;
  for (int s = 0; s < k; ++s) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && beats(v[i], e, bv, bi)) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (beats(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == s) {
      my_v = bv;
      my_i = bi;
    }
  }
  const float m = __shfl_sync(0xffffffffu, my_v, 0);  // slot 0 holds the maximum
  float num = (lane < k) ? expf(my_v - m) : 0.f;
  float den;
  if (renormalize) {
    den = num;
  } else {
    den = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (lane + 32 * i < E) den += expf(v[i] - m);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  if (lane < k) {
    ids[(size_t)t * k + lane] = my_i;
    w[(size_t)t * k + lane] = num / den;
  }
}

__global__ void __launch_bounds__(256) gating_kernel(const float* __restrict__ src, int splits,
                                                     int T, int E, int k, int renormalize,
                                                     int32_t* __restrict__ ids,
                                                     float* __restrict__ w, GatingRouting fuse,
                                                     int* status) {
  __shared__ RoutingSmem<8> rsm;
  __shared__ int s_last;
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t < T) {
    gating_token(src, splits, t, T, E, k, renormalize, ids, w, lane);
  }
  if (fuse.counter == nullptr) return;
  // Fused init_routing: the last CTA to finish its tokens routes all P pairs.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(fuse.counter, 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const RouteMap rm{0, fuse.E_routed > 0 ? fuse.E_routed : E, E};
  routing_single_cta(ids, T * k, rm, fuse.counts, fuse.offsets, fuse.eri, fuse.sri, fuse.done,
                     status, rsm);
  if (threadIdx.x == 0) *fuse.counter = 0;  // ready for the next call
}

}  // namespace

RouterPlan router_plan(int T, int H, int E) {
  RouterPlan p;
  p.t_tiles = (T + kRT - 1) / kRT;
  p.small = (p.t_tiles <= 2 && H % kSmallRows == 0);
  if (p.small) {
    p.e_tiles = (E + kSmallExp - 1) / kSmallExp;
    p.splits = H / kSmallRows;
    return p;
  }
  p.e_tiles = (E + kRE - 1) / kRE;
  const int tiles = p.t_tiles * p.e_tiles;
  int s = 1;
  // split H until there are ~128 CTAs, keeping each split a multiple of kRK rows
  while (s < 16 && tiles * s * 2 <= 128 && (H / kRK) % (s * 2) == 0) s *= 2;
  p.splits = s;
  return p;
}

template <typename XT>
cudaError_t launch_router_t(const XT* x, const float* Wg, int T, int H, int E,
                            const RouterPlan& plan, float* out, int* zero_word, cudaStream_t s,
                            const void* l2_hint = nullptr, size_t l2_hint_bytes = 0) {
  if (plan.small) {
    dim3 grid(plan.e_tiles, plan.splits, plan.t_tiles);
    const size_t chunks = l2_hint != nullptr ? l2_hint_bytes / kPrefetchChunk : 0;
    return launch_pdl(router_small_kernel<XT>, grid, dim3(256), 0, s, x, Wg, T, H, E, out,
                      zero_word, static_cast<const uint8_t*>(l2_hint), chunks);
  }
  dim3 grid(plan.t_tiles, plan.e_tiles, plan.splits);
  return launch_pdl(router_kernel<XT>, grid, dim3(256), 0, s, x, Wg, T, H, E, H / plan.splits,
                    out, zero_word);
}

cudaError_t launch_router(const uint16_t* x, const float* Wg, int T, int H, int E,
                          const RouterPlan& plan, float* out, int* zero_word, cudaStream_t s,
                          const void* l2_hint, size_t l2_hint_bytes) {
  return launch_router_t(x, Wg, T, H, E, plan, out, zero_word, s, l2_hint, l2_hint_bytes);
}

cudaError_t launch_router_f32(const float* x, const float* Wg, int T, int H, int E,
                              const RouterPlan& plan, float* out, int* zero_word, cudaStream_t s,
                              const void* l2_hint, size_t l2_hint_bytes) {
  return launch_router_t(x, Wg, T, H, E, plan, out, zero_word, s, l2_hint, l2_hint_bytes);
}

cudaError_t launch_router_reduce(const float* partial, int splits, int T, int E, float* logits,
                                 cudaStream_t s) {
  const size_t n = (size_t)T * E;
  const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  router_reduce_kernel<<<blocks, 256, 0, s>>>(partial, splits, n, logits);
  return cudaGetLastError();
}

cudaError_t launch_gating(const float* src, int splits, int T, int E, int k, int renormalize,
                          int32_t* ids, float* w, const GatingRouting* fuse, int* status,
                          cudaStream_t s) {
  const int blocks = (T + 7) / 8;
  GatingRouting f{};
  if (fuse != nullptr) f = *fuse;
  return launch_pdl(gating_kernel, dim3(blocks), dim3(256), 0, s, src, splits, T, E, k,
                    renormalize, ids, w, f, status);
}

}  // namespace moe
