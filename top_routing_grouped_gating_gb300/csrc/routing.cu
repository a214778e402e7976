// init_routing, compute_expert_tokens and finalize_routing
// (page "基于Atlas A3、950训练/推理集群的Qwen3-MoE模型低时延推理性能优化实践",
// §高效排序和token路由).
//
// init_routing is a stable counting sort of the P = T*k token-expert pairs by
// expert id.  Pairs are taken in chunks of consecutive j; a chunk's rows for
// expert e start at offsets[e] + (pairs of e in earlier chunks).  Inside a chunk,
// pairs are ranked in rounds of blockDim consecutive j: __match_any_sync gives
// the rank among equal ids inside a warp, and per-warp counts in shared memory
// give the rank across the round's warps.  Every position is therefore the
// unique stable one and the result is deterministic.
//
// Small P (decode) runs histogram, scan and scatter in one CTA; large P uses a
// per-chunk histogram kernel, a one-CTA scan and a per-chunk scatter kernel.
#include "common.cuh"
#include "internal.h"
#include "routing_dev.cuh"

namespace moe {

namespace {

constexpr int kRouteThreads = 1024;
constexpr int kSingleCtaMaxPairs = 4096;
constexpr int kChunkPairs = 2048;

__global__ void __launch_bounds__(kRouteThreads) routing_single_cta_kernel(
    const int32_t* __restrict__ ids, int P, RouteMap rm, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ eri, int32_t* __restrict__ sri,
    int* __restrict__ zero_counter, int* status) {
  __shared__ RoutingSmem<kRouteThreads / 32> sm;
  routing_single_cta(ids, P, rm, counts, offsets, eri, sri, zero_counter, status, sm);
}

__global__ void __launch_bounds__(kRouteThreads) routing_hist_kernel(
    const int32_t* __restrict__ ids, int P, RouteMap rm, int chunk_pairs,
    int32_t* __restrict__ chunk_hist, int* status) {
  __shared__ int s_hist[kMaxExperts];
  const int tid = threadIdx.x;
  const int E = rm.E;
  for (int i = tid; i < E; i += blockDim.x) s_hist[i] = 0;
  __syncthreads();
  const int j0 = blockIdx.x * chunk_pairs;
  const int j1 = min(P, j0 + chunk_pairs);
  bool bad = false;
  for (int j = j0 + tid; j < j1; j += blockDim.x) {
    const int e = local_id(ids[j], rm);
    if (e >= 0) atomicAdd(&s_hist[e], 1);
    else if (e == -3) bad = true;
  }
  if (bad) flag_status(status, MOE_DEV_BAD_EXPERT_ID);
  __syncthreads();
  for (int i = tid; i < E; i += blockDim.x) chunk_hist[(size_t)blockIdx.x * E + i] = s_hist[i];
}

// chunk_hist[c][e] (counts) -> chunk_hist[c][e] (first row of e for chunk c).  Thread
// e walks the chunks in groups of eight, loading a group before storing any of it, so
// eight loads are in flight instead of one L2 round trip per chunk.
__global__ void __launch_bounds__(256) routing_scan_kernel(int32_t* __restrict__ chunk_hist,
                                                           int chunks, int E,
                                                           int32_t* __restrict__ counts,
                                                           int32_t* __restrict__ offsets,
                                                           int* __restrict__ zero_counter) {
  __shared__ int s_tmp[8];
  const int e = threadIdx.x;
  int run = 0;
  if (e < E) {
    for (int c0 = 0; c0 < chunks; c0 += 8) {
      int h[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) h[i] = c0 + i < chunks ? chunk_hist[(size_t)(c0 + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) run += h[i];
    }
  }
  int total = 0;
  const int off = block_excl_scan_256(e < E ? run : 0, s_tmp, &total);
  if (e < E) {
    if (counts != nullptr) counts[e] = run;
    offsets[e] = off;
    if (zero_counter != nullptr) zero_counter[e] = 0;
    if (zero_counter != nullptr && e == 0) zero_counter[E] = 0;
    int base = off;
    for (int c0 = 0; c0 < chunks; c0 += 8) {
      int h[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) h[i] = c0 + i < chunks ? chunk_hist[(size_t)(c0 + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (c0 + i < chunks) chunk_hist[(size_t)(c0 + i) * E + e] = base;
        base += h[i];
      }
    }
  }
  if (e == 0) offsets[E] = total;
}

__global__ void __launch_bounds__(kRouteThreads) routing_scatter_kernel(
    const int32_t* __restrict__ ids, int P, RouteMap rm, int chunk_pairs,
    const int32_t* __restrict__ chunk_base, int32_t* __restrict__ eri, int32_t* __restrict__ sri) {
  __shared__ int s_base[kMaxExperts];
  __shared__ int s_wcnt[(kRouteThreads / 32) * kMaxExperts];
  const int tid = threadIdx.x;
  const int E = rm.E;
  for (int i = tid; i < E; i += blockDim.x) s_base[i] = chunk_base[(size_t)blockIdx.x * E + i];
  for (int i = tid; i < (kRouteThreads / 32) * E; i += blockDim.x) s_wcnt[i] = 0;
  __syncthreads();
  const int j0 = blockIdx.x * chunk_pairs;
  scatter_range(ids, j0, min(P, j0 + chunk_pairs), rm, s_base, s_wcnt, eri, sri);
}

// expanded_x[p] = x[sri[p] / k] for p < offsets[E]; one warp per row, 16-byte copies.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ sri,
                                                          const int32_t* __restrict__ offsets,
                                                          int E, int P, int H, int k,
                                                          uint16_t* __restrict__ xe) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int p = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (p >= P || p >= offsets[E]) return;
  const int t = sri[p] / k;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  uint4* dst = reinterpret_cast<uint4*>(xe + (size_t)p * H);
  const int nv = H / 8;
  int v = lane;
  for (; v + 96 < nv; v += 128) {  // four independent 16-byte loads in flight per lane
    const uint4 a = src[v], b = src[v + 32], c = src[v + 64], d = src[v + 96];
    dst[v] = a;
    dst[v + 32] = b;
    dst[v + 64] = c;
    dst[v + 96] = d;
  }
  for (; v < nv; v += 32) dst[v] = src[v];
}

// expanded_x[eri[t * k + j]] = x[t] for every pair with eri >= 0: the same rows as
// the gather above, but each token row is read once, in row order.  (Gathering by
// sorted row reads each token row k times, far apart in time; at prefill sizes the
// expanded rows streaming through L2 evict x in between.)  One warp per token and
// 2 KB column chunk of its row: each lane loads four 16-byte pieces, then stores them
// to each of the token's expanded rows.
__global__ void __launch_bounds__(256) scatter_rows_kernel(const uint16_t* __restrict__ x,
                                                           const int32_t* __restrict__ eri, int T,
                                                           int k, int H,
                                                           uint16_t* __restrict__ xe) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nv = H / 8;                       // 16-byte pieces per row
  const int chunks = (nv + 127) / 128;
  const long long t = w / chunks;
  if (t >= T) return;
  const int v0 = static_cast<int>(w - t * chunks) * 128 + lane;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  uint4 a[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (v0 + 32 * i < nv) a[i] = src[v0 + 32 * i];
  const int my_p = lane < k ? eri[(size_t)t * k + lane] : -1;
  for (int j = 0; j < k; ++j) {
    const int p = __shfl_sync(0xffffffffu, my_p, j);
    if (p < 0) continue;
    uint4* dst = reinterpret_cast<uint4*>(xe + (size_t)p * H);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (v0 + 32 * i < nv) dst[v0 + 32 * i] = a[i];
  }
}

__global__ void __launch_bounds__(kRouteThreads) expert_tokens_kernel(
    const int32_t* __restrict__ ids, int P, int E, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int* status) {
  __shared__ int s_hist[kMaxExperts];
  __shared__ int s_tmp[8];
  const int tid = threadIdx.x;
  for (int i = tid; i < kMaxExperts; i += blockDim.x) s_hist[i] = 0;
  __syncthreads();
  bool bad = false;
  for (int j = tid; j < P; j += blockDim.x) {
    const int e = ids[j];
    if (e >= 0 && e < E) atomicAdd(&s_hist[e], 1);
    else bad = true;
  }
  if (bad) flag_status(status, MOE_DEV_BAD_EXPERT_ID);
  __syncthreads();
  int total = 0;
  const int c = (tid < E) ? s_hist[tid] : 0;
  const int off = block_excl_scan_256(c, s_tmp, &total);
  if (tid < E) {
    counts[tid] = c;
    if (offsets != nullptr) offsets[tid] = off;
  }
  if (tid == 0 && offsets != nullptr) offsets[E] = total;
}

// out[t] = sum_s w[t,s] * y2[eri[t*k+s]] in fp32, slot order; one CTA per token and
// chunk of blockDim.x * 8 columns (gridDim.y chunks).
__global__ void __launch_bounds__(256) finalize_kernel(const uint16_t* __restrict__ y2,
                                                       const float* __restrict__ w,
                                                       const int32_t* __restrict__ eri, int k,
                                                       int H, uint16_t* __restrict__ out) {
  __shared__ int s_row[32];
  __shared__ float s_w[32];
  pdl_wait();
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    s_row[threadIdx.x] = eri[(size_t)t * k + threadIdx.x];
    s_w[threadIdx.x] = w[(size_t)t * k + threadIdx.x];
  }
  __syncthreads();
  for (int v = blockIdx.y * blockDim.x + threadIdx.x; v < H / 8; v += gridDim.y * blockDim.x) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    // eight slots' loads in flight at once, then the fp32 sum in slot order
    for (int s0 = 0; s0 < k; s0 += 8) {
      uint4 q[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int p = s0 + i < k ? s_row[s0 + i] : -1;
        q[i] = p >= 0 ? reinterpret_cast<const uint4*>(y2 + (size_t)p * H)[v] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (s0 + i >= k || s_row[s0 + i] < 0) continue;
        const float ws = s_w[s0 + i];
        const uint32_t u[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[2 * j] = fmaf(ws, bf16_lo(u[j]), acc[2 * j]);
          acc[2 * j + 1] = fmaf(ws, bf16_hi(u[j]), acc[2 * j + 1]);
        }
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(out + (size_t)t * H)[v] = o;
  }
}

}  // namespace

RoutingPlan routing_plan(int P, int E) {
  (void)E;
  RoutingPlan r;
  r.single_cta = P <= kSingleCtaMaxPairs;
  r.chunk_pairs = kChunkPairs;
  r.chunks = r.single_cta ? 1 : (P + kChunkPairs - 1) / kChunkPairs;
  return r;
}

size_t routing_ws_bytes(int P, int E) {
  const RoutingPlan r = routing_plan(P, E);
  return r.single_cta ? 0 : (size_t)r.chunks * E * sizeof(int32_t);
}

cudaError_t launch_routing(const int32_t* ids, int P, int E, int32_t* counts, int32_t* offsets,
                           int32_t* eri, int32_t* sri, void* ws, int* zero_counter, int* status,
                           cudaStream_t s) {
  return launch_routing_range(ids, P, 0, E, E, counts, offsets, eri, sri, ws, zero_counter, status,
                              s);
}

cudaError_t launch_routing_range(const int32_t* ids, int P, int e_begin, int E, int E_total,
                                 int32_t* counts, int32_t* offsets, int32_t* eri, int32_t* sri,
                                 void* ws, int* zero_counter, int* status, cudaStream_t s) {
  const RoutingPlan r = routing_plan(P, E);
  const RouteMap rm{e_begin, E, E_total};
  if (r.single_cta) {
    routing_single_cta_kernel<<<1, kRouteThreads, 0, s>>>(ids, P, rm, counts, offsets, eri, sri,
                                                          zero_counter, status);
    return cudaGetLastError();
  }
  int32_t* chunk_hist = static_cast<int32_t*>(ws);
  routing_hist_kernel<<<r.chunks, kRouteThreads, 0, s>>>(ids, P, rm, r.chunk_pairs, chunk_hist,
                                                         status);
  routing_scan_kernel<<<1, 256, 0, s>>>(chunk_hist, r.chunks, E, counts, offsets, zero_counter);
  routing_scatter_kernel<<<r.chunks, kRouteThreads, 0, s>>>(ids, P, rm, r.chunk_pairs, chunk_hist,
                                                            eri, sri);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* sri, const int32_t* offsets,
                               int E, int P, int H, int k, uint16_t* xe, cudaStream_t s) {
  const int blocks = (P + 7) / 8;
  return launch_pdl(gather_rows_kernel, dim3(blocks), dim3(256), 0, s, x, sri, offsets, E, P, H, k,
                    xe);
}

cudaError_t launch_expand_rows(const uint16_t* x, const int32_t* eri, const int32_t* sri,
                               const int32_t* offsets, int E, int T, int H, int k, uint16_t* xe,
                               cudaStream_t s) {
  if (T < kScatterMinTokens) return launch_gather_rows(x, sri, offsets, E, T * k, H, k, xe, s);
  const long long warps = (long long)T * ((H / 8 + 127) / 128);
  const unsigned blocks = static_cast<unsigned>((warps + 7) / 8);
  return launch_pdl(scatter_rows_kernel, dim3(blocks), dim3(256), 0, s, x, eri, T, k, H, xe);
}

cudaError_t launch_expert_tokens(const int32_t* ids, int P, int E, int32_t* counts,
                                 int32_t* offsets, int* status, cudaStream_t s) {
  expert_tokens_kernel<<<1, kRouteThreads, 0, s>>>(ids, P, E, counts, offsets, status);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const uint16_t* y2, const float* w, const int32_t* eri, int T, int k,
                            int H, uint16_t* out, cudaStream_t s) {
  // one CTA per token; with few tokens, each token's columns are spread over several
  // CTAs (about two per SM in all), so more SMs have the slot rows' loads in flight
  const int groups = H / 8;
  int threads = groups >= 256 ? 256 : ((groups + 31) / 32) * 32;
  int ysplit = 1;
  const int want = 2 * device_sm_count();
  if (T < want) {
    const int max_split = (groups + 127) / 128;   // at least 128 threads per CTA
    ysplit = (want + T - 1) / T < max_split ? (want + T - 1) / T : max_split;
    threads = ((groups + ysplit - 1) / ysplit + 31) / 32 * 32;
    ysplit = (groups + threads - 1) / threads;
  }
  return launch_pdl(finalize_kernel, dim3(T, ysplit), dim3(threads), 0, s, y2, w, eri, k, H, out);
}

}  // namespace moe
