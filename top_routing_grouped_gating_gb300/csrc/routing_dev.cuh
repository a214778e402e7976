// Device-side pieces of init_routing shared by the routing kernels and by the
// gating kernel's fused decode path (page "基于Atlas A3、950训练/推理集群的Qwen3-MoE
// 模型低时延推理性能优化实践", §高效排序和token路由): a block-wide exclusive scan
// over up to 256 experts, the stable in-order scatter of a range of pairs, and the
// whole one-CTA routing (histogram, scan, scatter) for small P.
#pragma once

#include "common.cuh"

namespace moe {
namespace {

constexpr int kMaxExperts = 256;

// Which ids this routing call sorts: local experts [begin, begin + E) out of ids
// [0, E_total).  Other valid ids (another rank's experts, zero-computation
// experts) are skipped without error; ids outside [0, E_total) are invalid.
struct RouteMap {
  int begin;
  int E;
  int E_total;
};

// >= 0: local expert; -2: skipped; -3: invalid id.
__device__ __forceinline__ int local_id(int id, const RouteMap& rm) {
  if (id < 0 || id >= rm.E_total) return -3;
  const int l = id - rm.begin;
  return (l >= 0 && l < rm.E) ? l : -2;
}

// Exclusive scan of one value per thread for threads [0, 256); every thread of
// the block must call it.  s_tmp: 8 ints.  Returns the exclusive prefix; *total
// receives the sum of all 256 values.
__device__ __forceinline__ int block_excl_scan_256(int v, int* s_tmp, int* total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int x = tid < kMaxExperts ? v : 0;
  int inc = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += y;
  }
  if (warp < 8 && lane == 31) s_tmp[warp] = inc;
  __syncthreads();
  int pre = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const int c = s_tmp[w];
    if (w < warp) pre += c;
    tot += c;
  }
  __syncthreads();
  *total = tot;
  return pre + inc - x;
}

// Scatter pairs [j_begin, j_end) in order.  s_base[e] = first free row of e for
// this range (advanced as rounds complete); s_wcnt = (warps x E) zeros.
__device__ __forceinline__ void scatter_range(const int32_t* __restrict__ ids, int j_begin, int j_end,
                                              const RouteMap& rm,
                              int* s_base, int* s_wcnt, int32_t* __restrict__ eri,
                              int32_t* __restrict__ sri) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int E = rm.E;
  for (int j0 = j_begin; j0 < j_end; j0 += blockDim.x) {
    const int j = j0 + tid;
    int e = -1;                       // -1: no pair in this slot
    if (j < j_end) {
      e = local_id(__ldcg(ids + j), rm);  // ids may come from other CTAs of this grid
      if (e < 0) e = -2;                  // not routed here: pair dropped
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) s_wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += s_wcnt[w * E + e];
      const int p = s_base[e] + before + rank;
      eri[j] = p;
      sri[p] = j;
    } else if (e == -2) {
      eri[j] = -1;
    }
    __syncthreads();
    for (int x = tid; x < E; x += blockDim.x) {
      int s = 0;
      for (int w = 0; w < nwarps; ++w) {
        s += s_wcnt[w * E + x];
        s_wcnt[w * E + x] = 0;
      }
      s_base[x] += s;
    }
    __syncthreads();
  }
}

// Shared memory of the one-CTA routing for a block of NWARPS warps.
template <int NWARPS>
struct RoutingSmem {
  int hist[kMaxExperts];
  int base[kMaxExperts];
  int tmp[8];
  int wcnt[NWARPS * kMaxExperts];
};

// Histogram, exclusive scan and stable scatter of all P pairs by one CTA
// (blockDim.x == 32 * NWARPS >= 256) for the local experts of rm.  zero_counter
// (rm.E + 1 ints, may be null) is cleared on the way.
template <int NWARPS>
__device__ __forceinline__ void routing_single_cta(const int32_t* __restrict__ ids, int P,
                                                   const RouteMap& rm,
                                                   int32_t* __restrict__ counts,
                                                   int32_t* __restrict__ offsets,
                                                   int32_t* __restrict__ eri,
                                                   int32_t* __restrict__ sri,
                                                   int* __restrict__ zero_counter, int* status,
                                                   RoutingSmem<NWARPS>& sm) {
  const int tid = threadIdx.x;
  const int E = rm.E;
  for (int i = tid; i < kMaxExperts; i += blockDim.x) sm.hist[i] = 0;
  for (int i = tid; i < NWARPS * E; i += blockDim.x) sm.wcnt[i] = 0;
  if (zero_counter != nullptr)
    for (int i = tid; i <= E; i += blockDim.x) zero_counter[i] = 0;
  __syncthreads();
  bool bad = false;
  for (int j = tid; j < P; j += blockDim.x) {
    const int e = local_id(__ldcg(ids + j), rm);
    if (e >= 0) atomicAdd(&sm.hist[e], 1);
    else if (e == -3) bad = true;
  }
  if (bad) flag_status(status, MOE_DEV_BAD_EXPERT_ID);
  __syncthreads();
  int total = 0;
  const int c = (tid < E) ? sm.hist[tid] : 0;
  const int off = block_excl_scan_256(c, sm.tmp, &total);
  if (tid < E) {
    sm.base[tid] = off;
    offsets[tid] = off;
    if (counts != nullptr) counts[tid] = c;
  }
  if (tid == 0) offsets[E] = total;
  __syncthreads();
  scatter_range(ids, 0, P, rm, sm.base, sm.wcnt, eri, sri);
}

}  // namespace
}  // namespace moe
