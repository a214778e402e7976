// Kernels of the "next" rows around the MoE layer:
//  - fused residual add + RMSNorm + cast with two outputs, fp32 for the router and
//    bf16 for the experts (page "基于Atlas A3、950训练/推理集群的Qwen3-MoE模型低时延
//    推理性能优化实践", §融合RMSNorm Cast);
//  - finalize with zero-computation experts, whose output is their input (page
//    "基于Atlas A3集群的LongCat-Flash模型推理性能优化实践", §MoE模块实现Expert Parallel:
//    copy_expert_num, MoE(ori_x) = ori_x);
//  - re-routing of tokens received by an expert-parallel AlltoAll, grouped by
//    source rank then local expert, into expert-major order (first page,
//    §计算分解 Double Routing方案, npu_moe_re_routing).
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

// One CTA per token row, 8 consecutive elements per thread and iteration.
__global__ void __launch_bounds__(256) add_rmsnorm_cast_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ r, const uint16_t* __restrict__ w,
    float eps, int H, uint16_t* __restrict__ residual_out, float* __restrict__ y32_out,
    uint16_t* __restrict__ ybf_out) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float srow[];
  __shared__ float s_red[8];
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t base = (size_t)t * H;
  float ss = 0.f;
  for (int c = tid * 8; c < H; c += 256 * 8) {
    const uint4 xv = *reinterpret_cast<const uint4*>(x + base + c);
    uint4 rv = make_uint4(0u, 0u, 0u, 0u);
    if (r != nullptr) rv = *reinterpret_cast<const uint4*>(r + base + c);
    const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w}, ra[4] = {rv.x, rv.y, rv.z, rv.w};
    float s[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s[2 * i] = bf16_lo(xa[i]) + bf16_lo(ra[i]);
      s[2 * i + 1] = bf16_hi(xa[i]) + bf16_hi(ra[i]);
    }
    if (residual_out != nullptr)
      *reinterpret_cast<uint4*>(residual_out + base + c) =
          make_uint4(pack_bf16x2(s[0], s[1]), pack_bf16x2(s[2], s[3]), pack_bf16x2(s[4], s[5]),
                     pack_bf16x2(s[6], s[7]));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      srow[c + i] = s[i];
      ss = fmaf(s[i], s[i], ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) s_red[warp] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) tot += s_red[i];
  const float rstd = rsqrtf(tot / static_cast<float>(H) + eps);
  for (int c = tid * 8; c < H; c += 256 * 8) {
    const uint4 wv = *reinterpret_cast<const uint4*>(w + c);
    const uint32_t wa[4] = {wv.x, wv.y, wv.z, wv.w};
    float y[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      y[2 * i] = srow[c + 2 * i] * rstd * bf16_lo(wa[i]);
      y[2 * i + 1] = srow[c + 2 * i + 1] * rstd * bf16_hi(wa[i]);
    }
    if (y32_out != nullptr) {
      float4* dst = reinterpret_cast<float4*>(y32_out + base + c);
      dst[0] = make_float4(y[0], y[1], y[2], y[3]);
      dst[1] = make_float4(y[4], y[5], y[6], y[7]);
    }
    *reinterpret_cast<uint4*>(ybf_out + base + c) =
        make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                   pack_bf16x2(y[6], y[7]));
  }
}

// out[t] = sum_s w[t,s] * (eri[j] >= 0 ? y2[eri[j]] : (ids[j] in [E, E_total) ? xin[t] : 0)),
// j = t*k + s, fp32 in slot order.  One CTA per token.
__global__ void __launch_bounds__(256) finalize_v2_kernel(const uint16_t* __restrict__ y2,
                                                          const float* __restrict__ w,
                                                          const int32_t* __restrict__ eri,
                                                          const int32_t* __restrict__ ids,
                                                          const uint16_t* __restrict__ xin,
                                                          int k, int H, int E, int E_total,
                                                          uint16_t* __restrict__ out) {
  __shared__ int s_row[32];
  __shared__ float s_w[32];
  __shared__ int s_copy[32];
  pdl_wait();
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    const size_t j = (size_t)t * k + threadIdx.x;
    s_row[threadIdx.x] = eri[j];
    s_w[threadIdx.x] = w[j];
    const int id = ids != nullptr ? ids[j] : -1;
    s_copy[threadIdx.x] = (id >= E && id < E_total) ? 1 : 0;
  }
  __syncthreads();
  for (int v = threadIdx.x; v < H / 8; v += blockDim.x) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    // eight slots' loads in flight at once, then the fp32 sum in slot order
    for (int s0 = 0; s0 < k; s0 += 8) {
      uint4 q[8];
      bool use[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int s = s0 + i;
        const int p = s < k ? s_row[s] : -1;
        const uint16_t* src = p >= 0 ? y2 + (size_t)p * H
                                     : ((s < k && s_copy[s]) ? xin + (size_t)t * H : nullptr);
        use[i] = src != nullptr;
        q[i] = use[i] ? reinterpret_cast<const uint4*>(src)[v] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (!use[i]) continue;
        const float ws = s_w[s0 + i];
        const uint32_t u[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[2 * j] = fmaf(ws, bf16_lo(u[j]), acc[2 * j]);
          acc[2 * j + 1] = fmaf(ws, bf16_hi(u[j]), acc[2 * j + 1]);
        }
      }
    }
    reinterpret_cast<uint4*>(out + (size_t)t * H)[v] =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                   pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
  }
}

// Re-routing tables (one CTA).  cnt[R][El] rows arrive rank-major; in_base[r*El+e]
// is the first received row of (r, e) and out_base[r*El+e] its first output row
// in expert-major order; offsets[e] = first output row of expert e.
__global__ void __launch_bounds__(256) reroute_tables_kernel(const int32_t* __restrict__ cnt, int R,
                                                             int El, int32_t* __restrict__ in_base,
                                                             int32_t* __restrict__ out_base,
                                                             int32_t* __restrict__ offsets) {
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int r = 0; r < R; ++r)
      for (int e = 0; e < El; ++e) {
        in_base[r * El + e] = acc;
        acc += cnt[r * El + e];
      }
    in_base[R * El] = acc;
    acc = 0;
    for (int e = 0; e < El; ++e) {
      offsets[e] = acc;
      for (int r = 0; r < R; ++r) {
        out_base[r * El + e] = acc;
        acc += cnt[r * El + e];
      }
    }
    offsets[El] = acc;
  }
}

// Received row i -> output row perm[i]; the row is copied.  One warp per row.
__global__ void __launch_bounds__(256) reroute_rows_kernel(const uint16_t* __restrict__ xin, int N,
                                                           int H, int RE,
                                                           const int32_t* __restrict__ in_base,
                                                           const int32_t* __restrict__ out_base,
                                                           uint16_t* __restrict__ xout,
                                                           int32_t* __restrict__ perm) {
  const int lane = threadIdx.x & 31;
  const int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (i >= N) return;
  int lo = 0, hi = RE;  // in_base[lo] <= i < in_base[hi]; empty segments skipped by the search
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (in_base[mid] <= i) lo = mid;
    else hi = mid;
  }
  const int o = out_base[lo] + (i - in_base[lo]);
  if (lane == 0) perm[i] = o;
  if (xin != nullptr) {
    const uint4* src = reinterpret_cast<const uint4*>(xin + (size_t)i * H);
    uint4* dst = reinterpret_cast<uint4*>(xout + (size_t)o * H);
    for (int v = lane; v < H / 8; v += 32) dst[v] = src[v];
  }
}

}  // namespace

cudaError_t launch_add_rmsnorm_cast(const uint16_t* x, const uint16_t* r, const uint16_t* w,
                                    float eps, int T, int H, uint16_t* residual_out,
                                    float* y32_out, uint16_t* ybf_out, cudaStream_t s) {
  const size_t smem = (size_t)H * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(add_rmsnorm_cast_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(add_rmsnorm_cast_kernel, dim3(T), dim3(256), smem, s, x, r, w, eps, H,
                    residual_out, y32_out, ybf_out);
}

cudaError_t launch_finalize_v2(const uint16_t* y2, const float* w, const int32_t* eri,
                               const int32_t* ids, const uint16_t* xin, int T, int k, int H, int E,
                               int E_total, uint16_t* out, cudaStream_t s) {
  const int threads = (H / 8) >= 256 ? 256 : ((H / 8 + 31) / 32) * 32;
  return launch_pdl(finalize_v2_kernel, dim3(T), dim3(threads), 0, s, y2, w, eri, ids, xin, k, H,
                    E, E_total, out);
}

size_t reroute_ws_bytes(int R, int El) {
  return ((size_t)2 * R * El + 1) * sizeof(int32_t);
}

cudaError_t launch_re_routing(const uint16_t* xin, const int32_t* cnt, int R, int El, int N, int H,
                              uint16_t* xout, int32_t* perm, int32_t* offsets, void* ws,
                              cudaStream_t s) {
  int32_t* in_base = static_cast<int32_t*>(ws);
  int32_t* out_base = in_base + R * El + 1;
  reroute_tables_kernel<<<1, 32, 0, s>>>(cnt, R, El, in_base, out_base, offsets);
  if (N > 0)
    reroute_rows_kernel<<<(N + 7) / 8, 256, 0, s>>>(xin, N, H, R * El, in_base, out_base, xout,
                                                     perm);
  return cudaGetLastError();
}

}  // namespace moe
