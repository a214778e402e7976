// MXFP8 kernels: fused residual add + RMSNorm + dynamic MX quantisation, the
// standalone dynamic MX quantiser, MX pre-quantisation of the expert weights, and
// the expert-sorted expansion of quantised activations.
//
// Page "基于Atlas A3、950训练/推理集群的Qwen3-MoE模型低时延推理性能优化实践":
// §融合RMSNorm MX量化 fuses the residual add, RMSNorm and MXFP8 dynamic quantisation
// (round mode "rint", data type float8_e4m3fn) into one op; §融合RMSNorm Cast feeds
// the router with the fp32 normalised activations; §计算分解(AllGather方案) quantises
// hidden states with npu_dynamic_mx_quant.
//
// MX format (OCP Microscaling v1.0): blocks of 32 consecutive elements along the
// reduction axis share one E8M0 scale 2^X, X = floor(log2(max|v|)) - 8 (8 = the
// exponent of e4m3's largest normal), clamped to [-127, 127]; an all-zero block
// gets X = -127.  Elements are e4m3(v / 2^X), round to nearest even, saturating
// at +-448.  Scale byte = X + 127.
//
// Scale layout for the tensor core ("atoms").  A block-scaled MMA reads the scales
// of 128 rows x 4 blocks (one 128-element K step of fp8) from a 512-byte atom:
// byte (r % 32) * 16 + (r / 32) * 4 + kb holds the scale of row r, block kb.
// Weight scales are stored as atoms per (expert, 128-row block, K step); the
// expert-sorted activations are padded so every expert starts on a 128-row
// boundary and their scales are atoms per (128-row group, K step).
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"
#include "routing_dev.cuh"

namespace moe {

namespace {

MOE_DEVINL int mx_exponent(float amax) {
  const uint32_t bits = __float_as_uint(amax);
  const int ef = static_cast<int>((bits >> 23) & 0xFF);
  if (ef == 0) return -127;                // zero or subnormal block maximum
  int X = ef - 127 - 8;
  return X < -127 ? -127 : (X > 127 ? 127 : X);
}

MOE_DEVINL float exp2i(int e) {  // 2^e for e in [-126, 127]
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

MOE_DEVINL uint8_t to_e4m3(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// Quantise one value given its block's exponent X (v * 2^-X is exact).
MOE_DEVINL uint8_t mx_code(float v, int X) {
  // 2^-X can be 2^127 (X = -127): split in two exact power-of-two factors
  const int nx = -X;
  const int a = nx > 126 ? 126 : nx;
  return to_e4m3(v * exp2i(a) * exp2i(nx - a));
}

MOE_DEVINL int atom_offset(int row, int kb) { return (row & 31) * 16 + ((row >> 5) & 3) * 4 + kb; }

// ---------------------------------------------------------------------------
// One CTA per token row; 256 threads, 8 consecutive elements per thread and
// iteration, so an MX block of 32 spans 4 adjacent lanes.
__global__ void __launch_bounds__(256) add_rmsnorm_mxquant_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ r, const uint16_t* __restrict__ w,
    float eps, int H, uint16_t* __restrict__ residual_out, float* __restrict__ y32_out,
    uint16_t* __restrict__ ys_out, uint8_t* __restrict__ q, uint8_t* __restrict__ scale) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float srow[];  // H floats: s = x + r
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
    uint4 o;
    o.x = pack_bf16x2(s[0], s[1]);
    o.y = pack_bf16x2(s[2], s[3]);
    o.z = pack_bf16x2(s[4], s[5]);
    o.w = pack_bf16x2(s[6], s[7]);
    if (residual_out != nullptr) *reinterpret_cast<uint4*>(residual_out + base + c) = o;
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
    if (ys_out != nullptr) store_split3_x8(y, ys_out + 3 * base + c, H);
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(y[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int X = mx_exponent(amax);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) lo |= static_cast<uint32_t>(mx_code(y[i], X)) << (8 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) hi |= static_cast<uint32_t>(mx_code(y[4 + i], X)) << (8 * i);
    *reinterpret_cast<uint2*>(q + base + c) = make_uint2(lo, hi);
    if ((lane & 3) == 0) scale[(size_t)t * (H / 32) + c / 32] = static_cast<uint8_t>(X + 127);
  }
}

// Standalone dynamic MX quantisation of an fp32 (rows, n) matrix along its rows.
__global__ void __launch_bounds__(256) mx_quantize_kernel(const float* __restrict__ y, int rows,
                                                          int n, uint8_t* __restrict__ q,
                                                          uint8_t* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const size_t blocks = (size_t)rows * (n / 32);
  // one warp per 4 blocks: 8 lanes x 4 elements per block
  const size_t gw = (blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5;
  const size_t b = gw * 4 + (lane >> 3);
  if (b >= blocks) return;
  const size_t row = b / (n / 32), blk = b % (n / 32);
  const size_t off = row * n + blk * 32 + (lane & 7) * 4;
  const float4 v = *reinterpret_cast<const float4*>(y + off);
  float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  const int X = mx_exponent(amax);
  const uint32_t c = static_cast<uint32_t>(mx_code(v.x, X)) |
                     (static_cast<uint32_t>(mx_code(v.y, X)) << 8) |
                     (static_cast<uint32_t>(mx_code(v.z, X)) << 16) |
                     (static_cast<uint32_t>(mx_code(v.w, X)) << 24);
  *reinterpret_cast<uint32_t*>(q + off) = c;
  if ((lane & 7) == 0) scale[row * (n / 32) + blk] = static_cast<uint8_t>(X + 127);
}

// MX pre-quantisation of logical weights W (E, K, Ncols) along K into K-major fp8
// rows of the packed order plus scale atoms.  w13's packed order is the bf16
// packing's: in 128-row block b, the 32-row quarter q holds the 16 gate rows of
// features 64b + 16q .. 64b + 16q + 15 and then their 16 up rows, so that one TMEM
// lane quarter of the GEMM accumulator pairs them within a warp.  Tile: 128 K values
// x 32 packed rows per CTA (32 x 8 threads).
template <bool kW13>
__global__ void __launch_bounds__(256) pack_mx_kernel(const uint16_t* __restrict__ w, int K,
                                                      int ncols, int I, uint8_t* __restrict__ q,
                                                      uint8_t* __restrict__ sf) {
  __shared__ float tile[128][33];
  const int k0 = blockIdx.x * 128, r0 = blockIdx.y * 32, e = blockIdx.z;
  const int tx = threadIdx.x, ty = threadIdx.y;
  // this thread's logical column: for w13, packed row 32q + i of 128-row block b holds
  // gate feature 64b + 16q + i (i < 16) or the matching up feature (i >= 16)
  const int col = kW13 ? (r0 / 128) * 64 + ((r0 % 128) / 32) * 16 + (tx & 15) + (tx < 16 ? 0 : I)
                       : r0 + tx;
  for (int i = ty; i < 128; i += 8)
    tile[i][tx] =
        __uint_as_float(static_cast<uint32_t>(w[((size_t)e * K + k0 + i) * ncols + col]) << 16);
  __syncthreads();
  const int rows_total = ncols;  // packed rows per expert
  const int ksteps = K / 128;
  for (int rr = 0; rr < 4; ++rr) {
    const int lr = ty * 4 + rr;       // local packed row 0..31
    const int row = r0 + lr;
    for (int kb = 0; kb < 4; ++kb) {
      const float v = tile[kb * 32 + tx][lr];
      float amax = fabsf(v);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const int X = mx_exponent(amax);
      q[((size_t)e * rows_total + row) * K + k0 + kb * 32 + tx] = mx_code(v, X);
      if (tx == 0) {
        const size_t atom = ((size_t)e * (rows_total / 128) + row / 128) * ksteps + k0 / 128;
        sf[atom * 512 + atom_offset(row & 127, kb)] = static_cast<uint8_t>(X + 127);
      }
    }
  }
}

// MXFP4 (e2m1 + E8M0/32) pre-quantisation of weights along K, same row order and
// scale atoms as pack_mx_kernel: X = floor(log2 amax) - 2 (6 = 1.5 * 2^2 is e2m1's
// largest value), codes e2m1(v / 2^X) nearest-even, saturating.  Codes are packed
// two per byte, element 2i in the low nibble, and stored tile-major: the 128 rows
// x 128 K-elements of one (expert, 128-row block, K step) tile are 8 KB of
// consecutive memory, row after row (64 bytes each), so the GEMM reads every
// weight tile as one contiguous block.
template <bool kW13>
__global__ void __launch_bounds__(256) pack_mx4_kernel(const uint16_t* __restrict__ w, int K,
                                                       int ncols, int I, uint8_t* __restrict__ q,
                                                       uint8_t* __restrict__ sf) {
  __shared__ float tile[128][33];
  const int k0 = blockIdx.x * 128, r0 = blockIdx.y * 32, e = blockIdx.z;
  const int tx = threadIdx.x, ty = threadIdx.y;
  // this thread's logical column: for w13, packed row 32q + i of 128-row block b holds
  // gate feature 64b + 16q + i (i < 16) or the matching up feature (i >= 16)
  const int col = kW13 ? (r0 / 128) * 64 + ((r0 % 128) / 32) * 16 + (tx & 15) + (tx < 16 ? 0 : I)
                       : r0 + tx;
  for (int i = ty; i < 128; i += 8)
    tile[i][tx] =
        __uint_as_float(static_cast<uint32_t>(w[((size_t)e * K + k0 + i) * ncols + col]) << 16);
  __syncthreads();
  const int rows_total = ncols;
  const int ksteps = K / 128;
  for (int rr = 0; rr < 4; ++rr) {
    const int lr = ty * 4 + rr;
    const int row = r0 + lr;
    for (int kb = 0; kb < 4; ++kb) {
      const float v = tile[kb * 32 + tx][lr];
      float amax = fabsf(v);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const uint32_t bits = __float_as_uint(amax);
      const int ef = static_cast<int>((bits >> 23) & 0xFF);
      int X = ef == 0 ? -127 : ef - 127 - 2;
      X = X < -127 ? -127 : (X > 127 ? 127 : X);
      const int nx = -X, a = nx > 126 ? 126 : nx;
      const float scaled = v * exp2i(a) * exp2i(nx - a);
      const uint32_t c =
          static_cast<uint32_t>(__nv_cvt_float_to_fp4(scaled, __NV_E2M1, cudaRoundNearest)) & 15u;
      const uint32_t hi = __shfl_down_sync(0xffffffffu, c, 1);
      if ((tx & 1) == 0)
        q[(((size_t)e * (rows_total / 128) + row / 128) * ksteps + k0 / 128) * 8192 +
          (row & 127) * 64 + (kb * 32 + tx) / 2] =
            static_cast<uint8_t>(c | (hi << 4));
      if (tx == 0) {
        const size_t atom = ((size_t)e * (rows_total / 128) + row / 128) * ksteps + k0 / 128;
        sf[atom * 512 + atom_offset(row & 127, kb)] = static_cast<uint8_t>(X + 127);
      }
    }
  }
}

// Expert-sorted, padded expansion of MX activations: pair j (token t = j/k, expert
// e, unpadded row p = eri[j]) goes to padded row
//   prow = poff[e] + (p - off[e]),  poff[e] = sum_{e' < e} roundup(count[e'], pad),
// pad = 128 (one scale atom per 128 rows) or 32 (one atom per 32 rows, only its
// first 32-row group used: the narrow-tile GEMM shape).  Copies the H code bytes of
// token t and its H/32 scales (into atoms), and records prow in eri_pad[j].  One
// warp per pair.
__global__ void __launch_bounds__(256) mx_expand_kernel(
    const uint8_t* __restrict__ xq, const uint8_t* __restrict__ xs, const int32_t* __restrict__ ids,
    const int32_t* __restrict__ eri, const int32_t* __restrict__ offsets, int E, int P, int H, int k,
    int pad, uint8_t* __restrict__ xe, uint8_t* __restrict__ xe_sf, int32_t* __restrict__ eri_pad) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_poff[257];
  __shared__ int s_off[257];
  const int tid = threadIdx.x, lane = tid & 31;
  __shared__ int s_tmp[8];
  for (int i = tid; i <= E; i += blockDim.x) s_off[i] = offsets[i];
  __syncthreads();
  {
    // padded expert starts: exclusive block scan of the counts rounded up to pad
    // (E <= 256 = blockDim.x)
    const int c = tid < E ? ((s_off[tid + 1] - s_off[tid] + pad - 1) / pad) * pad : 0;
    int total = 0;
    const int pre = block_excl_scan_256(c, s_tmp, &total);
    if (tid < E) s_poff[tid] = pre;
    if (tid == 0) s_poff[E] = total;
  }
  __syncthreads();
  const int j = (blockIdx.x * blockDim.x + tid) >> 5;
  if (j >= P) return;
  const int p = eri[j];
  const int e = ids[j];
  if (p < 0 || e < 0 || e >= E) {
    if (lane == 0) eri_pad[j] = -1;
    return;
  }
  const int prow = s_poff[e] + (p - s_off[e]);
  if (lane == 0) eri_pad[j] = prow;
  const int t = j / k;
  const uint4* src = reinterpret_cast<const uint4*>(xq + (size_t)t * H);
  uint4* dst = reinterpret_cast<uint4*>(xe + (size_t)prow * H);
  for (int v = lane; v < H / 16; v += 32) dst[v] = src[v];
  const int ksteps = H / 128;
  uint8_t* atoms = xe_sf + (size_t)(prow / pad) * ksteps * 512;
  for (int b = lane; b < H / 32; b += 32)
    atoms[(size_t)(b / 4) * 512 + atom_offset(prow % pad, b & 3)] = xs[(size_t)t * (H / 32) + b];
}

// Expert-sorted MX rows (row p of expert e = the e-th block of `offsets`, codes (P, K)
// and row-major scales (P, K/32)) into the padded layout of mx_expand_kernel.
// row_map[p] = padded row.  One warp per row; rows at or past offsets[E] are skipped.
__global__ void __launch_bounds__(256) mx_pad_sorted_kernel(
    const uint8_t* __restrict__ q, const uint8_t* __restrict__ sc,
    const int32_t* __restrict__ offsets, int E, int P, int K, int pad, uint8_t* __restrict__ out_q,
    uint8_t* __restrict__ out_sf, int32_t* __restrict__ row_map) {
  __shared__ int s_poff[257];
  __shared__ int s_off[257];
  const int tid = threadIdx.x, lane = tid & 31;
  __shared__ int s_tmp[8];
  for (int i = tid; i <= E; i += blockDim.x) s_off[i] = offsets[i];
  __syncthreads();
  {
    // padded expert starts: exclusive block scan of the counts rounded up to pad
    // (E <= 256 = blockDim.x)
    const int c = tid < E ? ((s_off[tid + 1] - s_off[tid] + pad - 1) / pad) * pad : 0;
    int total = 0;
    const int pre = block_excl_scan_256(c, s_tmp, &total);
    if (tid < E) s_poff[tid] = pre;
    if (tid == 0) s_poff[E] = total;
  }
  __syncthreads();
  const int p = (blockIdx.x * blockDim.x + tid) >> 5;
  if (p >= P || p >= s_off[E]) return;
  int lo = 0, hi = E;  // s_off[lo] <= p < s_off[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_off[mid] <= p) lo = mid;
    else hi = mid;
  }
  const int prow = s_poff[lo] + (p - s_off[lo]);
  if (lane == 0) row_map[p] = prow;
  const uint4* src = reinterpret_cast<const uint4*>(q + (size_t)p * K);
  uint4* dst = reinterpret_cast<uint4*>(out_q + (size_t)prow * K);
  for (int v = lane; v < K / 16; v += 32) dst[v] = src[v];
  const int ksteps = K / 128;
  uint8_t* atoms = out_sf + (size_t)(prow / pad) * ksteps * 512;
  for (int b = lane; b < K / 32; b += 32)
    atoms[(size_t)(b / 4) * 512 + atom_offset(prow % pad, b & 3)] = sc[(size_t)p * (K / 32) + b];
}

// The inverse for GEMM outputs: padded MX rows (codes + scale atoms) or padded bf16
// rows back to expert-sorted rows p < offsets[E].  One warp per row.
__global__ void __launch_bounds__(256) mx_unpad_kernel(
    const uint8_t* __restrict__ pq, const uint8_t* __restrict__ psf,
    const uint16_t* __restrict__ pbf, const int32_t* __restrict__ row_map,
    const int32_t* __restrict__ offsets_end, int P, int N, int pad, uint8_t* __restrict__ q,
    uint8_t* __restrict__ sc, uint16_t* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int p = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (p >= P || p >= *offsets_end) return;
  const int prow = row_map[p];
  if (pbf != nullptr) {
    const uint4* src = reinterpret_cast<const uint4*>(pbf + (size_t)prow * N);
    uint4* dst = reinterpret_cast<uint4*>(y + (size_t)p * N);
    for (int v = lane; v < N / 8; v += 32) dst[v] = src[v];
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(pq + (size_t)prow * N);
  uint4* dst = reinterpret_cast<uint4*>(q + (size_t)p * N);
  for (int v = lane; v < N / 16; v += 32) dst[v] = src[v];
  const int ksteps = N / 128;
  const uint8_t* atoms = psf + (size_t)(prow / pad) * ksteps * 512;
  for (int b = lane; b < N / 32; b += 32)
    sc[(size_t)p * (N / 32) + b] = atoms[(size_t)(b / 4) * 512 + atom_offset(prow % pad, b & 3)];
}

}  // namespace

cudaError_t launch_mx_pad_sorted(const uint8_t* q, const uint8_t* sc, const int32_t* offsets,
                                 int E, int P, int K, int pad, uint8_t* out_q, uint8_t* out_sf,
                                 int32_t* row_map, cudaStream_t s) {
  if (pad != 32 && pad != 128) return cudaErrorInvalidValue;
  mx_pad_sorted_kernel<<<(P + 7) / 8, 256, 0, s>>>(q, sc, offsets, E, P, K, pad, out_q, out_sf,
                                                    row_map);
  return cudaGetLastError();
}

cudaError_t launch_mx_unpad(const uint8_t* pq, const uint8_t* psf, const uint16_t* pbf,
                            const int32_t* row_map, const int32_t* offsets_end, int P, int N,
                            int pad, uint8_t* q, uint8_t* sc, uint16_t* y, cudaStream_t s) {
  if (pad != 32 && pad != 128) return cudaErrorInvalidValue;
  mx_unpad_kernel<<<(P + 7) / 8, 256, 0, s>>>(pq, psf, pbf, row_map, offsets_end, P, N, pad, q, sc,
                                               y);
  return cudaGetLastError();
}

cudaError_t launch_add_rmsnorm_mxquant(const uint16_t* x, const uint16_t* r, const uint16_t* w,
                                       float eps, int T, int H, uint16_t* residual_out,
                                       float* y32_out, uint16_t* ys_out, uint8_t* q,
                                       uint8_t* scale, cudaStream_t s) {
  const size_t smem = (size_t)H * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(add_rmsnorm_mxquant_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(add_rmsnorm_mxquant_kernel, dim3(T), dim3(256), smem, s, x, r, w, eps, H,
                    residual_out, y32_out, ys_out, q, scale);
}

cudaError_t launch_mx_quantize(const float* y, int rows, int n, uint8_t* q, uint8_t* scale,
                               cudaStream_t s) {
  const size_t blocks = (size_t)rows * (n / 32);
  const size_t warps = (blocks + 3) / 4;
  const unsigned grid = (unsigned)((warps * 32 + 255) / 256);
  mx_quantize_kernel<<<grid, 256, 0, s>>>(y, rows, n, q, scale);
  return cudaGetLastError();
}

cudaError_t launch_pack_mx(const uint16_t* w13, const uint16_t* down, int E, int H, int I,
                           uint8_t* w13q, uint8_t* w13sf, uint8_t* downq, uint8_t* downsf,
                           cudaStream_t s) {
  dim3 block(32, 8);
  if (w13 != nullptr) {
    dim3 grid(H / 128, 2 * I / 32, E);
    pack_mx_kernel<true><<<grid, block, 0, s>>>(w13, H, 2 * I, I, w13q, w13sf);
  }
  if (down != nullptr) {
    dim3 grid(I / 128, H / 32, E);
    pack_mx_kernel<false><<<grid, block, 0, s>>>(down, I, H, I, downq, downsf);
  }
  return cudaGetLastError();
}

cudaError_t launch_pack_mx4(const uint16_t* w13, const uint16_t* down, int E, int H, int I,
                            uint8_t* w13q, uint8_t* w13sf, uint8_t* downq, uint8_t* downsf,
                            cudaStream_t s) {
  dim3 block(32, 8);
  if (w13 != nullptr) {
    dim3 grid(H / 128, 2 * I / 32, E);
    pack_mx4_kernel<true><<<grid, block, 0, s>>>(w13, H, 2 * I, I, w13q, w13sf);
  }
  if (down != nullptr) {
    dim3 grid(I / 128, H / 32, E);
    pack_mx4_kernel<false><<<grid, block, 0, s>>>(down, I, H, I, downq, downsf);
  }
  return cudaGetLastError();
}

cudaError_t launch_mx_expand(const uint8_t* xq, const uint8_t* xs, const int32_t* ids,
                             const int32_t* eri, const int32_t* offsets, int E, int P, int H,
                             int k, int pad, uint8_t* xe, uint8_t* xe_sf, int32_t* eri_pad,
                             cudaStream_t s) {
  if (pad != 32 && pad != 128) return cudaErrorInvalidValue;
  const int blocks = (P + 7) / 8;
  return launch_pdl(mx_expand_kernel, dim3(blocks), dim3(256), 0, s, xq, xs, ids, eri, offsets, E,
                    P, H, k, pad, xe, xe_sf, eri_pad);
}

}  // namespace moe
