// Router logits on the tensor cores for prefill-size token counts.
//
// The page "基于Atlas A3、950训练/推理集群的Qwen3-MoE模型低时延推理性能优化实践"
// (§融合RMSNorm Cast) keeps the gate computation in FP32.  On CUDA cores that costs
// 2*T*H*E fp32 FMAs, which at prefill sizes takes longer than the rest of the
// layer apart from the expert GEMMs.  Here it runs as a bf16 tensor-core GEMM with
// fp32 accumulation without giving up the fp32 operands: each fp32 router weight is
// split exactly into three bf16 pieces, W = W1 + W2 + W3 (8 + 8 + 8 significand
// bits), and the bf16 activations times each piece are exact in fp32, so
//   logits = x.W1 + x.W2 + x.W3
// is one GEMM with K = 3H whose only rounding is the fp32 accumulation.  fp32
// activations (the MXFP8 layer routes on the fp32 RMSNorm output) are split the same
// way and the six products with combined weight above 2^-24 are kept:
//   (x1,W1) (x1,W2) (x2,W1) (x1,W3) (x2,W2) (x3,W1).
// The GEMM is the grouped-GEMM kernel with a single "expert" (all T tokens), the
// router weights as its 128-row A operand, K split into `splits` units that write
// fp32 partial sums part[s][T][E]; the gating kernel adds them in split order.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kTcMinTokens = 65;    // below: CUDA-core decode router

// Wg (H, E) fp32 -> A (mrows, nseg * H) bf16: row e = the weight pieces of expert e
// in segment order (bf16 activations: W1 W2 W3; fp32: W1 W2 W1 W3 W2 W1); rows
// e >= E are zero.  Also writes the one-expert offsets {0, T} and clears zero_word.
__global__ void __launch_bounds__(256) router_pack_kernel(const float* __restrict__ Wg, int H,
                                                          int E, int nseg, int T,
                                                          uint16_t* __restrict__ A,
                                                          int32_t* __restrict__ offs2,
                                                          int* __restrict__ zero_word) {
  pdl_wait();
  pdl_trigger();
  __shared__ float tile[32][33];
  const int h0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;
  for (int i = ty; i < 32; i += 8) {
    const int h = h0 + i, e = e0 + tx;
    tile[i][tx] = (h < H && e < E) ? Wg[(size_t)h * E + e] : 0.f;
  }
  __syncthreads();
  const size_t kp = (size_t)nseg * H;
  for (int i = ty; i < 32; i += 8) {
    const int e = e0 + i, h = h0 + tx;
    if (h >= H) continue;
    uint16_t p[3];
    split3_bf16(tile[tx][i], p);
    uint16_t* row = A + (size_t)e * kp + h;
    if (nseg == 3) {
      row[0] = p[0];
      row[H] = p[1];
      row[2 * (size_t)H] = p[2];
    } else {
      row[0] = p[0];
      row[H] = p[1];
      row[2 * (size_t)H] = p[0];
      row[3 * (size_t)H] = p[2];
      row[4 * (size_t)H] = p[1];
      row[5 * (size_t)H] = p[0];
    }
  }
  if (blockIdx.x == 0 && blockIdx.y == 0 && tx == 0 && ty == 0) {
    offs2[0] = 0;
    offs2[1] = T;
    if (zero_word != nullptr) *zero_word = 0;
  }
}

// y (T, H) fp32 -> ys (T, 3H) bf16 = [y1 | y2 | y3], the exact three-piece split.
// Grid (ceil(H / 8 / 256), min(T, 65535)): each thread splits 8 consecutive elements
// of rows blockIdx.y, + gridDim.y, ... (two 16-byte loads, three 16-byte stores per
// row; H % 64 == 0 on this path).
__global__ void __launch_bounds__(256) split_f32_kernel(const float* __restrict__ y, int T, int H,
                                                        uint16_t* __restrict__ ys) {
  pdl_wait();
  pdl_trigger();
  const int g = blockIdx.x * blockDim.x + threadIdx.x;   // 8-element group of a row
  if (g >= H / 8) return;
  for (int t = blockIdx.y; t < T; t += gridDim.y) {
    const float4* src = reinterpret_cast<const float4*>(y + (size_t)t * H) + 2 * g;
    const float4 a = src[0], b = src[1];
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    store_split3_x8(v, ys + (size_t)t * 3 * H + 8 * g, H);
  }
}

size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

}  // namespace

RouterPlan router_plan_ex(int T, int H, int E, bool f32in) {
  RouterPlan p = router_plan(T, H, E);
  p.tc = false;
  p.nseg = 0;
  p.extra_bytes = 0;
  if (T < kTcMinTokens || H % 64 != 0) return p;
  p.tc = true;
  p.small = false;
  p.nseg = f32in ? 6 : 3;
  const int mrows = ((E + 127) / 128) * 128;
  const int tblocks = (T + 255) / 256;
  const int kblocks = p.nseg * H / 64;
  // about one wave of units: fewer K splits halve the fp32 partials the gating
  // kernel then sums (two waves measured slower on the 4096-token Zipf layer)
  int s = 152 / (tblocks * (mrows / 128));
  s = s < 1 ? 1 : (s > 16 ? 16 : s);
  while (kblocks % s != 0) --s;
  p.splits = s;
  p.extra_bytes = align256((size_t)mrows * p.nseg * H * 2) + 256 +
                  (f32in ? align256((size_t)T * 3 * H * 2) : 0);
  return p;
}

size_t router_ws_bytes(int T, int H, int E, bool f32in) {
  const RouterPlan p = router_plan_ex(T, H, E, f32in);
  return align256((size_t)p.splits * T * E * sizeof(float)) + p.extra_bytes;
}

uint16_t* router_split_rows(void* extra, const RouterPlan& plan, int H, int E) {
  const int mrows = ((E + 127) / 128) * 128;
  return reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(extra) +
                                     align256((size_t)mrows * plan.nseg * H * 2) + 256);
}

cudaError_t launch_router_tc(const void* x, bool f32in, bool presplit, const float* Wg, int T,
                             int H, int E, const RouterPlan& plan, float* partial, void* extra,
                             int* zero_word, int* status, cudaStream_t s) {
  const int mrows = ((E + 127) / 128) * 128;
  const int kp = plan.nseg * H;
  uint8_t* base = static_cast<uint8_t*>(extra);
  uint16_t* A = reinterpret_cast<uint16_t*>(base);
  int32_t* offs2 = reinterpret_cast<int32_t*>(base + align256((size_t)mrows * kp * 2));
  uint16_t* ys = router_split_rows(extra, plan, H, E);
  cudaError_t err = launch_pdl(router_pack_kernel, dim3((H + 31) / 32, mrows / 32), dim3(32, 8), 0,
                               s, Wg, H, E, plan.nseg, T, A, offs2, zero_word);
  if (err != cudaSuccess) return err;
  const uint16_t* B = static_cast<const uint16_t*>(x);
  if (f32in && presplit) {
    B = ys;   // written by the producing kernel
  } else if (f32in) {
    const dim3 grid((unsigned)((H / 8 + 255) / 256), (unsigned)(T < 65535 ? T : 65535));
    err = launch_pdl(split_f32_kernel, grid, dim3(256), 0, s, static_cast<const float*>(x), T, H,
                     ys);
    if (err != cudaSuccess) return err;
    B = ys;
  }
  GemmPhase ph{};
  ph.A_weights = A;
  ph.B_act = B;
  ph.out = nullptr;
  ph.K = kp;
  ph.MW = mrows;
  ph.n_out = E;
  ph.epi = 2;
  ph.ksplit = plan.splits;
  ph.b_inner = f32in ? 3 * H : H;
  ph.bseg = H;
  ph.bmap = f32in ? (0u | (0u << 3) | (1u << 6) | (0u << 9) | (1u << 12) | (2u << 15)) : 0u;
  ph.out_f32 = partial;
  ph.mvalid = E;
  ph.rows_total = T;
  return launch_grouped_gemm(&ph, nullptr, offs2, 1, T, T, nullptr, status, s);
}

}  // namespace moe
