// Block-scaled MXFP8 grouped GEMM (tcgen05.mma kind::mxf8f6f4, E8M0 scales per 32
// K-elements in TMEM) for the MXFP8 expert MLPs of the page "基于Atlas A3、950训练/
// 推理集群的Qwen3-MoE模型低时延推理性能优化实践" (§融合RMSNorm MX量化 feeds MXFP8
// activations to the grouped matmul; §高性能专家计算; SwiGLU from §计算分解).
//
// Same orientation, unit order, warp roles and phase dependency as the bf16 grouped
// GEMM (gmm.cu): D[128 weight rows][<=128 tokens] per unit, weights as the A
// operand.  Differences:
//  - operands are e4m3 bytes, so one 128-byte swizzle row holds 128 K-elements and
//    a pipeline stage covers K = 128 = four MMAs of K = 32;
//  - each stage also carries the 512-byte scale atoms of its A and B tiles (128
//    rows x 4 blocks each, loaded with 1-D bulk copies); the MMA thread copies them
//    into a per-stage TMEM slot with tcgen05.cp before the stage's four MMAs, and
//    MMA kk uses byte kk of each scale word;
//  - the expert-sorted activations are padded so each expert starts on a kPad-row
//    boundary, with one scale atom per kPad-row block and K step;
//  - two tile shapes: 128 x 128 with 128-row activation boxes and kPad = 128 for
//    prefill, and a decode shape of 128 x 32 with 16-row boxes, a deeper ring and
//    kPad = 32.  With kPad = 32 a tile's B scales always sit in the first TMEM
//    column of the copied atom, so the MMA's scale address is never offset by a
//    32-row group (a one-column offset was rejected as a misaligned address);
//  - the gate/up epilogue applies SwiGLU and MX-quantises h along I (a warp's 32
//    lanes hold one 32-feature block of one token), writing e4m3 codes and scale
//    atoms that the down projection then reads.
#include <cuda_fp8.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 128;                          // fp8 elements per stage (128 bytes)
constexpr int kThreads = 256;
constexpr int kMaxE = 256;
// A CTA's units are decoded once in the prologue into shared memory, so a unit
// boundary costs each role one shared-memory load instead of a binary search and
// divisions; a longer list is decoded on the fly.
constexpr int kMaxUnits = 512;
constexpr int kABytes = kBM * kBK;                // 16 KB
constexpr int kSfBytes = 512;                     // one scale atom
// epilogue shared memory: four 32 x 32 bf16 transpose tiles (down projection), which
// also hold the two warp pairs' block-maximum swap areas of the gate/up projection
constexpr int kEpiBytes = 4 * 32 * 32 * 2;
static_assert(kEpiBytes >= 2 * 128 * 4, "block-maximum swap areas");

// Tile shape: kBN tokens per unit, kStages pipeline stages, B boxes of kBoxRows rows.
// With kAbsorb > 0 an expert's last token block takes up to kAbsorb rows beyond kBN
// (instead of a separate, nearly empty block whose MMAs would cost as much issue time
// as a full one); those rows come in one extra kAbsorb-row box, and their B scales
// are the next 128-row atom, copied into the next four TMEM columns.
template <int BN_, int STAGES_, int BOX_, int PAD_, bool PAIR_, int ABSORB_>
struct MxShape {
  static constexpr int kBN = BN_;
  static constexpr int kAbsorb = ABSORB_;
  static constexpr int kMaxRows = kBN + kAbsorb;      // largest token block
  // Stage release and scale readiness signalled per pair of stages (fewer barrier
  // operations on the MMA thread, but a shorter producer lookahead).
  static constexpr bool kPair = PAIR_;
  static constexpr int kGroup = kPair ? 2 : 1;
  static constexpr int kPad = PAD_;                    // row padding of each expert block
  static constexpr int kStages = STAGES_;
  static constexpr int kBoxRows = BOX_;
  static constexpr int kBBytes = kMaxRows * kBK;
  static constexpr int kBoxBytes = kBoxRows * kBK;
  // B scale atoms per stage (one per 128 rows of the largest block), plus one for A
  static constexpr int kSfAtoms = 1 + (kMaxRows + 127) / 128;
  static constexpr int kSfStageCols = 4 * kSfAtoms;
  // TMEM: accumulator 1 starts kAccStride columns after accumulator 0 (a power of two);
  // the scale slots sit after accumulator 0 when kMaxRows is not a power of two
  static constexpr bool kPow2 = (kMaxRows & (kMaxRows - 1)) == 0;
  static constexpr int kAccStride = kPow2 ? kMaxRows : 256;
  static constexpr int kSfCol = kPow2 ? 2 * kMaxRows : kMaxRows;
  static constexpr int kColsUsed = kPow2 ? kSfCol + kSfStageCols * kStages : kAccStride + kMaxRows;
  static constexpr int kTmemCols = kColsUsed <= 128 ? 128 : (kColsUsed <= 256 ? 256 : 512);
  // smem layout
  static constexpr int kA = 0;
  static constexpr int kB = kA + kStages * kABytes;
  static constexpr int kSf = kB + kStages * kBBytes;   // per stage: SFA, SFB atoms
  static constexpr int kEpi = kSf + kStages * kSfAtoms * kSfBytes;
  static constexpr int kBar = kEpi + kEpiBytes;
  static constexpr int kNumBars = kStages + 2 * (kStages / kGroup) + 6;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kTables = kMisc + 16;
  static constexpr int kUnits = kTables + (4 * (kMaxE + 1) + 8) * 4;
  static constexpr int kEnd = kUnits + kMaxUnits * 8;
  static_assert(kUnits % 8 == 0, "unit list alignment");
  static constexpr int kSmemBytes = kEnd + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kColsUsed <= 512, "tensor memory budget");
  static_assert(kPow2 || kSfCol + kSfStageCols * kStages <= kAccStride, "scale slots fit");
  static_assert(kBN % 32 == 0 && kPad == kBN && kBN % kBoxRows == 0, "tile shape");
  static_assert(kAbsorb % 16 == 0 && kAbsorb < kBN && kMaxRows <= 256, "absorbed rows");
  static_assert(kBBytes % 1024 == 0 && kBoxBytes % 1024 == 0 && (kBN * kBK) % 1024 == 0,
                "swizzle atoms");
  static_assert(kStages % kGroup == 0, "stages are released and signalled in pairs");
};
using ShapePrefill = MxShape<128, 5, 128, 128, false, 32>;
// e4m3 decode is bound by HBM bytes in flight (more stages); e2m1 decode moves half
// the bytes per stage and is bound by the MMA thread's issue rate (paired barriers)
using ShapeDecode = MxShape<32, 9, 16, 32, false, 0>;
using ShapeDecodeFp4 = MxShape<32, 8, 16, 32, true, 0>;

// Token blocks of an expert with m rows: blocks of kBN, the last one taking up to
// kAbsorb more (never empty: (nb - 1) * kBN < m - kAbsorb when nb > 1).
template <int kBN, int kAbsorb>
__host__ __device__ constexpr int token_blocks(int m) {
  return m <= 0 ? 0
                : (kAbsorb ? ((m - kAbsorb + kBN - 1) / kBN > 1 ? (m - kAbsorb + kBN - 1) / kBN : 1)
                           : (m + kBN - 1) / kBN);
}
static_assert(token_blocks<128, 32>(0) == 0 && token_blocks<128, 32>(1) == 1 &&
                  token_blocks<128, 32>(160) == 1 && token_blocks<128, 32>(161) == 2 &&
                  token_blocks<128, 32>(288) == 2 && token_blocks<128, 32>(289) == 3 &&
                  token_blocks<32, 0>(33) == 2,
              "token blocks");

struct MxArgs {
  const int32_t* offsets;
  int E;
  int K[2];
  int MW[2];
  int ld[2];
  int active[2];
  int a_fp4[2];             // A is e2m1 (TMA-unpacked to 16-byte groups) instead of e4m3
  const uint8_t* a_sf[2];   // weight scale atoms [E][MW/128][K/128][512]
  const uint8_t* b_sf[2];   // activation scale atoms [Ppad/128][K/128][512]
  uint8_t* hq;              // phase-0 output codes (Ppad, ld0)
  uint8_t* h_sf;            // phase-0 output scale atoms [Ppad/128][ld0/128][512]
  uint16_t* y;              // phase-1 output (Ppad, ld1) bf16
  int* done;
  int* sched;               // CTA pairs: counter the pairs draw units from (or null)
  int* status;
};

struct Unit {
  int ph, e, mb, nb, row0, rows;   // row0: padded row of the token block
};

struct Tables {
  const int* off;
  const int* poff;
  const int* uoff[2];
  int E;
};

template <int kBN, int kAbsorb>
__device__ __forceinline__ Unit decode_unit(int u, const Tables& tb) {
  Unit r;
  const int total0 = tb.uoff[0][tb.E];
  r.ph = (u < total0) ? 0 : 1;
  if (r.ph) u -= total0;
  const int* uo = tb.uoff[r.ph];
  int lo = 0, hi = tb.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (uo[mid] <= u) lo = mid;
    else hi = mid;
  }
  r.e = lo;
  const int local = u - uo[lo];
  const int m = tb.off[lo + 1] - tb.off[lo];
  const int nb = token_blocks<kBN, kAbsorb>(m);
  r.mb = local / nb;
  r.nb = local - r.mb * nb;
  r.row0 = tb.poff[lo] + r.nb * kBN;
  r.rows = r.nb == nb - 1 ? m - r.nb * kBN : kBN;
  return r;
}

// A unit in two words: row0; ph | e << 1 | mb << 10 | rows << 20 (e < 512 and
// mb < 1024 hold for every shape the entry points accept; rows <= 160).
__device__ __forceinline__ uint2 pack_unit(const Unit& t) {
  return make_uint2(static_cast<uint32_t>(t.row0),
                    static_cast<uint32_t>(t.ph) | (static_cast<uint32_t>(t.e) << 1) |
                        (static_cast<uint32_t>(t.mb) << 10) | (static_cast<uint32_t>(t.rows) << 20));
}
__device__ __forceinline__ Unit unpack_unit(uint2 w) {
  Unit t;
  t.row0 = static_cast<int>(w.x);
  t.ph = static_cast<int>(w.y & 1u);
  t.e = static_cast<int>((w.y >> 1) & 511u);
  t.mb = static_cast<int>((w.y >> 10) & 1023u);
  t.rows = static_cast<int>(w.y >> 20);
  t.nb = 0;
  return t;
}

__device__ __forceinline__ bool wait_counter(const int* p, int need, const volatile int* abort) {
  if (ld_acquire_gpu(p) >= need) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    __nanosleep(64);
    if (ld_acquire_gpu(p) >= need) return true;
    if ((i & 15u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > kWaitLimitNs) return false;
    }
  }
}

__device__ __forceinline__ uint16_t f2bf(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&b);
}

__device__ __forceinline__ int mx_exponent(float amax) {
  const int ef = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF);
  if (ef == 0) return -127;
  const int X = ef - 127 - 8;
  return X < -127 ? -127 : (X > 127 ? 127 : X);
}

__device__ __forceinline__ uint8_t mx_code(float v, int X) {
  const int nx = -X;
  const int a = nx > 126 ? 126 : nx;
  const float f = v * __uint_as_float(static_cast<uint32_t>(a + 127) << 23) *
                  __uint_as_float(static_cast<uint32_t>(nx - a + 127) << 23);
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(f, __NV_SATFINITE, __NV_E4M3));
}

// One 32-token chunk of a gate/up accumulator: SwiGLU, then MX quantisation of h
// along I into the down projection's activation layout.  The warp reads TMEM lane
// quarter q of the CTA's 128-row weight block mb (whose features are mb * 64 ..
// mb * 64 + 63): lanes 0-15 hold the gate rows of features 16q .. 16q + 15 of the
// block and lanes 16-31 their up rows, v[j] being token c0 + j.  One shuffle pairs
// gate and up, so lanes 0-15 finish tokens c0 .. c0 + 15 and lanes 16-31 tokens
// c0 + 16 .. c0 + 31, each for feature 16q + (lane & 15).  An MX block (32 features)
// spans quarters q and q ^ 1: each half-warp takes its 16 per-token maxima over its
// 16 lanes by a butterfly (16 values halved over lane offsets 8, 4, 2, 1, after which
// lane t holds token c0 + t's maximum), the two warps swap them through xs (a
// [2 slots][2 warps][32] float area of the warp pair, the slot alternating with the
// pair's chunk count) after a named barrier of the pair, and every lane then writes
// its code byte of each of its 16 token rows; the even warp of the pair writes the
// scale bytes.
template <int kPad>
__device__ __forceinline__ void swiglu_mx_chunk(const MxArgs& args, const float (&v)[32], int row0,
                                                int c0, int rows, int mb, int q, int lane,
                                                float* xs, int slot, uint32_t bar_id) {
  const bool lo = lane < 16;
  float h[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float send = lo ? v[16 + j] : v[j];
    const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
    const float g = lo ? v[j] : recv;
    const float up = lo ? recv : v[16 + j];
    h[j] = g / (1.0f + __expf(-g)) * up;
  }
  float m[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) m[j] = fabsf(h[j]);
#pragma unroll
  for (int o = 8, n = 16; o >= 1; o >>= 1, n >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < n / 2; ++k) {
      const float send = upper ? m[k] : m[k + n / 2];
      const float keep = upper ? m[k + n / 2] : m[k];
      m[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
    }
  }
  xs[(slot * 2 + (q & 1)) * 32 + lane] = m[0];
  named_bar_sync(bar_id, 64);
  const int Xmine = mx_exponent(fmaxf(m[0], xs[(slot * 2 + ((q & 1) ^ 1)) * 32 + lane]));
  const int ld = args.ld[0];
  if ((q & 1) == 0 && c0 + lane < rows) {
    const int prow = row0 + c0 + lane;
    const int kbq = (mb & 1) * 2 + (q >> 1);   // 32-feature block within the 128-feature step
    uint8_t* atom = args.h_sf + ((size_t)(prow / kPad) * (ld / 128) + mb / 2) * kSfBytes;
    atom[(prow & 31) * 16 + ((prow % kPad) >> 5) * 4 + kbq] = static_cast<uint8_t>(Xmine + 127);
  }
  uint8_t* hcol = args.hq + mb * 64 + 16 * q + (lane & 15);
  const int tb0 = c0 + (lo ? 0 : 16);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int X = __shfl_sync(0xffffffffu, Xmine, (lane & 16) + j);
    if (tb0 + j < rows) hcol[(size_t)(row0 + tb0 + j) * ld] = mx_code(h[j], X);
  }
}

template <class S>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA0,
                           const __grid_constant__ CUtensorMap tmB0,
                           const __grid_constant__ CUtensorMap tmA1,
                           const __grid_constant__ CUtensorMap tmB1,
                           const __grid_constant__ CUtensorMap tmX0,   // absorbed-row boxes
                           const __grid_constant__ CUtensorMap tmX1, const MxArgs args) {
  constexpr int kBN = S::kBN, kStages = S::kStages, kBoxRows = S::kBoxRows, kPad = S::kPad;
  constexpr int kAbsorb = S::kAbsorb, kSfAtoms = S::kSfAtoms, kSfStageCols = S::kSfStageCols;
  constexpr int kBBytes = S::kBBytes, kBoxBytes = S::kBoxBytes;
  constexpr int kAccStride = S::kAccStride, kSfCol = S::kSfCol, kTmemCols = S::kTmemCols;
  using L = S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem + L::kA;
  uint8_t* sB = smem + L::kB;
  uint8_t* sSF = smem + L::kSf;
  uint8_t* sEpi = smem + L::kEpi;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* empty = full + kStages;
  // empty[g] / sfready[g] cover the stages of group g (one stage, or the pair 2g, 2g + 1)
  constexpr int kG = S::kGroup, kNG = kStages / kG;
  uint64_t* sfready = empty + kNG;
  uint64_t* tfull = sfready + kNG;
  uint64_t* tempty = tfull + 2;
  uint64_t* fin = tempty + 2;            // MMA issuer's drain on abort
  uint64_t* fin_sf = fin + 1;            // scale copier's drain on abort
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  int* s_off = reinterpret_cast<int*>(smem + L::kTables);
  int* s_poff = s_off + (kMaxE + 1);
  int* s_uoff0 = s_poff + (kMaxE + 1);
  int* s_uoff1 = s_uoff0 + (kMaxE + 1);
  int* s_tmp = s_uoff1 + (kMaxE + 1);
  uint2* s_units = reinterpret_cast<uint2*>(smem + L::kUnits);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = args.E;
  pdl_trigger();

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 2);  // weight + activation producer
    for (int g = 0; g < kNG; ++g) {
      mbar_init(&empty[g], 1);
      mbar_init(&sfready[g], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(fin, 1);
    mbar_init(fin_sf, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA0);
    tma_prefetch_desc(&tmB0);
    tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB1);
    if (kAbsorb) {
      tma_prefetch_desc(&tmX0);
      tma_prefetch_desc(&tmX1);
    }
  }
  if (warp == 2) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  for (int i = tid; i <= E; i += kThreads) s_off[i] = args.offsets[i];
  __syncthreads();

  // units per expert (per phase) and the 128-row padded offsets, by block scans
  {
    int v[3] = {0, 0, 0};
    if (tid < E) {
      const int m = s_off[tid + 1] - s_off[tid];
      const int nb = token_blocks<kBN, kAbsorb>(m);
      v[0] = args.active[0] ? nb * (args.MW[0] / kBM) : 0;
      v[1] = args.active[1] ? nb * (args.MW[1] / kBM) : 0;
      v[2] = ((m + kPad - 1) / kPad) * kPad;
    }
    int* dsts[3] = {s_uoff0, s_uoff1, s_poff};
    for (int p = 0; p < 3; ++p) {
      int inc = v[p];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      if (lane == 31) s_tmp[warp] = inc;
      __syncthreads();
      int pre = 0, tot = 0;
      for (int w = 0; w < kThreads / 32; ++w) {
        if (w < warp) pre += s_tmp[w];
        tot += s_tmp[w];
      }
      if (tid < E) dsts[p][tid] = pre + inc - v[p];
      if (tid == 0) dsts[p][E] = tot;
      __syncthreads();
    }
  }
  tc_fence_after_sync();
  const uint32_t tmem_base = *s_tmem;
  Tables tb;
  tb.off = s_off;
  tb.poff = s_poff;
  tb.uoff[0] = s_uoff0;
  tb.uoff[1] = s_uoff1;
  tb.E = E;
  const int total = s_uoff0[E] + s_uoff1[E];
  const int my_units =
      (int)blockIdx.x < total ? (total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  const bool use_list = my_units <= kMaxUnits;   // the same in every thread of the CTA
  if (use_list) {
    for (int i = tid; i < my_units; i += kThreads)
      s_units[i] = pack_unit(decode_unit<kBN, kAbsorb>((int)blockIdx.x + i * (int)gridDim.x, tb));
    __syncthreads();
  }

  // Each tcgen05 / TMA instruction costs its issuing thread tens of clocks, so the
  // per-stage issue work is spread over four single-thread roles: weight loads
  // (warp 0), activation loads (warp 2), scale-atom copies into TMEM (warp 3) and
  // the MMAs (warp 1).  A stage is full when both producers' bytes have landed.
  // Scale readiness and stage release are signalled per group of kG stages (with
  // pairs, one commit and one wait per pair instead of per stage): sfready[g] when
  // the copier's tcgen05.cp of the group are done, empty[g] when its MMAs are done
  // (that also retires the copies, which ran before them).  A CTA's last stage
  // closes its group even when the group is not complete.
  int my_stages = 0;   // stages this CTA runs (closes the last pair)
  {
    const int total0 = s_uoff0[E];
    const int g = gridDim.x, b = blockIdx.x;
    const int mine = b < total ? (total - b + g - 1) / g : 0;
    const int mine0 = b < total0 ? (total0 - b + g - 1) / g : 0;
    my_stages = mine0 * (args.K[0] / kBK) + (mine - mine0) * (args.K[1] / kBK);
  }
  if ((warp == 0 || warp == 2) && lane == 0) {
    // ------------------------------------------------------ TMA producers --
    const bool weights = warp == 0;
    // weight tiles are re-read by every token block of their expert
    const uint64_t pol_w = kBN <= 32 ? l2_policy_evict_first() : l2_policy_evict_normal();
    const uint64_t pol_x = l2_policy_evict_last();
    int stage = 0;
    uint32_t par = 0;
    uint32_t issued_mask = 0, issued_par = 0;
    bool ok = true;
    for (int u = blockIdx.x, ui = 0; u < total && ok; u += gridDim.x, ++ui) {
      const Unit t = use_list ? unpack_unit(s_units[ui]) : decode_unit<kBN, kAbsorb>(u, tb);
      if (!weights && t.ph == 1 && args.done != nullptr) {
        // the down projection's activations are h of this expert's gate/up units
        const int m = s_off[t.e + 1] - s_off[t.e];
        const int need = token_blocks<kBN, kAbsorb>(m) * (args.MW[0] / kBM);
        if (!wait_counter(args.done + t.e, need, s_abort)) {
          ok = false;
          break;
        }
        fence_proxy_async_global();
      }
      const int K = args.K[t.ph];
      const int nk = K / kBK;
      const int nbox = (min(t.rows, kBN) + kBoxRows - 1) / kBoxRows;
      const bool tail = kAbsorb > 0 && t.rows > kBN;   // absorbed rows in a second atom
      // an e2m1 tile fills the same 16 KB of smem as an e4m3 one (each 16-code group
      // padded to 16 bytes), but only its 8 KB of packed codes count as transferred
      const uint32_t abytes = args.a_fp4[t.ph] ? kABytes / 2 : kABytes;
      const uint32_t bytes =
          weights ? abytes + kSfBytes
                  : nbox * kBoxBytes + (tail ? kAbsorb * kBK + 2 * kSfBytes : kSfBytes);
      const CUtensorMap* tm = weights ? (t.ph ? &tmA1 : &tmA0) : (t.ph ? &tmB1 : &tmB0);
      const int arow = t.e * args.MW[t.ph] + t.mb * kBM;
      const int atile0 = (t.e * (args.MW[t.ph] / kBM) + t.mb) * nk;
      const uint8_t* sfsrc =
          weights ? args.a_sf[t.ph] + ((size_t)(t.e * (args.MW[t.ph] / kBM) + t.mb) * nk) * kSfBytes
                  : args.b_sf[t.ph] + ((size_t)(t.row0 / kPad) * nk) * kSfBytes;
      for (int kb = 0; kb < nk; ++kb) {
        if (stage % kG == 0 && !mbar_wait(&empty[stage / kG], par ^ 1u, s_abort)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[stage], bytes);
        uint8_t* sf = sSF + stage * kSfAtoms * kSfBytes + (weights ? 0 : kSfBytes);
        if (weights) {
          if (args.a_fp4[t.ph])  // tile-major e2m1: tile (e, mb, kb) is rows [128 * tile, +128)
            tma_load_2d(sA + stage * kABytes, tm, &full[stage], 0, (atile0 + kb) * kBM, pol_w);
          else
            tma_load_2d(sA + stage * kABytes, tm, &full[stage], kb * kBK, arow, pol_w);
          bulk_load_1d(sf, sfsrc + (size_t)kb * kSfBytes, kSfBytes, &full[stage], pol_w);
        } else {
          for (int j = 0; j < nbox; ++j)
            tma_load_2d(sB + stage * kBBytes + j * kBoxBytes, tm, &full[stage], kb * kBK,
                        t.row0 + j * kBoxRows, pol_x);
          bulk_load_1d(sf, sfsrc + (size_t)kb * kSfBytes, kSfBytes, &full[stage], pol_x);
          if (tail) {
            tma_load_2d(sB + stage * kBBytes + kBN * kBK, t.ph ? &tmX1 : &tmX0, &full[stage],
                        kb * kBK, t.row0 + kBN, pol_x);
            // the next 128-row block's atom for the same K step
            bulk_load_1d(sf + kSfBytes, sfsrc + ((size_t)nk + kb) * kSfBytes, kSfBytes,
                         &full[stage], pol_x);
          }
        }
        issued_mask |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (par << stage);
        if (++stage == kStages) {
          stage = 0;
          par ^= 1u;
        }
      }
    }
    if (ok && weights) {
      // all stage groups released: no MMA still reads this CTA's shared memory
      if (stage % kG) stage += kG - stage % kG;   // a partly used group was closed early
      if (stage == kStages) {
        stage = 0;
        par ^= 1u;
      }
      for (int i = 0; i < kNG; ++i) {
        if (!mbar_wait(&empty[stage / kG], par ^ 1u, s_abort)) {
          ok = false;
          break;
        }
        stage += kG;
        if (stage == kStages) {
          stage = 0;
          par ^= 1u;
        }
      }
    }
    if (!ok) {
      *s_abort = 1;
      flag_status(args.status, MOE_DEV_WAIT_TIMEOUT);
      // let this thread's copies land before the CTA can exit (bounded waits)
      for (int s2 = 0; s2 < kStages; ++s2)
        if ((issued_mask >> s2) & 1u) mbar_wait(&full[s2], (issued_par >> s2) & 1u, nullptr);
    }
  } else if (warp == 3 && lane == 0) {
    // --------------------------------------------------- scale-atom copier --
    int stage = 0, done_stages = 0;
    uint32_t par = 0;
    bool ok = true;
    for (int u = blockIdx.x, ui = 0; u < total && ok; u += gridDim.x, ++ui) {
      const Unit t = use_list ? unpack_unit(s_units[ui]) : decode_unit<kBN, kAbsorb>(u, tb);
      const int nk = args.K[t.ph] / kBK;
      const bool tail = kAbsorb > 0 && t.rows > kBN;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait(&full[stage], par, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t sfa_t = tmem_base + static_cast<uint32_t>(kSfCol + stage * kSfStageCols);
        const uint32_t sf_s = smem_u32(sSF + stage * kSfAtoms * kSfBytes);
        tc_cp_32x128b_warpx4(sfa_t, smem_desc_noswz(sf_s, 128));
        tc_cp_32x128b_warpx4(sfa_t + 4, smem_desc_noswz(sf_s + kSfBytes, 128));
        if (tail) tc_cp_32x128b_warpx4(sfa_t + 8, smem_desc_noswz(sf_s + 2 * kSfBytes, 128));
        ++done_stages;
        if (stage % kG == kG - 1 || done_stages == my_stages) tc_commit(&sfready[stage / kG]);
        if (++stage == kStages) {
          stage = 0;
          par ^= 1u;
        }
      }
    }
    if (!ok) {
      *s_abort = 1;
      flag_status(args.status, MOE_DEV_WAIT_TIMEOUT);
      tc_commit(fin_sf);
      mbar_wait(fin_sf, 0, nullptr);
    }
  } else if (warp == 1 && lane == 0) {
    // -------------------------------------------------------- MMA issuer --
    int stage = 0, acc = 0, done_stages = 0;
    uint32_t par = 0, apar = 0;
    bool ok = true;
    for (int u = blockIdx.x, ui = 0; u < total && ok; u += gridDim.x, ++ui) {
      const Unit t = use_list ? unpack_unit(s_units[ui]) : decode_unit<kBN, kAbsorb>(u, tb);
      const int n = (t.rows + 15) & ~15;
      const uint32_t idesc0 = idesc_mxf8_f32(kBM, n, 0, 0) | (args.a_fp4[t.ph] ? (5u << 7) : 0u);
      if (!mbar_wait(&tempty[acc], apar ^ 1u, s_abort)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kAccStride);
      const int nk = args.K[t.ph] / kBK;
      for (int kb = 0; kb < nk; ++kb) {
        // the scales' copy completing implies the stages' operands have landed
        if (stage % kG == 0 && !mbar_wait(&sfready[stage / kG], par, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t sfa_t = tmem_base + static_cast<uint32_t>(kSfCol + stage * kSfStageCols);
        const uint64_t adesc = smem_desc_sw128(smem_u32(sA + stage * kABytes));
        const uint64_t bdesc = smem_desc_sw128(smem_u32(sB + stage * kBBytes));
#pragma unroll
        for (int kk = 0; kk < kBK / 32; ++kk)   // +32 bytes along K = +2 in the start field
          tc_mma_mxf8(d, adesc + 2 * kk, bdesc + 2 * kk, idesc0 | idesc_sf_ids(kk, kk), sfa_t,
                      sfa_t + 4, (kb | kk) ? 1u : 0u);
        ++done_stages;
        if (stage % kG == kG - 1 || done_stages == my_stages) tc_commit(&empty[stage / kG]);
        if (++stage == kStages) {
          stage = 0;
          par ^= 1u;
        }
      }
      if (!ok) break;
      tc_commit(&tfull[acc]);
      acc ^= 1;
      if (acc == 0) apar ^= 1u;
    }
    if (!ok) {
      *s_abort = 1;
      flag_status(args.status, MOE_DEV_WAIT_TIMEOUT);
      tc_commit(fin);
      mbar_wait(fin, 0, nullptr);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue --
    const int q = warp & 3;
    const int et = tid - 128;
    int* s_flag = s_tmp;
    int acc = 0, nchunk = 0;
    uint32_t apar = 0;
    for (int u = blockIdx.x, ui = 0; u < total; u += gridDim.x, ++ui) {
      const Unit t = use_list ? unpack_unit(s_units[ui]) : decode_unit<kBN, kAbsorb>(u, tb);
      if (et == 0) s_flag[0] = mbar_wait(&tfull[acc], apar, s_abort) ? 1 : 0;
      named_bar_sync(1, 128);
      const int ok = s_flag[0];
      named_bar_sync(1, 128);
      if (!ok) {
        if (et == 0) {
          *s_abort = 1;
          flag_status(args.status, MOE_DEV_WAIT_TIMEOUT);
        }
        break;
      }
      tc_fence_after_sync();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * kAccStride);
      if (t.ph == 0) {
        // SwiGLU and MX quantisation of h, a 32-token chunk at a time; warps q and q ^ 1
        // (the two halves of one 32-feature MX block) swap block maxima through xs
        float* xs = reinterpret_cast<float*>(sEpi) + (q >> 1) * 128;
        for (int c0 = 0; c0 < t.rows; c0 += 32) {
          float v[32];
          tmem_ld_32x32b_x32(tbase + c0, v);
          swiglu_mx_chunk<kPad>(args, v, t.row0, c0, t.rows, t.mb, q, lane, xs, nchunk & 1,
                                2 + (q >> 1));
          ++nchunk;
        }
      } else {
        uint16_t* tbw = reinterpret_cast<uint16_t*>(sEpi) + q * 32 * 32;
        const int ld = args.ld[1];
        for (int c0 = 0; c0 < t.rows; c0 += 32) {
          float v[32];
          tmem_ld_32x32b_x32(tbase + c0, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) tbw[j * 32 + lane] = f2bf(v[j]);
          __syncwarp();
#pragma unroll
          for (int it = 0; it < 4; ++it) {
            const int idx = lane + 32 * it;
            const int j = idx >> 2, c = idx & 3;
            if (c0 + j < t.rows) {
              const uint4 val = *reinterpret_cast<const uint4*>(tbw + j * 32 + c * 8);
              *reinterpret_cast<uint4*>(args.y + (size_t)(t.row0 + c0 + j) * ld + t.mb * kBM +
                                        q * 32 + c * 8) = val;
            }
          }
          __syncwarp();
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (t.ph == 0 && args.done != nullptr) {
        __threadfence();
        fence_proxy_async_global();
        named_bar_sync(1, 128);
        if (et == 0) red_release_add_gpu(args.done + t.e, 1);
      }
      acc ^= 1;
      if (acc == 0) apar ^= 1u;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------- CTA pairs --
// Prefill on pairs of SMs (clusters of two CTAs) with 256-token units.  One
// tcgen05.mma.cta_group::2 of M = 256 covers both CTAs' 128-row weight blocks (CTA r
// holds block 2 * pb + r of A) and up to 256 tokens, of which CTA r holds rows
// [r * N/2, (r + 1) * N/2) of B; each CTA's TMEM receives the 128 x N fp32 accumulator
// of its own weight block.  Per SM an instruction then does 128 x 256 x 32, twice the
// one-CTA kernel's 128 x 128 x 32, for the same issue work and for half the shared-
// memory operand traffic per FLOP (the bounds of the one-CTA kernel).  An expert's last
// unit absorbs up to 32 rows beyond 256 through a second MMA of N = 32 per K step
// (each CTA holding 16 of those rows), writing accumulator columns 256..287, so that
// experts of 257..288 rows need no second, nearly empty unit.
//
// TMEM: one accumulator of 288 columns and five 16-column scale slots (SFA, then the
// B scale atoms of rows 0-127, 128-255 and the absorbed rows) do not leave room for a
// second accumulator, so the MMAs of a unit wait until both CTAs' epilogues have read
// the previous one.  Eight epilogue warps (two per TMEM lane quarter, each taking
// every other 32-token chunk) keep that drain short.
//
// Roles (384 threads): warp 0 lane 0 loads the weight tile and its scale atom, warp 2
// lane 0 the token rows (this CTA's half) and the token block's B scale atoms (in both
// CTAs); in the even CTA warp 3 lane 0 copies each stage's scale atoms into both
// CTAs' TMEM (tcgen05.cp.cta_group::2, each CTA from its own shared memory) and warp 1
// lane 0 issues the MMAs; in the odd CTA warp 3 lane 0 passes each landed stage on to
// the even CTA's `full` barrier (a relaxed remote arrive).  Stage release and
// accumulator completion are committed to both CTAs (multicast); the accumulator's
// `tempty` barrier lives in the even CTA and counts the epilogue warps of both.
struct PairMx {
  static constexpr int kBN = 256;                  // tokens of a unit's main MMA
  static constexpr int kTail = 32;                 // rows the last unit of an expert absorbs
  static constexpr int kMaxRows = kBN + kTail;
  static constexpr int kPad = 128;                 // row padding of the expert blocks
  static constexpr int kStages = 6;
  static constexpr int kEpiGroups = 3;             // epilogue warps per TMEM lane quarter
  static constexpr int kEpiWarps = 4 * kEpiGroups;
  static constexpr int kThreads = 32 * (4 + kEpiWarps);
  static constexpr int kChunks = (kMaxRows / 32 + kEpiGroups - 1) / kEpiGroups;  // per warp
  static constexpr int kBBytes = (kBN / 2) * kBK;  // this CTA's half of the main token block
  static constexpr int kTBytes = (kTail / 2) * kBK;// this CTA's half of the absorbed rows
  static constexpr int kSfAtoms = 4;               // SFA, SFB rows 0-127, 128-255, absorbed
  static constexpr int kSfStageCols = 4 * kSfAtoms;
  static constexpr int kSfCol = kMaxRows;          // scale slots follow the accumulator
  static constexpr int kTmemCols = 512;
  static constexpr int kEpiGroupBytes = 2 * 128 * 4;          // block-maximum swaps, phase 0
  static constexpr int kEpiBytes = kEpiGroups * kEpiGroupBytes;
  static constexpr int kMaxUnits = 256;
  // registers: 65536 / 512 at launch; the epilogue warpgroups hold kChunks x 32 values
  static constexpr int kLaunchRegs = 128;
  static constexpr int kRoleRegs = 56, kEpiRegs = 152;
  static constexpr int kA = 0;
  static constexpr int kB = kA + kStages * kABytes;
  static constexpr int kT = kB + kStages * kBBytes;
  static constexpr int kSf = kT + kStages * kTBytes;
  static constexpr int kEpi = kSf + kStages * kSfAtoms * kSfBytes;
  static constexpr int kBar = kEpi + kEpiBytes;
  static constexpr int kNumBars = 3 * kStages + 4;  // full, empty, sfready; tfull, tempty, fin, fin_sf
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kTables = kMisc + 16;
  static constexpr int kUnits = kTables + (4 * (kMaxE + 1) + 16) * 4;  // scan scratch: 16 warps
  static constexpr int kEnd = kUnits + kMaxUnits * 8;
  static constexpr int kSmemBytes = kEnd + 1024;
  static_assert(kBar % 8 == 0 && kUnits % 8 == 0, "barrier and unit list alignment");
  static_assert(kB % 1024 == 0 && kT % 1024 == 0 && kBBytes % 1024 == 0 && kTBytes % 1024 == 0,
                "swizzle atoms");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kSfCol + kSfStageCols * kStages <= kTmemCols, "tensor memory budget");
  static_assert(kThreads * kLaunchRegs <= 65536, "launch registers");
  static_assert(128 * kRoleRegs + 32 * kEpiWarps * kEpiRegs <= kThreads * kLaunchRegs,
                "register split within the launch's registers");
  static_assert(kChunks * kEpiGroups * 32 >= kMaxRows, "chunks cover a unit");
};
static_assert(token_blocks<256, 32>(256) == 1 && token_blocks<256, 32>(288) == 1 &&
                  token_blocks<256, 32>(289) == 2 && token_blocks<256, 32>(544) == 2 &&
                  token_blocks<256, 32>(545) == 3,
              "pair token blocks");

// The 32-token chunks an epilogue warp reads: chunk i holds the tokens
// c0 = 32 * (g + kEpiGroups * i) of the warp's 32 TMEM lanes (quarter q).
constexpr int kPairChunks = PairMx::kChunks;

// The epilogue's work on the chunks it has read (the accumulator is free again by
// then).  Phase 0 applies SwiGLU and MX-quantises h along I.  Warps q and q + 2 of a
// group hold the gate and up rows of the same 32 features (lanes); they swap half of
// each chunk through shared memory, so the gate warp finishes tokens 0-15 of the
// chunk and the up warp tokens 16-31, each lane one feature.  Each token's block
// maximum over the warp's 32 lanes comes from a butterfly (16 values halved over
// lane offsets 16, 8, 4, 2, then combined over offset 1: lanes 2t and 2t + 1 end
// with token t's maximum), the scale exponent is broadcast back, and every lane
// writes its code byte of each token row (32 consecutive bytes per token).  Phase 1
// writes y in bf16 through a 32 x 32 transpose.
__device__ __forceinline__ void pair_epilogue(const MxArgs& args, const Unit& t,
                                              float (&acc)[kPairChunks][32], uint8_t* sEpi,
                                              int q, int g, int lane, int& nchunk) {
  constexpr int kPad = PairMx::kPad, kG = PairMx::kEpiGroups;
  if (t.ph == 0) {
    float* xs = reinterpret_cast<float*>(sEpi) + (g * 2 + (q >> 1)) * 128;
#pragma unroll
    for (int i = 0; i < kPairChunks; ++i) {
      const int c0 = 32 * (g + kG * i);
      if (c0 >= t.rows) break;
      swiglu_mx_chunk<kPad>(args, acc[i], t.row0, c0, t.rows, t.mb, q, lane, xs, nchunk & 1,
                            2 + (q >> 1) + 2 * g);
      ++nchunk;
    }
  } else {
    // lane l holds output feature q * 32 + l of the CTA's weight block for 32 tokens;
    // one shuffle per token pair gives the even lanes two neighbouring features of
    // token j and the odd lanes two of token j + 1, so each store writes 64 bytes of
    // each of two rows
    const int ld = args.ld[1];
    const bool even = (lane & 1) == 0;
    uint16_t* ycol = args.y + t.mb * kBM + q * 32 + (lane & ~1);
#pragma unroll
    for (int i = 0; i < kPairChunks; ++i) {
      const int c0 = 32 * (g + kG * i);
      if (c0 >= t.rows) break;
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float x = __shfl_xor_sync(0xffffffffu, even ? acc[i][j + 1] : acc[i][j], 1);
        const uint32_t pk = even ? pack_bf16x2(acc[i][j], x) : pack_bf16x2(x, acc[i][j + 1]);
        const int tok = c0 + j + (even ? 0 : 1);
        if (tok < t.rows) *reinterpret_cast<uint32_t*>(ycol + (size_t)(t.row0 + tok) * ld) = pk;
      }
    }
  }
}

// Pair unit u: phase, expert, the pair's 256-row weight block (mb; the units per
// expert are counted in 256-row blocks), token block of up to 256 + 32 rows.
__device__ __forceinline__ Unit decode_pair_unit(int u, const Tables& tb) {
  return decode_unit<PairMx::kBN, PairMx::kTail>(u, tb);
}

// The units a pair runs, in increasing unit order.  Round-robin (units pair,
// pair + npairs, ...) unless the launch has a unit counter: then a pair's first two
// units are those of the round-robin walk and each further one is drawn from the
// counter (unit 2 * npairs + ticket) by the even CTA's weight producer, which draws
// the entry after next at the start of each unit and publishes the next one then, in
// both CTAs' lists, so pairs whose units ran faster take more of them.  An entry is
// one 64-bit word (pending until published; an end entry closes the list), written
// and polled with relaxed accesses at cluster scope: the word is its own flag.  Every
// role walks the same list, and a pair's list increases like a round-robin one, so a
// down-projection unit still only waits for gate/up units that pairs drew before it.
struct PairList {
  uint32_t units_addr;   // shared::cta address of the CTA's list
  int pair, npairs, total;
  bool drawn, use_list;
};

// 1: unit ui is in t; 0: the list ended before ui; -1: the wait for entry ui ran
// out (or the CTA is aborting).
__device__ __forceinline__ int pair_unit(const PairList& pl, const Tables& tb, int ui, Unit& t,
                                         const volatile int* abort) {
  if (!pl.drawn) {
    const int u = pl.pair + ui * pl.npairs;
    if (u >= pl.total) return 0;
    if (pl.use_list) {
      const uint64_t v = ld_relaxed_cluster_u64(pl.units_addr + 8u * static_cast<uint32_t>(ui));
      t = unpack_unit(make_uint2(static_cast<uint32_t>(v), static_cast<uint32_t>(v >> 32)));
    } else {
      t = decode_pair_unit(u, tb);
    }
    return 1;
  }
  const uint32_t a = pl.units_addr + 8u * static_cast<uint32_t>(ui);
  uint64_t v = ld_relaxed_cluster_u64(a);
  if (static_cast<uint32_t>(v >> 32) == kPendingUnitWord) {
    const unsigned long long t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
      __nanosleep(32);
      v = ld_relaxed_cluster_u64(a);
      if (static_cast<uint32_t>(v >> 32) != kPendingUnitWord) break;
      if ((n & 15u) == 0 && (*abort || globaltimer() - t0 > kWaitLimitNs)) return -1;
    }
  }
  if (static_cast<uint32_t>(v >> 32) == kEndUnitWord) return 0;
  t = unpack_unit(make_uint2(static_cast<uint32_t>(v), static_cast<uint32_t>(v >> 32)));
  return 1;
}

__global__ void __launch_bounds__(PairMx::kThreads, 1)
    grouped_gemm_mx_pair_kernel(const __grid_constant__ CUtensorMap tmA0,
                                const __grid_constant__ CUtensorMap tmB0,
                                const __grid_constant__ CUtensorMap tmA1,
                                const __grid_constant__ CUtensorMap tmB1,
                                const __grid_constant__ CUtensorMap tmX0,   // 16-row tail boxes
                                const __grid_constant__ CUtensorMap tmX1, const MxArgs args) {
  using S = PairMx;
  constexpr int kStages = S::kStages, kSfAtoms = S::kSfAtoms, kSfStageCols = S::kSfStageCols;
  constexpr int kSfCol = S::kSfCol, kBN = S::kBN, kTail = S::kTail, kPad = S::kPad;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem + S::kA;
  uint8_t* sB = smem + S::kB;
  uint8_t* sT = smem + S::kT;
  uint8_t* sSF = smem + S::kSf;
  uint8_t* sEpi = smem + S::kEpi;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBar);
  uint64_t* empty = full + kStages;
  uint64_t* sfready = empty + kStages;   // used in the even CTA only
  uint64_t* tfull = sfready + kStages;
  uint64_t* tempty = tfull + 1;          // waited on in the even CTA only
  uint64_t* fin = tempty + 1;
  uint64_t* fin_sf = fin + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + S::kMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + S::kMisc + 4);
  int* s_off = reinterpret_cast<int*>(smem + S::kTables);
  int* s_poff = s_off + (kMaxE + 1);
  int* s_uoff0 = s_poff + (kMaxE + 1);
  int* s_uoff1 = s_uoff0 + (kMaxE + 1);
  int* s_tmp = s_uoff1 + (kMaxE + 1);
  uint2* s_units = reinterpret_cast<uint2*>(smem + S::kUnits);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = args.E;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(blockIdx.x >> 1), npairs = static_cast<int>(gridDim.x >> 1);
  pdl_trigger();

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      // even CTA: its two producers + the odd CTA's forwarded arrival
      mbar_init(&full[s], leader ? 3 : 2);
      mbar_init(&empty[s], 1);
      mbar_init(&sfready[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 2 * S::kEpiWarps);   // the epilogue warps of both CTAs
    mbar_init(fin, 1);
    mbar_init(fin_sf, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA0);
    tma_prefetch_desc(&tmB0);
    tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB1);
    tma_prefetch_desc(&tmX0);
    tma_prefetch_desc(&tmX1);
  }
  if (warp == 2) {
    tmem_alloc_pair(s_tmem, S::kTmemCols);
    tmem_relinquish_pair();
  }
  for (int i = tid; i <= E; i += S::kThreads) s_off[i] = args.offsets[i];
  __syncthreads();

  // pair units per expert (per phase) and the 128-row padded offsets, by block scans
  {
    int v[3] = {0, 0, 0};
    if (tid < E) {
      const int m = s_off[tid + 1] - s_off[tid];
      const int nb = token_blocks<kBN, kTail>(m);
      v[0] = args.active[0] ? nb * (args.MW[0] / (2 * kBM)) : 0;
      v[1] = args.active[1] ? nb * (args.MW[1] / (2 * kBM)) : 0;
      v[2] = ((m + kPad - 1) / kPad) * kPad;
    }
    int* dsts[3] = {s_uoff0, s_uoff1, s_poff};
    for (int p = 0; p < 3; ++p) {
      int inc = v[p];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      if (lane == 31) s_tmp[warp] = inc;
      __syncthreads();
      int pre = 0, tot = 0;
      for (int w = 0; w < S::kThreads / 32; ++w) {
        if (w < warp) pre += s_tmp[w];
        tot += s_tmp[w];
      }
      if (tid < E) dsts[p][tid] = pre + inc - v[p];
      if (tid == 0) dsts[p][E] = tot;
      __syncthreads();
    }
  }
  Tables tb;
  tb.off = s_off;
  tb.poff = s_poff;
  tb.uoff[0] = s_uoff0;
  tb.uoff[1] = s_uoff1;
  tb.E = E;
  const int total = s_uoff0[E] + s_uoff1[E];
  const int my_units = pair < total ? (total - pair + npairs - 1) / npairs : 0;
  // the same in every thread of the grid.  A drawn list holds at most kMaxUnits - 1
  // units; at most half of the pairs can fill theirs, so the others draw the rest.
  PairList pl;
  pl.units_addr = smem_u32(s_units);
  pl.pair = pair;
  pl.npairs = npairs;
  pl.total = total;
  pl.drawn = args.sched != nullptr && total <= (S::kMaxUnits - 1) * (npairs / 2);
  pl.use_list = pl.drawn || my_units <= S::kMaxUnits;
  if (pl.drawn) {
    // entries 0 and 1 are the round-robin walk's, the others pending; both CTAs
    // write theirs before the cluster barrier below, ahead of any published entry
    for (int i = tid; i < S::kMaxUnits; i += S::kThreads) {
      const int u = pair + i * npairs;
      s_units[i] = i >= 2            ? make_uint2(0, kPendingUnitWord)
                   : u < total ? pack_unit(decode_pair_unit(u, tb))
                               : make_uint2(0, kEndUnitWord);
    }
  } else if (pl.use_list) {
    for (int i = tid; i < my_units; i += S::kThreads)
      s_units[i] = pack_unit(decode_pair_unit(pair + i * npairs, tb));
  }
  __syncthreads();
  tc_fence_after_sync();
  // both CTAs' barriers are initialised, their lists started and TMEM allocated
  // before any remote arrive or store
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = *s_tmem;
  const uint32_t lead_full0 = mapa_shared(smem_u32(&full[0]), 0);
  const uint32_t lead_tempty = mapa_shared(smem_u32(tempty), 0);
  // Registers: the role warpgroup needs few, the epilogue warpgroups hold up to
  // kPairChunks x 32 accumulator values each (kRoleRegs and kEpiRegs share out the
  // launch's kThreads x kLaunchRegs); each warpgroup's setmaxnreg opens its branch.
  if (warp < 4) {
    setmaxnreg_dec<S::kRoleRegs>();
    if ((warp == 0 || warp == 2) && lane == 0) {
      // ------------------------------------------------------ TMA producers --
      const bool weights = warp == 0;
      const uint64_t pol_w_reused = l2_policy_evict_normal();
      const uint64_t pol_w_once = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      int stage = 0;
      uint32_t par = 0;
      uint32_t issued_mask = 0, issued_par = 0;
      bool ok = true;
      // the even CTA's weight producer draws the units of a drawn list: at the start
      // of unit ui it publishes entry ui + 1 (drawn one unit earlier; entries 0 and 1
      // are the round-robin walk's) and draws entry ui + 2 (the list's last entry is
      // kept for the end entry)
      const bool drawer = pl.drawn && leader && weights;
      bool open = drawer && pair + npairs < total;   // entry 1 is a unit
      int ticket = 0;
      for (int ui = 0; ok; ++ui) {
        Unit t;
        const int got = pair_unit(pl, tb, ui, t, s_abort);
        if (got <= 0) {
          ok = got == 0;
          break;
        }
        if (open) {
          if (ui >= 1) {
            const int un = ticket >= 0 ? 2 * npairs + ticket : total;
            const uint64_t w = un < total ? unit_word(pack_unit(decode_pair_unit(un, tb)))
                                          : unit_word(make_uint2(0, kEndUnitWord));
            const uint32_t entry = pl.units_addr + 8u * static_cast<uint32_t>(ui + 1);
            st_relaxed_cluster_u64(mapa_shared(entry, 1), w);
            st_relaxed_cluster_u64(mapa_shared(entry, 0), w);
            open = un < total;
          }
          if (open) ticket = ui + 2 <= S::kMaxUnits - 2 ? atomicAdd(args.sched, 1) : -1;
        }
        if (!weights && t.ph == 1 && args.done != nullptr) {
          // the down projection's activations are h of this expert's gate/up units
          const int m = s_off[t.e + 1] - s_off[t.e];
          const int need = token_blocks<kBN, kTail>(m) * (args.MW[0] / kBM);
          if (!wait_counter(args.done + t.e, need, s_abort)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
        }
        const int nk = args.K[t.ph] / kBK;
        const int mb = 2 * t.mb + static_cast<int>(rank);      // this CTA's 128-row block
        const bool tail = t.rows > kBN;
        const int nmain = tail ? kBN : ((t.rows + 15) & ~15);
        const int half = nmain >> 1;
        // weight tiles of an expert with one token block are read once: stream them
        const uint64_t pol_w =
            token_blocks<kBN, kTail>(s_off[t.e + 1] - s_off[t.e]) == 1 ? pol_w_once : pol_w_reused;
        const int nsfb = nmain > 128 ? 2 : 1;
        const uint32_t abytes = args.a_fp4[t.ph] ? kABytes / 2 : kABytes;
        const uint32_t bytes = weights ? abytes + kSfBytes
                                       : S::kBBytes + nsfb * kSfBytes + (tail ? S::kTBytes + kSfBytes : 0);
        const int arow = t.e * args.MW[t.ph] + mb * kBM;
        const int atile0 = (t.e * (args.MW[t.ph] / kBM) + mb) * nk;
        const uint8_t* sfsrc =
            weights ? args.a_sf[t.ph] + ((size_t)(t.e * (args.MW[t.ph] / kBM) + mb) * nk) * kSfBytes
                    : args.b_sf[t.ph] + ((size_t)(t.row0 / kPad) * nk) * kSfBytes;
        const int hrow0 = t.row0 + static_cast<int>(rank) * half;
        const int trow0 = t.row0 + kBN + static_cast<int>(rank) * (kTail / 2);
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&empty[stage], par ^ 1u, s_abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], bytes);
          uint8_t* sf = sSF + stage * kSfAtoms * kSfBytes;
          if (weights) {
            if (args.a_fp4[t.ph])  // tile-major e2m1: tile (e, mb, kb) is rows [128 * tile, +128)
              tma_load_2d(sA + stage * kABytes, t.ph ? &tmA1 : &tmA0, &full[stage], 0,
                          (atile0 + kb) * kBM, pol_w);
            else
              tma_load_2d(sA + stage * kABytes, t.ph ? &tmA1 : &tmA0, &full[stage], kb * kBK, arow,
                          pol_w);
            bulk_load_1d(sf, sfsrc + (size_t)kb * kSfBytes, kSfBytes, &full[stage], pol_w);
          } else {
            tma_load_2d(sB + stage * S::kBBytes, t.ph ? &tmB1 : &tmB0, &full[stage], kb * kBK, hrow0,
                        pol_x);
            // the token block's B scales, in both CTAs (each CTA's MMA scales all N columns)
            bulk_load_1d(sf + kSfBytes, sfsrc + (size_t)kb * kSfBytes, kSfBytes, &full[stage], pol_x);
            if (nsfb == 2)
              bulk_load_1d(sf + 2 * kSfBytes, sfsrc + ((size_t)nk + kb) * kSfBytes, kSfBytes,
                           &full[stage], pol_x);
            if (tail) {
              tma_load_2d(sT + stage * S::kTBytes, t.ph ? &tmX1 : &tmX0, &full[stage], kb * kBK,
                          trow0, pol_x);
              bulk_load_1d(sf + 3 * kSfBytes, sfsrc + ((size_t)2 * nk + kb) * kSfBytes, kSfBytes,
                           &full[stage], pol_x);
            }
          }
          issued_mask |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (par << stage);
          if (++stage == kStages) {
            stage = 0;
            par ^= 1u;
          }
        }
      }
      if (ok && weights) {
        // every stage released by the pair's MMAs (their multicast commits have landed)
        for (int i = 0; i < kStages; ++i) {
          if (!mbar_wait(&empty[stage], par ^ 1u, s_abort)) {
            ok = false;
            break;
          }
          if (++stage == kStages) {
            stage = 0;
            par ^= 1u;
          }
        }
      }
      if (!ok) {
        *s_abort = 1;
        flag_status(args.status, MOE_DEV_WAIT_TIMEOUT);
        // let this thread's copies land before the CTA can exit (bounded waits)
        for (int s2 = 0; s2 < kStages; ++s2)
          if ((issued_mask >> s2) & 1u) mbar_wait(&full[s2], (issued_par >> s2) & 1u, nullptr);
      }
    } else if (warp == 3 && lane == 0) {
      // ------------ even CTA: scale copier; odd CTA: forwarder of its landed stages --
      int stage = 0;
      uint32_t par = 0;
      bool ok = true;
      for (int ui = 0; ok; ++ui) {
        Unit t;
        const int got = pair_unit(pl, tb, ui, t, s_abort);
        if (got <= 0) {
          ok = got == 0;
          break;
        }
        const int nk = args.K[t.ph] / kBK;
        const bool tail = t.rows > kBN;
        const bool two = tail || t.rows > 128;
        for (int kb = 0; kb < nk; ++kb) {
          if (leader) {
            if (!mbar_wait_cluster(&full[stage], par, s_abort)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t sfa_t = tmem_base + static_cast<uint32_t>(kSfCol + stage * kSfStageCols);
            const uint32_t sf_s = smem_u32(sSF + stage * kSfAtoms * kSfBytes);
            tc_cp_pair_32x128b_warpx4(sfa_t, smem_desc_noswz(sf_s, 128));
            tc_cp_pair_32x128b_warpx4(sfa_t + 4, smem_desc_noswz(sf_s + kSfBytes, 128));
            if (two) tc_cp_pair_32x128b_warpx4(sfa_t + 8, smem_desc_noswz(sf_s + 2 * kSfBytes, 128));
            if (tail)
              tc_cp_pair_32x128b_warpx4(sfa_t + 12, smem_desc_noswz(sf_s + 3 * kSfBytes, 128));
            tc_commit_pair(&sfready[stage], 1);
          } else {
            if (!mbar_wait(&full[stage], par, s_abort)) {
              ok = false;
              break;
            }
            // this stage's bytes are in this CTA's shared memory (observed above)
            mbar_arrive_cluster_relaxed(lead_full0 + stage * 8);
          }
          if (++stage == kStages) {
            stage = 0;
            par ^= 1u;
          }
        }
      }
      if (!ok) {
        *s_abort = 1;
        flag_status(args.status, MOE_DEV_WAIT_TIMEOUT);
        if (leader) {
          tc_commit_pair(fin_sf, 1);
          mbar_wait(fin_sf, 0, nullptr);
        }
      }
    } else if (warp == 1 && lane == 0 && leader) {
      // ----------------------------------------------- even CTA: MMA issuer --
      int stage = 0;
      uint32_t par = 0, apar = 0;
      bool ok = true;
      for (int ui = 0; ok; ++ui) {
        Unit t;
        const int got = pair_unit(pl, tb, ui, t, s_abort);
        if (got <= 0) {
          ok = got == 0;
          break;
        }
        const bool tail = t.rows > kBN;
        const int nmain = tail ? kBN : ((t.rows + 15) & ~15);
        const uint32_t fp4 = args.a_fp4[t.ph] ? (5u << 7) : 0u;
        const uint32_t idesc_main = idesc_mxf8_f32(2 * kBM, nmain, 0, 0) | fp4;
        const uint32_t idesc_tail = idesc_mxf8_f32(2 * kBM, kTail, 0, 0) | fp4;
        // both CTAs' epilogues have read the previous unit's accumulator
        if (!mbar_wait_cluster(tempty, apar ^ 1u, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d = tmem_base;
        const int nk = args.K[t.ph] / kBK;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&sfready[stage], par, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sfa_t = tmem_base + static_cast<uint32_t>(kSfCol + stage * kSfStageCols);
          const uint64_t adesc = smem_desc_sw128(smem_u32(sA + stage * kABytes));
          const uint64_t bdesc = smem_desc_sw128(smem_u32(sB + stage * S::kBBytes));
  #pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk)   // +32 bytes along K = +2 in the start field
            tc_mma_pair_mxf8(d, adesc + 2 * kk, bdesc + 2 * kk, idesc_main | idesc_sf_ids(kk, kk),
                             sfa_t, sfa_t + 4, (kb | kk) ? 1u : 0u);
          if (tail) {
            const uint64_t tdesc = smem_desc_sw128(smem_u32(sT + stage * S::kTBytes));
  #pragma unroll
            for (int kk = 0; kk < kBK / 32; ++kk)
              tc_mma_pair_mxf8(d + kBN, adesc + 2 * kk, tdesc + 2 * kk,
                               idesc_tail | idesc_sf_ids(kk, kk), sfa_t, sfa_t + 12,
                               (kb | kk) ? 1u : 0u);
          }
          tc_commit_pair(&empty[stage], 3);
          if (++stage == kStages) {
            stage = 0;
            par ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair(tfull, 3);
        apar ^= 1u;
      }
      // the last unit's epilogues (the odd CTA's arrivals are remote) finish before exit
      if (ok && !mbar_wait_cluster(tempty, apar ^ 1u, s_abort)) ok = false;
      if (!ok) {
        *s_abort = 1;
        flag_status(args.status, MOE_DEV_WAIT_TIMEOUT);
        tc_commit_pair(fin, 1);
        mbar_wait(fin, 0, nullptr);
      }
    }
  } else {
    setmaxnreg_inc<S::kEpiRegs>();
    // ------------------------------------------------------------ epilogue --
    const int q = warp & 3;                  // TMEM lane quarter
    const int g = (warp - 4) >> 2;           // chunk group: 32-token chunks g, g + 3, ...
    const int et = tid - 128;
    int* s_flag = s_tmp;
    int nchunk = 0;                          // gate/up chunks so far (the xs slot parity)
    uint32_t apar = 0;
    for (int ui = 0;; ++ui) {
      // one thread waits for the unit and its accumulator; s_flag[0]: 1 go, 0 the
      // list has ended, -1 a wait ran out
      if (et == 0) {
        Unit t0;
        int st = pair_unit(pl, tb, ui, t0, s_abort);
        if (st == 1) {
          if (!mbar_wait(tfull, apar, s_abort)) st = -1;
          const uint2 w = pack_unit(t0);
          s_flag[1] = static_cast<int>(w.x);
          s_flag[2] = static_cast<int>(w.y);
        }
        s_flag[0] = st;
      }
      named_bar_sync(1, 32 * S::kEpiWarps);
      const int st = s_flag[0];
      Unit t = unpack_unit(make_uint2(static_cast<uint32_t>(s_flag[1]), static_cast<uint32_t>(s_flag[2])));
      named_bar_sync(1, 32 * S::kEpiWarps);
      if (st <= 0) {
        if (st < 0 && et == 0) {
          *s_abort = 1;
          flag_status(args.status, MOE_DEV_WAIT_TIMEOUT);
        }
        break;
      }
      t.mb = 2 * t.mb + static_cast<int>(rank);
      tc_fence_after_sync();
      // read this warp's chunks into registers, then hand the accumulator back to the
      // MMA thread before working on them
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      float acc[kPairChunks][32];
#pragma unroll
      for (int i = 0; i < kPairChunks; ++i) {
        const int c0 = 32 * (g + S::kEpiGroups * i);
        if (c0 < t.rows) tmem_ld_32x32b_x32_nowait(tbase + c0, acc[i]);
      }
      tmem_wait_ld();
      tc_fence_before_sync();
      __syncwarp();
      // the TMEM reads are complete (tcgen05.wait::ld above), so the odd CTA's remote
      // arrive needs no release: a release at cluster scope would first wait for this
      // thread's global stores of the previous unit
      if (lane == 0) {
        if (leader) mbar_arrive(tempty);
        else mbar_arrive_cluster_relaxed(lead_tempty);
      }
      pair_epilogue(args, t, acc, sEpi, q, g, lane, nchunk);
      if (t.ph == 0 && args.done != nullptr) {
        __threadfence();
        fence_proxy_async_global();
        named_bar_sync(1, 32 * S::kEpiWarps);
        if (et == 0) red_release_add_gpu(args.done + t.e, 1);
      }
      apar ^= 1u;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();
  if (warp == 2) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, S::kTmemCols);
  }
}

bool encode_tmap_2d_u8(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t rows,
                       uint32_t box_inner, uint32_t box_rows) {
  return encode_tmap_2d(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, inner, rows, box_inner,
                        box_rows);
}

// Tile-major packed e2m1 weights seen as (E * MW * K / 128) rows of 128 codes (64
// bytes); TMA unpacks each 16-code group into 8 data bytes + 8 gap bytes, so a
// 128 x 128 box fills the same 16 KB of 128-byte smem rows as an e4m3 tile.
bool encode_tmap_2d_fp4(CUtensorMap* tm, const void* base, uint64_t rows) {
  return encode_tmap_2d_strided(tm, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, base, kBK, rows,
                                kBK / 2, kBK, kBM);
}

template <class S>
cudaError_t launch_shape(const GemmPhaseMx* ph0, const GemmPhaseMx* ph1, const int32_t* offsets,
                         int E, int P_pad_rows, int* done, int* status, cudaStream_t s) {
  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
      err = cudaFuncSetAttribute(grouped_gemm_mx_kernel<S>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
      if (err != cudaSuccess) return err;
      attr_set[dev] = true;
    }
  }
  MxArgs a{};
  a.offsets = offsets;
  a.E = E;
  a.done = (ph0 && ph1) ? done : nullptr;
  a.status = status;
  CUtensorMap tm[6];   // A0, B0, A1, B1, then the absorbed-row B boxes of both phases
  const GemmPhaseMx* phs[2] = {ph0, ph1};
  for (int p = 0; p < 2; ++p) {
    const GemmPhaseMx* g = phs[p] ? phs[p] : (ph0 ? ph0 : ph1);
    a.active[p] = phs[p] != nullptr;
    a.K[p] = g->K;
    a.MW[p] = g->MW;
    a.ld[p] = g->n_out;
    a.a_sf[p] = g->A_sf;
    a.b_sf[p] = g->B_sf;
    a.a_fp4[p] = g->a_fp4 ? 1 : 0;
    const bool ok_a =
        g->a_fp4 ? encode_tmap_2d_fp4(&tm[2 * p], g->A_q, (uint64_t)E * g->MW * (g->K / kBK))
                 : encode_tmap_2d_u8(&tm[2 * p], g->A_q, (uint64_t)g->K, (uint64_t)E * g->MW, kBK,
                                     kBM);
    if (!ok_a) return cudaErrorInvalidValue;
    if (!encode_tmap_2d_u8(&tm[2 * p + 1], g->B_q, (uint64_t)g->K, (uint64_t)P_pad_rows, kBK,
                           S::kBoxRows))
      return cudaErrorInvalidValue;
    if (S::kAbsorb > 0) {
      if (!encode_tmap_2d_u8(&tm[4 + p], g->B_q, (uint64_t)g->K, (uint64_t)P_pad_rows, kBK,
                             S::kAbsorb))
        return cudaErrorInvalidValue;
    } else {
      tm[4 + p] = tm[2 * p + 1];
    }
  }
  if (ph0) {
    a.hq = ph0->out_q;
    a.h_sf = ph0->out_sf;
  }
  if (ph1) a.y = ph1->out_bf16;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(device_sm_count(), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = S::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = a.done != nullptr ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_mx_kernel<S>, tm[0], tm[1], tm[2], tm[3], tm[4],
                            tm[5], a);
}

cudaError_t launch_pair_mx(const GemmPhaseMx* ph0, const GemmPhaseMx* ph1, const int32_t* offsets,
                           int E, int P_pad_rows, int* done, int* status, cudaStream_t s) {
  using S = PairMx;
  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
      err = cudaFuncSetAttribute(grouped_gemm_mx_pair_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
      if (err != cudaSuccess) return err;
      attr_set[dev] = true;
    }
  }
  MxArgs a{};
  a.offsets = offsets;
  a.E = E;
  a.done = (ph0 && ph1) ? done : nullptr;
  a.sched = a.done != nullptr ? done + E : nullptr;   // zeroed with the dependency counters
  a.status = status;
  CUtensorMap tm[6];   // A0, B0, A1, B1 (128-row boxes), then the 16-row tail boxes
  const GemmPhaseMx* phs[2] = {ph0, ph1};
  for (int p = 0; p < 2; ++p) {
    const GemmPhaseMx* g = phs[p] ? phs[p] : (ph0 ? ph0 : ph1);
    a.active[p] = phs[p] != nullptr;
    a.K[p] = g->K;
    a.MW[p] = g->MW;
    a.ld[p] = g->n_out;
    a.a_sf[p] = g->A_sf;
    a.b_sf[p] = g->B_sf;
    a.a_fp4[p] = g->a_fp4 ? 1 : 0;
    const bool ok_a =
        g->a_fp4 ? encode_tmap_2d_fp4(&tm[2 * p], g->A_q, (uint64_t)E * g->MW * (g->K / kBK))
                 : encode_tmap_2d_u8(&tm[2 * p], g->A_q, (uint64_t)g->K, (uint64_t)E * g->MW, kBK,
                                     kBM);
    if (!ok_a) return cudaErrorInvalidValue;
    if (!encode_tmap_2d_u8(&tm[2 * p + 1], g->B_q, (uint64_t)g->K, (uint64_t)P_pad_rows, kBK,
                           S::kBN / 2) ||
        !encode_tmap_2d_u8(&tm[4 + p], g->B_q, (uint64_t)g->K, (uint64_t)P_pad_rows, kBK,
                           S::kTail / 2))
      return cudaErrorInvalidValue;
  }
  if (ph0) {
    a.hq = ph0->out_q;
    a.h_sf = ph0->out_sf;
  }
  if (ph1) a.y = ph1->out_bf16;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(device_sm_count() & ~1, 1, 1);
  cfg.blockDim = dim3(S::kThreads, 1, 1);
  cfg.dynamicSmemBytes = S::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  // co-residency for the phase dependency; profilers refuse cooperative cluster
  // launches, so profiling may ask for a plain cluster launch instead
  attr[1].val.cooperative = (a.done != nullptr && !pair_launch_noncooperative()) ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_mx_pair_kernel, tm[0], tm[1], tm[2], tm[3], tm[4],
                            tm[5], a);
}

// The pair kernel takes weight matrices that split into 256-row blocks.
bool pairable_mx(const GemmPhaseMx* g) { return g == nullptr || g->MW % (2 * kBM) == 0; }

}  // namespace

cudaError_t launch_grouped_gemm_mx(const GemmPhaseMx* ph0, const GemmPhaseMx* ph1,
                                   const int32_t* offsets, int E, int pad, int P_pad_rows,
                                   int* done, int* status, cudaStream_t s) {
  // few tokens per expert: narrow tiles and a deeper ring keep more weight bytes in flight
  if (pad == ShapeDecode::kPad) {
    const bool fp4 = (ph0 ? ph0->a_fp4 : false) || (ph1 ? ph1->a_fp4 : false);
    if (fp4) return launch_shape<ShapeDecodeFp4>(ph0, ph1, offsets, E, P_pad_rows, done, status, s);
    return launch_shape<ShapeDecode>(ph0, ph1, offsets, E, P_pad_rows, done, status, s);
  }
  if (pad != ShapePrefill::kPad) return cudaErrorInvalidValue;
  // Prefill-size tiles on CTA pairs where the shapes allow.  When the driver refuses
  // the cooperative cluster launch (not every SM free for a cluster, e.g. under a
  // profiler or next to another context), this call runs the one-CTA kernel; a device
  // that never accepted it is not asked again.
  static std::atomic<int> pair_state[64];  // 0 unknown, 1 launched, 2 refused
  int dev = 0;
  if (pairable_mx(ph0) && pairable_mx(ph1) && device_sm_count() >= 2 &&
      cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64 && pair_state[dev].load() != 2) {
    const cudaError_t err = launch_pair_mx(ph0, ph1, offsets, E, P_pad_rows, done, status, s);
    if (err == cudaSuccess) {
      pair_state[dev].store(1);
      return err;
    }
    (void)cudaGetLastError();   // a refused launch configuration is not a sticky error
    if (pair_state[dev].load() != 1) pair_state[dev].store(2);
  }
  return launch_shape<ShapePrefill>(ph0, ph1, offsets, E, P_pad_rows, done, status, s);
}

}  // namespace moe
