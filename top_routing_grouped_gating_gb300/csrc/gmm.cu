// Persistent grouped GEMM on the sm_103a tensor cores (tcgen05 + TMEM + TMA) for
// the expert MLPs of the page "基于Atlas A3、950训练/推理集群的Qwen3-MoE模型低时延
// 推理性能优化实践": §高性能专家计算 (grouped_matmul over all experts at once) with
// §计算分解's SwiGLU fused into the epilogue of the gate/up projection.
//
// Orientation.  Every tile is  D[128 weight rows][N tokens] = W_tile . X_tile^T :
// the packed weights are the MMA's A operand (M = 128 output features), the
// expert's token rows are the B operand (N = 16..BN tokens, a multiple of 16 set
// per tile from the expert's row count).  Decode-size experts (a few rows) then
// cost one thin MMA per K step while the 128-row weight tiles stream from HBM;
// prefill-size experts use N up to BN = 256 so each weight tile is reused by 256
// tokens.
//
// Work unit = (phase, expert, 128-row weight block, token block).  Phase 0 is the
// gate/up projection (weights packed so each 32-row quarter of a 128-row block
// holds 16 gate rows and the 16 matching up rows, paired by a warp shuffle in the
// epilogue); phase 1 is the down projection.  Units are numbered
// phase-major, expert-major, weight-block-major, token-block-minor and handed to
// CTAs round-robin (grid = SM count, one CTA per SM).  When both phases run in one
// launch, a phase-1 unit waits until every phase-0 unit of its expert has
// published its rows of h (per-expert counter, release/acquire + async-proxy
// fence); phase-0 units never wait, so the wait always ends.
//
// Warp roles (256 threads): warp 0 lane 0 = TMA producer; warp 1 lane 0 = MMA
// issuer; warp 2 = TMEM allocator; warps 4-7 = epilogue (warp w reads TMEM lanes
// 32*(w%4) .. +31).  Shared memory holds a STAGES-deep ring of (A 128x64, B BNx64)
// bf16 tiles in the 128-byte-swizzled K-major layout TMA writes; TMEM holds two
// 128 x BN fp32 accumulators so the epilogue of one unit overlaps the MMAs of the
// next.  Prefill-size token tiles run on the CTA-pair variant further down
// (grouped_gemm_pair_kernel): the same unit order and phase dependency on 256-row
// weight blocks, with a second pipeline for the experts that hold only a few tokens.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kBM = 128;         // weight rows per tile (MMA M)
constexpr int kBK = 64;          // K per stage: one 128-byte swizzle row of bf16
constexpr int kThreads = 256;
constexpr int kMaxE = 256;
// A CTA's units are decoded once in the prologue into shared memory, so a unit
// boundary costs each role one shared-memory load instead of a binary search and
// divisions; a longer list is decoded on the fly.
constexpr int kMaxUnits = 512;
constexpr int kABytes = kBM * kBK * 2;          // 16 KB
constexpr int kEpiBytes = 4 * 32 * 32 * 2;  // per epilogue warp: 32 tokens x 32 bf16

struct GemmArgs {
  const int32_t* offsets;
  int E;
  int K[2];
  int MW[2];
  int ld[2];
  int epi[2];       // 0: SwiGLU -> bf16, 1: bf16, 2: fp32 split-K partials
  int active[2];
  int ksplit[2];    // units per (expert, weight block, token block) along K
  int bseg[2];      // > 0: B's K coordinate = piece(k / bseg) * bseg + k % bseg
  uint32_t bmap[2]; // 3 bits per K segment: the piece of B it reads
  int mvalid[2];    // epi 2: valid weight rows (columns of the partial)
  int rows_total[2];// epi 2: rows of one partial slab
  uint16_t* out[2];
  float* out_f32[2];
  int* done;        // per-expert count of finished phase-0 units, or null
  int* sched;       // CTA pairs: counter the pairs draw heavy units from, or null
  int* status;
  // Test hook of the one-CTA kernel (moe_debug_set_gemm_stall): a producer that
  // reaches its stall_stage-th stage issues nothing more and waits for another role
  // to give up; every wait of the launch is bounded by wait_ns.  stall_stage < 0:
  // off (the normal case); wait_ns is then the library-wide limit.
  int stall_stage;
  unsigned long long wait_ns;
  // Pair kernel: 0 decides on the device whether experts of at most 32 rows run on
  // the light pipeline; 1 runs them there whenever there are any; 2 never.
  int light_mode;
};

template <int BN, int STAGES, int BOX>
struct Layout {
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kBoxBytes = BOX * kBK * 2;
  static constexpr int kA = 0;
  static constexpr int kB = kA + STAGES * kABytes;
  static constexpr int kEpi = kB + STAGES * kBBytes;
  static constexpr int kBar = kEpi + kEpiBytes;              // 8-byte aligned
  static constexpr int kNumBars = 2 * STAGES + 5;            // full, empty, tfull[2], tempty[2], fin
  static constexpr int kMisc = kBar + kNumBars * 8;          // tmem addr, abort flag
  static constexpr int kTables = kMisc + 16;                 // off, uoff0, uoff1 (kMaxE+1 each), scan tmp
  static constexpr int kUnits = kTables + ((3 * (kMaxE + 1) + 8) * 4 + 7) / 8 * 8;
  static constexpr int kEnd = kUnits + kMaxUnits * 8;
  static_assert(kUnits % 8 == 0, "unit list alignment");
  static constexpr int kSmemBytes = kEnd + 1024;             // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct Unit {
  int ph, e, mb, ks, row0, rows;
};

struct Tables {
  const int* off;
  const int* uoff[2];
  int ksplit[2];
  int E;
};

template <int BN>
__device__ __forceinline__ Unit decode_unit(int u, const Tables& tb) {
  Unit r;
  const int total0 = tb.uoff[0][tb.E];
  r.ph = (u < total0) ? 0 : 1;
  if (r.ph) u -= total0;
  const int* uo = tb.uoff[r.ph];
  int lo = 0, hi = tb.E;  // uo[lo] <= u < uo[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (uo[mid] <= u) lo = mid;
    else hi = mid;
  }
  r.e = lo;
  const int S = tb.ksplit[r.ph];
  const int local = u - uo[lo];
  r.ks = local % S;
  const int rest = local / S;
  const int m = tb.off[lo + 1] - tb.off[lo];
  const int nb = (m + BN - 1) / BN;
  r.mb = rest / nb;
  const int b = rest - r.mb * nb;
  r.row0 = tb.off[lo] + b * BN;
  r.rows = min(BN, tb.off[lo + 1] - r.row0);
  return r;
}

// A unit in two words: row0; ph | e << 1 | mb << 10 | rows << 19 | ks << 28 (e < 512,
// mb < 512, rows <= 256 and ks < 16 hold for every shape the entry points accept).
__device__ __forceinline__ uint2 pack_unit(const Unit& t) {
  return make_uint2(static_cast<uint32_t>(t.row0),
                    static_cast<uint32_t>(t.ph) | (static_cast<uint32_t>(t.e) << 1) |
                        (static_cast<uint32_t>(t.mb) << 10) | (static_cast<uint32_t>(t.rows) << 19) |
                        (static_cast<uint32_t>(t.ks) << 28));
}
__device__ __forceinline__ Unit unpack_unit(uint2 w) {
  Unit t;
  t.row0 = static_cast<int>(w.x);
  t.ph = static_cast<int>(w.y & 1u);
  t.e = static_cast<int>((w.y >> 1) & 511u);
  t.mb = static_cast<int>((w.y >> 10) & 511u);
  t.rows = static_cast<int>((w.y >> 19) & 511u);
  t.ks = static_cast<int>(w.y >> 28);
  return t;
}

__device__ __forceinline__ bool wait_counter(const int* p, int need, const volatile int* abort,
                                             unsigned long long limit_ns = kWaitLimitNs) {
  if (ld_acquire_gpu(p) >= need) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    __nanosleep(64);
    if (ld_acquire_gpu(p) >= need) return true;
    if ((i & 15u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > limit_ns) return false;
    }
  }
}

__device__ __forceinline__ uint16_t f2bf(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&b);
}

// Drains one accumulator (this warp's 32 TMEM lanes, t.rows token columns) into
// the unit's output: SwiGLU to bf16 h (epi 0), bf16 (epi 1) or fp32 split-K
// partials (epi 2).  Warp q of the epilogue group owns TMEM lanes 32q..32q+31.
__device__ __forceinline__ void epilogue_tile(const GemmArgs& args, const Unit& t,
                                              uint32_t tbase, uint8_t* sEpi, int q,
                                              int lane) {
  uint16_t* out = args.out[t.ph];
  const int ld = args.ld[t.ph];
  if (args.epi[t.ph] == 2) {
    // fp32 split-K partial: part[ks][row][col], col = weight row of this lane
    const int col = t.mb * kBM + q * 32 + lane;
    float* part = args.out_f32[t.ph] + (size_t)t.ks * args.rows_total[t.ph] * ld;
    for (int c0 = 0; c0 < t.rows; c0 += 32) {
      float v[32];
      tmem_ld_32x32b_x32(tbase + c0, v);
      if (col < args.mvalid[t.ph]) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c0 + j < t.rows) part[(size_t)(t.row0 + c0 + j) * ld + col] = v[j];
      }
    }
  } else if (args.epi[t.ph] == 0) {
    // Each 32-lane TMEM quarter holds 16 gate rows (lanes 0-15) and the 16
    // matching up rows (lanes 16-31).  One shuffle across the half-warps pairs
    // them: lanes 0-15 finish tokens 0-15 of the chunk, lanes 16-31 tokens 16-31,
    // for feature t.mb*64 + q*16 + (lane % 16).
    uint16_t* hw = reinterpret_cast<uint16_t*>(sEpi) + q * 32 * 16;  // [32 tok][16] bf16
    const bool lo = lane < 16;
    const int f = lane & 15;
    for (int c0 = 0; c0 < t.rows; c0 += 32) {
      float v[32];
      tmem_ld_32x32b_x32(tbase + c0, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float send = lo ? v[16 + j] : v[j];
        const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
        const float g = lo ? v[j] : recv;
        const float up = lo ? recv : v[16 + j];
        const float h = g / (1.0f + __expf(-g)) * up;
        hw[(lo ? j : 16 + j) * 16 + f] = f2bf(h);
      }
      __syncwarp();
      if (c0 + lane < t.rows) {
        const uint4* src = reinterpret_cast<const uint4*>(hw + lane * 16);
        uint4* dst = reinterpret_cast<uint4*>(out + (size_t)(t.row0 + c0 + lane) * ld +
                                              t.mb * 64 + q * 16);
        dst[0] = src[0];
        dst[1] = src[1];
      }
      __syncwarp();
    }
  } else {
    uint16_t* tbw = reinterpret_cast<uint16_t*>(sEpi) + q * 32 * 32;  // [32 tok][32] bf16
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
          *reinterpret_cast<uint4*>(out + (size_t)(t.row0 + c0 + j) * ld + t.mb * kBM +
                                    q * 32 + c * 8) = val;
        }
      }
      __syncwarp();
    }
  }
}

template <int BN, int STAGES, int BOX>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0,
                        const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmA1,
                        const __grid_constant__ CUtensorMap tmB1, const GemmArgs args) {
  using L = Layout<BN, STAGES, BOX>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem + L::kA;
  uint8_t* sB = smem + L::kB;
  uint8_t* sEpi = smem + L::kEpi;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* fin = tempty + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  int* s_off = reinterpret_cast<int*>(smem + L::kTables);
  int* s_uoff0 = s_off + (kMaxE + 1);
  int* s_uoff1 = s_uoff0 + (kMaxE + 1);
  int* s_tmp = s_uoff1 + (kMaxE + 1);
  uint2* s_units = reinterpret_cast<uint2*>(smem + L::kUnits);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = args.E;
  pdl_trigger();  // the finalize launch may start and wait for this grid to finish

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(fin, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA0);
    tma_prefetch_desc(&tmB0);
    tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB1);
  }
  if (warp == 2) {
    tmem_alloc(s_tmem, 2 * BN);
    tmem_relinquish();
  }
  for (int i = tid; i <= E; i += kThreads) s_off[i] = args.offsets[i];
  __syncthreads();

  // Units per expert and their exclusive prefix, per phase (E <= 256 = threads).
  {
    int u[2] = {0, 0};
    if (tid < E) {
      const int m = s_off[tid + 1] - s_off[tid];
      const int nb = (m + BN - 1) / BN;
      u[0] = args.active[0] ? nb * (args.MW[0] / kBM) * args.ksplit[0] : 0;
      u[1] = args.active[1] ? nb * (args.MW[1] / kBM) * args.ksplit[1] : 0;
    }
    for (int p = 0; p < 2; ++p) {
      int inc = u[p];
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
      int* dst = p ? s_uoff1 : s_uoff0;
      if (tid < E) dst[tid] = pre + inc - u[p];
      if (tid == 0) dst[E] = tot;
      __syncthreads();
    }
  }
  tc_fence_after_sync();
  const uint32_t tmem_base = *s_tmem;
  Tables tb;
  tb.off = s_off;
  tb.uoff[0] = s_uoff0;
  tb.uoff[1] = s_uoff1;
  tb.ksplit[0] = args.ksplit[0];
  tb.ksplit[1] = args.ksplit[1];
  tb.E = E;
  const int total = s_uoff0[E] + s_uoff1[E];
  const int my_units =
      (int)blockIdx.x < total ? (total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  const bool use_list = my_units <= kMaxUnits;   // the same in every thread of the CTA
  if (use_list) {
    for (int i = tid; i < my_units; i += kThreads)
      s_units[i] = pack_unit(decode_unit<BN>((int)blockIdx.x + i * (int)gridDim.x, tb));
    __syncthreads();
  }

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ TMA producer --
      // weights: read once per unit in the thin-tile (decode) variant, so stream
      // them past L2; wide token tiles re-read a weight tile for every token block
      // of its expert, so keep them cacheable
      const uint64_t pol_w = BN <= 32 ? l2_policy_evict_first() : l2_policy_evict_normal();
      const uint64_t pol_x = l2_policy_evict_last();
      const unsigned long long wait_ns = args.wait_ns;
      int stage = 0;
      uint32_t par = 0;
      uint32_t issued_mask = 0, issued_par = 0;
      int nissued = 0;
      bool ok = true, stalled = false;
      for (int u = blockIdx.x, ui = 0; u < total && ok && !stalled; u += gridDim.x, ++ui) {
        const Unit t = use_list ? unpack_unit(s_units[ui]) : decode_unit<BN>(u, tb);
        if (t.ph == 1 && args.done != nullptr) {
          const int m = s_off[t.e + 1] - s_off[t.e];
          const int need = ((m + BN - 1) / BN) * (args.MW[0] / kBM) * args.ksplit[0];
          if (!wait_counter(args.done + t.e, need, s_abort, wait_ns)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
        }
        const CUtensorMap* ta = t.ph ? &tmA1 : &tmA0;
        const CUtensorMap* tbm = t.ph ? &tmB1 : &tmB0;
        const int nbox = (t.rows + BOX - 1) / BOX;
        const uint32_t bytes = kABytes + nbox * L::kBoxBytes;
        const int arow = t.e * args.MW[t.ph] + t.mb * kBM;
        const int nks = args.K[t.ph] / kBK / args.ksplit[t.ph];
        const int bseg = args.bseg[t.ph];
        const uint32_t bmap = args.bmap[t.ph];
        for (int kb = t.ks * nks; kb < (t.ks + 1) * nks; ++kb) {
          if (nissued == args.stall_stage) {
            // test hook: nothing is issued for this stage or after it; the MMA
            // thread's wait for it runs out (nothing of this CTA is in flight then)
            stalled = true;
            break;
          }
          if (!mbar_wait(&empty[stage], par ^ 1u, s_abort, wait_ns)) {
            ok = false;
            break;
          }
          const int ka = kb * kBK;
          int kx = ka;
          if (bseg > 0) {
            const int seg = ka / bseg;
            kx = static_cast<int>((bmap >> (3 * seg)) & 7u) * bseg + (ka - seg * bseg);
          }
          mbar_arrive_expect_tx(&full[stage], bytes);
          tma_load_2d(sA + stage * kABytes, ta, &full[stage], ka, arow, pol_w);
          for (int j = 0; j < nbox; ++j)
            tma_load_2d(sB + stage * L::kBBytes + j * L::kBoxBytes, tbm, &full[stage], kx,
                        t.row0 + j * BOX, pol_x);
          issued_mask |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (par << stage);
          ++nissued;
          if (++stage == STAGES) {
            stage = 0;
            par ^= 1u;
          }
        }
      }
      if (stalled) {
        // wait (bounded) for the role whose wait ran out to raise the abort flag
        const unsigned long long t0 = globaltimer();
        while (!*s_abort && globaltimer() - t0 < 4 * wait_ns) __nanosleep(256);
        ok = false;
      }
      if (ok) {
        // producer tail: wait until the MMA unit has released every stage, so no
        // commit-arrive is still in flight when the CTA exits
        for (int i = 0; i < STAGES; ++i) {
          if (!mbar_wait(&empty[stage], par ^ 1u, s_abort, wait_ns)) {
            ok = false;
            break;
          }
          if (++stage == STAGES) {
            stage = 0;
            par ^= 1u;
          }
        }
      }
      if (!ok) {
        *s_abort = 1;
        flag_status(args.status, MOE_DEV_WAIT_TIMEOUT);
        // let copies already in flight land before the CTA's shared memory goes away
        for (int s = 0; s < STAGES; ++s)
          if ((issued_mask >> s) & 1u) mbar_wait(&full[s], (issued_par >> s) & 1u, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------- MMA issuer --
      const unsigned long long wait_ns = args.wait_ns;
      int stage = 0, acc = 0;
      uint32_t par = 0, apar = 0;
      bool ok = true;
      for (int u = blockIdx.x, ui = 0; u < total && ok; u += gridDim.x, ++ui) {
        const Unit t = use_list ? unpack_unit(s_units[ui]) : decode_unit<BN>(u, tb);
        const int n = (t.rows + 15) & ~15;
        const uint32_t idesc = idesc_bf16_f32(kBM, n);
        if (!mbar_wait(&tempty[acc], apar ^ 1u, s_abort, wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
        const int nk = args.K[t.ph] / kBK / args.ksplit[t.ph];
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&full[stage], par, s_abort, wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a0 = smem_u32(sA + stage * kABytes);
          const uint32_t b0 = smem_u32(sB + stage * L::kBBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            tc_mma_bf16(d, smem_desc_sw128(a0 + kk * 32), smem_desc_sw128(b0 + kk * 32), idesc,
                        (kb | kk) ? 1u : 0u);
          tc_commit(&empty[stage]);
          if (++stage == STAGES) {
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
        tc_commit(fin);  // drain this thread's outstanding MMAs before TMEM is freed
        mbar_wait(fin, 0, nullptr);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue --
    const int q = warp & 3;          // TMEM lane quarter
    const int et = tid - 128;        // 0..127
    int* s_flag = s_tmp;             // broadcast of the elected wait's result
    int acc = 0;
    uint32_t apar = 0;
    for (int u = blockIdx.x, ui = 0; u < total; u += gridDim.x, ++ui) {
      const Unit t = use_list ? unpack_unit(s_units[ui]) : decode_unit<BN>(u, tb);
      if (et == 0) s_flag[0] = mbar_wait(&tfull[acc], apar, s_abort, args.wait_ns) ? 1 : 0;
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
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      epilogue_tile(args, t, tbase, sEpi, q, lane);
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
    tmem_dealloc(tmem_base, 2 * BN);
  }
}

// ------------------------------------------------------------ CTA pairs --
// Prefill variant on pairs of SMs (a cluster of two CTAs).  A pair unit is
// (phase, expert, 256-row weight block, token block): one tcgen05.mma.cta_group::2
// of M = 256 covers both CTAs' 128-row weight blocks (CTA r holds block 2*pb + r of
// A) and the token block's N columns, of which CTA r holds rows [r*N/2, (r+1)*N/2)
// of B.  Each CTA's TMEM receives the full 128 x N accumulator of its own weight
// block.  Per SM and stage the ring holds 16 KB of weights and at most 16 KB of
// tokens, so six stages fit.
//
// Two pipelines share the pair.  Experts with at most kLightRows tokens (the cold
// experts of a skewed router) stream a whole weight matrix for a handful of
// tokens: their stages cost the MMA thread as much issue time as full ones while
// the tensor pipe idles, and their weights come from HBM.  They run on a light
// pipeline of their own (a second producer, MMA thread, forwarder and epilogue
// group, a two-stage ring with 16-row token slots and two 32-column accumulators),
// so that their weight streaming overlaps the heavy units' tensor work instead of
// adding to it.  The other experts' units run on the heavy pipeline.  An expert's
// units all go to one pipeline, so the down projection's wait for h never crosses
// pipelines.  The kernel uses the light pipeline only when its per-stage cost
// estimates say the overlap pays (see the prologue); then the heavy accumulators
// narrow to 224 columns (TMEM columns 0 and 256; the light ones sit at 224 and 480)
// and the heavy token slots to 112 rows per CTA.  Otherwise every expert runs on the
// heavy pipeline with 256-token blocks and 128-row slots, and the light roles find no
// units.
//
// Roles (512 threads): in each CTA, warp 0 lane 0 loads the heavy tiles and warp 2
// lane 0 the light ones, each onto its own ring's `full` barrier; in the even CTA
// warp 1 lane 0 issues the heavy MMAs and warp 3 lane 0 the light ones, committing
// each stage's release and each accumulator's completion to both CTAs (multicast
// commit); in the odd CTA warps 3 and 1 forward the heavy and light stage arrivals
// to the even CTA (a relaxed remote arrive).  Warps 4-11 drain the heavy
// accumulators (two per TMEM lane quarter, alternating 32-token chunks) and warps
// 12-15 the light ones, storing from registers, and arrive on the even CTA's `tempty`.
constexpr int kPairBN = 256;         // token rows per heavy unit without light experts
constexpr int kPairBNL = 224;        // ... and next to light experts
constexpr int kLightRows = 32;       // experts with at most this many tokens run light
constexpr int kLightBox = 16;        // B rows per CTA of a light unit (N <= 32)
constexpr int kPairBoxS = 16;        // B box rows of heavy units whose half is <= 16 rows
constexpr int kPairThreads = 512;
constexpr int kPairStages = 6;       // heavy ring
constexpr int kLightStages = 2;
constexpr int kHeavyEpiWarps = 8;
constexpr int kLightEpiWarps = 4;
constexpr int kPairMaxUnits = 256;   // per pipeline list in shared memory
constexpr int kPairTmemCols = 512;

struct PairLayout {
  static constexpr int kHStride = kABytes + 128 * kBK * 2;     // heavy stage: A, 128 B rows
  static constexpr int kHStrideL = kABytes + (kPairBNL / 2) * kBK * 2;   // 112 B rows
  static constexpr int kLStride = kABytes + kLightBox * kBK * 2;         // light stage
  static constexpr int kL = kPairStages * kHStrideL;           // light ring after the heavy one
  static constexpr int kRing = (kL + kLightStages * kLStride) > kPairStages * kHStride
                                   ? kL + kLightStages * kLStride
                                   : kPairStages * kHStride;
  static constexpr int kBar = kRing;
  // heavy full/empty, light full/empty, and per pipeline tfull[2], tempty[2], fin
  static constexpr int kNumBars = 2 * kPairStages + 2 * kLightStages + 2 * 5;
  static constexpr int kMisc = kBar + kNumBars * 8;            // TMEM address, abort, heavy BN
  static constexpr int kTables = kMisc + 16;   // off, unit offsets (heavy and light, both phases)
  static constexpr int kTmpInts = 32;          // scan words (16 warps), epilogue flags
  static constexpr int kUnits = kTables + ((5 * (kMaxE + 1) + kTmpInts) * 4 + 7) / 8 * 8;
  static constexpr int kEnd = kUnits + 2 * kPairMaxUnits * 8;
  static_assert(kL % 1024 == 0 && kLStride % 1024 == 0 && kHStrideL % 1024 == 0 &&
                    kHStride % 1024 == 0,
                "swizzle atoms");
  static_assert(kUnits % 8 == 0, "unit list alignment");
  static constexpr int kSmemBytes = kEnd + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};
static_assert(kPairBNL + kLightRows <= kPairBN && 2 * kPairBN <= kPairTmemCols,
              "a light accumulator fits beside each narrowed heavy one");

// decode_unit with a token-block size chosen at run time.
__device__ __forceinline__ Unit decode_unit_rows(int u, const int* off, const int* uoff0,
                                                 const int* uoff1, int E, int BN) {
  Unit r;
  const int total0 = uoff0[E];
  r.ph = (u < total0) ? 0 : 1;
  if (r.ph) u -= total0;
  const int* uo = r.ph ? uoff1 : uoff0;
  int lo = 0, hi = E;  // uo[lo] <= u < uo[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (uo[mid] <= u) lo = mid;
    else hi = mid;
  }
  r.e = lo;
  r.ks = 0;
  const int local = u - uo[lo];
  const int m = off[lo + 1] - off[lo];
  const int nb = (m + BN - 1) / BN;
  r.mb = local / nb;
  const int b = local - r.mb * nb;
  r.row0 = off[lo] + b * BN;
  r.rows = min(BN, off[lo + 1] - r.row0);
  return r;
}

// Exclusive prefix sum over the kPairThreads threads of a CTA (s_tmp: 16 ints).
__device__ __forceinline__ int pair_scan_excl(int v, int* s_tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) s_tmp[warp] = inc;
  __syncthreads();
  int pre = 0, tot = 0;
  for (int w = 0; w < kPairThreads / 32; ++w) {
    if (w < warp) pre += s_tmp[w];
    tot += s_tmp[w];
  }
  __syncthreads();
  *total = tot;
  return pre + inc - v;
}

// One pipeline of the pair kernel as its roles see it.
struct PairPipe {
  uint8_t* ring;           // stage s: A at ring + s * stride, B kABytes after it
  int stride;
  int stages;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tfull;
  uint64_t* tempty;
  uint64_t* fin;
  uint32_t lead_full0;     // full[0] of the even CTA (cluster address)
  uint32_t lead_tempty0;   // tempty[0] of the even CTA
  const uint2* units;      // this pair's units, or null: decoded on the fly
  bool drawn;              // units after the first two are drawn from args.sched
  const int* off;
  const int* uoff0;
  const int* uoff1;
  int E;
  int bn;                  // token rows per unit
  int total;               // units of the pipeline (both phases)
  uint32_t acc_base;       // accumulator a at TMEM column acc_base + a * kPairBN
  int epi_warps;           // epilogue warps per CTA (a multiple of 4)
  int bar_id;              // named barrier of the epilogue group
  int* flag;               // the epilogue group's broadcast word
};

// A pipeline's units, in increasing unit order: round-robin (units pair, pair +
// npairs, ...), or, for a drawn list, the round-robin walk's first two and then units
// 2 * npairs + ticket drawn from a counter by the even CTA's producer, which at the
// start of each unit publishes the next entry (drawn one unit earlier) in both CTAs'
// lists and draws the one after, so pairs whose units ran faster take more of them.
// A pair's list increases like a round-robin one, so a down-projection unit still
// only waits for gate/up units that pairs drew before it.
// Returns 1 with unit ui in t, 0 when the list ended before ui, -1 when the wait
// for a drawn entry ran out (or the CTA is aborting).
// The roles are instantiated for round-robin (kDrawn false) and drawn lists.
template <bool kDrawn>
__device__ __forceinline__ int pipe_unit(const PairPipe& p, int pair, int npairs, int ui, Unit& t,
                                         const volatile int* abort) {
  if (!kDrawn) {
    const int u = pair + ui * npairs;
    if (u >= p.total) return 0;
    t = p.units != nullptr ? unpack_unit(p.units[ui])
                           : decode_unit_rows(u, p.off, p.uoff0, p.uoff1, p.E, p.bn);
    return 1;
  }
  const uint32_t a = smem_u32(p.units + ui);
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

// TMA producer of one pipeline in one CTA: this CTA's weight block and token half.
template <bool kDrawn>
__device__ __forceinline__ void pair_producer(const PairPipe& p, const GemmArgs& args,
                                              const CUtensorMap* tmA0, const CUtensorMap* tmA1,
                                              const CUtensorMap* tmW0, const CUtensorMap* tmW1,
                                              int wide_rows, const CUtensorMap* tmS0,
                                              const CUtensorMap* tmS1, int pair, int npairs,
                                              uint32_t rank, volatile int* s_abort) {
  const uint64_t pol_w_reused = l2_policy_evict_normal();
  const uint64_t pol_w_once = l2_policy_evict_first();
  const uint64_t pol_x = l2_policy_evict_last();
  int stage = 0;
  uint32_t par = 0;
  uint32_t issued_mask = 0, issued_par = 0;
  bool ok = true;
  // the even CTA's producer of a drawn list: entry ui + 1 is published at the start
  // of unit ui (entries 0 and 1 are the round-robin walk's), entry ui + 2 drawn then
  // (the list's last entry is kept for the end entry)
  bool open = kDrawn && rank == 0 && pair + npairs < p.total;   // entry 1 is a unit
  int ticket = 0;
  for (int ui = 0; ok; ++ui) {
    Unit t;
    const int got = pipe_unit<kDrawn>(p, pair, npairs, ui, t, s_abort);
    if (got <= 0) {
      ok = got == 0;
      break;
    }
    if (open) {
      if (ui >= 1) {
        const int un = ticket >= 0 ? 2 * npairs + ticket : p.total;
        const uint64_t w =
            un < p.total ? unit_word(pack_unit(decode_unit_rows(un, p.off, p.uoff0, p.uoff1, p.E, p.bn)))
                         : unit_word(make_uint2(0, kEndUnitWord));
        const uint32_t entry = smem_u32(p.units + ui + 1);
        st_relaxed_cluster_u64(mapa_shared(entry, 1), w);
        st_relaxed_cluster_u64(mapa_shared(entry, 0), w);
        open = un < p.total;
      }
      if (open) ticket = ui + 2 <= kPairMaxUnits - 2 ? atomicAdd(args.sched, 1) : -1;
    }
    const int m = p.off[t.e + 1] - p.off[t.e];
    if (t.ph == 1 && args.done != nullptr) {
      // the down projection reads h of this expert's gate/up units (same pipeline)
      const int need = ((m + p.bn - 1) / p.bn) * (args.MW[0] / kBM);
      if (!wait_counter(args.done + t.e, need, s_abort)) {
        ok = false;
        break;
      }
      fence_proxy_async_global();
    }
    const int half = ((t.rows + 15) & ~15) >> 1;          // this CTA's B rows (N / 2)
    const bool thin = half <= kPairBoxS;
    const CUtensorMap* ta = t.ph ? tmA1 : tmA0;
    const CUtensorMap* tbm = thin ? (t.ph ? tmS1 : tmS0) : (t.ph ? tmW1 : tmW0);
    const uint32_t bytes = kABytes + (thin ? kPairBoxS : wide_rows) * kBK * 2;
    const int arow = t.e * args.MW[t.ph] + (2 * t.mb + static_cast<int>(rank)) * kBM;
    const int brow = t.row0 + static_cast<int>(rank) * half;
    const int nk = args.K[t.ph] / kBK;
    // weight tiles of an expert with one token block are read once: stream them
    const uint64_t pol_w = m <= p.bn ? pol_w_once : pol_w_reused;
    for (int kb = 0; kb < nk; ++kb) {
      if (!mbar_wait(&p.empty[stage], par ^ 1u, s_abort)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(&p.full[stage], bytes);
      uint8_t* sa = p.ring + stage * p.stride;
      tma_load_2d(sa, ta, &p.full[stage], kb * kBK, arow, pol_w);
      tma_load_2d(sa + kABytes, tbm, &p.full[stage], kb * kBK, brow, pol_x);
      issued_mask |= 1u << stage;
      issued_par = (issued_par & ~(1u << stage)) | (par << stage);
      if (++stage == p.stages) {
        stage = 0;
        par ^= 1u;
      }
    }
  }
  if (ok) {
    // every stage released by the pair's MMAs: no multicast commit is still on
    // its way to this CTA's barriers when it exits
    for (int i = 0; i < p.stages; ++i) {
      if (!mbar_wait(&p.empty[stage], par ^ 1u, s_abort)) {
        ok = false;
        break;
      }
      if (++stage == p.stages) {
        stage = 0;
        par ^= 1u;
      }
    }
  }
  if (!ok) {
    *s_abort = 1;
    flag_status(args.status, MOE_DEV_WAIT_TIMEOUT);
    for (int s = 0; s < p.stages; ++s)
      if ((issued_mask >> s) & 1u) mbar_wait(&p.full[s], (issued_par >> s) & 1u, nullptr);
  }
}

// Odd CTA: passes each of its landed stages on to the even CTA's `full` barrier.
template <bool kDrawn>
__device__ __forceinline__ void pair_forwarder(const PairPipe& p, const GemmArgs& args, int pair,
                                               int npairs, volatile int* s_abort) {
  int stage = 0;
  uint32_t par = 0;
  bool ok = true;
  for (int ui = 0; ok; ++ui) {
    Unit t;
    const int got = pipe_unit<kDrawn>(p, pair, npairs, ui, t, s_abort);
    if (got <= 0) {
      ok = got == 0;
      break;
    }
    const int nk = args.K[t.ph] / kBK;
    for (int kb = 0; kb < nk; ++kb) {
      if (!mbar_wait(&p.full[stage], par, s_abort)) {
        ok = false;
        break;
      }
      // the stage's bytes are in this CTA's shared memory (observed above)
      mbar_arrive_cluster_relaxed(p.lead_full0 + stage * 8);
      if (++stage == p.stages) {
        stage = 0;
        par ^= 1u;
      }
    }
  }
  if (!ok) {
    *s_abort = 1;
    flag_status(args.status, MOE_DEV_WAIT_TIMEOUT);
  }
}

// Even CTA: the pipeline's MMA issuer.
template <bool kDrawn>
__device__ __forceinline__ void pair_mma(const PairPipe& p, const GemmArgs& args, uint32_t tmem_base,
                                         int pair, int npairs, volatile int* s_abort) {
  int stage = 0, acc = 0;
  uint32_t par = 0, apar = 0;
  bool ok = true;
  for (int ui = 0; ok; ++ui) {
    Unit t;
    const int got = pipe_unit<kDrawn>(p, pair, npairs, ui, t, s_abort);
    if (got <= 0) {
      ok = got == 0;
      break;
    }
    const int n = (t.rows + 15) & ~15;
    const uint32_t idesc = idesc_bf16_f32(2 * kBM, n);
    // both CTAs' epilogues have drained this accumulator
    if (!mbar_wait_cluster(&p.tempty[acc], apar ^ 1u, s_abort)) {
      ok = false;
      break;
    }
    tc_fence_after_sync();
    const uint32_t d = tmem_base + p.acc_base + static_cast<uint32_t>(acc * kPairBN);
    const int nk = args.K[t.ph] / kBK;
    for (int kb = 0; kb < nk; ++kb) {
      if (!mbar_wait_cluster(&p.full[stage], par, s_abort)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t a0 = smem_u32(p.ring + stage * p.stride);
      const uint32_t b0 = a0 + kABytes;
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)
        tc_mma_pair_bf16(d, smem_desc_sw128(a0 + kk * 32), smem_desc_sw128(b0 + kk * 32), idesc,
                         (kb | kk) ? 1u : 0u);
      tc_commit_pair(&p.empty[stage], 3);
      if (++stage == p.stages) {
        stage = 0;
        par ^= 1u;
      }
    }
    if (!ok) break;
    tc_commit_pair(&p.tfull[acc], 3);
    acc ^= 1;
    if (acc == 0) apar ^= 1u;
  }
  if (ok) {
    // the odd CTA's last remote tempty arrivals land before this CTA may exit
    for (int i = 0; i < 2; ++i) {
      if (!mbar_wait_cluster(&p.tempty[acc], apar ^ 1u, s_abort)) {
        ok = false;
        break;
      }
      acc ^= 1;
      if (acc == 0) apar ^= 1u;
    }
  }
  if (!ok) {
    *s_abort = 1;
    flag_status(args.status, MOE_DEV_WAIT_TIMEOUT);
    tc_commit_pair(p.fin, 1);  // drain this thread's outstanding MMAs before TMEM is freed
    mbar_wait(p.fin, 0, nullptr);
  }
}

// One 32-token chunk of an accumulator, stored from registers.  The warp reads TMEM
// lane quarter q of the CTA's 128-row weight block t.mb.  Gate/up (epi 0): lanes 0-15
// hold the gate rows of features 16q .. 16q + 15 of the block and lanes 16-31 the
// matching up rows (the packed w13 layout), so one shuffle pairs them and lanes 0-15
// finish tokens c0 .. c0 + 15, lanes 16-31 tokens c0 + 16 .. c0 + 31, each for feature
// 16q + (lane & 15).  Down (epi 1): lane l holds output feature 32q + l of the block.
// In both, a second shuffle between neighbouring lanes gives each lane two adjacent
// features of one token, so every store writes 4 bytes and one warp-wide store covers
// whole 32- or 64-byte row segments of two tokens.
__device__ __forceinline__ void pair_store_chunk(const GemmArgs& args, const Unit& t,
                                                 uint32_t tbase, int c0, int q, int lane) {
  uint16_t* out = args.out[t.ph];
  const int ld = args.ld[t.ph];
  const bool odd = (lane & 1) != 0;
  float v[32];
  tmem_ld_32x32b_x32(tbase + c0, v);
  if (args.epi[t.ph] == 0) {
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
    // even lane f: features (f, f + 1) of token j; odd lane: (f - 1, f) of token j + 1
    uint16_t* col = out + (size_t)t.mb * 64 + q * 16 + (lane & 14);
    const int tb = c0 + (lo ? 0 : 16);
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      const float x = __shfl_xor_sync(0xffffffffu, odd ? h[j] : h[j + 1], 1);
      const int tok = tb + j + (odd ? 1 : 0);
      const uint32_t pk = odd ? (uint32_t)f2bf(x) | ((uint32_t)f2bf(h[j + 1]) << 16)
                              : (uint32_t)f2bf(h[j]) | ((uint32_t)f2bf(x) << 16);
      if (tok < t.rows) *reinterpret_cast<uint32_t*>(col + (size_t)(t.row0 + tok) * ld) = pk;
    }
  } else {
    uint16_t* col = out + (size_t)t.mb * kBM + q * 32 + (lane & 30);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const float x = __shfl_xor_sync(0xffffffffu, odd ? v[j] : v[j + 1], 1);
      const int tok = c0 + j + (odd ? 1 : 0);
      const uint32_t pk = odd ? (uint32_t)f2bf(x) | ((uint32_t)f2bf(v[j + 1]) << 16)
                              : (uint32_t)f2bf(v[j]) | ((uint32_t)f2bf(x) << 16);
      if (tok < t.rows) *reinterpret_cast<uint32_t*>(col + (size_t)(t.row0 + tok) * ld) = pk;
    }
  }
}

// An epilogue group: p.epi_warps warps per CTA, warp ew taking TMEM lane quarter
// ew % 4 and every (p.epi_warps / 4)-th 32-token chunk from chunk ew / 4.
template <bool kDrawn>
__device__ __forceinline__ void pair_epilogue(const PairPipe& p, const GemmArgs& args,
                                              uint32_t tmem_base, int pair, int npairs,
                                              uint32_t rank, int ew, int lane,
                                              volatile int* s_abort) {
  const bool leader = rank == 0;
  const int q = ew & 3, g = ew >> 2, ng = p.epi_warps >> 2;
  const int nthr = 32 * p.epi_warps;
  const int et = ew * 32 + lane;
  int acc = 0;
  uint32_t apar = 0;
  for (int ui = 0;; ++ui) {
    // one thread waits for the unit and its accumulator; p.flag[0]: 1 go, 0 the
    // list has ended, -1 a wait ran out
    if (et == 0) {
      Unit t0;
      int st = pipe_unit<kDrawn>(p, pair, npairs, ui, t0, s_abort);
      if (st == 1) {
        const uint2 w = pack_unit(t0);
        p.flag[1] = static_cast<int>(w.x);
        p.flag[2] = static_cast<int>(w.y);
        if (!mbar_wait(&p.tfull[acc], apar, s_abort)) st = -1;
      }
      p.flag[0] = st;
    }
    named_bar_sync(p.bar_id, nthr);
    const int st = p.flag[0];
    Unit t = unpack_unit(make_uint2(static_cast<uint32_t>(p.flag[1]), static_cast<uint32_t>(p.flag[2])));
    named_bar_sync(p.bar_id, nthr);
    if (st <= 0) {
      if (st < 0 && et == 0) {
        *s_abort = 1;
        flag_status(args.status, MOE_DEV_WAIT_TIMEOUT);
      }
      break;
    }
    t.mb = 2 * t.mb + static_cast<int>(rank);   // this CTA's 128-row weight block
    tc_fence_after_sync();
    const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + p.acc_base +
                           static_cast<uint32_t>(acc * kPairBN);
    for (int c0 = 32 * g; c0 < t.rows; c0 += 32 * ng) pair_store_chunk(args, t, tbase, c0, q, lane);
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) {
      if (leader) mbar_arrive(&p.tempty[acc]);
      else mbar_arrive_cluster(p.lead_tempty0 + acc * 8);
    }
    if (t.ph == 0 && args.done != nullptr) {
      // this unit's h rows are read by TMA (the async proxy) in the down projection;
      // after the group's barrier, one release covers every thread's stores
      fence_proxy_async_global();
      named_bar_sync(p.bar_id, nthr);
      if (et == 0) red_release_add_gpu(args.done + t.e, 1);
    }
    acc ^= 1;
    if (acc == 0) apar ^= 1u;
  }
}

__global__ void __launch_bounds__(kPairThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA0,
                             const __grid_constant__ CUtensorMap tmA1,
                             const __grid_constant__ CUtensorMap tmB0,   // 128-row B boxes
                             const __grid_constant__ CUtensorMap tmB1,
                             const __grid_constant__ CUtensorMap tmH0,   // 112-row B boxes
                             const __grid_constant__ CUtensorMap tmH1,
                             const __grid_constant__ CUtensorMap tmS0,   // 16-row B boxes
                             const __grid_constant__ CUtensorMap tmS1, const GemmArgs args) {
  using L = PairLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* h_full = bars;
  uint64_t* h_empty = h_full + kPairStages;
  uint64_t* l_full = h_empty + kPairStages;
  uint64_t* l_empty = l_full + kLightStages;
  uint64_t* h_tfull = l_empty + kLightStages;   // [2]
  uint64_t* h_tempty = h_tfull + 2;             // [2], waited on in the even CTA only
  uint64_t* l_tfull = h_tempty + 2;             // [2]
  uint64_t* l_tempty = l_tfull + 2;             // [2], waited on in the even CTA only
  uint64_t* h_fin = l_tempty + 2;
  uint64_t* l_fin = h_fin + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  int* s_hbn = reinterpret_cast<int*>(smem + L::kMisc + 8);
  int* s_off = reinterpret_cast<int*>(smem + L::kTables);
  int* s_uh0 = s_off + (kMaxE + 1);
  int* s_uh1 = s_uh0 + (kMaxE + 1);
  int* s_ul0 = s_uh1 + (kMaxE + 1);
  int* s_ul1 = s_ul0 + (kMaxE + 1);
  int* s_tmp = s_ul1 + (kMaxE + 1);   // 16 scan words, then the two epilogue groups' words
  uint2* s_hunits = reinterpret_cast<uint2*>(smem + L::kUnits);
  uint2* s_lunits = s_hunits + kPairMaxUnits;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = args.E;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(blockIdx.x >> 1), npairs = static_cast<int>(gridDim.x >> 1);
  pdl_trigger();

  if (tid == 0) {
    // even CTA: its own producer + the odd CTA's forwarded arrival
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&h_full[s], leader ? 2 : 1);
      mbar_init(&h_empty[s], 1);
    }
    for (int s = 0; s < kLightStages; ++s) {
      mbar_init(&l_full[s], leader ? 2 : 1);
      mbar_init(&l_empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&h_tfull[a], 1);
      mbar_init(&h_tempty[a], 2 * kHeavyEpiWarps);   // the group's warps in both CTAs
      mbar_init(&l_tfull[a], 1);
      mbar_init(&l_tempty[a], 2 * kLightEpiWarps);
    }
    mbar_init(h_fin, 1);
    mbar_init(l_fin, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA0);
    tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB0);
    tma_prefetch_desc(&tmB1);
    tma_prefetch_desc(&tmH0);
    tma_prefetch_desc(&tmH1);
    tma_prefetch_desc(&tmS0);
    tma_prefetch_desc(&tmS1);
  }
  if (warp == 2) {
    tmem_alloc_pair(s_tmem, kPairTmemCols);
    tmem_relinquish_pair();
  }
  for (int i = tid; i <= E; i += kPairThreads) s_off[i] = args.offsets[i];
  __syncthreads();

  // Units per expert and pipeline, and their exclusive prefix per phase.  The light
  // pipeline pays off when the light experts' weight streaming can hide under the
  // heavy units' tensor work; when light stages dominate (small skewed batches) its
  // two-stage ring is slower than running every expert on the heavy pipeline.  Per
  // stage (measured): ~1700 clocks on the light ring, ~690 on the heavy ring beside
  // it (224-token units), ~660 on a heavy ring of its own (256-token units).
  {
    const int m = tid < E ? s_off[tid + 1] - s_off[tid] : 0;
    const bool small = m > 0 && m <= kLightRows;
    int stg = 0;                                   // stages of one token block
    for (int ph = 0; ph < 2; ++ph)
      if (args.active[ph]) stg += args.MW[ph] / (2 * kBM) * (args.K[ph] / kBK);
    int l_st = 0, h224 = 0, h256 = 0;
    pair_scan_excl(small ? stg : 0, s_tmp, &l_st);
    pair_scan_excl(small ? 0 : (m + kPairBNL - 1) / kPairBNL * stg, s_tmp, &h224);
    pair_scan_excl((m + kPairBN - 1) / kPairBN * stg, s_tmp, &h256);
    const long long t_split = 1700LL * l_st > 690LL * h224 ? 1700LL * l_st : 690LL * h224;
    const bool with_light_run =
        l_st > 0 && (args.light_mode == 1 || (args.light_mode == 0 && t_split < 660LL * h256));
    const bool light = small && with_light_run;
    const int hb = with_light_run ? kPairBNL : kPairBN;
    if (tid == 0) *s_hbn = hb;
    int uh[2] = {0, 0}, ul[2] = {0, 0};
    if (tid < E) {
      const int nb = light ? 0 : (m + hb - 1) / hb;
      for (int ph = 0; ph < 2; ++ph) {
        const int pb = args.active[ph] ? args.MW[ph] / (2 * kBM) : 0;
        uh[ph] = nb * pb;
        ul[ph] = light ? pb : 0;
      }
    }
    int* dst[4] = {s_uh0, s_uh1, s_ul0, s_ul1};
    const int val[4] = {uh[0], uh[1], ul[0], ul[1]};
    for (int i = 0; i < 4; ++i) {
      int tot = 0;
      const int pre = pair_scan_excl(val[i], s_tmp, &tot);
      if (tid < E) dst[i][tid] = pre;
      if (tid == 0) dst[i][E] = tot;
    }
    __syncthreads();
  }
  const int hb = *s_hbn;

  PairPipe hp, lp;
  hp.ring = smem;
  hp.stride = hb == kPairBN ? L::kHStride : L::kHStrideL;
  hp.stages = kPairStages;
  hp.full = h_full;
  hp.empty = h_empty;
  hp.tfull = h_tfull;
  hp.tempty = h_tempty;
  hp.fin = h_fin;
  hp.lead_full0 = mapa_shared(smem_u32(&h_full[0]), 0);
  hp.lead_tempty0 = mapa_shared(smem_u32(&h_tempty[0]), 0);
  hp.off = s_off;
  hp.uoff0 = s_uh0;
  hp.uoff1 = s_uh1;
  hp.E = E;
  hp.bn = hb;
  hp.total = s_uh0[E] + s_uh1[E];
  hp.acc_base = 0;                  // columns 0 and 256
  hp.epi_warps = kHeavyEpiWarps;
  hp.bar_id = 1;
  hp.flag = s_tmp + 16;             // three words each

  lp.ring = smem + L::kL;
  lp.stride = L::kLStride;
  lp.stages = kLightStages;
  lp.full = l_full;
  lp.empty = l_empty;
  lp.tfull = l_tfull;
  lp.tempty = l_tempty;
  lp.fin = l_fin;
  lp.lead_full0 = mapa_shared(smem_u32(&l_full[0]), 0);
  lp.lead_tempty0 = mapa_shared(smem_u32(&l_tempty[0]), 0);
  lp.off = s_off;
  lp.uoff0 = s_ul0;
  lp.uoff1 = s_ul1;
  lp.E = E;
  lp.bn = kLightRows;
  lp.total = s_ul0[E] + s_ul1[E];
  lp.acc_base = kPairBNL;           // columns 224 and 480
  lp.epi_warps = kLightEpiWarps;
  lp.bar_id = 2;
  lp.flag = s_tmp + 20;

  // Each pair's units of both lists, decoded once (the same in every thread).  The
  // heavy list is drawn when the launch has a unit counter, the light pipeline does
  // not run (beside it, drawing measured slower) and at most half of the pairs can
  // fill a list (kPairMaxUnits - 1 units), so that the others draw the rest.
  const int h_my = pair < hp.total ? (hp.total - pair + npairs - 1) / npairs : 0;
  const int l_my = pair < lp.total ? (lp.total - pair + npairs - 1) / npairs : 0;
  hp.drawn = args.sched != nullptr && lp.total == 0 &&
             hp.total <= (kPairMaxUnits - 1) * (npairs / 2);
  lp.drawn = false;
  hp.units = hp.drawn || h_my <= kPairMaxUnits ? s_hunits : nullptr;
  lp.units = l_my <= kPairMaxUnits ? s_lunits : nullptr;
  if (hp.drawn) {
    // entries 0 and 1 are the round-robin walk's, the others pending; both CTAs
    // write theirs before the cluster barrier below, ahead of any published entry
    for (int i = tid; i < kPairMaxUnits; i += kPairThreads) {
      const int u = pair + i * npairs;
      s_hunits[i] = i >= 2 ? make_uint2(0, kPendingUnitWord)
                    : u < hp.total
                        ? pack_unit(decode_unit_rows(u, s_off, s_uh0, s_uh1, E, hp.bn))
                        : make_uint2(0, kEndUnitWord);
    }
  } else if (hp.units != nullptr) {
    for (int i = tid; i < h_my; i += kPairThreads)
      s_hunits[i] = pack_unit(decode_unit_rows(pair + i * npairs, s_off, s_uh0, s_uh1, E, hp.bn));
  }
  if (lp.units != nullptr)
    for (int i = tid; i < l_my; i += kPairThreads)
      s_lunits[i] = pack_unit(decode_unit_rows(pair + i * npairs, s_off, s_ul0, s_ul1, E, lp.bn));
  __syncthreads();
  tc_fence_after_sync();
  // both CTAs' barriers are initialised, their lists started and TMEM allocated
  // before any remote arrive or store
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = *s_tmem;

  const CUtensorMap* hw0 = hb == kPairBN ? &tmB0 : &tmH0;
  const CUtensorMap* hw1 = hb == kPairBN ? &tmB1 : &tmH1;
  if (lane == 0 && warp == 0) {
    if (hp.drawn)
      pair_producer<true>(hp, args, &tmA0, &tmA1, hw0, hw1, hb / 2, &tmS0, &tmS1, pair, npairs,
                          rank, s_abort);
    else
      pair_producer<false>(hp, args, &tmA0, &tmA1, hw0, hw1, hb / 2, &tmS0, &tmS1, pair, npairs,
                           rank, s_abort);
  } else if (lane == 0 && warp == 2) {
    pair_producer<false>(lp, args, &tmA0, &tmA1, &tmS0, &tmS1, kLightBox, &tmS0, &tmS1, pair,
                         npairs, rank, s_abort);
  } else if (lane == 0 && warp == 1) {
    if (!leader) pair_forwarder<false>(lp, args, pair, npairs, s_abort);
    else if (hp.drawn) pair_mma<true>(hp, args, tmem_base, pair, npairs, s_abort);
    else pair_mma<false>(hp, args, tmem_base, pair, npairs, s_abort);
  } else if (lane == 0 && warp == 3) {
    if (leader) pair_mma<false>(lp, args, tmem_base, pair, npairs, s_abort);
    else if (hp.drawn) pair_forwarder<true>(hp, args, pair, npairs, s_abort);
    else pair_forwarder<false>(hp, args, pair, npairs, s_abort);
  } else if (warp >= 4 && warp < 4 + kHeavyEpiWarps) {
    if (hp.drawn)
      pair_epilogue<true>(hp, args, tmem_base, pair, npairs, rank, warp - 4, lane, s_abort);
    else
      pair_epilogue<false>(hp, args, tmem_base, pair, npairs, rank, warp - 4, lane, s_abort);
  } else if (warp >= 4 + kHeavyEpiWarps) {
    pair_epilogue<false>(lp, args, tmem_base, pair, npairs, rank, warp - 4 - kHeavyEpiWarps, lane,
                         s_abort);
  }

  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();
  if (warp == 2) {
    __syncwarp();   // lane 0 ran the light producer: the warp is converged for dealloc
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kPairTmemCols);
  }
}

// Packed w13: per expert 2I rows of H.  Row block b (128 rows) covers features
// 64b..64b+63; its quarter q (rows 32q..32q+31) holds gate columns 64b+16q+i in
// rows 32q+i and the matching up columns I+64b+16q+i in rows 32q+16+i (i < 16), so
// one TMEM lane quarter of the accumulator holds both halves of 16 features.
// Tiled 32x32 transpose.
__global__ void pack_w13_kernel(const uint16_t* __restrict__ w13, int H, int I,
                                uint16_t* __restrict__ out) {
  __shared__ uint16_t tile[32][33];
  const int h0 = blockIdx.x * 32, r0 = blockIdx.y * 32, e = blockIdx.z;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int blk = r0 / 128, q = (r0 % 128) / 32;
  const int col = tx < 16 ? blk * 64 + q * 16 + tx : I + blk * 64 + q * 16 + (tx - 16);
  const size_t n2 = 2 * (size_t)I;
  for (int i = ty; i < 32; i += 8) tile[i][tx] = w13[((size_t)e * H + h0 + i) * n2 + col];
  __syncthreads();
  for (int i = ty; i < 32; i += 8)
    out[((size_t)e * n2 + r0 + i) * H + h0 + tx] = tile[tx][i];
}

// Packed down: per expert H rows of I (down^T).
__global__ void pack_down_kernel(const uint16_t* __restrict__ down, int H, int I,
                                 uint16_t* __restrict__ out) {
  __shared__ uint16_t tile[32][33];
  const int i0 = blockIdx.x * 32, n0 = blockIdx.y * 32, e = blockIdx.z;
  const int tx = threadIdx.x, ty = threadIdx.y;
  for (int i = ty; i < 32; i += 8) tile[i][tx] = down[((size_t)e * I + i0 + i) * H + n0 + tx];
  __syncthreads();
  for (int i = ty; i < 32; i += 8)
    out[((size_t)e * H + n0 + i) * I + i0 + tx] = tile[tx][i];
}

// Test hook state (moe_debug_set_gemm_stall); read at each one-CTA launch.
std::atomic<int> g_stall_stage{-1};
// Test hook state (moe_debug_set_pair_light); read at each CTA-pair launch.
std::atomic<int> g_pair_light{0};
std::atomic<unsigned long long> g_stall_wait_ns{kWaitLimitNs};

template <int BN, int STAGES, int BOX>
cudaError_t launch_impl(const GemmPhase* ph0, const GemmPhase* ph1, const int32_t* offsets, int E,
                        int P, int* done, int* status, cudaStream_t s) {
  using L = Layout<BN, STAGES, BOX>;
  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
      err = cudaFuncSetAttribute(grouped_gemm_kernel<BN, STAGES, BOX>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
      if (err != cudaSuccess) return err;
      attr_set[dev] = true;
    }
  }
  GemmArgs a{};
  a.offsets = offsets;
  a.E = E;
  a.done = (ph0 && ph1) ? done : nullptr;
  a.status = status;
  a.stall_stage = g_stall_stage.load();
  a.wait_ns = a.stall_stage >= 0 ? g_stall_wait_ns.load() : kWaitLimitNs;
  CUtensorMap tm[4];
  const GemmPhase* phs[2] = {ph0, ph1};
  for (int p = 0; p < 2; ++p) {
    const GemmPhase* g = phs[p] ? phs[p] : (ph0 ? ph0 : ph1);
    a.active[p] = phs[p] != nullptr;
    a.K[p] = g->K;
    a.MW[p] = g->MW;
    a.ld[p] = g->n_out;
    a.epi[p] = g->epi;
    a.ksplit[p] = g->ksplit > 0 ? g->ksplit : 1;
    a.bseg[p] = g->bseg;
    a.bmap[p] = g->bmap;
    a.mvalid[p] = g->mvalid;
    a.rows_total[p] = g->rows_total;
    a.out[p] = g->out;
    a.out_f32[p] = g->out_f32;
    const uint64_t binner = g->b_inner > 0 ? (uint64_t)g->b_inner : (uint64_t)g->K;
    if (!encode_tmap_2d_bf16(&tm[2 * p], g->A_weights, (uint64_t)g->K, (uint64_t)E * g->MW, kBK,
                             kBM))
      return cudaErrorInvalidValue;
    if (!encode_tmap_2d_bf16(&tm[2 * p + 1], g->B_act, binner, (uint64_t)P, kBK, BOX))
      return cudaErrorInvalidValue;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(device_sm_count(), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = a.done != nullptr ? 1 : 0;  // co-residency for the phase dependency
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<BN, STAGES, BOX>, tm[0], tm[1], tm[2], tm[3],
                            a);
}

cudaError_t launch_pair_impl(const GemmPhase* ph0, const GemmPhase* ph1, const int32_t* offsets,
                             int E, int P, int* done, int* status, cudaStream_t s) {
  using L = PairLayout;
  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
      err = cudaFuncSetAttribute(grouped_gemm_pair_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
      if (err != cudaSuccess) return err;
      attr_set[dev] = true;
    }
  }
  GemmArgs a{};
  a.offsets = offsets;
  a.E = E;
  a.done = (ph0 && ph1) ? done : nullptr;
  a.sched = a.done != nullptr ? done + E : nullptr;   // zeroed with the dependency counters
  a.status = status;
  a.stall_stage = -1;
  a.wait_ns = kWaitLimitNs;
  a.light_mode = g_pair_light.load();
  // A0, A1, then per phase the B boxes of 128 rows (256-token units), 112 rows
  // (224-token units) and kPairBoxS rows (thin and light units)
  CUtensorMap tm[8];
  const GemmPhase* phs[2] = {ph0, ph1};
  for (int p = 0; p < 2; ++p) {
    const GemmPhase* g = phs[p] ? phs[p] : (ph0 ? ph0 : ph1);
    a.active[p] = phs[p] != nullptr;
    a.K[p] = g->K;
    a.MW[p] = g->MW;
    a.ld[p] = g->n_out;
    a.epi[p] = g->epi;
    a.ksplit[p] = 1;
    a.out[p] = g->out;
    if (!encode_tmap_2d_bf16(&tm[p], g->A_weights, (uint64_t)g->K, (uint64_t)E * g->MW, kBK,
                             kBM) ||
        !encode_tmap_2d_bf16(&tm[2 + p], g->B_act, (uint64_t)g->K, (uint64_t)P, kBK,
                             kPairBN / 2) ||
        !encode_tmap_2d_bf16(&tm[4 + p], g->B_act, (uint64_t)g->K, (uint64_t)P, kBK,
                             kPairBNL / 2) ||
        !encode_tmap_2d_bf16(&tm[6 + p], g->B_act, (uint64_t)g->K, (uint64_t)P, kBK, kPairBoxS))
      return cudaErrorInvalidValue;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(device_sm_count() & ~1, 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kSmemBytes;
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
  return cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel, tm[0], tm[1], tm[2], tm[3], tm[4],
                            tm[5], tm[6], tm[7], a);
}

// The pair kernel takes plain expert GEMMs (SwiGLU or bf16 epilogue, whole K per
// unit, B rows of length K) whose weight matrices split into 256-row blocks.
bool pairable(const GemmPhase* g) {
  return g == nullptr || (g->epi != 2 && (g->ksplit <= 1) && g->bseg == 0 &&
                          (g->b_inner == 0 || g->b_inner == g->K) && g->MW % (2 * kBM) == 0);
}

}  // namespace

void set_pair_light(int mode) { g_pair_light.store(mode); }

void set_gemm_stall(int stage, unsigned long long wait_ns) {
  g_stall_wait_ns.store(stage >= 0 ? wait_ns : kWaitLimitNs);
  g_stall_stage.store(stage >= 0 ? stage : -1);
}

cudaError_t launch_grouped_gemm(const GemmPhase* ph0, const GemmPhase* ph1,
                                const int32_t* offsets, int E, int P, int max_rows_hint,
                                int* done_counter, int* status, cudaStream_t s) {
  (void)max_rows_hint;
  // Thin token tiles when the mean expert load is small (decode), wide ones else.
  if ((long long)P <= 16LL * E)
    return launch_impl<32, 10, 16>(ph0, ph1, offsets, E, P, done_counter, status, s);
  // Wide tiles on CTA pairs where the shapes allow.  When the driver refuses the
  // cooperative cluster launch (not every SM free for a cluster, e.g. under a
  // profiler or next to another context), this call runs the one-CTA kernel; a
  // device that never accepted it is not asked again.
  static std::atomic<int> pair_state[64];  // 0 unknown, 1 launched, 2 refused
  int dev = 0;
  if (pairable(ph0) && pairable(ph1) && device_sm_count() >= 2 && cudaGetDevice(&dev) == cudaSuccess &&
      dev >= 0 && dev < 64 && pair_state[dev].load() != 2) {
    const cudaError_t err = launch_pair_impl(ph0, ph1, offsets, E, P, done_counter, status, s);
    if (err == cudaSuccess) {
      pair_state[dev].store(1);
      return err;
    }
    (void)cudaGetLastError();   // a refused launch configuration is not a sticky error
    if (pair_state[dev].load() != 1) pair_state[dev].store(2);
  }
  return launch_impl<256, 4, 128>(ph0, ph1, offsets, E, P, done_counter, status, s);
}

cudaError_t launch_pack_w13(const uint16_t* w13, int E, int H, int I, uint16_t* out,
                            cudaStream_t s) {
  dim3 grid(H / 32, 2 * I / 32, E), block(32, 8);
  pack_w13_kernel<<<grid, block, 0, s>>>(w13, H, I, out);
  return cudaGetLastError();
}

cudaError_t launch_pack_down(const uint16_t* down, int E, int H, int I, uint16_t* out,
                             cudaStream_t s) {
  dim3 grid(I / 32, H / 32, E), block(32, 8);
  pack_down_kernel<<<grid, block, 0, s>>>(down, H, I, out);
  return cudaGetLastError();
}

}  // namespace moe
