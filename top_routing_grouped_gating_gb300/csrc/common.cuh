// Shared device helpers for the sm_103a MoE-layer kernels: bf16 packing, the
// device status word, and thin inline-PTX wrappers for mbarrier, TMA (bulk
// tensor copies) and the 5th-generation tensor core (tcgen05 + TMEM).
//
// Every wait on an mbarrier or on a global flag is bounded in wall-clock time
// (%globaltimer).  A wait that runs out sets MOE_DEV_WAIT_TIMEOUT in the status
// word and returns false; callers then unwind without trapping.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_gb300.h"

#define MOE_DEVINL __device__ __forceinline__

namespace moe {

// Wall-clock limit of any single device-side wait (ns).  Far above any legal
// wait (a whole grouped GEMM takes milliseconds), far below a watchdog.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

MOE_DEVINL void flag_status(int* status, int bits) {
  if (status != nullptr) atomicOr(status, bits);
}

MOE_DEVINL uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

MOE_DEVINL unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------- bf16 ----
MOE_DEVINL float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
MOE_DEVINL float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
MOE_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);  // .x = lo (low 16 bits)
  return *reinterpret_cast<uint32_t*>(&p);
}
// Exact three-piece bf16 split v = p0 + p1 + p2 (8 + 8 + 8 significand bits): each
// piece is the bf16 rounding of what the pieces before it left over.
MOE_DEVINL void split3_bf16(float v, uint16_t (&p)[3]) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  p[0] = *reinterpret_cast<uint16_t*>(&b);
  const float r1 = v - bf16_lo(p[0]);
  b = __float2bfloat16_rn(r1);
  p[1] = *reinterpret_cast<uint16_t*>(&b);
  const float r2 = r1 - bf16_lo(p[1]);
  b = __float2bfloat16_rn(r2);
  p[2] = *reinterpret_cast<uint16_t*>(&b);
}
// Eight consecutive fp32 values split into three rows of eight bf16 pieces, stored
// at dst, dst + stride and dst + 2 * stride (16-byte aligned).
MOE_DEVINL void store_split3_x8(const float (&v)[8], uint16_t* dst, size_t stride) {
  uint32_t w[3][4];
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    uint16_t p0[3], p1[3];
    split3_bf16(v[i], p0);
    split3_bf16(v[i + 1], p1);
#pragma unroll
    for (int s = 0; s < 3; ++s)
      w[s][i / 2] = static_cast<uint32_t>(p0[s]) | (static_cast<uint32_t>(p1[s]) << 16);
  }
#pragma unroll
  for (int s = 0; s < 3; ++s)
    *reinterpret_cast<uint4*>(dst + s * stride) = make_uint4(w[s][0], w[s][1], w[s][2], w[s][3]);
}

// ------------------------------------------------------------- mbarrier ----
MOE_DEVINL void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
MOE_DEVINL void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
MOE_DEVINL void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
MOE_DEVINL void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
MOE_DEVINL bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false
// if the time limit (limit_ns) passed or *abort became non-zero (another role gave up).
MOE_DEVINL bool mbar_wait(uint64_t* bar, uint32_t parity, const volatile int* abort,
                          unsigned long long limit_ns = kWaitLimitNs) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(a, parity)) return true;
    if ((i & 63u) == 0) {
      if (abort != nullptr && *abort) return false;
      if (globaltimer() - t0 > limit_ns) return false;
    }
  }
}

// Named barrier among a subset of the CTA's warps (id 0 is __syncthreads).
MOE_DEVINL void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ TMA ----
MOE_DEVINL void tma_prefetch_desc(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}
// Asks the memory system to bring [p, p + bytes) into L2; nothing waits for it.
// p 16-byte aligned, bytes a multiple of 16, the range inside one allocation.
MOE_DEVINL void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)),
               "r"(bytes)
               : "memory");
}
MOE_DEVINL uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
MOE_DEVINL uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
MOE_DEVINL uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 2-D tiled bulk tensor load global -> shared, completion counted in bytes on bar.
// x (innermost coordinate, elements) must keep x*elem_size a multiple of 16 bytes.
MOE_DEVINL void tma_load_2d(void* smem_dst, const CUtensorMap* tm, uint64_t* bar, int x, int y,
                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size multiple of 16).
MOE_DEVINL void bulk_load_1d(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                             uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

MOE_DEVINL void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// -------------------------------------------------------- tcgen05 / TMEM ----
// Allocation is a whole-warp operation; the TMEM address lands in shared memory.
MOE_DEVINL void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
MOE_DEVINL void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MOE_DEVINL void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
MOE_DEVINL void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
MOE_DEVINL void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive once on bar when every tcgen05 op issued so far by this thread is done.
MOE_DEVINL void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// D(tmem) (+)= A(smem desc) x B(smem desc)^T, bf16 inputs, fp32 accumulate.
MOE_DEVINL void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA with
// 128-byte swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms stacked
// along M/N.  Leading-byte offset is unused for this layout; stride = 1024 bytes.
// The tile base must be 1024-byte aligned; stepping K inside the 128-byte row is
// done by adding the byte offset to the start address.
MOE_DEVINL uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address, bits 0-13
  d |= static_cast<uint64_t>(1) << 16;                   // leading byte offset (16 B, unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                   // descriptor version (sm_100 family)
  d |= static_cast<uint64_t>(2) << 61;                   // swizzle mode: 128-byte
  return d;
}

// Shared-memory descriptor of a K-major tile without swizzle: 8-row x 16-byte core
// matrices, `sbo` bytes apart along M/N (used for the 32 x 16-byte scale atoms).
MOE_DEVINL uint64_t smem_desc_noswz(uint32_t saddr, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// Copy a 32-row x 128-bit shared-memory tile into TMEM columns [taddr, taddr+4),
// replicated into all four 32-lane quarters (the scale-factor atom layout).
MOE_DEVINL void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Block-scaled MMA: D (+)= (A . 2^SFA) x (B . 2^SFB)^T, A and B e4m3, scales E8M0
// per 32 K-elements read from TMEM, fp32 accumulate.  K = 32 per instruction.
MOE_DEVINL void tc_mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Instruction descriptor, kind::mxf8f6f4 with block scaling: A and B e4m3, both
// K-major, E8M0 scales; sf ids pick the byte of each 32-bit scale word.
__host__ __device__ constexpr uint32_t idesc_mxf8_f32(int M, int N, uint32_t sfa_id,
                                                      uint32_t sfb_id) {
  return (sfb_id << 4)                               // B scale-factor byte
         | (0u << 7) | (0u << 10)                    // A, B format: e4m3
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (1u << 23)                                // scale format: E8M0
         | (static_cast<uint32_t>(M >> 4) << 24)     // M / 16
         | (sfa_id << 29);                           // A scale-factor byte
}

// The scale-factor byte fields of a kind::mxf8f6f4 instruction descriptor alone.
__host__ __device__ constexpr uint32_t idesc_sf_ids(uint32_t sfa_id, uint32_t sfb_id) {
  return (sfb_id << 4) | (sfa_id << 29);
}
static_assert((idesc_mxf8_f32(128, 64, 0, 0) | idesc_sf_ids(3, 2)) == idesc_mxf8_f32(128, 64, 3, 2),
              "scale-factor id fields");

// Instruction descriptor, kind::f16: D f32, A and B bf16, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                                   // D format: f32
         | (1u << 7)                                 // A format: bf16
         | (1u << 10)                                // B format: bf16
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// 32 consecutive TMEM columns of this warp's 32 lanes (lane i of the warp reads
// TMEM lane (taddr.lane + i)); waits for the load before returning.
MOE_DEVINL void tmem_ld_32x32b_x32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// The same load without the wait: the registers hold the values only after a later
// tmem_wait_ld() in this thread (several loads can be in flight before one wait).
MOE_DEVINL void tmem_ld_32x32b_x32_nowait(uint32_t taddr, float (&v)[32]) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
MOE_DEVINL void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Per-warpgroup register budget (all four warps of a warpgroup execute it): the
// block's launch-time registers are shared out anew; the shares must add up to at
// most the block's threads x registers per thread at launch.
template <int N>
MOE_DEVINL void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
MOE_DEVINL void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Global flag helpers (acquire/release at GPU scope) for cross-CTA dependencies.
MOE_DEVINL int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
MOE_DEVINL void red_release_add_gpu(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ------------------------------------------------------- CTA pairs (2-SM) --
// A cluster of two CTAs on two SMs whose tensor cores run one cta_group::2 MMA:
// the even CTA issues it; each CTA holds half of the M rows of A and half of the
// N rows of B in its own shared memory, and its 128 lanes of the accumulator.
MOE_DEVINL uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The shared::cluster address of `addr` (a shared::cta address) in CTA `rank`.
MOE_DEVINL uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier of another CTA of the cluster (release, cluster scope).
MOE_DEVINL void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// Relaxed remote arrive, for passing on that bytes this thread has already seen
// land in its own shared memory (through its own mbarrier) are there; a release
// at cluster scope costs the issuing thread over a thousand clocks.
MOE_DEVINL void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// Unit lists that a CTA pair's even CTA publishes into both CTAs' shared memory
// while the pair runs: an entry is one 64-bit word (a packed unit, whose high word
// is never one of the two markers below), stored and polled with relaxed accesses
// at cluster scope, so that the word is its own flag and the publishing thread waits
// for nothing.
constexpr uint32_t kEndUnitWord = 0xFFFFFFFFu;       // high word of a list's end entry
constexpr uint32_t kPendingUnitWord = 0xFFFFFFFEu;   // high word of an entry not yet published
MOE_DEVINL uint64_t ld_relaxed_cluster_u64(uint32_t cta_addr) {
  uint64_t v;
  asm volatile("ld.relaxed.cluster.shared::cta.u64 %0, [%1];" : "=l"(v) : "r"(cta_addr) : "memory");
  return v;
}
MOE_DEVINL void st_relaxed_cluster_u64(uint32_t cluster_addr, uint64_t v) {
  asm volatile("st.relaxed.cluster.shared::cluster.u64 [%0], %1;" ::"r"(cluster_addr), "l"(v)
               : "memory");
}
MOE_DEVINL uint64_t unit_word(uint2 w) {
  return static_cast<uint64_t>(w.x) | (static_cast<uint64_t>(w.y) << 32);
}
MOE_DEVINL bool mbar_try_wait_cluster(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait with cluster-scope acquire (for a barrier with remote arrivals).
MOE_DEVINL bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, const volatile int* abort) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait_cluster(a, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(a, parity)) return true;
    if ((i & 63u) == 0) {
      if (abort != nullptr && *abort) return false;
      if (globaltimer() - t0 > kWaitLimitNs) return false;
    }
  }
}
// Every thread of both CTAs.
MOE_DEVINL void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
MOE_DEVINL void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
MOE_DEVINL void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
MOE_DEVINL void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Arrive once on the mbarrier at this shared::cta offset in every CTA of `mask` when
// the pair operations issued so far by this thread are done.
MOE_DEVINL void tc_commit_pair(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}
// Scale-atom copy for a pair MMA, issued by the even CTA: each CTA's 32 x 128-bit
// shared-memory tile (same offset in both) lands in its own TMEM columns
// [taddr, taddr + 4), replicated into all four lane quarters.
MOE_DEVINL void tc_cp_pair_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}
// Block-scaled MMA over the pair: M = 256 (128 weight rows per CTA), B's N rows split
// between the CTAs (N/2 each), E8M0 scales from each CTA's own TMEM, fp32 accumulate.
MOE_DEVINL void tc_mma_pair_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                 uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// bf16 MMA over the pair: M = 256 (128 rows of A per CTA), B's N rows split
// between the CTAs (N/2 each), fp32 accumulators in each CTA's TMEM.
MOE_DEVINL void tc_mma_pair_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// ------------------------------------------- programmatic dependent launch ----
// A kernel launched with programmatic stream serialization may start before its
// predecessor in the stream has finished; it must call pdl_wait() before touching
// anything the predecessor writes.  pdl_trigger() lets this kernel's own successor
// start launching early (its pdl_wait still waits for this grid to complete).
MOE_DEVINL void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_DEVINL void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Host: launch with programmatic stream serialization allowed.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace moe
