// init_routing without caller-provided scratch.
//
// moe_init_routing needs a small device workspace (per-chunk expert histograms,
// and the counts when the caller does not want them).  Some callers cannot hand
// one over: code that runs inside a host framework which owns all device memory
// and exposes no allocator, or a latency-critical serving loop whose policy is to
// never allocate after start-up.  For them this file keeps the scratch in a
// fixed-size array in the library's own device memory.
//
// Set-up: the first call on each device (with that device current) looks up the
// array's device address with cudaGetSymbolAddress and caches it; in host code
// the array's name is only a host-side stand-in and must never be passed to a
// kernel.  Make that first call before any stream capture on the device.  The
// cached address belongs to the device's primary context: like the library's other
// per-device state, it assumes that context is not destroyed (cudaDeviceReset)
// while the library stays loaded.  Device indices 0..63 are supported.
//
// Sharing: every call on a device uses the same array, which keeps whatever the
// last call left in it.  Calls that can overlap on the GPU (different streams
// without ordering between them) race on it; serialise them.  Each call
// overwrites every entry it reads before reading it, so nothing needs clearing.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe_gb300.h"
#include "internal.h"

namespace {

constexpr int kChunkPairs = 2048;  // pairs per histogram chunk of the routing kernels
constexpr int kMaxChunks = (MOE_NOALLOC_MAX_PAIRS + kChunkPairs - 1) / kChunkPairs;
constexpr int kMaxExperts = 256;
constexpr int kScratchInts = kMaxChunks * kMaxExperts + kMaxExperts;

// 33 KB per device, held until the process exits.
static __device__ __align__(256) int32_t g_routing_scratch[kScratchInts];

std::mutex g_mu;
int32_t* g_scratch_addr[64] = {};

// Device address of g_routing_scratch on the current device (looked up once).
moe_status scratch_address(int32_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED_ARCH;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_routing_scratch) != cudaSuccess) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_init_routing_noalloc(const moe_bf16* x, const int32_t* topk_ids, int T,
                                               int H, int E, int k, moe_bf16* expanded_x,
                                               int32_t* expanded_row_idx,
                                               int32_t* sorted_row_idx, int32_t* expert_offsets,
                                               int32_t* counts, moe_stream_t stream) {
  if (!topk_ids || !expanded_row_idx || !sorted_row_idx || !expert_offsets)
    return MOE_ERR_INVALID_ARG;
  if (expanded_x && (!x || (reinterpret_cast<uintptr_t>(x) & 15u) ||
                     (reinterpret_cast<uintptr_t>(expanded_x) & 15u)))
    return MOE_ERR_INVALID_ARG;
  if (T < 1 || E < 1 || E > kMaxExperts || k < 1 || k > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((long long)T * k > MOE_NOALLOC_MAX_PAIRS) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (expanded_x && (H < 8 || H % 8 != 0)) return MOE_ERR_UNSUPPORTED_SHAPE;
  int major = 0, minor = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED_ARCH;
  int32_t* scratch = nullptr;
  const moe_status st = scratch_address(&scratch);
  if (st != MOE_OK) return st;
  const int P = T * k;
  if (moe::routing_ws_bytes(P, E) > sizeof(int32_t) * kMaxChunks * kMaxExperts)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  int32_t* cnt = counts ? counts : scratch + kMaxChunks * kMaxExperts;
  int32_t* dev_status = moe::device_status_ptr();
  if (moe::launch_routing(topk_ids, P, E, cnt, expert_offsets, expanded_row_idx, sorted_row_idx,
                          scratch, nullptr, dev_status, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (expanded_x &&
      moe::launch_expand_rows(x, expanded_row_idx, sorted_row_idx, expert_offsets, E, T, H, k,
                              expanded_x, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
