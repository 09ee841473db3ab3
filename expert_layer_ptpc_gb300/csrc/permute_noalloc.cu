// moe_permute_noalloc: the expert permutation without a caller-supplied
// workspace, for callers that cannot allocate device memory.
//
// Who needs this: a host that embeds this layer inside another framework
// which has already reserved the device's memory in its own arena (no free
// memory left for cudaMalloc, and no handle to that arena), or a latency-
// critical serving loop that may not call cudaMalloc/cudaFree at all because
// those calls synchronise the device. Such a caller passes only its inputs
// and outputs; the scratch lives in the fixed array below.
//
// The scratch is a file-scope device array of kNoAllocScratchInts int32
// (1 MiB). Every GPU that loads the library holds it until the process exits.
// It holds the per-chunk expert histograms of the multi-block path; that path
// writes every entry it later reads, so nothing has to start at zero, and the
// array keeps whatever the last call left in it. All calls share the one
// array: calls whose kernels overlap on the GPU (different streams, or
// different host threads on one device) race on it and must be serialised by
// the caller.
//
// Host code may not hand the array's name to a kernel: on the host that name
// is only a stand-in, not a device address. The first call on each device,
// with that device current, looks up the array's device address with
// cudaGetSymbolAddress and caches it; make that first call before any stream
// capture on the device. The cache lives as long as the process: after a
// cudaDeviceReset the module is loaded again at another address, and this
// entry point must not be used on that device any more.
#include <mutex>

#include "../../include/moe_ptpc.h"
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int64_t kNoAllocScratchInts = 262144;   // 1 MiB of int32

static __device__ __align__(256) int g_permute_scratch[kNoAllocScratchInts];

constexpr int kMaxDevices = 64;

// Device address of g_permute_scratch on the current device, looked up once
// per device. Returns nullptr (and leaves *err set) if the lookup fails.
int* scratch_on_current_device(cudaError_t* err) {
  static std::mutex mu;
  static int* addr[kMaxDevices] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = static_cast<int*>(p);
  }
  *err = cudaSuccess;
  return addr[dev];
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_permute_noalloc(const int32_t* topk_ids, int T, int E, int k,
                                   int32_t* expert_counts,
                                   int32_t* expert_offsets,
                                   int32_t* sorted_to_flat,
                                   int32_t* flat_to_sorted,
                                   moe_stream_t stream) {
  if (T < 0 || E <= 0 || k < 1 || k > E || k > kMaxTopK)
    return MOE_ERR_INVALID_ARG;
  if (E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)T * k >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  if (!expert_counts || !expert_offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_ids || !sorted_to_flat || !flat_to_sorted))
    return MOE_ERR_INVALID_ARG;
  const int64_t R = (int64_t)T * k;
  // larger problems need more histogram scratch than the fixed array holds
  if (permute_ws_bytes(R, E) > (size_t)kNoAllocScratchInts * sizeof(int))
    return MOE_ERR_UNSUPPORTED;
  cudaError_t err;
  int* scratch = scratch_on_current_device(&err);
  if (scratch == nullptr) return MOE_ERR_CUDA;
  err = launch_permute(topk_ids, R, E, expert_counts, expert_offsets,
                       sorted_to_flat, flat_to_sorted, -1, scratch,
                       static_cast<cudaStream_t>(stream), false);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
