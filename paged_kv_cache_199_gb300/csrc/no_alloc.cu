// Allocation-free GQA decode entry point.
//
// paged_decode_run needs a caller-provided workspace (work list, split
// counters, split partial states). Some callers cannot obtain one: code
// that must not call cudaMalloc at all, for example an inference runtime
// that reserves all device memory at start-up and forbids allocation
// afterwards, a plugin whose host framework owns the device allocator, or
// a real-time path where an allocation's latency or failure is not
// acceptable. paged_decode_run_no_alloc serves them: the workspace is a
// fixed-size array in the library's own device memory (a file-scope
// __device__ array, present on every GPU that loads the library for the
// life of the process), and the call allocates nothing.
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"
#include "paged_decode.h"
#include "plan_internal.h"

namespace pd {
namespace {

// The largest workspace the allocation-free entry point can serve.
constexpr size_t kNoAllocScratchBytes = PD_NO_ALLOC_MAX_WORKSPACE_BYTES;

__device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device. In host code
// the array's name is only a host-side stand-in, so the address is looked
// up once per device with that device current, and cached. The cache
// belongs to the runtime's primary context of each device: after
// cudaDeviceReset, or under another driver context, the cached address is
// no longer the array's.
pd_status scratch_for_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "scratch device query");
  if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice, "scratch device query");
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_no_alloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "scratch symbol lookup");
    if (ptr == nullptr) return cuda_fail(cudaErrorInvalidSymbol, "scratch symbol lookup");
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return PD_OK;
}

}  // namespace
}  // namespace pd

extern "C" pd_status paged_decode_run_no_alloc(const pd_plan* plan, const void* q, const void* k_pool,
                                               const void* v_pool, const int32_t* block_tables,
                                               const int32_t* seq_lens, const int32_t* q_indptr,
                                               float sm_scale, const float* k_scale,
                                               const float* v_scale, void* out, float* lse,
                                               pd_stream_t stream) {
  if (!plan || plan->prob.kind != PD_ATTN_GQA) return PD_ERR_INVALID_ARG;
  // a plan whose workspace exceeds the array is refused before anything runs
  if (paged_decode_workspace_size(plan) > pd::kNoAllocScratchBytes) return PD_ERR_WORKSPACE_TOO_SMALL;
  if (plan->items.empty()) return PD_OK;   // an empty batch: nothing to enqueue
  // the argument rules of paged_decode_run, checked before the plan copy so
  // that a refused call enqueues nothing
  auto misaligned = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; };
  if (!q || !k_pool || !v_pool || !block_tables || !seq_lens || !out) return PD_ERR_INVALID_ARG;
  if (misaligned(q) || misaligned(k_pool) || misaligned(v_pool) || misaligned(out)) return PD_ERR_INVALID_ARG;
  if (plan->prob.kv_dtype == PD_KV_FP8_E4M3 && (!k_scale || !v_scale)) return PD_ERR_INVALID_ARG;
  if (!(sm_scale == sm_scale)) return PD_ERR_INVALID_ARG;
  void* scratch = nullptr;
  pd_status st = pd::scratch_for_current_device(&scratch);
  if (st != PD_OK) return st;
  // The array keeps whatever the previous call left in it, so every call
  // rewrites the plan image, which also zeroes the split counters, the
  // queue counters and the error word.
  st = paged_decode_plan_upload(plan, scratch, pd::kNoAllocScratchBytes, stream);
  if (st != PD_OK) return st;
  return paged_decode_run(plan, q, k_pool, v_pool, block_tables, seq_lens, q_indptr, sm_scale,
                          k_scale, v_scale, out, lse, scratch, pd::kNoAllocScratchBytes, stream);
}
