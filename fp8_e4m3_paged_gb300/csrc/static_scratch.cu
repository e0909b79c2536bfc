// Split + combine for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code running inside a memory
// manager that owns every byte of the device heap, plugins that are handed
// only input/output buffers by a host runtime, or latency-critical paths that
// forbid allocator calls.  fp8kv_attn_forward_static lets them run the whole
// attention without a caller-provided workspace: the FP32 partials and the
// status word live in a file-scope device array of fixed size, which every
// GPU that loads this library holds until the process exits.
//
// Host code cannot use the array's name as a device address; its address is
// looked up once per device with cudaGetSymbolAddress (with that device
// current) on the first call made on that device.  That first call should
// therefore happen before any stream capture.  The address is cached for the
// life of the process, so a device reset (cudaDeviceReset) between calls is
// not supported.  Every call shares the one array: calls whose kernels overlap
// on the GPU (different streams, or two host threads) race on it and must be
// serialised by the caller.
#include <atomic>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "fp8kv_attn.h"
#include "internal.h"

namespace fp8kv {
namespace {

__device__ __align__(256) uint8_t g_scratch[FP8KV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace fp8kv

extern "C" int fp8kv_attn_forward_static(const fp8kv_attn_plan_t* plan, const fp8kv_attn_args* a,
                                         fp8kv_stream_t stream) {
  using namespace fp8kv;
  if (!plan || !a) return FP8KV_EINVAL;
  if (plan->revision != FP8KV_ATTN_REVISION) return FP8KV_EVERSION;
  if (plan->workspace_bytes > (int64_t)FP8KV_STATIC_SCRATCH_BYTES) return FP8KV_EWORKSPACE;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return FP8KV_ECUDA;
  // Same arguments, with the static array as the workspace.
  fp8kv_attn_args s = *a;
  s.workspace = scratch;
  s.workspace_bytes = FP8KV_STATIC_SCRATCH_BYTES;
  Params p;
  int rc = build_params(plan, &s, &p);
  if (rc != FP8KV_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (p.B == 0) {
    // nothing to run; a caller's status word still reads "no anomaly"
    if (a->workspace && a->workspace_bytes >= 4 && cudaMemsetAsync(a->workspace, 0, 4, st) != cudaSuccess)
      return FP8KV_ECUDA;
    return FP8KV_OK;
  }
  // The array keeps the previous call's contents: the sticky status word
  // must start at zero; every partial the combine reads is rewritten first.
  if (cudaMemsetAsync(scratch, 0, 4, st) != cudaSuccess) return FP8KV_ECUDA;
  cudaError_t e;
  switch (plan->kernel) {
    case kGeneric: e = launch_split_generic(plan, p, st); break;
    case kTc:
    case kTcSmall: e = launch_split_tc(plan, p, st); break;
    default: return FP8KV_EINVAL;
  }
  if (e != cudaSuccess) return FP8KV_ECUDA;
  e = launch_combine(plan, p, st);
  if (e != cudaSuccess) return FP8KV_ECUDA;
  // Optional: the call's status word, for callers that pass a 4-byte buffer.
  if (a->workspace && a->workspace_bytes >= 4) {
    if (cudaMemcpyAsync(a->workspace, scratch, 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
      return FP8KV_ECUDA;
  }
  return FP8KV_OK;
}
