// Tensor-core (tcgen05) split kernel.  Not selected by the planner yet.
#include <cuda_runtime.h>

#include "internal.h"

namespace fp8kv {

cudaError_t launch_split_tc(const fp8kv_attn_plan_t*, const Params&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace fp8kv
