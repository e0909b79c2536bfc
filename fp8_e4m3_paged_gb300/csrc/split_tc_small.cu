// Instantiations of the transposed tensor-core split kernel for groups of at
// most 16 query vectors per (request, KV head) (decode and small verify
// groups), specialised on the number of live query vectors the softmax
// handles per token (4, 8 or 16).  The kernel is in split_tc_kernel.cuh.
#include "split_tc_kernel.cuh"

namespace fp8kv {
namespace {

template <int FMT, int NL>
cudaError_t launch_nl(const fp8kv_attn_plan_t* plan, const Params& p, cudaStream_t st) {
  if (p.D == 256)
    return p.mode == FP8KV_MODE_DENSE ? launch<256, FP8KV_MODE_DENSE, FMT, true, NL>(plan, p, st)
                                      : launch<256, FP8KV_MODE_SPARSE_PAGE4, FMT, true, NL>(plan, p, st);
  if (p.D == 128)
    return p.mode == FP8KV_MODE_DENSE ? launch<128, FP8KV_MODE_DENSE, FMT, true, NL>(plan, p, st)
                                      : launch<128, FP8KV_MODE_SPARSE_PAGE4, FMT, true, NL>(plan, p, st);
  return cudaErrorInvalidValue;
}

template <int FMT>
cudaError_t launch_fmt(const fp8kv_attn_plan_t* plan, const Params& p, cudaStream_t st) {
  if (p.row_chunk <= 4) return launch_nl<FMT, 4>(plan, p, st);
  if (p.row_chunk <= 8) return launch_nl<FMT, 8>(plan, p, st);
  return launch_nl<FMT, kN>(plan, p, st);
}

}  // namespace

cudaError_t launch_split_tc_small(const fp8kv_attn_plan_t* plan, const Params& p, cudaStream_t st) {
  return p.kv_format == FP8KV_KV_E5M2 ? launch_fmt<FP8KV_KV_E5M2>(plan, p, st)
                                      : launch_fmt<FP8KV_KV_E4M3>(plan, p, st);
}

}  // namespace fp8kv
