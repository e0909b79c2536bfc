// Instantiations of the tensor-core split kernel whose MMA rows are the
// query vectors (up to 64 per CTA), the shared-memory sizes of both variants,
// and the dispatch of a plan to its variant (the kernel is in
// split_tc_kernel.cuh).
#include "split_tc_kernel.cuh"

namespace fp8kv {

int tc_smem_bytes(int D, bool small_group) {
  if (small_group) return D == 256 ? Cfg<256, true>::kSmem : Cfg<128, true>::kSmem;
  return D == 256 ? Cfg<256, false>::kSmem : Cfg<128, false>::kSmem;
}

namespace {

template <int FMT>
cudaError_t launch_rows(const fp8kv_attn_plan_t* plan, const Params& p, cudaStream_t st) {
  if (p.D == 256)
    return p.mode == FP8KV_MODE_DENSE ? launch<256, FP8KV_MODE_DENSE, FMT, false, kN>(plan, p, st)
                                      : launch<256, FP8KV_MODE_SPARSE_PAGE4, FMT, false, kN>(plan, p, st);
  if (p.D == 128)
    return p.mode == FP8KV_MODE_DENSE ? launch<128, FP8KV_MODE_DENSE, FMT, false, kN>(plan, p, st)
                                      : launch<128, FP8KV_MODE_SPARSE_PAGE4, FMT, false, kN>(plan, p, st);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_split_tc(const fp8kv_attn_plan_t* plan, const Params& p, cudaStream_t st) {
  if (plan->kernel == kTcSmall) return launch_split_tc_small(plan, p, st);
  return p.kv_format == FP8KV_KV_E5M2 ? launch_rows<FP8KV_KV_E5M2>(plan, p, st)
                                      : launch_rows<FP8KV_KV_E4M3>(plan, p, st);
}

}  // namespace fp8kv
