// Cross-rank merge of (FP32 output, base-2 LSE) pairs: the context-parallel
// combine of "Qualify calibrated E4M3 and disk PLE with QSA DCP2" (ranks
// expose base-2 LSE and FP32 partial output; an all-to-all or an all-gather
// of the LSEs plus a reduce-scatter of the outputs merges them).
//
//   L = log2(sum_r 2^lse_r),  out = sum_r 2^(lse_r - L) o_r
//
// D/4 threads per vector, each owning four columns; every thread of a vector
// reads the R LSEs (L1 broadcast), then one float4 per rank.  A few MB per
// call at most: latency-bound, one pass over the inputs.
#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace fp8kv {
namespace {

constexpr int kMergeThreads = 256;

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const fp8kv_merge_args a, int32_t scale_rank) {
  const int tpv = a.head_dim / 4;                 // threads per vector
  const int vpc = kMergeThreads / tpv;            // vectors per CTA
  const int64_t i = (int64_t)blockIdx.x * vpc + threadIdx.x / tpv;
  const int c4 = threadIdx.x % tpv;
  if (threadIdx.x >= vpc * tpv || i >= a.num_vectors) return;
  const int R = a.num_ranks;
  float L = -INFINITY;
  for (int r = 0; r < R; ++r) L = fmaxf(L, a.lses[r * a.rank_stride_lse + i]);
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  float W = 0.f;
  if (L != -INFINITY) {
    for (int r = 0; r < R; ++r) W += exp2f(a.lses[r * a.rank_stride_lse + i] - L);
    const float inv = 1.f / W;
    if (scale_rank >= 0) {
      // this rank's own output, weighted for the reduce-scatter sum
      const float w = exp2f(a.lses[scale_rank * a.rank_stride_lse + i] - L) * inv;
      const float4 x = *reinterpret_cast<const float4*>(a.outs + i * a.head_dim + c4 * 4);
      o = make_float4(w * x.x, w * x.y, w * x.z, w * x.w);
    } else {
      for (int r = 0; r < R; ++r) {
        const float w = exp2f(a.lses[r * a.rank_stride_lse + i] - L) * inv;
        if (w == 0.f) continue;  // a rank that saw nothing (its o is never read)
        const float4 x = *reinterpret_cast<const float4*>(a.outs + r * a.rank_stride_out + i * a.head_dim + c4 * 4);
        o.x = fmaf(w, x.x, o.x);
        o.y = fmaf(w, x.y, o.y);
        o.z = fmaf(w, x.z, o.z);
        o.w = fmaf(w, x.w, o.w);
      }
    }
  }
  if (a.out_f32) *reinterpret_cast<float4*>(a.out_f32 + i * a.head_dim + c4 * 4) = o;
  if (a.out) {
    const __half2 h01 = __floats2half2_rn(o.x, o.y), h23 = __floats2half2_rn(o.z, o.w);
    uint2 pk;
    pk.x = *reinterpret_cast<const uint32_t*>(&h01);
    pk.y = *reinterpret_cast<const uint32_t*>(&h23);
    *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(a.out) + i * a.head_dim + c4 * 4) = pk;
  }
  if (a.lse_out && c4 == 0) a.lse_out[i] = (L == -INFINITY) ? -INFINITY : L + log2f(W);
}

}  // namespace

cudaError_t launch_merge(const fp8kv_merge_args& a, int32_t scale_rank, cudaStream_t st) {
  const int tpv = a.head_dim / 4;
  const int vpc = kMergeThreads / tpv;
  const int64_t grid = (a.num_vectors + vpc - 1) / vpc;
  merge_kernel<<<(unsigned)grid, kMergeThreads, 0, st>>>(a, scale_rank);
  return cudaGetLastError();
}

}  // namespace fp8kv
