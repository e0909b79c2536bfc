// Combine kernel: merge the split-KV partitions of every query vector in FP32.
//
//   M = max_s m_s over partitions with l_s > 0
//   w_s = 2^(m_s - M),  L = sum_s w_s l_s,  out = v_scale * sum_s w_s acc_s / L
//
// written as fp16 with round-to-nearest-even.  A query vector whose total L is
// 0 (dead row, or nothing visible) gets +0.0.  Partitions with l_s = 0 are
// skipped by a branch, so their numerators are never read ("DFlash2 E4M3
// attention with FP32 state", intro paragraph 4: FP32 combination, FP16 final
// activation; "Qwen4Exp: fp8_e4m3 main KV cache on the QSA path", review:
// v_scale acts as the output scale).
#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace fp8kv {
namespace {

constexpr int CT = 128;  // threads per combine CTA

// One CTA per output vector (b, r, h); thread handles d = tid + k*CT.
template <int D>
__global__ void __launch_bounds__(CT) combine_kernel(Params p) {
  constexpr int PER = (D + CT - 1) / CT;
  const int idx = blockIdx.x;  // (b*q_max + r)*Hq + h
  const int h = idx % p.Hq;
  const int r = (idx / p.Hq) % p.q_max;
  const int b = idx / (p.Hq * p.q_max);
  const int g = h / p.G;
  const int i = r * p.G + (h % p.G);
  const int64_t base = (((int64_t)b * p.Hkv + g) * p.S) * p.rows + i;
  const float2* ml = p.ml + base;
  const float* acc = p.partial + base * D;
  const int64_t sstride = p.rows;  // partitions of one query vector are rows apart

  float M = -INFINITY;
  for (int s = 0; s < p.S; ++s) {
    const float2 v = ml[s * sstride];
    if (v.y > 0.f) M = fmaxf(M, v.x);
  }
  float L = 0.f;
  float o[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) o[k] = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < p.S; ++s) {
      const float2 v = ml[s * sstride];
      if (v.y > 0.f) {
        const float w = exp2_int(v.x - M);  // maxima are integers: exact
        L = fmaf(w, v.y, L);
        const float* a = acc + (int64_t)s * sstride * D;
#pragma unroll
        for (int k = 0; k < PER; ++k) {
          const int d = threadIdx.x + k * CT;
          if (d < D) o[k] = fmaf(w, a[d], o[k]);
        }
      }
    }
  }
  const float vs = p.v_scale_dev ? *p.v_scale_dev : p.v_scale;
  const float f = (L > 0.f) ? vs / L : 0.f;
  uint16_t* out = p.out + (int64_t)idx * D;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int d = threadIdx.x + k * CT;
    if (d < D) {
      const float y = (L > 0.f) ? o[k] * f : 0.f;
      out[d] = __half_as_ushort(__float2half_rn(y));
    }
  }
}

}  // namespace

cudaError_t launch_combine(const fp8kv_attn_plan_t* plan, const Params& p, cudaStream_t st) {
  const int n = p.B * p.q_max * p.Hq;
  if (n == 0) return cudaSuccess;
  switch (p.D) {
    case 64: combine_kernel<64><<<n, CT, 0, st>>>(p); break;
    case 128: combine_kernel<128><<<n, CT, 0, st>>>(p); break;
    case 256: combine_kernel<256><<<n, CT, 0, st>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  (void)plan;
  return cudaGetLastError();
}

}  // namespace fp8kv
