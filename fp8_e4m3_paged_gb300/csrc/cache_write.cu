// Cache write: new fp16 / bf16 K and V rows -> E4M3 (or E5M2) bytes in the
// paged cache.
//
//   byte = E4M3(fp32(x) / scale)        (E5M2 likewise)
//
// with the division correctly rounded in FP32 and the conversion done by the
// hardware's cvt.rn.satfinite.e4m3x2.f32 / .e5m2x2.f32 (round to nearest
// even, saturating to +-448 / +-57344).  The quotient only matters through its E4M3 rounding, so the
// kernel multiplies by the reciprocal and divides exactly only where that
// could change the code (see quot()).  This is the write path that fills the cache the attention
// reads, with the layer's per-tensor scales ("Qwen4Exp: fp8_e4m3 main KV
// cache on the QSA path", PR description).
//
// One thread per (token, KV head, two 16-element chunks) writes both the K
// and the V chunks: 16-byte loads and stores, all coalesced along d.  The op moves 4 bytes in and 2 bytes out per element
// pair (K and V) and is bound by HBM; the grid is one wave of resident CTAs
// (a multiple of the SM count) with a grid-stride loop.
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "fp8_encode.cuh"
#include "internal.h"

namespace fp8kv {
namespace {

constexpr int kCwThreads = 256;

// One work item = CPT consecutive 16-element chunks of one (token, head), K
// and V.  The slot of the next item is loaded one iteration ahead, so the
// input loads never wait for it.
template <int DT, int CPT, int FMT>
__global__ void __launch_bounds__(kCwThreads) cache_write_kernel(const fp8kv_cache_write_args a) {
  const float ks = a.k_scale_dev ? *a.k_scale_dev : a.k_scale;
  const float vs = a.v_scale_dev ? *a.v_scale_dev : a.v_scale;
  const float kr = __frcp_rn(ks), vr = __frcp_rn(vs);
  const int items_per_head = a.head_dim / (16 * CPT);
  const int64_t per_token = (int64_t)a.num_kv_heads * items_per_head;
  const int64_t total = (int64_t)a.num_tokens * per_token;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const uint16_t* k = reinterpret_cast<const uint16_t*>(a.k);
  const uint16_t* v = reinterpret_cast<const uint16_t*>(a.v);
  int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t slot_next = idx < total ? __ldg(a.slot_mapping + idx / per_token) : -1;
  for (; idx < total; idx += stride) {
    const int64_t slot = slot_next;
    if (idx + stride < total) slot_next = __ldg(a.slot_mapping + (idx + stride) / per_token);
    if (slot < 0) continue;
    const int64_t n = idx / per_token;
    const int rem = (int)(idx - n * per_token);
    const int h = rem / items_per_head;
    const int c0 = (rem - h * items_per_head) * CPT;
    const int64_t blk = slot / a.page_size, off = slot % a.page_size;
    if (blk >= a.num_kv_blocks) {
      if (c0 == 0 && h == 0 && a.status) set_status(a.status, FP8KV_STATUS_BAD_BLOCK);
      continue;
    }
    const uint4* kp = reinterpret_cast<const uint4*>(k + n * a.k_stride_token + h * a.k_stride_head + c0 * 16);
    const uint4* vp = reinterpret_cast<const uint4*>(v + n * a.v_stride_token + h * a.v_stride_head + c0 * 16);
    uint4 kx[CPT][2], vx[CPT][2];
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      kx[j][0] = __ldg(kp + 2 * j);
      kx[j][1] = __ldg(kp + 2 * j + 1);
      vx[j][0] = __ldg(vp + 2 * j);
      vx[j][1] = __ldg(vp + 2 * j + 1);
    }
    uint8_t* kd = a.k_cache + blk * a.kc_stride_block + off * a.kc_stride_token + h * a.kc_stride_head + c0 * 16;
    uint8_t* vd = a.v_cache + blk * a.vc_stride_block + off * a.vc_stride_token + h * a.vc_stride_head + c0 * 16;
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      *reinterpret_cast<uint4*>(kd + 16 * j) = quant16<DT, FMT>(kx[j], ks, kr);
      *reinterpret_cast<uint4*>(vd + 16 * j) = quant16<DT, FMT>(vx[j], vs, vr);
    }
  }
}

}  // namespace

cudaError_t launch_cache_write(const fp8kv_cache_write_args& a, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const bool two = (a.head_dim / 16) % 2 == 0;  // two chunks per item when the row splits evenly
  void (*fn)(const fp8kv_cache_write_args);
  constexpr int E4 = FP8KV_KV_E4M3, E5 = FP8KV_KV_E5M2, F16 = FP8KV_DTYPE_F16, BF16 = FP8KV_DTYPE_BF16;
  const bool e5 = a.kv_format == E5;
  if (a.dtype == F16)
    fn = e5 ? (two ? cache_write_kernel<F16, 2, E5> : cache_write_kernel<F16, 1, E5>)
            : (two ? cache_write_kernel<F16, 2, E4> : cache_write_kernel<F16, 1, E4>);
  else
    fn = e5 ? (two ? cache_write_kernel<BF16, 2, E5> : cache_write_kernel<BF16, 1, E5>)
            : (two ? cache_write_kernel<BF16, 2, E4> : cache_write_kernel<BF16, 1, E4>);
  // one wave of resident CTAs (grid-stride loop over the items)
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kCwThreads, 0);
  if (e != cudaSuccess) return e;
  const int64_t total = (int64_t)a.num_tokens * a.num_kv_heads * (a.head_dim / (two ? 32 : 16));
  const int64_t need = (total + kCwThreads - 1) / kCwThreads;
  const int64_t cap = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
  const unsigned grid = (unsigned)(need < cap ? need : cap);
  fn<<<grid, kCwThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace fp8kv
