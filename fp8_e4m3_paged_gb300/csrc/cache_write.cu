// Cache write: new fp16 / bf16 K and V rows -> E4M3 bytes in the paged cache.
//
//   byte = E4M3(fp32(x) / scale)
//
// with the division correctly rounded in FP32 and the conversion done by the
// hardware's cvt.rn.satfinite.e4m3x2.f32 (round to nearest even, saturating
// to +-448).  The quotient only matters through its E4M3 rounding, so the
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
#include "internal.h"

namespace fp8kv {
namespace {

constexpr int kCwThreads = 256;

// Four floats (memory order) -> four E4M3 bytes, little-endian in a word.
// The instruction puts its first source in the upper byte of the pair.
__device__ __forceinline__ uint32_t e4m3x4(float x0, float x1, float x2, float x3) {
  uint32_t w;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(w)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
  return w;
}

// Two 2-byte elements (one 32-bit word) -> two floats.
template <int DT>
__device__ __forceinline__ float2 to_f32x2(uint32_t w) {
  if (DT == FP8KV_DTYPE_F16) return __half22float2(*reinterpret_cast<const __half2*>(&w));
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
}

// x / s as far as its E4M3 code is concerned.  q = x * r with r = fl(1/s)
// is within 2 fp32 ulps of the correctly rounded quotient fl(x/s) (one
// rounding of r, one of the product).  The E4M3 code of a normal value is
// decided by the 20 fp32 mantissa bits below its 3 kept bits against the
// halfway pattern 0x80000, so when those bits of q are more than 4 ulps
// from it, q and fl(x/s) lie strictly on the same side of the same
// rounding boundary and convert to the same code.  Within 4 ulps of a
// boundary, below the E4M3 normal range (2^-6), or for non-finite q the
// exact quotient is computed.
__device__ __forceinline__ float quot(float x, float s, float r) {
  const float q = x * r;
  const float aq = fabsf(q);
  const uint32_t low = __float_as_uint(q) & 0xFFFFFu;
  const bool exact = !(aq >= 0.015625f && aq <= 3.0e38f) || (low - 0x7FFFCu) <= 8u;
  return exact ? __fdiv_rn(x, s) : q;
}

// 16 elements (two 16-byte words) / scale -> 16 E4M3 bytes.
template <int DT>
__device__ __forceinline__ uint4 quant16(const uint4 (&x)[2], float scale, float rcp) {
  uint32_t in[8] = {x[0].x, x[0].y, x[0].z, x[0].w, x[1].x, x[1].y, x[1].z, x[1].w};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 a = to_f32x2<DT>(in[2 * j]), b = to_f32x2<DT>(in[2 * j + 1]);
    o[j] = e4m3x4(quot(a.x, scale, rcp), quot(a.y, scale, rcp), quot(b.x, scale, rcp), quot(b.y, scale, rcp));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// One work item = CPT consecutive 16-element chunks of one (token, head), K
// and V.  The slot of the next item is loaded one iteration ahead, so the
// input loads never wait for it.
template <int DT, int CPT>
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
      *reinterpret_cast<uint4*>(kd + 16 * j) = quant16<DT>(kx[j], ks, kr);
      *reinterpret_cast<uint4*>(vd + 16 * j) = quant16<DT>(vx[j], vs, vr);
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
  if (a.dtype == FP8KV_DTYPE_F16)
    fn = two ? cache_write_kernel<FP8KV_DTYPE_F16, 2> : cache_write_kernel<FP8KV_DTYPE_F16, 1>;
  else
    fn = two ? cache_write_kernel<FP8KV_DTYPE_BF16, 2> : cache_write_kernel<FP8KV_DTYPE_BF16, 1>;
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
