// FP32 -> FP8 encoding of new K/V rows (round to nearest even, saturating),
// shared by the cache write and the split kernels' fused write of the new
// tokens.  The quotient x / scale only matters through its FP8 code; see
// quot().
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fp8kv_attn.h"

namespace fp8kv {

// Four floats (memory order) -> four E4M3 (FMT = FP8KV_KV_E4M3) or E5M2
// bytes, little-endian in a word.  The instruction puts its first source in
// the upper byte of the pair.
template <int FMT>
__device__ __forceinline__ uint32_t fp8x4(float x0, float x1, float x2, float x3) {
  uint32_t w;
  if (FMT == FP8KV_KV_E5M2)
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e5m2x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e5m2x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(w)
        : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
  else
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

// x / s as far as its FP8 code is concerned.  q = x * r with r = fl(1/s)
// is within 2 fp32 ulps of the correctly rounded quotient fl(x/s) (one
// rounding of r, one of the product).  The E4M3 code of a normal value is
// decided by the 20 fp32 mantissa bits below its 3 kept bits against the
// halfway pattern 0x80000 (E5M2: the 21 bits below its 2 kept bits against
// 0x100000), so when those bits of q are more than 4 ulps from it, q and
// fl(x/s) lie strictly on the same side of the same rounding boundary and
// convert to the same code.  Within 4 ulps of a boundary, below the normal
// range (E4M3 2^-6, E5M2 2^-14), or for non-finite q the exact quotient is
// computed.
template <int FMT>
__device__ __forceinline__ float quot(float x, float s, float r) {
  const float q = x * r;
  const float aq = fabsf(q);
  bool exact;
  if (FMT == FP8KV_KV_E5M2) {
    const uint32_t low = __float_as_uint(q) & 0x1FFFFFu;
    exact = !(aq >= 6.103515625e-05f && aq <= 3.0e38f) || (low - 0xFFFFCu) <= 8u;
  } else {
    const uint32_t low = __float_as_uint(q) & 0xFFFFFu;
    exact = !(aq >= 0.015625f && aq <= 3.0e38f) || (low - 0x7FFFCu) <= 8u;
  }
  return exact ? __fdiv_rn(x, s) : q;
}

// 16 elements (two 16-byte words) / scale -> 16 FP8 bytes.
template <int DT, int FMT>
__device__ __forceinline__ uint4 quant16(const uint4 (&x)[2], float scale, float rcp) {
  uint32_t in[8] = {x[0].x, x[0].y, x[0].z, x[0].w, x[1].x, x[1].y, x[1].z, x[1].w};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 a = to_f32x2<DT>(in[2 * j]), b = to_f32x2<DT>(in[2 * j + 1]);
    o[j] = fp8x4<FMT>(quot<FMT>(a.x, scale, rcp), quot<FMT>(a.y, scale, rcp), quot<FMT>(b.x, scale, rcp),
                      quot<FMT>(b.y, scale, rcp));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace fp8kv
