// Device helpers shared by the split and combine kernels.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

namespace fp8kv {

// tok / page_size for 0 <= tok < 2^31, given page_div = ceil(2^64 /
// page_size) (0 for page size 1): the high word of one 64-bit multiply
// instead of an integer division, whose long dependent instruction sequence
// is costly on the copy-issuing threads (exact for every numerator below
// 2^32: Lemire, Kaser and Kurz, "Faster remainder by direct computation").
__device__ __forceinline__ int div_page(int tok, int page_size, unsigned long long page_div) {
  return page_size == 1 ? tok : (int)__umul64hi(page_div, (unsigned long long)(unsigned)tok);
}

// log2(e): logits are kept in base-2 units so that softmax uses exp2.
constexpr float kLog2e = 1.4426950408889634f;

// The base-2 logit factor softmax_scale * k_scale * log2(e) as an unevaluated
// sum hi + lo of two FP32 values: the product is formed in double once per
// CTA, so an exponent built from both parts keeps the precision of the exact
// factor (a single FP32 factor carries a relative error of up to ~2^-23,
// which shifts every weight by a few units in the last place).
struct LogitScale {
  float hi, lo;
};
__device__ __forceinline__ LogitScale logit_scale(float softmax_scale, float k_scale) {
  const double c = (double)softmax_scale * (double)k_scale * 1.4426950408889634074;
  const float hi = (float)c;
  return {hi, (float)(c - (double)hi)};
}

// Exact E4M3 -> FP32 for the four bytes of w (little-endian order).
//
// An E4M3 byte s.eeee.mmm placed so that eeee lands in the low four bits of
// the FP32 exponent field and mmm in the top of the FP32 mantissa encodes
// dec(b) * 2^-120 exactly (normal codes: 2^(e-127) * 1.mmm; subnormal codes
// e = 0: m * 2^-129 as an FP32 denormal); multiplying by 2^120 is exact.
// The two NaN codes give NaN (the placement alone would give 480).  Every
// byte the kernels read but must not use is excluded by selection, never by
// arithmetic, so a NaN code only matters in a token some row attends.
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float (&o)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t b = (w >> (8 * k)) & 0xFFu;
    const uint32_t bits = ((b & 0x80u) << 24) | ((b & 0x7Fu) << 20);
    // 0x7F / 0xFF are NaN in E4M3FN (the bit placement would give 480)
    o[k] = ((b & 0x7Fu) == 0x7Fu) ? __uint_as_float(0x7FC00000u) : __uint_as_float(bits) * 0x1p120f;
  }
}

// Four E5M2 bytes -> four floats: an E5M2 byte is the upper byte of the
// IEEE binary16 with the same value (infinities and NaNs included).
__device__ __forceinline__ void e5m2x4_to_f32(uint32_t w, float (&o)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const unsigned short h = (unsigned short)(((w >> (8 * k)) & 0xFFu) << 8);
    o[k] = __half2float(__ushort_as_half(h));
  }
}

// Byte lanes of the 16 cache bytes in w that hold a non-finite code, as the
// top bit of each byte of the four words OR-ed together (0: all finite).
// E4M3: 0x7F / 0xFF (NaN); E5M2: exponent field all ones (infinity or NaN).
// For b' = b & 0x7F (E4M3) or b & 0x7C (E5M2), b' + 1 (+ 4) carries into bit
// 7 exactly when b' is the all-ones pattern, and never into the next byte.
__device__ __forceinline__ uint32_t nonfinite_codes(const uint4& w, bool e5m2) {
  const uint32_t m = e5m2 ? 0x7C7C7C7Cu : 0x7F7F7F7Fu;
  const uint32_t a = e5m2 ? 0x04040404u : 0x01010101u;
  return (((w.x & m) + a) | ((w.y & m) + a) | ((w.z & m) + a) | ((w.w & m) + a)) & 0x80808080u;
}

// Nonzero iff one of the eight bf16 values in w is an infinity or a NaN
// (exponent bits all ones): per 16-bit half, (h & 0x7F80) + 0x80 reaches bit
// 15 only from 0x7F80, and no carry crosses the halves.
__device__ __forceinline__ uint32_t nonfinite_bf16(const uint4& w) {
  const uint32_t m = 0x7F807F80u, a = 0x00800080u;
  return (((w.x & m) + a) | ((w.y & m) + a) | ((w.z & m) + a) | ((w.w & m) + a)) & 0x80008000u;
}

// The four bytes of x with every non-finite code replaced by 0.
__device__ __forceinline__ uint32_t zap_nonfinite(uint32_t x, bool e5m2) {
  const uint32_t m = e5m2 ? 0x7C7C7C7Cu : 0x7F7F7F7Fu;
  const uint32_t a = e5m2 ? 0x04040404u : 0x01010101u;
  const uint32_t top = ((x & m) + a) & 0x80808080u;  // bit 7 of each non-finite byte
  return x & ~((top >> 7) * 0xFFu);
}

// Sparse visibility: query row r sees token t of an entry iff bit 4r + t of
// its mask word (rows 0..7) or bit 4(r - 8) + t of its second word (rows
// 8..15, absent with 8 or fewer rows) is set.
__device__ __forceinline__ uint32_t sparse_bit(uint32_t lo, uint32_t hi, int r, int t) {
  return ((r < 8 ? lo : hi) >> (4 * (r & 7) + t)) & 1u;
}
// The second mask word of entry e of request b (0 without one).
__device__ __forceinline__ uint32_t mask_hi_of(const uint32_t* mask_hi, int64_t stride, int b, int e) {
  return mask_hi ? mask_hi[(int64_t)b * stride + e] : 0u;
}

__device__ __forceinline__ void set_status(unsigned int* status, unsigned int bit) {
  atomicOr(status, bit);
}

// hi + lo += x without rounding loss in the hi/lo pair (Knuth's TwoSum: the
// rounding error of hi + x is recovered exactly and folded into lo).  When
// the sum is not finite the error term is meaningless (inf - inf) and is
// dropped, so an infinity stays an infinity and a NaN stays a NaN in hi.
__device__ __forceinline__ void two_sum_acc(float& hi, float& lo, float x) {
  const float s = __fadd_rn(hi, x);
  const float bp = __fsub_rn(s, hi);
  const float ap = __fsub_rn(s, bp);
  const float err = __fadd_rn(__fsub_rn(hi, ap), __fsub_rn(x, bp));
  hi = s;
  lo = __fadd_rn(lo, fabsf(s) < INFINITY ? err : 0.f);
}

// 2^x for an integer-valued x <= 0 (running maxima are kept integral), exact.
__device__ __forceinline__ float exp2_int(float x) {
  return x < -200.f ? 0.f : ldexpf(1.0f, (int)x);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace fp8kv
