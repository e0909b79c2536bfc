// Combine kernel: merge the split-KV partitions of every query vector in FP32.
//
//   M = max_s m_s over partitions with l_s > 0
//   w_s = 2^(m_s - M),  L = sum_s w_s l_s,  out = v_scale * sum_s w_s acc_s / L
//
// written as fp16 with round-to-nearest-even.  A query vector whose total L is
// 0 (dead row, or nothing visible) gets +0.0.  Partitions with l_s = 0 are
// dropped by selection, so their numerators are never used; a NaN l_s (a NaN
// byte in a token some row sees) is kept, so the NaN reaches the output as
// the exact softmax would have it.  The partition
// maxima are integers (base-2 units), so every w_s is an exact power of two
// ("DFlash2 E4M3 attention with FP32 state", intro paragraph 4: FP32
// combination, FP16 final activation; "Qwen4Exp: fp8_e4m3 main KV cache on
// the QSA path", review: v_scale acts as the output scale).
//
// The weighted numerators are summed with TwoSum into a hi + lo pair (the
// weights are powers of two, so each product is exact): an output that
// cancels across partitions keeps the precision of its partials.
//
// One CTA per (query vector, 64-wide slice of D); its 256 threads are 16
// partition lanes x 16 float4 columns.  The kernel is latency-bound (a few
// MB in total), so the (m, l) pairs of all partitions and the numerators a
// lane needs (up to NB per lane) are loaded in one trip to memory, before
// the weights are known.  The lanes are reduced in shared memory in a fixed
// order.
#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace fp8kv {
namespace {

constexpr int CT = 256;
constexpr int SL = 16;      // partition lanes
constexpr int DW = 64;      // d slice per CTA
constexpr int MAXS = 1024;  // partitions whose weights are staged per pass
constexpr int KR = MAXS / CT;  // (m, l) pairs a thread holds
constexpr int NB = 12;      // numerator loads in flight per lane (S <= 192 in one trip)

// LSE = false: fp16 output.  LSE = true: FP32 output and the vector's
// base-2 log-sum-exp M + log2(L) (-inf when nothing is visible), the pair a
// context-parallel rank hands to the cross-rank merge ("Qualify calibrated
// E4M3 and disk PLE with QSA DCP2", commit exposing base-2 LSE and FP32
// partial output).
template <bool LSE>
__global__ void __launch_bounds__(CT) combine_kernel(Params p) {
  __shared__ float red_m[CT / 32];
  __shared__ float s_w[MAXS];       // weight 2^(m_s - M) of live partitions (0 = dead)
  __shared__ float s_l[MAXS];
  __shared__ float4 red_o[SL][DW / 4];
  __shared__ float4 red_lo[SL][DW / 4];
  __shared__ float red_l[SL];
  const int D = p.D;
  const int n_slices = D / DW;
  const int idx = blockIdx.x / n_slices;  // (b*q_max + r)*Hq + h
  const int slice = blockIdx.x % n_slices;
  const int h = idx % p.Hq;
  const int r = (idx / p.Hq) % p.q_max;
  const int b = idx / (p.Hq * p.q_max);
  const int g = h / p.G;
  const int i = r * p.G + (h % p.G);
  const int64_t base = (((int64_t)b * p.Hkv + g) * p.S) * p.rows + i;
  const float2* ml = p.ml + base;           // partition s at ml[s * rows]
  const int64_t sstride = p.rows;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = p.S;

  const int sl = tid / (DW / 4), c4 = tid % (DW / 4);
  const float* acc = p.partial + base * D + slice * DW + c4 * 4;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f), ol = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  float M = -INFINITY;
  for (int s0 = 0; s0 < S; s0 += MAXS) {
    const int ns = min(MAXS, S - s0);
    // one trip to memory: the (m, l) pairs of this pass and, speculatively,
    // the numerators this lane will need (a dead partition's numerator may
    // hold anything: it is dropped by selection below, never multiplied)
    float mv[KR], lv[KR];
#pragma unroll
    for (int k = 0; k < KR; ++k) {
      const int kk = tid + k * CT;
      mv[k] = -INFINITY;
      lv[k] = 0.f;
      if (kk < ns) {
        const float2 v = ml[(s0 + kk) * sstride];
        mv[k] = v.x;
        lv[k] = v.y;
      }
    }
    float4 a[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const int k = sl + j * SL;
      a[j] = (k < ns) ? *reinterpret_cast<const float4*>(acc + (int64_t)(s0 + k) * sstride * D)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (s0 == 0) {
      // global max over live partitions (later passes re-read their pairs)
      float M0 = -INFINITY;
#pragma unroll
      for (int k = 0; k < KR; ++k)
        if (lv[k] != 0.f) M0 = fmaxf(M0, mv[k]);
      for (int s = tid + MAXS; s < S; s += CT) {
        const float2 v = ml[s * sstride];
        if (v.y != 0.f) M0 = fmaxf(M0, v.x);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) M0 = fmaxf(M0, __shfl_xor_sync(0xffffffffu, M0, off));
      if (lane == 0) red_m[warp] = M0;
    } else {
      __syncthreads();  // the previous pass is done with s_w / s_l
    }
    __syncthreads();
    M = red_m[0];
#pragma unroll
    for (int k = 1; k < CT / 32; ++k) M = fmaxf(M, red_m[k]);
    if (M == -INFINITY) break;  // nothing visible for this vector
#pragma unroll
    for (int k = 0; k < KR; ++k) {
      const int kk = tid + k * CT;
      if (kk < ns) {
        const bool live = lv[k] != 0.f;
        s_w[kk] = live ? exp2_int(mv[k] - M) : 0.f;  // integer maxima: exact
        s_l[kk] = live ? lv[k] : 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const int k = sl + j * SL;
      const float w = (k < ns) ? s_w[k] : 0.f;
      if (w != 0.f) {
        two_sum_acc(o.x, ol.x, w * a[j].x);
        two_sum_acc(o.y, ol.y, w * a[j].y);
        two_sum_acc(o.z, ol.z, w * a[j].z);
        two_sum_acc(o.w, ol.w, w * a[j].w);
        L = fmaf(w, s_l[k], L);
      }
    }
    // partitions beyond SL * NB per pass: the remaining loads of this lane
    for (int k0 = sl + SL * NB; k0 < ns; k0 += SL * NB) {
      float4 b4[NB];
      float w[NB];
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        const int k = k0 + j * SL;
        w[j] = (k < ns) ? s_w[k] : 0.f;
        b4[j] = (w[j] != 0.f) ? *reinterpret_cast<const float4*>(acc + (int64_t)(s0 + k) * sstride * D)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        const int k = k0 + j * SL;
        if (w[j] != 0.f) {
          two_sum_acc(o.x, ol.x, w[j] * b4[j].x);
          two_sum_acc(o.y, ol.y, w[j] * b4[j].y);
          two_sum_acc(o.z, ol.z, w[j] * b4[j].z);
          two_sum_acc(o.w, ol.w, w[j] * b4[j].w);
          L = fmaf(w[j], s_l[k], L);
        }
      }
    }
  }
  red_o[sl][c4] = o;
  red_lo[sl][c4] = ol;
  if (c4 == 0) red_l[sl] = L;
  __syncthreads();
  if (tid < DW / 4) {
    float4 t = red_o[0][tid], tl = red_lo[0][tid];
    float Lt = red_l[0];
#pragma unroll
    for (int k = 1; k < SL; ++k) {
      const float4 u = red_o[k][tid], ul = red_lo[k][tid];
      two_sum_acc(t.x, tl.x, u.x);
      two_sum_acc(t.y, tl.y, u.y);
      two_sum_acc(t.z, tl.z, u.z);
      two_sum_acc(t.w, tl.w, u.w);
      tl.x += ul.x;
      tl.y += ul.y;
      tl.z += ul.z;
      tl.w += ul.w;
      Lt += red_l[k];
    }
    t.x += tl.x;
    t.y += tl.y;
    t.z += tl.z;
    t.w += tl.w;
    const float vs = p.v_scale_dev ? *p.v_scale_dev : p.v_scale;
    const bool any = Lt != 0.f;  // NaN (a NaN byte in a seen token) propagates
    const float f = any ? vs / Lt : 0.f;
    const float y0 = any ? t.x * f : 0.f;
    const float y1 = any ? t.y * f : 0.f;
    const float y2 = any ? t.z * f : 0.f;
    const float y3 = any ? t.w * f : 0.f;
    if (LSE) {
      *reinterpret_cast<float4*>(p.out_f32 + (int64_t)idx * D + slice * DW + tid * 4) = make_float4(y0, y1, y2, y3);
      if (slice == 0 && tid == 0) p.lse[idx] = any ? M + log2f(Lt) : -INFINITY;
      return;
    }
    const __half2 h01 = __floats2half2_rn(y0, y1);
    const __half2 h23 = __floats2half2_rn(y2, y3);
    uint2 pk;
    pk.x = *reinterpret_cast<const uint32_t*>(&h01);
    pk.y = *reinterpret_cast<const uint32_t*>(&h23);
    *reinterpret_cast<uint2*>(p.out + (int64_t)idx * D + slice * DW + tid * 4) = pk;
  }
}

}  // namespace

cudaError_t launch_combine(const fp8kv_attn_plan_t* plan, const Params& p, cudaStream_t st) {
  const int64_t n = (int64_t)p.B * p.q_max * p.Hq * (p.D / DW);
  if (n == 0) return cudaSuccess;
  if (p.D % DW) return cudaErrorInvalidValue;
  (void)plan;
  if (p.out_f32)
    combine_kernel<true><<<(unsigned)n, CT, 0, st>>>(p);
  else
    combine_kernel<false><<<(unsigned)n, CT, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace fp8kv
