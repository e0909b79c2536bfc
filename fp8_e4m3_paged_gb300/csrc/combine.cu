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
// Two shapes, by partition count S:
// * S <= 64 (batched decode, short contexts): one warp per (query vector, 8
//   columns of D), lane = 16 partition lanes x 2 float4 column groups (lane &
//   15 = partition lane, lane >> 4 = group).  A lane takes partitions sl, sl +
//   16, ...; the (max, sum) pairs and the numerators it needs are loaded in
//   one trip, before the weights are known.  The maximum and the final sum
//   over the 16 partition lanes are xor-butterflies of shuffles (symmetric
//   merges, so every lane ends with the same bits), with no shared memory and
//   no barrier; the loads per lane are a template parameter so that the
//   registers, and with them the resident warps, follow S.
// * S > 64 (one long context split over the whole GPU): one CTA per (query
//   vector, 32-column slice), 16 partition lanes x 8 float4 columns; the
//   (max, sum) pairs are loaded once per CTA and the weights staged in shared
//   memory, each numerator load instruction covers two partitions' 128-byte
//   rows, and the 16 lanes are merged by a tree in shared memory.
// Both reduce in a fixed order: replays are bitwise identical.
#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace fp8kv {
namespace {

constexpr int kWarps = 8;  // warps per CTA
constexpr int SL = 16;     // partition lanes

// (hi, lo) += (hi2, lo2): TwoSum of the high parts, then the low parts and
// the rounding error added.  Symmetric in its two arguments.
__device__ __forceinline__ void merge_pair(float& hi, float& lo, float hi2, float lo2) {
  const float lsum = __fadd_rn(lo, lo2);
  lo = 0.f;
  two_sum_acc(hi, lo, hi2);
  lo = __fadd_rn(lo, lsum);
}

constexpr int MAXS = 1024;  // partitions whose weights a CTA stages per pass
constexpr int NBS = 12;     // numerator loads in flight per lane (S <= 192 in one trip)

// Many partitions (S > 64): one CTA per (query vector, DW-wide slice of D);
// its threads are 16 partition lanes x DW/4 float4 columns.  The (m, l)
// pairs of all partitions and the numerators a lane needs (up to NBS per
// lane) are loaded in one trip, the weights are staged in shared memory
// once per CTA, and the 16 lanes are merged by a tree in shared memory.
template <bool LSE, int DW>
__global__ void __launch_bounds__(SL * DW / 4) combine_slices(Params p) {
  constexpr int CT = SL * DW / 4;
  constexpr int KR = MAXS / CT;  // (m, l) pairs a thread holds
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
    float4 a[NBS];
#pragma unroll
    for (int j = 0; j < NBS; ++j) {
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
    for (int j = 0; j < NBS; ++j) {
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
    // partitions beyond SL * NBS per pass: the remaining loads of this lane
    for (int k0 = sl + SL * NBS; k0 < ns; k0 += SL * NBS) {
      float4 b4[NBS];
      float w[NBS];
#pragma unroll
      for (int j = 0; j < NBS; ++j) {
        const int k = k0 + j * SL;
        w[j] = (k < ns) ? s_w[k] : 0.f;
        b4[j] = (w[j] != 0.f) ? *reinterpret_cast<const float4*>(acc + (int64_t)(s0 + k) * sstride * D)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < NBS; ++j) {
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
  // tree over the 16 partition lanes (lane sl takes sl + w, w = 8, 4, 2, 1)
#pragma unroll
  for (int w = SL / 2; w > 0; w >>= 1) {
    if (sl < w) {
      float4 t = red_o[sl][c4], tl = red_lo[sl][c4];
      const float4 u = red_o[sl + w][c4], ul = red_lo[sl + w][c4];
      merge_pair(t.x, tl.x, u.x, ul.x);
      merge_pair(t.y, tl.y, u.y, ul.y);
      merge_pair(t.z, tl.z, u.z, ul.z);
      merge_pair(t.w, tl.w, u.w, ul.w);
      red_o[sl][c4] = t;
      red_lo[sl][c4] = tl;
      if (c4 == 0) red_l[sl] = __fadd_rn(red_l[sl], red_l[sl + w]);
    }
    __syncthreads();
  }
  if (tid < DW / 4) {
    float4 t = red_o[0][tid];
    const float4 tl = red_lo[0][tid];
    const float Lt = red_l[0];
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


// LSE = false: fp16 output.  LSE = true: FP32 output and the vector's
// base-2 log-sum-exp M + log2(L) (-inf when nothing is visible), the pair a
// context-parallel rank hands to the cross-rank merge ("Qualify calibrated
// E4M3 and disk PLE with QSA DCP2", commit exposing base-2 LSE and FP32
// partial output).
// Up to 64 partitions: one warp per (query vector, 8 columns of D), see the
// file header.
template <bool LSE, int NB>
__global__ void __launch_bounds__(32 * kWarps) combine_rows(Params p) {
  const int lane = threadIdx.x & 31;
  const int D = p.D;
  const int pairs = D / 8;  // 8-column units of a vector
  const int64_t gw = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int64_t n_vec = (int64_t)p.B * p.q_max * p.Hq;
  if (gw >= n_vec * pairs) return;  // whole warps only
  const int64_t idx = gw / pairs;   // (b*q_max + r)*Hq + h
  const int col = (int)(gw % pairs) * 8 + (lane >> 4) * 4;
  const int sl = lane & (SL - 1);
  const int h = (int)(idx % p.Hq);
  const int r = (int)((idx / p.Hq) % p.q_max);
  const int b = (int)(idx / ((int64_t)p.Hq * p.q_max));
  const int g = h / p.G;
  const int i = r * p.G + (h % p.G);
  const int64_t base = (((int64_t)b * p.Hkv + g) * p.S) * p.rows + i;
  const float2* ml = p.ml + base;  // partition s at ml[s * rows]
  const int64_t sstride = p.rows;
  const float* acc = p.partial + base * D + col;
  const int S = p.S;

  // one trip: (max, sum) pairs and, speculatively, the numerators (a dead
  // partition's numerator may hold anything: it is dropped by selection)
  float mv[NB], lv[NB];
  float4 a[NB];
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    const int s = sl + SL * j;
    mv[j] = -INFINITY;
    lv[j] = 0.f;
    a[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (s < S) {
      const float2 v = ml[(int64_t)s * sstride];
      mv[j] = v.x;
      lv[j] = v.y;
      a[j] = *reinterpret_cast<const float4*>(acc + (int64_t)s * sstride * D);
    }
  }
  float M = -INFINITY;
#pragma unroll
  for (int j = 0; j < NB; ++j)
    if (lv[j] != 0.f) M = fmaxf(M, mv[j]);
  for (int s = sl + SL * NB; s < S; s += SL) {  // more partitions than one trip holds
    const float2 v = ml[(int64_t)s * sstride];
    if (v.y != 0.f) M = fmaxf(M, v.x);
  }
#pragma unroll
  for (int off = SL / 2; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  float4 o = make_float4(0.f, 0.f, 0.f, 0.f), ol = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  if (M != -INFINITY) {
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      if (lv[j] != 0.f) {
        const float w = exp2_int(mv[j] - M);  // integer maxima: exact
        two_sum_acc(o.x, ol.x, w * a[j].x);
        two_sum_acc(o.y, ol.y, w * a[j].y);
        two_sum_acc(o.z, ol.z, w * a[j].z);
        two_sum_acc(o.w, ol.w, w * a[j].w);
        L = fmaf(w, lv[j], L);
      }
    }
    for (int s = sl + SL * NB; s < S; s += SL) {
      const float2 v = ml[(int64_t)s * sstride];
      if (v.y != 0.f) {
        const float4 x = *reinterpret_cast<const float4*>(acc + (int64_t)s * sstride * D);
        const float w = exp2_int(v.x - M);
        two_sum_acc(o.x, ol.x, w * x.x);
        two_sum_acc(o.y, ol.y, w * x.y);
        two_sum_acc(o.z, ol.z, w * x.z);
        two_sum_acc(o.w, ol.w, w * x.w);
        L = fmaf(w, v.y, L);
      }
    }
  }
  // the 16 partition lanes, butterfly
#pragma unroll
  for (int off = SL / 2; off > 0; off >>= 1) {
    merge_pair(o.x, ol.x, __shfl_xor_sync(0xffffffffu, o.x, off), __shfl_xor_sync(0xffffffffu, ol.x, off));
    merge_pair(o.y, ol.y, __shfl_xor_sync(0xffffffffu, o.y, off), __shfl_xor_sync(0xffffffffu, ol.y, off));
    merge_pair(o.z, ol.z, __shfl_xor_sync(0xffffffffu, o.z, off), __shfl_xor_sync(0xffffffffu, ol.z, off));
    merge_pair(o.w, ol.w, __shfl_xor_sync(0xffffffffu, o.w, off), __shfl_xor_sync(0xffffffffu, ol.w, off));
    L = __fadd_rn(L, __shfl_xor_sync(0xffffffffu, L, off));
  }
  if (sl != 0) return;
  o.x += ol.x;
  o.y += ol.y;
  o.z += ol.z;
  o.w += ol.w;
  const float vs = p.v_scale_dev ? *p.v_scale_dev : p.v_scale;
  const bool any = L != 0.f;  // NaN (a NaN byte in a seen token) propagates
  const float f = any ? vs / L : 0.f;
  const float y0 = any ? o.x * f : 0.f;
  const float y1 = any ? o.y * f : 0.f;
  const float y2 = any ? o.z * f : 0.f;
  const float y3 = any ? o.w * f : 0.f;
  if (LSE) {
    *reinterpret_cast<float4*>(p.out_f32 + idx * D + col) = make_float4(y0, y1, y2, y3);
    if (col == 0) p.lse[idx] = any ? M + log2f(L) : -INFINITY;
    return;
  }
  const __half2 h01 = __floats2half2_rn(y0, y1);
  const __half2 h23 = __floats2half2_rn(y2, y3);
  uint2 pk;
  pk.x = *reinterpret_cast<const uint32_t*>(&h01);
  pk.y = *reinterpret_cast<const uint32_t*>(&h23);
  *reinterpret_cast<uint2*>(p.out + idx * D + col) = pk;
}

constexpr int kSliceDW = 32;  // D slice of a many-partition CTA

template <bool LSE>
cudaError_t launch_lse(const Params& p, cudaStream_t st) {
  if (p.S > 4 * SL) {
    const int64_t n = (int64_t)p.B * p.q_max * p.Hq * (p.D / kSliceDW);
    combine_slices<LSE, kSliceDW><<<(unsigned)n, SL * kSliceDW / 4, 0, st>>>(p);
    return cudaGetLastError();
  }
  const int64_t warps = (int64_t)p.B * p.q_max * p.Hq * (p.D / 8);
  const unsigned grid = (unsigned)((warps + kWarps - 1) / kWarps);
  // loads per lane in the single trip: 2 cover 32 partitions, 4 cover 64
  if (p.S <= 2 * SL)
    combine_rows<LSE, 2><<<grid, 32 * kWarps, 0, st>>>(p);
  else
    combine_rows<LSE, 4><<<grid, 32 * kWarps, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(const fp8kv_attn_plan_t* plan, const Params& p, cudaStream_t st) {
  if ((int64_t)p.B * p.q_max * p.Hq == 0) return cudaSuccess;
  if (p.D % kSliceDW) return cudaErrorInvalidValue;
  (void)plan;
  return p.out_f32 ? launch_lse<true>(p, st) : launch_lse<false>(p, st);
}

}  // namespace fp8kv
