// Generic split kernel: FP32 CUDA-core path for every supported shape.
//
// One CTA handles one (partition s, KV head g, row chunk, request b).  It
// keeps up to 64 query vectors (query rows x heads of the group) in shared
// memory, streams its token range of the cache pages (E4M3 or E5M2 bytes, or
// bf16 values for A/B runs) in tiles of 32 tokens (dense) or 8 four-token
// microblocks (sparse) with 16-byte loads, decodes them exactly to FP32, and runs the online softmax with FP32 state:
//   s = (q . k) * softmax_scale * k_scale * log2(e)
//   m' = max(m, ceil(max_tile s));  acc = acc * 2^(m - m') + sum_t 2^(s_t - m') v_t
//   l  = l * 2^(m - m') + sum_t 2^(s_t - m')
// and finally stores the unnormalised FP32 numerators acc with (m, l)
// ("DFlash2 E4M3 attention with FP32 state", intro paragraph 4: FP32
// partition numerators, separate FP32 max/sum).  Masked tokens get s = -inf by
// selection and p = -0.0 (a visible token whose weight underflows gets +0.0).
// A tile whose V bytes hold no non-finite code takes the plain FMA loop (a
// masked token's -0.0 * v then adds nothing); a tile with a NaN (or E5M2
// infinity) code in V skips the tokens each row does not see, so the code
// reaches exactly the rows that see its token, as in the exact softmax.
#include <cstdint>
#include <type_traits>

#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"
#include "new_tokens.cuh"

namespace fp8kv {
namespace {

constexpr int NT = kGenericThreads;
constexpr int TT = kGenericTileTokens;

struct GenericSmem {
  // layout offsets (floats) for a given D and row chunk RC
  int q, k, v, p, alpha, nrow, mask;
  int total_bytes;
};

__host__ __device__ inline GenericSmem generic_layout(int D, int RC) {
  GenericSmem L;
  int off = 0;
  L.q = off;     off += D * RC;          // Qs[d][row]
  L.k = off;     off += TT * (D + 1);    // Ks[t][d] (padded rows)
  L.v = off;     off += TT * D;          // Vs[t][d]
  L.p = off;     off += TT * (RC + 1);   // Ps[t][row] (padded rows)
  L.alpha = off; off += RC;              // per-row rescale factor of this tile
  L.nrow = off;  off += RC;              // per-row live length (int) / row index
  L.mask = off;  off += 16;              // sparse: this tile's 8 masks, then their second words (uint)
  L.total_bytes = off * 4;
  return L;
}

// RPW: rows per warp in the score phase (row chunk = 8 * RPW, NT/32 = 8 warps).
template <int D, int MODE, int RPW>
__global__ void __launch_bounds__(NT) split_generic(Params p) {
  constexpr int RCMAX = 8 * RPW;
  constexpr int DG = D / 4;               // float4 column groups in the PV phase
  constexpr int RG = NT / DG;             // row groups in the PV phase
  constexpr int RPT = (RCMAX + RG - 1) / RG;  // rows per thread in the PV phase
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  const GenericSmem L = generic_layout(D, RCMAX);
  float* Qs = sm + L.q;
  float* Ks = sm + L.k;
  float* Vs = sm + L.v;
  float* Ps = sm + L.p;
  float* Al = sm + L.alpha;
  int* Nrow = reinterpret_cast<int*>(sm + L.nrow);
  uint32_t* Msk = reinterpret_cast<uint32_t*>(sm + L.mask);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.x;
  const int g = blockIdx.y / p.n_row_chunks;
  const int chunk = blockIdx.y % p.n_row_chunks;
  const int b = blockIdx.z;
  const int row0 = chunk * p.row_chunk;
  const int RC = min(p.row_chunk, p.rows - row0);

  // ---------------------------------------------------------- token range
  // Dense: union length U = max_r n_r; sparse: entry count E.  Partition s
  // covers a contiguous, tile-aligned slice of it.
  int U = 0;
  if (MODE == FP8KV_MODE_DENSE) {
    for (int r = 0; r < p.q_max; ++r) {
      int n = p.row_len[(int64_t)b * p.q_max + r];
      if (n < 0 || n > p.max_kv_len) {
        if (tid == 0) set_status(p.status, FP8KV_STATUS_BAD_LEN);
        n = min(max(n, 0), p.max_kv_len);
      }
      U = max(U, n);
    }
  } else {
    U = p.n_entries[b];
    if (U < 0 || U > p.max_blocks) {
      if (tid == 0) set_status(p.status, FP8KV_STATUS_BAD_ENTRIES);
      U = min(max(U, 0), p.max_blocks);
    }
  }
  const int unit = (MODE == FP8KV_MODE_DENSE) ? TT : TT / 4;  // tokens or entries per tile
  int per = max((U + p.S - 1) / p.S, p.min_part);
  per = (per + unit - 1) / unit * unit;
  const int u0 = s * per;
  const int u1 = min(U, u0 + per);

  const int64_t prow = (((int64_t)b * p.Hkv + g) * p.S + s) * p.rows + row0;
  float2* ml_out = p.ml + prow;
  float* acc_out = p.partial + prow * D;

  if (u0 >= u1) {
    for (int i = tid; i < RC; i += NT) ml_out[i] = make_float2(-INFINITY, 0.f);
    return;
  }
  // a verify step's new tokens in this partition, written before the tile
  // loop reads them (which then bypasses L1: fresh = true)
  const bool fresh = MODE == FP8KV_MODE_DENSE && p.n_new > 0;
  if (fresh) {
    if (u1 > U - p.n_new) {
      if (p.kv_format == FP8KV_KV_E5M2)
        write_new_tokens_and_fence<FP8KV_KV_E5M2>(p, b, g, U, u0, u1, tid, NT);
      else
        write_new_tokens_and_fence<FP8KV_KV_E4M3>(p, b, g, U, u0, u1, tid, NT);
    }
    __syncthreads();
  }

  // ---------------------------------------------------------- Q, row lengths
  const float ks = p.k_scale_dev ? *p.k_scale_dev : p.k_scale;
  const LogitScale cs = logit_scale(p.softmax_scale, ks);
  const float c = cs.hi;
  for (int idx = tid; idx < RCMAX * D; idx += NT) {
    const int i = idx / D, d = idx % D;
    float v = 0.f;
    if (i < RC) {
      const int rowi = row0 + i;
      const int r = rowi / p.G, h = g * p.G + rowi % p.G;
      v = __half2float(__ushort_as_half(p.q[(((int64_t)b * p.q_max + r) * p.Hq + h) * D + d]));
    }
    Qs[d * RCMAX + i] = v;
  }
  for (int i = tid; i < RCMAX; i += NT) {
    int n = 0;
    if (i < RC) {
      const int r = (row0 + i) / p.G;
      if (MODE == FP8KV_MODE_DENSE) {
        n = min(max(p.row_len[(int64_t)b * p.q_max + r], 0), p.max_kv_len);
      } else {
        n = r;  // sparse: the query row index selects the mask nibble
      }
    }
    Nrow[i] = (i < RC) ? n : -1;
  }

  // per-warp softmax state for rows warp*RPW + k (replicated in all lanes)
  float m_run[RPW], l_run[RPW];
#pragma unroll
  for (int k = 0; k < RPW; ++k) { m_run[k] = -INFINITY; l_run[k] = 0.f; }

  // PV accumulators: thread owns columns dg*4..+3 of rows rg + k*RG.  With
  // few rows per thread (the decode shapes this path serves) each tile is
  // summed in FP32 on its own and added to a compensated pair acc + acc_lo
  // (TwoSum), so the rounding of the running sum over a long partition is
  // recovered; larger row chunks accumulate in plain FP32.
  constexpr bool kComp = RPT <= 4;
  const int dg = tid % DG, rg = tid / DG;
  float4 acc[RPT], acc_lo[kComp ? RPT : 1];
#pragma unroll
  for (int k = 0; k < RPT; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < (kComp ? RPT : 1); ++k) acc_lo[k] = make_float4(0.f, 0.f, 0.f, 0.f);

  __syncthreads();

  for (int tb = u0; tb < u1; tb += unit) {
    bool vbad = false;  // this thread loaded a non-finite V code
    // ------------------------------------------------------ load + decode
    // 16-byte vectors: TT tokens x D/16 (FP8) or D/8 (bf16) vectors for K and for V.
    if (MODE == FP8KV_MODE_SPARSE_PAGE4 && tid < 8) {
      const int e = tb + tid;
      uint32_t mk = 0, mkh = 0;
      if (e < u1) {
        mk = p.entry_mask[(int64_t)b * p.entry_stride + e];
        mkh = mask_hi_of(p.entry_mask_hi, p.entry_stride, b, e);
        const int blk = p.entry_tbl[(int64_t)b * p.entry_stride + e];
        if ((mk | mkh) != 0u && (blk < 0 || blk >= p.num_kv_blocks)) {
          set_status(p.status, FP8KV_STATUS_BAD_BLOCK);
          mk = mkh = 0;
        }
      }
      Msk[tid] = mk;
      Msk[8 + tid] = mkh;
    }
    if (MODE == FP8KV_MODE_SPARSE_PAGE4) __syncthreads();
    // VPTL 16-byte vectors per token row: D/16 of FP8 bytes, D/8 of bf16
    auto load_tile = [&](auto vpt_c) {
    constexpr int VPTL = decltype(vpt_c)::value;
    for (int idx = tid; idx < TT * VPTL; idx += NT) {
      const int t = idx / VPTL, vv = idx % VPTL;
      bool ok = false;
      const uint8_t* kp = nullptr;
      const uint8_t* vp = nullptr;
      if (MODE == FP8KV_MODE_DENSE) {
        const int tok = tb + t;
        if (tok < u1) {
          const int page = div_page(tok, p.page_size, p.page_div);
          const int blk = p.block_table[(int64_t)b * p.bt_stride + page];
          const int slot = tok - page * p.page_size;
          if (blk >= 0 && blk < p.num_kv_blocks) {
            ok = true;
            kp = p.k_cache + blk * p.ksb + slot * p.kst + g * p.ksh;
            vp = p.v_cache + blk * p.vsb + slot * p.vst + g * p.vsh;
          } else if (vv == 0) {
            set_status(p.status, FP8KV_STATUS_BAD_BLOCK);
          }
        }
      } else {
        const int e = tb + t / 4, tk = t % 4;
        const uint32_t mk = Msk[t / 4] | Msk[8 + t / 4];
        // only tokens that at least one query row attends are read
        if (e < u1 && (mk & (0x11111111u << tk)) != 0u) {
          const int blk = p.entry_tbl[(int64_t)b * p.entry_stride + e];
          ok = true;
          kp = p.k_cache + blk * p.ksb + tk * p.kst + g * p.ksh;
          vp = p.v_cache + blk * p.vsb + tk * p.vst + g * p.vsh;
        }
      }
      uint4 kw = make_uint4(0, 0, 0, 0), vw = make_uint4(0, 0, 0, 0);
      if (ok) {
        if (fresh) {
          kw = __ldcg(reinterpret_cast<const uint4*>(kp) + vv);
          vw = __ldcg(reinterpret_cast<const uint4*>(vp) + vv);
        } else {
          kw = __ldg(reinterpret_cast<const uint4*>(kp) + vv);
          vw = __ldg(reinterpret_cast<const uint4*>(vp) + vv);
        }
      }
      if constexpr (VPTL == D / 8) {
        // bf16: the upper half of an FP32 word, exact
        vbad |= nonfinite_bf16(vw) != 0u;
        const uint32_t kwa[4] = {kw.x, kw.y, kw.z, kw.w};
        const uint32_t vwa[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          Ks[t * (D + 1) + vv * 8 + j * 2] = __uint_as_float(kwa[j] << 16);
          Ks[t * (D + 1) + vv * 8 + j * 2 + 1] = __uint_as_float(kwa[j] & 0xFFFF0000u);
          *reinterpret_cast<float2*>(&Vs[t * D + vv * 8 + j * 2]) =
              make_float2(__uint_as_float(vwa[j] << 16), __uint_as_float(vwa[j] & 0xFFFF0000u));
        }
      } else {
      float f[4];
      const uint32_t kwa[4] = {kw.x, kw.y, kw.z, kw.w};
      const uint32_t vwa[4] = {vw.x, vw.y, vw.z, vw.w};
      const bool e5 = p.kv_format == FP8KV_KV_E5M2;  // uniform
      vbad |= nonfinite_codes(vw, e5) != 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (e5)
          e5m2x4_to_f32(kwa[j], f);
        else
          e4m3x4_to_f32(kwa[j], f);
#pragma unroll
        for (int k = 0; k < 4; ++k) Ks[t * (D + 1) + vv * 16 + j * 4 + k] = f[k];
        if (e5)
          e5m2x4_to_f32(vwa[j], f);
        else
          e4m3x4_to_f32(vwa[j], f);
        *reinterpret_cast<float4*>(&Vs[t * D + vv * 16 + j * 4]) = make_float4(f[0], f[1], f[2], f[3]);
      }
      }
    }
    };
    if (p.kv_format == FP8KV_KV_BF16)
      load_tile(std::integral_constant<int, D / 8>{});
    else
      load_tile(std::integral_constant<int, D / 16>{});
    const bool vflag = __syncthreads_or(vbad) != 0;  // the tile holds a non-finite V code

    // ------------------------------------------------------ scores (lane = token)
    // Compensated QK: products q*k are exact in FP32 (11-bit x 4-bit
    // significands; 11 x 8 for bf16 K); they are summed in chunks of 8 and the chunk sums are
    // combined with an error-free TwoSum into hi + lo, so the logit keeps
    // more than FP32 precision.  The base-2 exponent is then formed as
    // fma(hi, c, -m) + lo*c, which rounds only the small difference to the
    // running max ("DFlash2 E4M3 attention with FP32 state", intro paragraph
    // 4: compensated QK accumulation).
    {
      float hi[RPW], lo[RPW];
#pragma unroll
      for (int k = 0; k < RPW; ++k) { hi[k] = 0.f; lo[k] = 0.f; }
      const float* kr = Ks + lane * (D + 1);
      const float* qr = Qs + warp * RPW;
#pragma unroll 1
      for (int d0 = 0; d0 < D; d0 += 8) {
        float ch[RPW];
#pragma unroll
        for (int k = 0; k < RPW; ++k) ch[k] = 0.f;
#pragma unroll
        for (int d = d0; d < d0 + 8; ++d) {
          const float kv = kr[d];
#pragma unroll
          for (int k = 0; k < RPW; ++k) ch[k] = fmaf(qr[d * RCMAX + k], kv, ch[k]);
        }
#pragma unroll
        for (int k = 0; k < RPW; ++k) two_sum_acc(hi[k], lo[k], ch[k]);
      }
      const int t = lane;
      const int tok = tb + ((MODE == FP8KV_MODE_DENSE) ? t : t / 4);
      const uint32_t mk = (MODE == FP8KV_MODE_DENSE) ? 0u : Msk[t / 4];
      const uint32_t mkh = (MODE == FP8KV_MODE_DENSE) ? 0u : Msk[8 + t / 4];
#pragma unroll
      for (int k = 0; k < RPW; ++k) {
        const int i = warp * RPW + k;
        const int n = Nrow[i];
        bool vis;
        if (MODE == FP8KV_MODE_DENSE)
          vis = (n >= 0) && (tok < u1) && (tok < n);
        else
          vis = (n >= 0) && (tok < u1) && sparse_bit(mk, mkh, n, t & 3);
        const float sv = vis ? fmaf(hi[k], c, lo[k] * c) : -INFINITY;
        float mt = sv;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
        // integer-valued running max: rescale factors 2^(m - m') and the
        // combine's partition weights are then exact powers of two
        const float m_new = fmaxf(m_run[k], ceilf(mt));
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float arg = fmaf(hi[k], cs.hi, -m_use) + fmaf(lo[k], cs.hi, hi[k] * cs.lo);
        const float pv = vis ? exp2f(arg) : -0.f;  // -0.0 marks "not seen"
        const float alpha = (m_run[k] == -INFINITY) ? 0.f : exp2_int(m_run[k] - m_use);
        float ps = pv;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        l_run[k] = l_run[k] * alpha + ps;
        m_run[k] = m_new;
        Ps[t * (RCMAX + 1) + i] = pv;
        if (lane == 0) Al[i] = alpha;
      }
    }
    __syncthreads();

    // ------------------------------------------------------ PV
    {
      float4 tt[RPT];  // this tile's sums (compensated path) or the running sums
#pragma unroll
      for (int k = 0; k < RPT; ++k) {
        const int i = rg + k * RG;
        const float a = (i < RCMAX) ? Al[i] : 1.f;
        acc[k].x *= a; acc[k].y *= a; acc[k].z *= a; acc[k].w *= a;
        if constexpr (kComp) {
          acc_lo[k].x *= a; acc_lo[k].y *= a; acc_lo[k].z *= a; acc_lo[k].w *= a;
          tt[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
          tt[k] = acc[k];
        }
      }
      if (!vflag) {
#pragma unroll 4
        for (int t = 0; t < TT; ++t) {
          const float4 v4 = *reinterpret_cast<const float4*>(&Vs[t * D + dg * 4]);
#pragma unroll
          for (int k = 0; k < RPT; ++k) {
            const int i = rg + k * RG;
            if (i < RCMAX) {
              const float pv = Ps[t * (RCMAX + 1) + i];
              tt[k].x = fmaf(pv, v4.x, tt[k].x);
              tt[k].y = fmaf(pv, v4.y, tt[k].y);
              tt[k].z = fmaf(pv, v4.z, tt[k].z);
              tt[k].w = fmaf(pv, v4.w, tt[k].w);
            }
          }
        }
      } else {
        // a NaN or infinite V value only reaches the rows that see its token
        for (int t = 0; t < TT; ++t) {
          const float4 v4 = *reinterpret_cast<const float4*>(&Vs[t * D + dg * 4]);
#pragma unroll
          for (int k = 0; k < RPT; ++k) {
            const int i = rg + k * RG;
            if (i < RCMAX) {
              const float pv = Ps[t * (RCMAX + 1) + i];
              if (__float_as_uint(pv) != 0x80000000u) {
                tt[k].x = fmaf(pv, v4.x, tt[k].x);
                tt[k].y = fmaf(pv, v4.y, tt[k].y);
                tt[k].z = fmaf(pv, v4.z, tt[k].z);
                tt[k].w = fmaf(pv, v4.w, tt[k].w);
              }
            }
          }
        }
      }
#pragma unroll
      for (int k = 0; k < RPT; ++k) {
        if constexpr (kComp) {
          two_sum_acc(acc[k].x, acc_lo[k].x, tt[k].x);
          two_sum_acc(acc[k].y, acc_lo[k].y, tt[k].y);
          two_sum_acc(acc[k].z, acc_lo[k].z, tt[k].z);
          two_sum_acc(acc[k].w, acc_lo[k].w, tt[k].w);
        } else {
          acc[k] = tt[k];
        }
      }
    }
    __syncthreads();
  }

  // ---------------------------------------------------------- epilogue
#pragma unroll
  for (int k = 0; k < RPT; ++k) {
    const int i = rg + k * RG;
    float4 o = acc[k];
    if constexpr (kComp) {
      o.x += acc_lo[k].x;
      o.y += acc_lo[k].y;
      o.z += acc_lo[k].z;
      o.w += acc_lo[k].w;
    }
    if (i < RC) reinterpret_cast<float4*>(acc_out + (int64_t)i * D)[dg] = o;
  }
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
      const int i = warp * RPW + k;
      if (i < RC) ml_out[i] = make_float2(m_run[k], l_run[k]);
    }
  }
}

template <int D, int MODE, int RPW>
cudaError_t launch_one(const fp8kv_attn_plan_t* plan, const Params& p, cudaStream_t st) {
  auto fn = split_generic<D, MODE, RPW>;
  const int smem = generic_layout(D, 8 * RPW).total_bytes;
  static DeviceOnce once;
  cudaError_t e = once.run([&] {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (e != cudaSuccess) return e;
  dim3 grid(plan->grid[0], plan->grid[1], plan->grid[2]);
  fn<<<grid, NT, smem, st>>>(p);
  return cudaGetLastError();
}

template <int D, int MODE>
cudaError_t launch_rpw(const fp8kv_attn_plan_t* plan, const Params& p, cudaStream_t st) {
  const int rc = p.row_chunk;
  if (rc <= 8) return launch_one<D, MODE, 1>(plan, p, st);
  if (rc <= 16) return launch_one<D, MODE, 2>(plan, p, st);
  if (rc <= 32) return launch_one<D, MODE, 4>(plan, p, st);
  return launch_one<D, MODE, 8>(plan, p, st);
}

template <int D>
cudaError_t launch_mode(const fp8kv_attn_plan_t* plan, const Params& p, cudaStream_t st) {
  if (p.mode == FP8KV_MODE_DENSE) return launch_rpw<D, FP8KV_MODE_DENSE>(plan, p, st);
  return launch_rpw<D, FP8KV_MODE_SPARSE_PAGE4>(plan, p, st);
}

}  // namespace

int generic_smem_bytes(int D, int row_chunk) {
  const int rpw = row_chunk <= 8 ? 1 : row_chunk <= 16 ? 2 : row_chunk <= 32 ? 4 : 8;
  return generic_layout(D, 8 * rpw).total_bytes;
}

cudaError_t launch_split_generic(const fp8kv_attn_plan_t* plan, const Params& p, cudaStream_t st) {
  switch (p.D) {
    case 64: return launch_mode<64>(plan, p, st);
    case 128: return launch_mode<128>(plan, p, st);
    case 256: return launch_mode<256>(plan, p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fp8kv
