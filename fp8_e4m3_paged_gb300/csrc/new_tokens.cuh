// Fused write of a verify step's new tokens, shared by the split kernels.
//
// The last n_new positions of request b (U - n_new .. U - 1, U its longest
// row length) receive the caller's new K and V rows, quantised to the
// cache's FP8 format exactly as the cache write does (fp8_encode.cuh).  A
// CTA writes the new positions inside its own partition [u0, u1) for its KV
// head, before it reads any of them: every CTA that attends to a new token
// has written that token itself (row chunks of one partition write the same
// bytes), so no CTA depends on another.
#pragma once

#include <cstdint>

#include "device_common.cuh"
#include "fp8_encode.cuh"
#include "internal.h"

namespace fp8kv {

template <int FMT>
__device__ __forceinline__ void write_new_tokens(const Params& p, int b, int g, int U, int u0, int u1, int tid,
                                                 int nthreads) {
  const int first = U - p.n_new;  // position of new token 0
  const int lo = max(u0, max(first, 0)), hi = min(u1, U);
  if (lo >= hi) return;
  const int chunks = p.D / 16;
  const int items = (hi - lo) * chunks * 2;  // (position, 16-element chunk, K or V)
  const float ks = p.k_scale_dev ? *p.k_scale_dev : p.k_scale;
  const float vs = p.v_scale_dev ? *p.v_scale_dev : p.v_scale;
  const float kr = __frcp_rn(ks), vr = __frcp_rn(vs);
  for (int it = tid; it < items; it += nthreads) {
    const bool is_v = it & 1;
    const int rest = it >> 1;
    const int c = rest % chunks, pos = lo + rest / chunks, j = pos - first;
    const int blk = p.block_table[(int64_t)b * p.bt_stride + pos / p.page_size];
    if (blk < 0 || blk >= p.num_kv_blocks) {
      if (c == 0 && !is_v) set_status(p.status, FP8KV_STATUS_BAD_BLOCK);
      continue;
    }
    const int64_t* s = is_v ? p.vn_s : p.kn_s;
    const uint4* src = reinterpret_cast<const uint4*>((is_v ? p.v_new : p.k_new) + b * s[0] + j * s[1] +
                                                      g * s[2] + c * 16);
    const uint4 x[2] = {src[0], src[1]};
    const float sc = is_v ? vs : ks, rc = is_v ? vr : kr;
    const uint4 q = p.new_dtype == FP8KV_DTYPE_F16 ? quant16<FP8KV_DTYPE_F16, FMT>(x, sc, rc)
                                                   : quant16<FP8KV_DTYPE_BF16, FMT>(x, sc, rc);
    uint8_t* dst = const_cast<uint8_t*>(is_v ? p.v_cache : p.k_cache) +
                   blk * (is_v ? p.vsb : p.ksb) + (pos % p.page_size) * (is_v ? p.vst : p.kst) +
                   g * (is_v ? p.vsh : p.ksh) + c * 16;
    *reinterpret_cast<uint4*>(dst) = q;
  }
}

// The new tokens of [u0, u1) written (if any) and ordered before the CTA's
// reads of them: device-scope fence, then for readers through the bulk-copy
// engine (async proxy) a proxy fence; the caller's CTA barrier follows.
template <int FMT>
__device__ __forceinline__ void write_new_tokens_and_fence(const Params& p, int b, int g, int U, int u0, int u1,
                                                           int tid, int nthreads) {
  write_new_tokens<FMT>(p, b, g, U, u0, u1, tid, nthreads);
  __threadfence();
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

}  // namespace fp8kv
