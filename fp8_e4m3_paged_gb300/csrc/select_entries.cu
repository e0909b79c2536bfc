// Grouped planner: token-ID selections -> four-token microblock entries with
// per-row masks, padded to a multiple of 8 with the null block ("Qualify
// calibrated E4M3 and disk PLE with QSA DCP2", commit "grouped page4
// null-block padding").
//
// One CTA per request.  The logical microblocks are taken in chunks (one
// chunk covers a 131072-token context with up to 8 query rows, 65536 with
// 9..16 rows, whose masks take two words): the chunk's masks are cleared in
// shared memory, every selection that falls in the chunk ORs its bit
// (4r + t%4; rows 8..15 in the second word) in with an atomic, a warp ballot per 32 microblocks turns
// the masks into a bitmap of non-empty microblocks, one prefix sum over the
// bitmap words' popcounts gives every word its first entry, and each thread
// writes the entries of its two words in microblock order.  Null entries
// then pad the count to a multiple of 8.  Nothing returns to the host, so
// the call is graph-capturable.
#include <cstdint>

#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace fp8kv {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kMaskWords = 32768;           // mask words per pass
constexpr int kSmem = kMaskWords * 4;       // the masks (dynamic shared memory)

// W mask words per microblock (1: up to 8 query rows, 2: up to 16).
template <int W>
__global__ void __launch_bounds__(kSelThreads) select_kernel(const fp8kv_select_args a) {
  constexpr int kChunk = kMaskWords / W;      // logical microblocks per pass
  constexpr int kWords = kChunk / 32;         // bitmap words per pass
  constexpr int kWordsPerThread = kWords / kSelThreads;
  static_assert(kWordsPerThread * kSelThreads == kWords && kWordsPerThread >= 1, "bitmap words per thread");
  extern __shared__ uint4 smem_masks[];
  uint32_t* masks = reinterpret_cast<uint32_t*>(smem_masks);  // microblock m: words m*W .. m*W+W-1
  __shared__ uint32_t words[kWords];
  __shared__ int warp_tot[kSelWarps];
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n_sel = (int64_t)a.q_max * a.topk;
  const int32_t* sel = a.sel + (int64_t)b * n_sel;
  const int32_t* bt = a.block_table + (int64_t)b * a.block_table_stride;
  int32_t* tbl = a.entry_tbl + (int64_t)b * a.entry_stride;
  uint32_t* msk = a.entry_mask + (int64_t)b * a.entry_stride;
  uint32_t* msk_hi = W == 2 ? a.entry_mask_hi + (int64_t)b * a.entry_stride : nullptr;
  const int64_t limit = 4ll * a.max_blocks;
  int base = 0;  // entries written so far (the same in every thread)
  bool bad = false;
  for (int lo = 0; lo < a.max_blocks; lo += kChunk) {
    const int n = min(kChunk, a.max_blocks - lo);
    const int nw = (n + 31) / 32;
    for (int i = tid; i < nw * 8 * W; i += kSelThreads) smem_masks[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    // selections, four loads in flight per thread before their atomics
    for (int64_t i0 = tid; i0 < n_sel; i0 += 4 * kSelThreads) {
      int32_t t4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t i = i0 + (int64_t)k * kSelThreads;
        t4[k] = (i < n_sel) ? __ldg(sel + i) : -1;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int32_t t = t4[k];
        if (t < 0) continue;
        if (t >= limit) {
          bad = true;
          continue;
        }
        const int m = t >> 2;
        if (m >= lo && m < lo + n) {
          const int r = (int)((i0 + (int64_t)k * kSelThreads) / a.topk);
          atomicOr(&masks[(m - lo) * W + (r >> 3)], 1u << (4 * (r & 7) + (t & 3)));
        }
      }
    }
    __syncthreads();
    // bitmap of non-empty microblocks: word w covers microblocks 32w..32w+31
    for (int w = warp; w < kWords; w += kSelWarps) {
      const int m = 32 * w + lane;
      const uint32_t any = W == 2 ? (masks[2 * m] | masks[2 * m + 1]) : masks[m];
      const uint32_t bits = __ballot_sync(0xffffffffu, m < n && any != 0u);
      if (lane == 0) words[w] = bits;
    }
    __syncthreads();
    // this thread owns words kWordsPerThread*tid ..: exclusive prefix of the counts
    uint32_t ws[kWordsPerThread];
    int mine = 0;
#pragma unroll
    for (int k = 0; k < kWordsPerThread; ++k) {
      ws[k] = words[kWordsPerThread * tid + k];
      mine += __popc(ws[k]);
    }
    int incl = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int k = 0; k < kSelWarps; ++k) {
      const int c = warp_tot[k];
      before += (k < warp) ? c : 0;
      total += c;
    }
    int pos = base + before + incl - mine;
#pragma unroll
    for (int k = 0; k < kWordsPerThread; ++k) {
      const uint32_t bits = ws[k];
      if (bits == 0u) continue;
      // the block-table entries of the word's non-empty microblocks: all
      // loads issued before the first store
      const int m0 = 32 * (kWordsPerThread * tid + k);
      int32_t phys[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) phys[j] = ((bits >> j) & 1u) ? __ldg(bt + lo + m0 + j) : 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if ((bits >> j) & 1u) {
          tbl[pos] = phys[j];
          msk[pos] = masks[(m0 + j) * W];
          if (W == 2) msk_hi[pos] = masks[(m0 + j) * W + 1];
          ++pos;
        }
      }
    }
    base += total;
    __syncthreads();  // masks, words and warp_tot are reused by the next pass
  }
  if (bad && a.status) set_status(a.status, FP8KV_STATUS_BAD_ENTRIES);
  const int padded = (base + 7) / 8 * 8;
  for (int j = base + tid; j < padded; j += kSelThreads) {
    tbl[j] = a.null_block;
    msk[j] = 0u;
    if (W == 2) msk_hi[j] = 0u;
  }
  if (tid == 0) a.n_entries[b] = padded;
}

}  // namespace

cudaError_t launch_select_to_entries(const fp8kv_select_args& a, cudaStream_t st) {
  auto fn = a.q_max > 8 ? select_kernel<2> : select_kernel<1>;
  static DeviceOnce once1, once2;
  cudaError_t e = (a.q_max > 8 ? once2 : once1).run([&] {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (e != cudaSuccess) return e;
  fn<<<(unsigned)a.batch, kSelThreads, kSmem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace fp8kv
