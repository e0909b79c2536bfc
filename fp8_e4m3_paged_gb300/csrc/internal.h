// Internal declarations shared by the library's translation units.
#pragma once

#include <atomic>
#include <cstdint>

#include <cuda_runtime.h>

#include "fp8kv_attn.h"

namespace fp8kv {

// Split-kernel variants a plan may choose.
enum Kernel : int32_t {
  kGeneric = FP8KV_KERNEL_GENERIC,  // CUDA-core FP32 path, any supported shape
  kTc = FP8KV_KERNEL_TC,            // tcgen05 tensor-core path (head_dim 128/256)
  kTcSmall = FP8KV_KERNEL_TC_SMALL, // tcgen05, transposed for row groups of at most 16 (decode)
};

constexpr int kGenericThreads = 256;
constexpr int kGenericTileTokens = 32;  // tokens (dense) or 8 entries (sparse)
constexpr int kMaxRowChunk = 64;        // query vectors per split CTA
constexpr int kGenericMaxPartTiles = 32; // longest partition of the generic path (tiles)

// Everything a split or combine kernel needs, resolved on the host.
struct Params {
  // problem
  int32_t mode, B, q_max, Hq, Hkv, D, G, rows, row_chunk, n_row_chunks, S;
  int32_t page_size, max_kv_len, max_blocks, num_kv_blocks;
  // ceil(2^64 / page_size) (page_size >= 2; 0 for 1): the split kernels
  // divide token indices by the page size with one multiply-high (Lemire,
  // Kaser and Kurz, "Faster remainder by direct computation", 2019: exact for
  // every numerator below 2^32 because 64 >= 32 + ceil(log2(page_size)))
  uint64_t page_div;
  int32_t kv_format;  // FP8KV_KV_E4M3 or FP8KV_KV_E5M2
  int32_t test_flags; // FP8KV_TEST_* (0 in production)
  int32_t min_part;   // shortest partition: tokens (dense) or entries (sparse), 0 = none
  // inputs
  const uint16_t* q;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  int64_t ksb, kst, ksh, vsb, vst, vsh;
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* row_len;
  const int32_t* entry_tbl;
  const uint32_t* entry_mask;
  const uint32_t* entry_mask_hi;  // sparse rows 8..15 (NULL with q_max <= 8)
  // fused write of the new tokens (n_new = 0: none); strides in elements
  const uint16_t* k_new;
  const uint16_t* v_new;
  int64_t kn_s[3], vn_s[3];  // request, token, head
  int32_t n_new, new_dtype;
  const int32_t* n_entries;
  int64_t entry_stride;
  // scales: logit factor = softmax_scale * k_scale * log2(e)
  float softmax_scale, k_scale, v_scale;
  const float* k_scale_dev;
  const float* v_scale_dev;
  // outputs / workspace
  uint16_t* out;
  unsigned int* status;
  float* partial;   // [B][Hkv][S][rows][D]
  float2* ml;       // [B][Hkv][S][rows]  (max in log2 units, sum)
  float* out_f32;   // combine with LSE: FP32 output [B][q_max][Hq][D] (NULL: fp16 out)
  float* lse;       // combine with LSE: base-2 LSE [B][q_max][Hq]
};

int build_params(const fp8kv_attn_plan_t* plan, const fp8kv_attn_args* a, Params* p, bool need_out = true);

cudaError_t launch_split_generic(const fp8kv_attn_plan_t* plan, const Params& p, cudaStream_t s);
cudaError_t launch_split_tc(const fp8kv_attn_plan_t* plan, const Params& p, cudaStream_t s);
cudaError_t launch_split_tc_small(const fp8kv_attn_plan_t* plan, const Params& p, cudaStream_t s);
cudaError_t launch_combine(const fp8kv_attn_plan_t* plan, const Params& p, cudaStream_t s);
cudaError_t launch_cache_write(const fp8kv_cache_write_args& a, cudaStream_t s);
cudaError_t launch_merge(const fp8kv_merge_args& a, int32_t scale_rank, cudaStream_t s);
cudaError_t launch_select_to_entries(const fp8kv_select_args& a, cudaStream_t s);

// Runs a setup call (a kernel attribute) once per device, on first use.
struct DeviceOnce {
  std::atomic<uint64_t> done{0};
  template <class F>
  cudaError_t run(F f) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = f();
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
  }
};

// Shared-memory bytes of the generic split kernel for a head dim and row chunk.
int generic_smem_bytes(int D, int row_chunk);

// Tensor-core path: shared-memory bytes (D = 128 or 256), threads, tile size.
int tc_smem_bytes(int D, bool small_group);
constexpr int kTcSmallRows = 16;     // query vectors per CTA of the small-group kernel
constexpr int kTcSmallAutoRows = 8;  // the planner's own choice of it: groups up to this size
constexpr int kTcThreads = 480;
constexpr int kTcTileTokens = 64;
constexpr int kTcRows = 64;
constexpr int kTcMaxPartTiles = 32;  // longest partition of the query-row tensor-core kernel (tiles)
// The small-group kernel drains each tile pair's PV into a compensated
// (TwoSum) master sum, so its error does not grow with the partition length:
// it takes longer partitions, hence fewer CTAs that each pay the pipeline
// fill and drain (64 decode requests: 850 -> 700 us per step at 6 instead of
// 23 partitions per request).
constexpr int kTcSmallMaxPartTiles = 128;

}  // namespace fp8kv
