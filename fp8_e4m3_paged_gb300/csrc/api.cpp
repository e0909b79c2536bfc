// C ABI entry points: planning (host only), argument validation, dispatch.
#include <cmath>
#include <cstdint>
#include <cstring>

#include <cuda_runtime.h>

#include "fp8kv_attn.h"
#include "internal.h"

using namespace fp8kv;

namespace {

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

}  // namespace

extern "C" int fp8kv_attn_version(void) { return FP8KV_ATTN_REVISION; }

extern "C" const char* fp8kv_attn_strerror(int code) {
  switch (code) {
    case FP8KV_OK: return "ok";
    case FP8KV_EINVAL: return "invalid argument (null or misaligned pointer, bad shape or stride)";
    case FP8KV_EUNSUPPORTED: return "unsupported shape (head_dim, q_max, or sparse page size)";
    case FP8KV_EWORKSPACE: return "workspace smaller than the plan requires";
    case FP8KV_EVERSION: return "plan was built by another library revision";
    case FP8KV_ECUDA: return "CUDA runtime error";
    default: return "unknown error code";
  }
}

extern "C" int fp8kv_attn_plan(const fp8kv_attn_desc* d, fp8kv_attn_plan_t* plan) {
  if (!d || !plan) return FP8KV_EINVAL;
  if (d->mode != FP8KV_MODE_DENSE && d->mode != FP8KV_MODE_SPARSE_PAGE4) return FP8KV_EINVAL;
  if (d->batch < 0 || d->num_q_heads < 1 || d->num_kv_heads < 1) return FP8KV_EINVAL;
  if (d->num_q_heads % d->num_kv_heads) return FP8KV_EINVAL;
  if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256) return FP8KV_EUNSUPPORTED;
  if (d->q_max < 1) return FP8KV_EINVAL;
  if (d->q_max > 16) return FP8KV_EUNSUPPORTED;
  if (d->page_size < 1 || d->max_kv_len < 0 || d->max_blocks < 0 || d->num_kv_blocks < 1)
    return FP8KV_EINVAL;
  if (d->num_sms < 0 || d->num_splits < 0) return FP8KV_EINVAL;
  if (d->kernel < FP8KV_KERNEL_AUTO || d->kernel > FP8KV_KERNEL_TC_SMALL) return FP8KV_EINVAL;
  if ((d->kernel == FP8KV_KERNEL_TC || d->kernel == FP8KV_KERNEL_TC_SMALL) && d->head_dim != 128 &&
      d->head_dim != 256)
    return FP8KV_EUNSUPPORTED;
  if (d->kv_format != FP8KV_KV_E4M3 && d->kv_format != FP8KV_KV_E5M2 && d->kv_format != FP8KV_KV_BF16)
    return FP8KV_EINVAL;
  // bf16 caches: the CUDA-core kernel only
  if (d->kv_format == FP8KV_KV_BF16 && d->kernel != FP8KV_KERNEL_AUTO && d->kernel != FP8KV_KERNEL_GENERIC)
    return FP8KV_EUNSUPPORTED;
  if (d->test_flags & ~FP8KV_TEST_STALL_PIPELINE) return FP8KV_EINVAL;
  if (d->mode == FP8KV_MODE_DENSE) {
    if ((int64_t)d->max_blocks * d->page_size < d->max_kv_len) return FP8KV_EINVAL;
  } else {
    if (d->page_size != 4) return FP8KV_EUNSUPPORTED;  // q_max <= 16: two mask words above 8 rows
  }

  int sms = d->num_sms;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8KV_ECUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FP8KV_ECUDA;
    if (sms < 1) return FP8KV_ECUDA;
  }

  fp8kv_attn_plan_t P;
  std::memset(&P, 0, sizeof(P));
  P.revision = FP8KV_ATTN_REVISION;
  P.mode = d->mode;
  P.batch = d->batch;
  P.q_max = d->q_max;
  P.num_q_heads = d->num_q_heads;
  P.num_kv_heads = d->num_kv_heads;
  P.head_dim = d->head_dim;
  P.page_size = d->page_size;
  P.max_kv_len = d->max_kv_len;
  P.max_blocks = d->max_blocks;
  P.num_kv_blocks = d->num_kv_blocks;
  P.group = d->num_q_heads / d->num_kv_heads;
  P.rows = d->q_max * P.group;
  P.num_sms = sms;
  P.kv_format = d->kv_format;
  P.test_flags = d->test_flags;

  // Kernel choice for D = 128 or 256: up to 8 query vectors per (request,
  // KV head) -- decode with GQA -- the transposed tcgen05 kernel (tokens as
  // the MMA rows); more, the tcgen05 kernel with the query vectors as the
  // MMA rows (up to 64 per CTA).  Measured over contexts of 1K..64K tokens:
  // with 4 or 8 vectors the two are within ~5 %, with 12 or 16 the
  // query-row kernel is 30-60 % faster (the transposed kernel's softmax then
  // carries 16 columns per token); the transposed kernel still takes up to 16
  // on request.  D = 64 and bf16 caches: the FP32 CUDA-core kernel, which
  // also serves every shape on request.
  const bool tc_dims = P.head_dim == 128 || P.head_dim == 256;
  int kind = d->kernel;
  if (kind == FP8KV_KERNEL_AUTO)
    kind = (!tc_dims || d->kv_format == FP8KV_KV_BF16)
               ? FP8KV_KERNEL_GENERIC
               : (P.rows <= kTcSmallAutoRows ? FP8KV_KERNEL_TC_SMALL : FP8KV_KERNEL_TC);
  int tile, ctas_per_sm, max_part_tiles;
  if (kind == FP8KV_KERNEL_TC || kind == FP8KV_KERNEL_TC_SMALL) {
    const bool small = kind == FP8KV_KERNEL_TC_SMALL;
    P.kernel = small ? kTcSmall : kTc;
    const int cap = small ? kTcSmallRows : kTcRows;
    P.row_chunk = P.rows < cap ? P.rows : cap;
    tile = kTcTileTokens;
    P.block_threads = kTcThreads;
    P.smem_bytes = tc_smem_bytes(P.head_dim, small);
    ctas_per_sm = 1;
    max_part_tiles = small ? kTcSmallMaxPartTiles : kTcMaxPartTiles;
  } else {
    P.kernel = kGeneric;
    P.row_chunk = P.rows < kMaxRowChunk ? P.rows : kMaxRowChunk;
    tile = kGenericTileTokens;
    P.block_threads = kGenericThreads;
    P.smem_bytes = generic_smem_bytes(P.head_dim, P.row_chunk);
    ctas_per_sm = 2;
    max_part_tiles = kGenericMaxPartTiles;
  }
  if (P.test_flags && P.kernel == kGeneric) return FP8KV_EINVAL;  // the switch targets the pipeline waits
  const int n_chunks = ceil_div(P.rows, P.row_chunk);
  P.tile_tokens = tile;

  // Split count: about one wave of CTAs (two for the generic path), never
  // more partitions than tiles of work (dense: tokens / tile, sparse: entries
  // / (tile / 4)), and partitions capped in length where FP32 accumulation
  // error grows with the number of tiles one partition sums (the query-row
  // and CUDA-core kernels; the small-group kernel's cap is far longer).
  const int64_t units = (int64_t)d->batch * d->num_kv_heads * n_chunks;
  const int max_tiles = d->mode == FP8KV_MODE_DENSE
                            ? (d->max_kv_len > 0 ? ceil_div(d->max_kv_len, tile) : 1)
                            : (d->max_blocks > 0 ? ceil_div(d->max_blocks, tile / 4) : 1);
  int S;
  if (d->num_splits > 0) {
    S = d->num_splits;
  } else {
    const int64_t target = (int64_t)ctas_per_sm * sms;
    S = units > 0 ? ceil_div(target, units) : 1;
    const int by_len = ceil_div(max_tiles, max_part_tiles);
    if (S < by_len) S = by_len;
    if (S > max_tiles) S = max_tiles;
    if (S < 1) S = 1;
  }
  P.num_splits = S;
  // A batch with more (request, KV head, row chunk) units than the GPU has
  // CTA slots is sized for its longest request; a partition of a short
  // request is then kept at 16 tiles or more, so that few CTAs spend their
  // fixed setup and pipeline fill on a tile or two (the rest exit at once).
  const int unit_tokens = d->mode == FP8KV_MODE_DENSE ? tile : tile / 4;
  P.min_part = units > (int64_t)ctas_per_sm * sms ? 16 * unit_tokens : 0;
  P.grid[0] = S;
  P.grid[1] = d->num_kv_heads * n_chunks;
  P.grid[2] = d->batch;

  const int64_t nvec = (int64_t)d->batch * d->num_kv_heads * S * P.rows;
  P.partial_offset = 256;
  P.ml_offset = align_up(P.partial_offset + nvec * P.head_dim * 4, 256);
  P.workspace_bytes = align_up(P.ml_offset + nvec * 8, 256);
  *plan = P;
  return FP8KV_OK;
}

int fp8kv::build_params(const fp8kv_attn_plan_t* plan, const fp8kv_attn_args* a, Params* p, bool need_out) {
  if (!plan || !a || !p) return FP8KV_EINVAL;
  if (plan->revision != FP8KV_ATTN_REVISION) return FP8KV_EVERSION;
  std::memset(p, 0, sizeof(*p));
  p->mode = plan->mode;
  p->B = plan->batch;
  p->q_max = plan->q_max;
  p->Hq = plan->num_q_heads;
  p->Hkv = plan->num_kv_heads;
  p->D = plan->head_dim;
  p->G = plan->group;
  p->rows = plan->rows;
  p->row_chunk = plan->row_chunk;
  p->n_row_chunks = plan->row_chunk > 0 ? (plan->rows + plan->row_chunk - 1) / plan->row_chunk : 0;
  p->S = plan->num_splits;
  p->page_size = plan->page_size;
  p->page_div = plan->page_size >= 2 ? ~0ull / (uint64_t)plan->page_size + 1 : 0ull;
  p->max_kv_len = plan->max_kv_len;
  p->max_blocks = plan->max_blocks;
  p->num_kv_blocks = plan->num_kv_blocks;
  p->kv_format = plan->kv_format;
  p->test_flags = plan->test_flags;
  p->min_part = plan->min_part;
  if (p->kv_format != FP8KV_KV_E4M3 && p->kv_format != FP8KV_KV_E5M2 && p->kv_format != FP8KV_KV_BF16)
    return FP8KV_EINVAL;
  if (p->kv_format == FP8KV_KV_BF16 && plan->kernel != kGeneric) return FP8KV_EINVAL;
  if (p->G < 1 || p->rows != p->q_max * p->G || p->S < 1 || p->row_chunk < 1) return FP8KV_EINVAL;

  if (!a->workspace || !aligned(a->workspace, 256)) return FP8KV_EINVAL;
  if ((int64_t)a->workspace_bytes < plan->workspace_bytes) return FP8KV_EWORKSPACE;
  if (p->B == 0) {
    p->status = reinterpret_cast<unsigned int*>(a->workspace);
    return FP8KV_OK;
  }
  if (!a->q || (need_out && !a->out) || !a->k_cache || !a->v_cache) return FP8KV_EINVAL;
  if (!aligned(a->q, 16) || (need_out && !aligned(a->out, 16)) || !aligned(a->k_cache, 16) ||
      !aligned(a->v_cache, 16))
    return FP8KV_EINVAL;
  const int64_t st[6] = {a->k_stride_block, a->k_stride_token, a->k_stride_head,
                         a->v_stride_block, a->v_stride_token, a->v_stride_head};
  for (int64_t s : st)
    if (s < 0 || (s % 16) != 0) return FP8KV_EINVAL;
  if (plan->mode == FP8KV_MODE_DENSE) {
    if (!a->block_table || !a->row_kv_len) return FP8KV_EINVAL;
    if (a->block_table_stride < plan->max_blocks || a->block_table_stride < 1) return FP8KV_EINVAL;
  } else {
    if (!a->entry_tbl || !a->entry_mask || !a->n_entries) return FP8KV_EINVAL;
    if (plan->q_max > 8 && !a->entry_mask_hi) return FP8KV_EINVAL;  // rows 8..15 need the second words
    if (a->entry_stride < plan->max_blocks || a->entry_stride < 1) return FP8KV_EINVAL;
  }
  if (!std::isfinite(a->softmax_scale)) return FP8KV_EINVAL;
  if (!a->k_scale_dev && !std::isfinite(a->k_scale)) return FP8KV_EINVAL;
  if (!a->v_scale_dev && !std::isfinite(a->v_scale)) return FP8KV_EINVAL;

  p->q = reinterpret_cast<const uint16_t*>(a->q);
  p->k_cache = a->k_cache;
  p->v_cache = a->v_cache;
  p->ksb = a->k_stride_block;
  p->kst = a->k_stride_token;
  p->ksh = a->k_stride_head;
  p->vsb = a->v_stride_block;
  p->vst = a->v_stride_token;
  p->vsh = a->v_stride_head;
  p->block_table = a->block_table;
  p->bt_stride = a->block_table_stride;
  p->row_len = a->row_kv_len;
  p->entry_tbl = a->entry_tbl;
  p->entry_mask = a->entry_mask;
  p->entry_mask_hi = plan->q_max > 8 ? a->entry_mask_hi : nullptr;
  p->n_entries = a->n_entries;
  p->entry_stride = a->entry_stride;
  p->softmax_scale = a->softmax_scale;
  p->k_scale = a->k_scale;
  p->v_scale = a->v_scale;
  p->k_scale_dev = a->k_scale_dev;
  p->v_scale_dev = a->v_scale_dev;
  p->out = reinterpret_cast<uint16_t*>(a->out);
  p->n_new = 0;
  p->k_new = p->v_new = nullptr;
  if (a->n_new != 0) {
    // fused write of the new tokens: dense FP8 caches, aligned rows
    if (a->n_new < 0 || a->n_new > plan->max_kv_len || plan->mode != FP8KV_MODE_DENSE) return FP8KV_EINVAL;
    if (plan->kv_format != FP8KV_KV_E4M3 && plan->kv_format != FP8KV_KV_E5M2) return FP8KV_EINVAL;
    if (a->new_dtype != FP8KV_DTYPE_F16 && a->new_dtype != FP8KV_DTYPE_BF16) return FP8KV_EINVAL;
    if (!a->k_new || !a->v_new || !aligned(a->k_new, 16) || !aligned(a->v_new, 16)) return FP8KV_EINVAL;
    const int64_t ns[6] = {a->k_new_stride_req, a->k_new_stride_token, a->k_new_stride_head,
                           a->v_new_stride_req, a->v_new_stride_token, a->v_new_stride_head};
    for (int64_t s : ns)
      if (s < 0 || (s % 8) != 0) return FP8KV_EINVAL;
    if (!a->k_scale_dev && !(a->k_scale > 0.f)) return FP8KV_EINVAL;
    if (!a->v_scale_dev && !(a->v_scale > 0.f)) return FP8KV_EINVAL;
    p->n_new = a->n_new;
    p->new_dtype = a->new_dtype;
    p->k_new = reinterpret_cast<const uint16_t*>(a->k_new);
    p->v_new = reinterpret_cast<const uint16_t*>(a->v_new);
    for (int i = 0; i < 3; ++i) {
      p->kn_s[i] = ns[i];
      p->vn_s[i] = ns[3 + i];
    }
  }
  char* ws = reinterpret_cast<char*>(a->workspace);
  p->status = reinterpret_cast<unsigned int*>(ws);
  p->partial = reinterpret_cast<float*>(ws + plan->partial_offset);
  p->ml = reinterpret_cast<float2*>(ws + plan->ml_offset);
  return FP8KV_OK;
}

extern "C" int fp8kv_attn_split(const fp8kv_attn_plan_t* plan, const fp8kv_attn_args* a,
                                fp8kv_stream_t stream) {
  Params p;
  const int rc = build_params(plan, a, &p);
  if (rc != FP8KV_OK) return rc;
  if (p.B == 0) return FP8KV_OK;
  cudaError_t e;
  switch (plan->kernel) {
    case kGeneric: e = launch_split_generic(plan, p, reinterpret_cast<cudaStream_t>(stream)); break;
    case kTc:
    case kTcSmall: e = launch_split_tc(plan, p, reinterpret_cast<cudaStream_t>(stream)); break;
    default: return FP8KV_EINVAL;
  }
  return e == cudaSuccess ? FP8KV_OK : FP8KV_ECUDA;
}

extern "C" int fp8kv_attn_combine(const fp8kv_attn_plan_t* plan, const fp8kv_attn_args* a,
                                  fp8kv_stream_t stream) {
  Params p;
  const int rc = build_params(plan, a, &p);
  if (rc != FP8KV_OK) return rc;
  if (p.B == 0) return FP8KV_OK;
  const cudaError_t e = launch_combine(plan, p, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FP8KV_OK : FP8KV_ECUDA;
}

extern "C" int fp8kv_attn_cache_write(const fp8kv_cache_write_args* a, fp8kv_stream_t stream) {
  if (!a) return FP8KV_EINVAL;
  if (a->num_tokens < 0 || a->num_kv_heads < 1 || a->page_size < 1 || a->num_kv_blocks < 1)
    return FP8KV_EINVAL;
  if (a->head_dim < 16 || a->head_dim > 1024 || (a->head_dim % 16) != 0) return FP8KV_EINVAL;
  if (a->dtype != FP8KV_DTYPE_F16 && a->dtype != FP8KV_DTYPE_BF16) return FP8KV_EINVAL;
  if (a->kv_format != FP8KV_KV_E4M3 && a->kv_format != FP8KV_KV_E5M2) return FP8KV_EINVAL;
  if (a->num_tokens == 0) return FP8KV_OK;
  if (!a->k || !a->v || !a->slot_mapping || !a->k_cache || !a->v_cache) return FP8KV_EINVAL;
  if (!aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->k_cache, 16) || !aligned(a->v_cache, 16))
    return FP8KV_EINVAL;
  const int64_t es[4] = {a->k_stride_token, a->k_stride_head, a->v_stride_token, a->v_stride_head};
  for (int64_t s : es)
    if (s < 0 || (s % 8) != 0) return FP8KV_EINVAL;
  const int64_t bs[6] = {a->kc_stride_block, a->kc_stride_token, a->kc_stride_head,
                         a->vc_stride_block, a->vc_stride_token, a->vc_stride_head};
  for (int64_t s : bs)
    if (s < 0 || (s % 16) != 0) return FP8KV_EINVAL;
  if (!a->k_scale_dev && !(std::isfinite(a->k_scale) && a->k_scale > 0.f)) return FP8KV_EINVAL;
  if (!a->v_scale_dev && !(std::isfinite(a->v_scale) && a->v_scale > 0.f)) return FP8KV_EINVAL;
  const cudaError_t e = launch_cache_write(*a, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FP8KV_OK : FP8KV_ECUDA;
}

extern "C" int fp8kv_attn_combine_lse(const fp8kv_attn_plan_t* plan, const fp8kv_attn_args* a, float* out_f32,
                                      float* lse, fp8kv_stream_t stream) {
  Params p;
  const int rc = build_params(plan, a, &p, false);
  if (rc != FP8KV_OK) return rc;
  if (p.B == 0) return FP8KV_OK;
  if (!out_f32 || !lse || !aligned(out_f32, 16) || !aligned(lse, 4)) return FP8KV_EINVAL;
  p.out_f32 = out_f32;
  p.lse = lse;
  const cudaError_t e = launch_combine(plan, p, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FP8KV_OK : FP8KV_ECUDA;
}

namespace {

int check_merge(const fp8kv_merge_args* a) {
  if (!a) return FP8KV_EINVAL;
  if (a->num_ranks < 1 || a->num_ranks > FP8KV_MERGE_MAX_RANKS || a->num_vectors < 0) return FP8KV_EINVAL;
  if (a->head_dim < 4 || a->head_dim > 1024 || (a->head_dim % 4) != 0) return FP8KV_EINVAL;
  if (a->num_vectors == 0) return FP8KV_OK;
  if (!a->outs || !aligned(a->outs, 16) || a->rank_stride_out < 0 || (a->rank_stride_out % 4) != 0)
    return FP8KV_EINVAL;
  if (!a->lses || a->rank_stride_lse < 0) return FP8KV_EINVAL;
  if ((a->out && !aligned(a->out, 8)) || (a->out_f32 && !aligned(a->out_f32, 16))) return FP8KV_EINVAL;
  return FP8KV_OK;
}

}  // namespace

extern "C" int fp8kv_attn_merge(const fp8kv_merge_args* a, fp8kv_stream_t stream) {
  const int rc = check_merge(a);
  if (rc != FP8KV_OK || a->num_vectors == 0) return rc;
  if (!a->out && !a->out_f32 && !a->lse_out) return FP8KV_EINVAL;
  const cudaError_t e = launch_merge(*a, -1, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FP8KV_OK : FP8KV_ECUDA;
}

extern "C" int fp8kv_attn_merge_scale(const fp8kv_merge_args* a, int32_t rank, fp8kv_stream_t stream) {
  const int rc = check_merge(a);
  if (rc != FP8KV_OK || a->num_vectors == 0) return rc;
  if (rank < 0 || rank >= a->num_ranks || !a->out_f32 || a->out || a->lse_out) return FP8KV_EINVAL;
  const cudaError_t e = launch_merge(*a, rank, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FP8KV_OK : FP8KV_ECUDA;
}

extern "C" int fp8kv_attn_select_to_entries(const fp8kv_select_args* a, fp8kv_stream_t stream) {
  if (!a) return FP8KV_EINVAL;
  if (a->batch < 0 || a->q_max < 1 || a->q_max > 16 || a->topk < 0 || a->max_blocks < 1) return FP8KV_EINVAL;
  if (a->q_max > 8 && !a->entry_mask_hi) return FP8KV_EINVAL;
  if (a->block_table_stride < a->max_blocks) return FP8KV_EINVAL;
  const int64_t cap = ((int64_t)a->q_max * a->topk + 7) / 8 * 8;
  if (a->entry_stride < cap || a->entry_stride < 1) return FP8KV_EINVAL;
  if (a->batch == 0) return FP8KV_OK;
  if ((a->topk > 0 && !a->sel) || !a->block_table || !a->entry_tbl || !a->entry_mask || !a->n_entries)
    return FP8KV_EINVAL;
  const cudaError_t e = launch_select_to_entries(*a, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FP8KV_OK : FP8KV_ECUDA;
}
