/*
 * fp8kv_attn.h -- C ABI of a paged-attention library for an FP8 E4M3 KV cache
 * (one GPU, sm_103a).
 *
 * What the calls compute
 * ----------------------
 * For every request b, query row r < q_max and query head h, with KV head
 * g = h / (Hq / Hkv), softmax attention over the tokens the row may see:
 *
 *   z_j   = softmax_scale * k_scale * <q[b][r][h], dec(K_j)>
 *   out   = v_scale * sum_j softmax(z)_j * dec(V_j)          (fp16, RNE)
 *
 * where dec() is the exact decode of the cache bytes: E4M3 (OCP E4M3FN), or
 * E5M2 when the plan's kv_format says so.
 *  - Dense mode: row r sees tokens [0, row_kv_len[b][r]); token t lives in
 *    physical block block_table[b][t / page_size], slot t % page_size.  A row
 *    length of 0 is a dead row and yields +0.0.  (Live per-query lengths
 *    including zero padding, runtime page stride: "DFlash2 E4M3 attention
 *    with FP32 state", intro paragraphs 3 and 5.)
 *  - Sparse mode (QSA): four-token microblocks.  Entry e < n_entries[b] names
 *    physical microblock entry_tbl[b][e]; bit (4*r + t) of entry_mask[b][e]
 *    says that query row r < 8 sees token t of it, and bit (4*(r-8) + t) of
 *    entry_mask_hi[b][e] the same for rows 8..15 (plans with q_max > 8).  Entries with mask 0 (the null
 *    padding entries) are never read, and unseen tokens contribute exactly
 *    zero whatever their bytes decode to, NaN included.  ("Qualify calibrated
 *    E4M3 and disk PLE with QSA DCP2", commit "grouped page4 null-block
 *    padding"; "Qwen4Exp: fp8_e4m3 main KV cache on the QSA path".)
 *  - Scales: the K scale is folded into the logit scale and the V scale is
 *    an output scale, both applied outside the token loop ("Qwen4Exp: fp8_e4m3
 *    main KV cache on the QSA path", review thread on host-side KV scales).
 *
 * Numerical contract ("DFlash2 E4M3 attention with FP32 state", intro
 * paragraph 4): FP32 QK and PV accumulation; split-KV partitions store FP32
 * unnormalised numerators with a separate FP32 running max and sum; an FP32
 * combine writes the FP16 output.
 *
 * Calls
 * -----
 *   fp8kv_attn_plan     host only: validates a shape and picks the split
 *                       count, grid and workspace size.
 *   fp8kv_attn_split    launches the split kernel (partials into workspace).
 *   fp8kv_attn_combine  launches the combine kernel (workspace -> out).
 *
 * split and combine must run on the same stream with the same workspace; one
 * workspace serves one stream at a time.  The library never allocates, frees,
 * synchronises, or reads device memory from the host, and keeps no state
 * between calls apart from a once-per-device kernel attribute setting, so a
 * split + combine pair can be captured in a CUDA graph and replayed with new
 * row lengths, masks or entry counts in the same device buffers.
 *
 * Errors: every call returns FP8KV_OK (0) or a negative FP8KV_E* code and
 * never aborts.  Device-side anomalies never trap: an out-of-range block id or
 * microblock id contributes nothing, a length or entry count above the planned
 * bound is clamped, and a sticky FP8KV_STATUS_* bit is OR-ed into the 32-bit
 * status word at byte offset 0 of the workspace.  The caller zeroes that word
 * (e.g. once, with the rest of the workspace) and may read it after a sync.
 */
#ifndef FP8KV_ATTN_H
#define FP8KV_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Capability revision: a plan records the revision that built it and the
 * launch calls refuse a plan from another revision (FP8KV_EVERSION), so a
 * stale plan cannot reach kernels with another partial layout ("DFlash2 E4M3
 * attention with FP32 state", intro paragraph 5: the wrapper requires a given
 * precision capability revision). */
#define FP8KV_ATTN_REVISION 5

/* Return codes. */
#define FP8KV_OK 0
#define FP8KV_EINVAL (-1)       /* null or misaligned pointer, bad shape or stride */
#define FP8KV_EUNSUPPORTED (-2) /* head_dim, q_max, or sparse with page_size != 4 */
#define FP8KV_EWORKSPACE (-3)   /* workspace smaller than plan->workspace_bytes */
#define FP8KV_EVERSION (-4)     /* plan built by another revision */
#define FP8KV_ECUDA (-5)        /* a CUDA runtime call or launch failed */

/* Modes. */
#define FP8KV_MODE_DENSE 0
#define FP8KV_MODE_SPARSE_PAGE4 1

/* Cache byte formats (desc.kv_format).  E4M3: OCP E4M3FN (no infinity,
 * 0x7F/0xFF NaN, largest 448).  E5M2: the upper byte of an IEEE binary16
 * (infinities and NaNs as in binary16, largest finite 57344) -- the legacy
 * format of the kernels "DFlash2 E4M3 attention with FP32 state" replaces. */
#define FP8KV_KV_E4M3 0
#define FP8KV_KV_E5M2 1
/* bf16 K/V (two bytes per element, little-endian; a token row is 2*head_dim
 * bytes): the unquantised cache for A/B runs against the FP8 path
 * ("DFlash2 E4M3 attention with FP32 state": the FP8 cache replaces a 16-bit
 * one).  Served by the FP32 CUDA-core kernel only (FP8KV_KERNEL_GENERIC;
 * asking for a tensor-core kernel gives FP8KV_EUNSUPPORTED).  The scales
 * apply as for the FP8 formats (1.0 for an unscaled cache). */
#define FP8KV_KV_BF16 2

/* Split-kernel choice (desc.kernel; the plan records the one chosen). */
#define FP8KV_KERNEL_AUTO 0
#define FP8KV_KERNEL_GENERIC 1 /* FP32 CUDA-core path: every supported shape */
#define FP8KV_KERNEL_TC 2      /* tcgen05 tensor-core path: head_dim 128/256 (else FP8KV_EUNSUPPORTED) */
#define FP8KV_KERNEL_TC_SMALL 3 /* tcgen05, transposed (tokens as the MMA rows, at most 16 query vectors
                                   per CTA): decode-sized groups; head_dim 128/256 */

/* Sticky device status bits (workspace word at byte offset 0). */
#define FP8KV_STATUS_BAD_BLOCK 0x1   /* block / microblock id outside [0, num_kv_blocks) */
#define FP8KV_STATUS_BAD_LEN 0x2     /* a row length < 0 or > max_kv_len (clamped) */
#define FP8KV_STATUS_BAD_ENTRIES 0x4 /* n_entries < 0 or > max_blocks (clamped) */
#define FP8KV_STATUS_TIMEOUT 0x8     /* a bounded pipeline wait gave up (results invalid) */

/* Test-only switches (desc.test_flags; 0 in production).
 * FP8KV_TEST_STALL_PIPELINE: the tensor-core split kernel's K producer holds
 * back its first arrival until another warp's bounded wait has given up, and
 * waits use a short poll budget, so that the give-up path (abort, drain of
 * issued copies and UMMAs, FP8KV_STATUS_TIMEOUT) runs on purpose.  Accepted
 * only with the tensor-core kernel; the launch's results are invalid. */
#define FP8KV_TEST_STALL_PIPELINE 0x1

/* cudaStream_t without including CUDA headers (same type). */
typedef struct CUstream_st* fp8kv_stream_t;

/* Problem shape (host memory, read only during fp8kv_attn_plan). */
typedef struct {
  int32_t mode;          /* FP8KV_MODE_* */
  int32_t batch;         /* B >= 0 requests (0: nothing to do) */
  int32_t q_max;         /* query rows per request: 1..16 (sparse above 8: args.entry_mask_hi) */
  int32_t num_q_heads;   /* Hq >= 1 */
  int32_t num_kv_heads;  /* Hkv >= 1, Hq % Hkv == 0 */
  int32_t head_dim;      /* D: 64, 128 or 256 */
  int32_t page_size;     /* tokens per physical block, >= 1 (sparse: 4) */
  int32_t max_kv_len;    /* dense: upper bound of every row_kv_len; sparse: unused */
  int32_t max_blocks;    /* dense: block-table columns used per request (>= ceil(max_kv_len/page_size));
                            sparse: entry slots per request (upper bound of n_entries) */
  int32_t num_kv_blocks; /* physical blocks in the page pool (for bounds checks), >= 1 */
  int32_t num_sms;       /* SMs to plan for; 0 = ask the current device */
  int32_t num_splits;    /* split-KV partitions per (request, KV head); 0 = planner's choice */
  int32_t kernel;        /* FP8KV_KERNEL_*: 0 = planner's choice */
  int32_t kv_format;     /* FP8KV_KV_*: 0 = E4M3 */
  int32_t test_flags;    /* FP8KV_TEST_*: 0 in production */
} fp8kv_attn_desc;

/* A plan: plain data, owned by the caller, nothing to free.  Fields other than
 * `reserved` are informational; pass the plan back unmodified. */
typedef struct {
  int32_t revision;      /* FP8KV_ATTN_REVISION of the library that planned it */
  int32_t mode, batch, q_max, num_q_heads, num_kv_heads, head_dim, page_size;
  int32_t max_kv_len, max_blocks, num_kv_blocks;
  int32_t group;         /* Hq / Hkv */
  int32_t rows;          /* q_max * group: query vectors per (request, KV head) */
  int32_t num_splits;    /* S */
  int32_t tile_tokens;   /* tokens per pipeline tile (dense) */
  int32_t kernel;        /* FP8KV_KERNEL_GENERIC or FP8KV_KERNEL_TC */
  int32_t grid[3];       /* split-kernel grid */
  int32_t block_threads; /* split-kernel block size */
  int32_t smem_bytes;    /* split-kernel dynamic shared memory */
  int32_t row_chunk;     /* query vectors per split CTA */
  int32_t num_sms;
  int64_t partial_offset;  /* byte offset of FP32 numerators in the workspace */
  int64_t ml_offset;       /* byte offset of FP32 (max, sum) pairs */
  int64_t workspace_bytes; /* minimum workspace size */
  int32_t kv_format;       /* FP8KV_KV_* of the cache bytes */
  int32_t test_flags;      /* FP8KV_TEST_* (0 in production) */
  int32_t min_part;        /* shortest non-empty partition: tokens (dense) or entries (sparse) */
  int32_t reserved[13];
} fp8kv_attn_plan_t;

/* Per-call arguments.  All pointers are device pointers owned by the caller,
 * except that the struct itself lives in host memory. */
typedef struct {
  const void* q;            /* fp16 [B][q_max][Hq][D], contiguous, 16-byte aligned */
  const uint8_t* k_cache;   /* E4M3 bytes; element (block, slot, kv head, d) at
                               k_cache + block*k_stride_block + slot*k_stride_token
                               + head*k_stride_head + d  (d contiguous) */
  const uint8_t* v_cache;   /* same addressing with the v_stride_* values */
  int64_t k_stride_block, k_stride_token, k_stride_head; /* bytes, multiples of 16 */
  int64_t v_stride_block, v_stride_token, v_stride_head; /* bytes, multiples of 16 */
  const int32_t* block_table;   /* dense: [B][block_table_stride] physical block ids */
  int64_t block_table_stride;   /* elements */
  const int32_t* row_kv_len;    /* dense: [B][q_max] live lengths (0 = dead row) */
  const int32_t* entry_tbl;     /* sparse: [B][entry_stride] microblock ids */
  const uint32_t* entry_mask;   /* sparse: [B][entry_stride] visibility bits (4*r + t) */
  const int32_t* n_entries;     /* sparse: [B] entries in use */
  int64_t entry_stride;         /* elements */
  float softmax_scale;          /* logit scale before the K scale */
  float k_scale;                /* host K scale (used when k_scale_dev is NULL) */
  float v_scale;                /* host V scale (used when v_scale_dev is NULL) */
  const float* k_scale_dev;     /* optional device scalar (one float), NULL = host */
  const float* v_scale_dev;     /* optional device scalar (one float), NULL = host */
  void* out;                    /* fp16 [B][q_max][Hq][D], contiguous */
  void* workspace;              /* >= plan->workspace_bytes, 256-byte aligned */
  size_t workspace_bytes;
  const uint32_t* entry_mask_hi; /* sparse with q_max > 8: [B][entry_stride] bits (4*(r-8) + t)
                                    of rows 8..15 (required there; ignored with q_max <= 8) */
  /* Fused cache write (dense mode, E4M3/E5M2 caches; n_new = 0: none).  The
   * last n_new positions of every request b -- U_b - n_new .. U_b - 1, with
   * U_b its longest row_kv_len -- receive these new K and V rows, quantised
   * in the cache's format with k_scale / v_scale exactly as
   * fp8kv_attn_cache_write does, inside fp8kv_attn_split and before any of
   * them is read: the verify step of speculative decoding writes its draft
   * tokens and attends over them in one launch.  The caches must then be
   * writable (k_cache / v_cache are written through).  Row j of request b,
   * head h: k_new + b*k_new_stride_req + j*k_new_stride_token +
   * h*k_new_stride_head (elements of new_dtype, d contiguous; strides
   * multiples of 8, base 16-byte aligned).  A position whose block is out
   * of range is not written and sets FP8KV_STATUS_BAD_BLOCK. */
  const void* k_new;
  const void* v_new;
  int64_t k_new_stride_req, k_new_stride_token, k_new_stride_head;
  int64_t v_new_stride_req, v_new_stride_token, v_new_stride_head;
  int32_t n_new;                /* new tokens per request, 0..max_kv_len (each U_b >= n_new) */
  int32_t new_dtype;            /* FP8KV_DTYPE_F16 (0) or FP8KV_DTYPE_BF16 (1) */
} fp8kv_attn_args;

/* Library revision (FP8KV_ATTN_REVISION). */
int fp8kv_attn_version(void);

/* Static text for a return code; never NULL. */
const char* fp8kv_attn_strerror(int code);

/* Validate `d` and fill `plan`.  Host only; touches no device memory.  When
 * d->num_sms is 0 it reads the current device's SM count (FP8KV_ECUDA if that
 * fails).  Returns FP8KV_EINVAL / FP8KV_EUNSUPPORTED for shapes it rejects. */
int fp8kv_attn_plan(const fp8kv_attn_desc* d, fp8kv_attn_plan_t* plan);

/* Launch the split kernel on `stream`: every (request, KV head, partition)
 * writes FP32 numerators and an FP32 (max, sum) pair per query vector into
 * the workspace.  Empty partitions write (max = -inf, sum = 0). */
int fp8kv_attn_split(const fp8kv_attn_plan_t* plan, const fp8kv_attn_args* a,
                     fp8kv_stream_t stream);

/* Launch the combine kernel on `stream`: merges the partitions of every query
 * vector in FP32 and writes fp16 `out` (rows whose total sum is 0 get +0.0). */
int fp8kv_attn_combine(const fp8kv_attn_plan_t* plan, const fp8kv_attn_args* a,
                       fp8kv_stream_t stream);

/* ------------------------------------------------------------------------
 * Cache write: quantise new K/V rows into the E4M3 pages.
 *
 * For every new token n < num_tokens with slot = slot_mapping[n] >= 0, block
 * slot / page_size, offset slot % page_size, and every KV head h, d < D:
 *
 *   k_cache[block][offset][h][d] = E4M3(fp32(k[n][h][d]) / k_scale)
 *   v_cache[block][offset][h][d] = E4M3(fp32(v[n][h][d]) / v_scale)
 *
 * with the division in FP32 (correctly rounded) and E4M3() rounding to the
 * nearest code, ties to even, magnitudes above 448 saturating to +-448 and
 * NaN giving a NaN code.  This is the write path that fills the cache the
 * attention reads, with the layer's per-tensor scales ("Qwen4Exp: fp8_e4m3
 * main KV cache on the QSA path", PR description: the uint8 cache is written
 * with the per-tensor scales and read back as e4m3).  Slots < 0 (padding
 * tokens) are not written; a slot whose block is outside [0, num_kv_blocks)
 * is not written either and sets FP8KV_STATUS_BAD_BLOCK in *status when
 * status is not NULL.  Two tokens that name the same slot race (last writer
 * unspecified), as in any scatter.
 * ------------------------------------------------------------------------ */
#define FP8KV_DTYPE_F16 0
#define FP8KV_DTYPE_BF16 1

typedef struct {
  int32_t num_tokens;     /* N >= 0 new tokens (0: nothing to do) */
  int32_t num_kv_heads;   /* Hkv >= 1 */
  int32_t head_dim;       /* D: a multiple of 16, 16..1024 */
  int32_t page_size;      /* tokens per physical block, >= 1 */
  int32_t num_kv_blocks;  /* physical blocks in the pool, >= 1 */
  int32_t dtype;          /* FP8KV_DTYPE_F16 or FP8KV_DTYPE_BF16 (k and v) */
  const void* k;          /* 2-byte elements; (n, h, d) at element n*k_stride_token + h*k_stride_head + d */
  const void* v;          /* same with the v_stride_* values */
  int64_t k_stride_token, k_stride_head;  /* elements, multiples of 8 (16-byte rows), >= 0 */
  int64_t v_stride_token, v_stride_head;
  const int64_t* slot_mapping;            /* [N] block * page_size + offset; < 0 = skip */
  uint8_t* k_cache;       /* same addressing as fp8kv_attn_args.k_cache */
  uint8_t* v_cache;
  int64_t kc_stride_block, kc_stride_token, kc_stride_head; /* bytes, multiples of 16 */
  int64_t vc_stride_block, vc_stride_token, vc_stride_head; /* bytes, multiples of 16 */
  float k_scale;          /* host K scale, > 0 (used when k_scale_dev is NULL) */
  float v_scale;          /* host V scale, > 0 (used when v_scale_dev is NULL) */
  const float* k_scale_dev; /* optional device scalar, NULL = host */
  const float* v_scale_dev;
  uint32_t* status;       /* optional device word for FP8KV_STATUS_BAD_BLOCK, NULL = none */
  int32_t kv_format;      /* FP8KV_KV_E4M3 (0, saturating to +-448) or FP8KV_KV_E5M2 (saturating to
                             +-57344); round to nearest even either way */
} fp8kv_cache_write_args;

/* Launch the cache write on `stream`.  k, v and the caches must be 16-byte
 * aligned.  Returns FP8KV_EINVAL for bad arguments, FP8KV_ECUDA if the launch
 * fails; never allocates or synchronises (graph-capturable). */
int fp8kv_attn_cache_write(const fp8kv_cache_write_args* a, fp8kv_stream_t stream);

/* ------------------------------------------------------------------------
 * Context-parallel merge ("Qualify calibrated E4M3 and disk PLE with QSA
 * DCP2": each rank holding a shard of the context exposes a base-2 LSE and
 * an FP32 partial output, merged across ranks by an all-gather of the LSEs
 * plus a reduce-scatter of the outputs, or by one all-to-all).
 *
 * fp8kv_attn_combine_lse is fp8kv_attn_combine for one rank's shard: instead
 * of the fp16 output it writes, per query vector, the FP32 output o (v_scale
 * applied) and lse = log2(sum_j 2^(log2(e) z_j)) over the shard's visible
 * tokens (o = 0, lse = -inf when the shard shows the vector nothing).
 * a->out is not used and may be NULL.
 *
 * fp8kv_attn_merge merges R ranks' (o_r, lse_r) pairs of n vectors:
 *   L = log2(sum_r 2^lse_r),  out = sum_r 2^(lse_r - L) o_r
 * (the attention over the union of the shards), writing any of: fp16 out
 * (RNE), FP32 out_f32, lse_out = L.  Vectors that no rank sees get +0.0 and
 * -inf.  The ranks are summed in order (bitwise deterministic).  With R = 1
 * and lses all finite it converts an FP32 output to fp16.
 *
 * fp8kv_attn_merge_scale is the all-gather + reduce-scatter shape: `outs`
 * holds this rank's own o (rank_stride_out unused), `lses` the all-gathered
 * LSEs of all R ranks, and out_f32 receives 2^(lse_rank - L) o_rank; summing
 * that over the ranks (the reduce-scatter) gives the merged FP32 output.
 * ------------------------------------------------------------------------ */
#define FP8KV_MERGE_MAX_RANKS 64

typedef struct {
  int32_t num_ranks;        /* R: 1..FP8KV_MERGE_MAX_RANKS */
  int32_t head_dim;         /* D: multiple of 4, 4..1024 */
  int64_t num_vectors;      /* n >= 0 (0: nothing to do) */
  const float* outs;        /* rank r's vector i at outs + r*rank_stride_out + i*D (16-byte aligned) */
  int64_t rank_stride_out;  /* elements, multiple of 4 */
  const float* lses;        /* rank r's vector i at lses + r*rank_stride_lse + i */
  int64_t rank_stride_lse;  /* elements */
  void* out;                /* fp16 [n][D] or NULL (8-byte aligned) */
  float* out_f32;           /* FP32 [n][D] or NULL (16-byte aligned) */
  float* lse_out;           /* [n] or NULL */
} fp8kv_merge_args;

int fp8kv_attn_combine_lse(const fp8kv_attn_plan_t* plan, const fp8kv_attn_args* a, float* out_f32,
                           float* lse, fp8kv_stream_t stream);
int fp8kv_attn_merge(const fp8kv_merge_args* a, fp8kv_stream_t stream);
int fp8kv_attn_merge_scale(const fp8kv_merge_args* a, int32_t rank, fp8kv_stream_t stream);

/* ------------------------------------------------------------------------
 * Grouped planner: token-ID selections -> the sparse mode's entries.
 *
 * For every request b: the distinct four-token logical microblocks
 * m = t / 4 that any query row selected (positions t >= 0, below
 * 4 * max_blocks), in increasing order, become entries with
 *   entry_tbl[b][e]  = block_table[b][m]          (physical microblock)
 *   entry_mask[b][e] = OR over selections t of row r < 8 in m of bit 4r + t%4
 *   entry_mask_hi[b][e] = the same for rows 8..15 (bit 4(r-8) + t%4; q_max > 8)
 * and null entries (null_block, mask 0) pad the count to a multiple of 8;
 * n_entries[b] is the padded count ("Qualify calibrated E4M3 and disk PLE
 * with QSA DCP2", commit "grouped page4 null-block padding").  Duplicate
 * selections are harmless; negative positions are unused slots; positions
 * at or past 4 * max_blocks are ignored and set FP8KV_STATUS_BAD_ENTRIES in
 * *status (when not NULL).  Entries past n_entries[b] are not written.
 * Device-side and graph-capturable: the counts never reach the host.
 * ------------------------------------------------------------------------ */
typedef struct {
  int32_t batch;                /* B >= 0 */
  int32_t q_max;                /* query rows per request, 1..16 (above 8: entry_mask_hi) */
  int32_t topk;                 /* selection slots per row, >= 0 */
  int32_t max_blocks;           /* logical microblocks per request, >= 1 */
  int32_t null_block;           /* physical microblock of padding entries */
  const int32_t* sel;           /* [B][q_max][topk] token positions, < 0 = unused */
  const int32_t* block_table;   /* [B][block_table_stride] logical -> physical microblock */
  int64_t block_table_stride;   /* elements, >= max_blocks */
  int32_t* entry_tbl;           /* [B][entry_stride] */
  uint32_t* entry_mask;         /* [B][entry_stride] */
  int64_t entry_stride;         /* elements, >= q_max * topk rounded up to 8 */
  int32_t* n_entries;           /* [B] */
  uint32_t* status;             /* optional status word, NULL = none */
  uint32_t* entry_mask_hi;      /* q_max > 8: [B][entry_stride] bits 4*(r-8) + t%4 of rows 8..15 */
} fp8kv_select_args;

int fp8kv_attn_select_to_entries(const fp8kv_select_args* a, fp8kv_stream_t stream);

/* Size of the library-owned device scratch used by fp8kv_attn_forward_static
 * (16 MiB; one copy per GPU that loads the library, held until exit). */
#define FP8KV_STATIC_SCRATCH_BYTES (16u << 20)

/* Split + combine without a caller-provided workspace, for callers that cannot
 * allocate device memory (a host runtime that hands a plugin only its input
 * and output buffers, a memory manager that owns the whole device heap, or a
 * path that forbids allocator calls).  This entry point has no counterpart in
 * the pages; it exists for those callers.
 *
 * The FP32 partials and the status word live in a file-scope device array of
 * FP8KV_STATIC_SCRATCH_BYTES; plans needing more return FP8KV_EWORKSPACE.
 * Nothing is allocated or freed.  `a` is used as for fp8kv_attn_split except
 * that a->workspace is not the scratch: if it is non-NULL and
 * a->workspace_bytes >= 4, the call's 32-bit status word is copied there (in
 * stream order) after the combine (with batch 0, the word is set to 0).  The
 * first call on a device looks the array's address up for that device; make
 * it before any stream capture.  The address is kept for the life of the
 * process: a device reset between calls is not supported.
 * Every call shares the one array: calls whose kernels may overlap on the GPU
 * (other streams, other host threads) race on it and must be serialised. */
int fp8kv_attn_forward_static(const fp8kv_attn_plan_t* plan, const fp8kv_attn_args* a,
                              fp8kv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8KV_ATTN_H */
