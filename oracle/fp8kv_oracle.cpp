// FP64 CPU oracle for paged attention over an FP8 E4M3 KV cache.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the library (fp8_e4m3_paged_gb300)
// may include, link or call this file; only the tests, the package smoke check
// and the benchmark's CPU-baseline leg use it.  It shares no code, header,
// table or constant with the CUDA path.
//
// What it computes is the plain definition of softmax attention over the
// exactly decoded E4M3 cache contents, in double precision:
//
//   z_j   = softmax_scale * k_scale * sum_d q[d] * dec(K_j[d])
//   w_j   = exp(z_j - max z) / sum_i exp(z_i - max z)
//   out_d = v_scale * sum_j w_j * dec(V_j[d])
//
// over the tokens j that a query row may see.  Sources:
//  * per-tensor scales fold into the logits and the output
//    ("Qwen4Exp: fp8_e4m3 main KV cache on the QSA path", review thread:
//    k_scale pre-multiplied into the softmax scale, v_scale as output scale;
//    Changes: the kernel dequantises K/V and folds the K and V scales);
//  * live per-query lengths, zero meaning a dead row
//    ("DFlash2 E4M3 attention with FP32 state", intro paragraph 3);
//  * runtime page stride / block table addressing (same page, paragraph 5;
//    "Qualify calibrated E4M3 and disk PLE with QSA DCP2", commit on packed
//    pages: kernels honour the block stride);
//  * four-token microblocks with 32-bit per-row visibility masks, mask-0
//    padding entries on the null block (same page, commit "grouped page4
//    null-block padding").
//  * the split-KV partition scheme (FP32 unnormalised numerators, separate
//    max and sum, then a combine) of "DFlash2 E4M3 attention with FP32 state",
//    intro paragraph 4 -- written here in FP64 as orc_attention_split.
//
// E4M3 is the OCP "E4M3FN" format: 1 sign, 4 exponent (bias 7), 3 mantissa
// bits, no infinities, 0x7F/0xFF are NaN, largest finite magnitude 448.
// The oracle reads only the bytes of visible tokens, so poisoned bytes of
// padding or unused page slots never reach it.
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off -fno-fast-math -shared -fPIC -pthread
//
// Parity pins: every function here is pinned by CPU tests (decode tables
// against the format definition and torch's converters; attention against an
// independent exact-rational evaluation on tiny inputs, closed forms and
// invariants).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>
#include <algorithm>

#define ORC_API extern "C"

typedef struct {
  int mode;  // 0 = dense paged, 1 = sparse four-token microblocks
  int B, q, Hq, Hkv, D;
  int page_size;                 // tokens per physical block (4 in sparse mode)
  const uint16_t* q_bits;        // [B][q][Hq][D] IEEE binary16 bit patterns
  const uint8_t* k_cache;        // E4M3 bytes
  const uint8_t* v_cache;
  int64_t k_stride[3];           // byte strides: block, token, head
  int64_t v_stride[3];
  const int32_t* block_table;    // dense: [B][bt_stride]
  int64_t bt_stride;
  const int32_t* row_len;        // dense: [B][q], 0 = dead row
  const int32_t* entry_tbl;      // sparse: [B][entry_stride]
  const uint32_t* entry_mask;    // sparse: [B][entry_stride]
  const int32_t* n_entries;      // sparse: [B]
  int64_t entry_stride;
  double softmax_scale, k_scale, v_scale;
  int kv_format;  // cache format: 0 = E4M3 (E4M3FN) bytes, 1 = E5M2 bytes, 2 = bf16 pairs
  const uint32_t* entry_mask_hi; // sparse rows 8..15: [B][entry_stride], NULL for q <= 8
} orc_problem;

// ORC_PLANT (compile-time, default 0 = none) plants one plausible mistake;
// only the test that checks that the pins catch such mistakes builds those
// variants.
#ifndef ORC_PLANT
#define ORC_PLANT 0
#endif

// ---------------------------------------------------------------- decoders

// E4M3 byte -> value, straight from the format definition.
ORC_API double orc_e4m3(uint8_t b) {
  const int s = b >> 7;
  const int e = (b >> 3) & 15;
  const int m = b & 7;
  if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
  double v;
  if (e == 0)
    v = std::ldexp((double)m, -9);                 // m/8 * 2^(1-7)
  else
    v = std::ldexp(1.0 + (double)m / 8.0, e - 7);
#if ORC_PLANT == 1
  if (e == 0) v = std::ldexp((double)m, -10);  // planted: wrong subnormal exponent
#endif
  return s ? -v : v;
}

ORC_API void orc_e4m3_table(double* out256) {
  for (int i = 0; i < 256; ++i) out256[i] = orc_e4m3((uint8_t)i);
}

// E5M2 byte -> value, from the format definition: 1 sign, 5 exponent bits
// (bias 15), 2 mantissa bits, subnormals, infinities (exponent 31, mantissa
// 0) and NaN (exponent 31, mantissa != 0) as in IEEE binary16, of which it
// is the upper byte -- the legacy cache format of "DFlash2 E4M3 attention
// with FP32 state" (the E5M2 kernels the page replaces).
ORC_API double orc_e5m2(uint8_t b) {
  const int s = b >> 7;
  const int e = (b >> 2) & 31;
  const int m = b & 3;
  double v;
  if (e == 31)
    v = m ? std::numeric_limits<double>::quiet_NaN() : std::numeric_limits<double>::infinity();
  else if (e == 0)
    v = std::ldexp((double)m, -16);  // m/4 * 2^(1-15)
  else
    v = std::ldexp(1.0 + (double)m / 4.0, e - 15);
#if ORC_PLANT == 14
  if (e != 0 && e != 31) v = std::ldexp(1.0 + (double)m / 4.0, e - 16);  // planted: bias 16
#endif
  return s ? -v : v;
}

ORC_API void orc_e5m2_table(double* out256) {
  for (int i = 0; i < 256; ++i) out256[i] = orc_e5m2((uint8_t)i);
}

// The problem's cache byte decode.
ORC_API double orc_bf16(uint16_t h);

// Element d of a K or V cache row: one E4M3 or E5M2 byte, or (kv_format 2) a
// little-endian bf16 pair.
static inline double dec(const orc_problem* p, const uint8_t* row, int d) {
  if (p->kv_format == 2) return orc_bf16((uint16_t)(row[2 * d] | (row[2 * d + 1] << 8)));
  return p->kv_format == 1 ? orc_e5m2(row[d]) : orc_e4m3(row[d]);
}

// IEEE binary16 bits -> value.
ORC_API double orc_f16(uint16_t h) {
  const int s = h >> 15;
  const int e = (h >> 10) & 31;
  const int m = h & 1023;
  double v;
  if (e == 31)
    v = m ? std::numeric_limits<double>::quiet_NaN() : std::numeric_limits<double>::infinity();
  else if (e == 0)
    v = std::ldexp((double)m, -24);
  else
    v = std::ldexp(1.0 + (double)m / 1024.0, e - 15);
  return s ? -v : v;
}

// ---------------------------------------------------------------- encoder

// Value -> E4M3 byte: the nearest representable value, ties to the code with
// an even mantissa (round to nearest, ties to even), magnitudes beyond the
// largest finite value 448 saturate to it (infinities included), the sign of
// zero and of values that round to zero is kept, NaN gives 0x7F.  The
// nearest value is found by comparing against all 127 finite magnitudes
// (exact in double: every candidate has at most 4 significant bits and the
// input has 24).  This is the cache write's rounding ("Qwen4Exp: fp8_e4m3
// main KV cache on the QSA path", PR description: the cache is written with
// the layer's per-tensor scales, round to nearest even with saturation to
// the finite range being the plain reading of an E4M3FN store).
ORC_API uint8_t orc_e4m3_encode(float y) {
  if (std::isnan(y)) return 0x7F;
  const uint8_t sign = std::signbit(y) ? 0x80 : 0x00;
  if (std::isinf(y)) return (uint8_t)(sign | 0x7E);
  const double a = std::fabs((double)y);
  int best = 0;
  double best_d = std::numeric_limits<double>::infinity();
  for (int c = 0; c < 0x7F; ++c) {  // magnitudes in increasing order, 0x7F is NaN
    const double d = std::fabs(a - orc_e4m3((uint8_t)c));
#if ORC_PLANT == 9
    if (d < best_d || (d == best_d && c > best)) {  // planted: ties away from zero
#else
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
#endif
      best_d = d;
      best = c;
    }
  }
#if ORC_PLANT == 10
  if (a > 448.0) return (uint8_t)(sign | 0x7F);  // planted: overflow to NaN instead of saturating
#endif
  return (uint8_t)(sign | best);
}

// float -> E5M2 byte, from the format definition: the nearest finite code
// (magnitudes 0x00..0x7B in increasing order; 0x7C is infinity, 0x7D..0x7F
// NaN), ties to the code with an even mantissa, so values past the largest
// finite 57344 (infinities included) saturate to it; NaN -> 0x7F.
ORC_API uint8_t orc_e5m2_encode(float y) {
  if (std::isnan(y)) return 0x7F;
  const uint8_t sign = std::signbit(y) ? 0x80 : 0x00;
  const double a = std::fabs((double)y);
  // past the largest finite value the nearest finite code is 57344 (an
  // explicit test: far out, the distances to the two largest codes are
  // equal in double precision and the even-code tie rule would pick 49152)
  if (std::isinf(y) || a >= 57344.0) return (uint8_t)(sign | 0x7B);
  int best = 0;
  double best_d = std::numeric_limits<double>::infinity();
  for (int c = 0; c <= 0x7B; ++c) {
    const double d = std::fabs(a - orc_e5m2((uint8_t)c));
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best_d = d;
      best = c;
    }
  }
  return (uint8_t)(sign | best);
}

// bfloat16 bits -> value (the upper half of a binary32).
ORC_API double orc_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// Cache write: for every new token n with slot = slot_mapping[n] >= 0, block
// slot / page_size, offset slot % page_size, and every KV head h and d < D:
//   k_cache[block, offset, h, d] = encode(fp32(k[n][h][d]) / fp32(k_scale))
// and the same for V (fp32 division, correctly rounded, then the encoder
// above).  Inputs are binary16 (dtype 0) or bfloat16 (dtype 1) bit patterns
// with element strides (token, head); caches use byte strides (block, token,
// head).  Slots whose block is outside [0, num_blocks) are skipped and
// counted in the return value.
ORC_API int orc_cache_write_fmt(int N, int Hkv, int D, int page_size, int num_blocks, int dtype,
                                const uint16_t* k, const uint16_t* v, const int64_t* k_es, const int64_t* v_es,
                                const int64_t* slot_mapping, float k_scale, float v_scale,
                                uint8_t* k_cache, uint8_t* v_cache, const int64_t* k_bs, const int64_t* v_bs,
                                int kv_format) {
  uint8_t (*enc)(float) = kv_format == 1 ? orc_e5m2_encode : orc_e4m3_encode;
  int bad = 0;
  for (int n = 0; n < N; ++n) {
    const int64_t slot = slot_mapping[n];
    if (slot < 0) continue;
    const int64_t blk = slot / page_size;
#if ORC_PLANT == 11
    const int64_t off = slot % page_size + 1;  // planted: slot offset off by one
#else
    const int64_t off = slot % page_size;
#endif
    if (blk >= num_blocks || off >= page_size) {
      ++bad;
      continue;
    }
    for (int h = 0; h < Hkv; ++h)
      for (int d = 0; d < D; ++d) {
        const uint16_t kb = k[n * k_es[0] + h * k_es[1] + d];
        const uint16_t vb = v[n * v_es[0] + h * v_es[1] + d];
        const float kx = (float)(dtype == 0 ? orc_f16(kb) : orc_bf16(kb));
        const float vx = (float)(dtype == 0 ? orc_f16(vb) : orc_bf16(vb));
        k_cache[blk * k_bs[0] + off * k_bs[1] + h * k_bs[2] + d] = enc(kx / k_scale);
        v_cache[blk * v_bs[0] + off * v_bs[1] + h * v_bs[2] + d] = enc(vx / v_scale);
      }
  }
  return bad;
}

// The E4M3 cache write (kv_format 0).
ORC_API int orc_cache_write(int N, int Hkv, int D, int page_size, int num_blocks, int dtype,
                            const uint16_t* k, const uint16_t* v, const int64_t* k_es, const int64_t* v_es,
                            const int64_t* slot_mapping, float k_scale, float v_scale,
                            uint8_t* k_cache, uint8_t* v_cache, const int64_t* k_bs, const int64_t* v_bs) {
  return orc_cache_write_fmt(N, Hkv, D, page_size, num_blocks, dtype, k, v, k_es, v_es, slot_mapping, k_scale,
                             v_scale, k_cache, v_cache, k_bs, v_bs, 0);
}

// ------------------------------------------------------- visible token set

struct Tok { int64_t k_off, v_off; };

// Tokens query row r of request b sees, for KV head g, in sequence order.
static void visible(const orc_problem* p, int b, int r, int g, std::vector<Tok>& out) {
  out.clear();
  if (p->mode == 0) {
    int n = p->row_len[(int64_t)b * p->q + r];
#if ORC_PLANT == 4
    if (n > 0) n -= 1;  // planted: off-by-one causal limit
#endif
    for (int j = 0; j < n; ++j) {
      const int64_t blk = p->block_table[(int64_t)b * p->bt_stride + j / p->page_size];
      const int64_t slot = j % p->page_size;
      out.push_back({blk * p->k_stride[0] + slot * p->k_stride[1] + (int64_t)g * p->k_stride[2],
                     blk * p->v_stride[0] + slot * p->v_stride[1] + (int64_t)g * p->v_stride[2]});
    }
  } else {
    const int ne = p->n_entries[b];
    for (int e = 0; e < ne; ++e) {
      const int64_t blk = p->entry_tbl[(int64_t)b * p->entry_stride + e];
      // rows 0..7: bit 4r + t of the first word; rows 8..15: bit 4(r - 8) + t
      // of the second
      const uint32_t msk = r < 8 ? p->entry_mask[(int64_t)b * p->entry_stride + e]
                                 : p->entry_mask_hi[(int64_t)b * p->entry_stride + e];
        for (int t = 0; t < 4; ++t) {
#if ORC_PLANT == 6
        if ((msk >> (8 * t + (r & 7))) & 1u) {  // planted: transposed mask bit layout
#else
        if ((msk >> (4 * (r & 7) + t)) & 1u) {
#endif
          out.push_back({blk * p->k_stride[0] + (int64_t)t * p->k_stride[1] + (int64_t)g * p->k_stride[2],
                         blk * p->v_stride[0] + (int64_t)t * p->v_stride[1] + (int64_t)g * p->v_stride[2]});
        }
      }
    }
  }
}

// ----------------------------------------------------------- one row-head

// Logits of query (b, r, h) over its visible tokens.
static void logits(const orc_problem* p, int b, int r, int h, const std::vector<Tok>& toks,
                   std::vector<double>& z) {
  const int D = p->D;
  const uint16_t* qv = p->q_bits + (((int64_t)b * p->q + r) * p->Hq + h) * D;
  std::vector<double> qd(D);
  for (int d = 0; d < D; ++d) qd[d] = orc_f16(qv[d]);
  z.resize(toks.size());
  for (size_t j = 0; j < toks.size(); ++j) {
    const uint8_t* kb = p->k_cache + toks[j].k_off;
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += qd[d] * dec(p, kb, d);
    double sc = p->softmax_scale * p->k_scale;
#if ORC_PLANT == 2
    sc = p->softmax_scale;  // planted: k_scale dropped
#endif
    z[j] = sc * dot;
  }
}

static int group_of(const orc_problem* p, int h) {
  const int G = p->Hq / p->Hkv;
#if ORC_PLANT == 3
  return h % p->Hkv;  // planted: interleaved head grouping
#endif
  return h / G;
}

// Softmax weights of query (b, r, h); returns the visible count.
ORC_API int orc_row_weights(const orc_problem* p, int b, int r, int h, double* w, int cap) {
  std::vector<Tok> toks;
  visible(p, b, r, group_of(p, h), toks);
  std::vector<double> z;
  logits(p, b, r, h, toks, z);
  const int n = (int)toks.size();
  if (n == 0) return 0;
  double M = -std::numeric_limits<double>::infinity();
  for (double v : z) M = std::max(M, v);
  double S = 0.0;
  for (double v : z) S += std::exp(v - M);
  for (int j = 0; j < n && j < cap; ++j) w[j] = std::exp(z[j] - M) / S;
  return n;
}

// Condition of each output element: v_scale * sum_j w_j |dec(V_j[d])|, the
// magnitude an FP32 evaluation's rounding errors scale with (a forward error
// bound for a weighted sum is proportional to the sum of |terms|).
static void row_head_abs(const orc_problem* p, int b, int r, int h, double* out) {
  const int D = p->D;
  std::vector<Tok> toks;
  visible(p, b, r, group_of(p, h), toks);
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (toks.empty()) return;
  std::vector<double> z;
  logits(p, b, r, h, toks, z);
  double M = -std::numeric_limits<double>::infinity();
  for (double v : z) M = std::max(M, v);
  double S = 0.0;
  for (double v : z) S += std::exp(v - M);
  std::vector<double> acc(D, 0.0);
  for (size_t j = 0; j < toks.size(); ++j) {
    const double w = std::exp(z[j] - M) / S;
    const uint8_t* vb = p->v_cache + toks[j].v_off;
    for (int d = 0; d < D; ++d) acc[d] += w * std::fabs(dec(p, vb, d));
  }
  for (int d = 0; d < D; ++d) out[d] = std::fabs(p->v_scale) * acc[d];
}

// Logit condition of each output element:
//   sum_j w_j a_j |v_scale dec(V_j[d]) - out[d]|,
//   a_j = |softmax_scale k_scale| sum_d' |q[d'] dec(K_j[d'])|.
// If every logit z_j carries an absolute error |dz_j| <= eps a_j (the a
// priori bound of a dot product evaluated in floating point is a small
// multiple of the unit roundoff times the sum of |products|), the softmax
// weights move by dw_j = w_j (dz_j - sum_k w_k dz_k), so the output moves by
// sum_j w_j dz_j (v_j - out) to first order: at most eps times this value.
static void row_head_logit_cond(const orc_problem* p, int b, int r, int h, double* out) {
  const int D = p->D;
  std::vector<Tok> toks;
  visible(p, b, r, group_of(p, h), toks);
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (toks.empty()) return;
  std::vector<double> z;
  logits(p, b, r, h, toks, z);
  double M = -std::numeric_limits<double>::infinity();
  for (double v : z) M = std::max(M, v);
  double S = 0.0;
  for (double v : z) S += std::exp(v - M);
  const uint16_t* qv = p->q_bits + (((int64_t)b * p->q + r) * p->Hq + h) * D;
  const double sc = std::fabs(p->softmax_scale * p->k_scale);
  std::vector<double> w(toks.size()), a(toks.size()), o(D, 0.0);
  for (size_t j = 0; j < toks.size(); ++j) {
    w[j] = std::exp(z[j] - M) / S;
    const uint8_t* kb = p->k_cache + toks[j].k_off;
    double s = 0.0;
    for (int d = 0; d < D; ++d) s += std::fabs(orc_f16(qv[d]) * dec(p, kb, d));
    a[j] = sc * s;
    const uint8_t* vb = p->v_cache + toks[j].v_off;
    for (int d = 0; d < D; ++d) o[d] += w[j] * p->v_scale * dec(p, vb, d);
  }
  for (size_t j = 0; j < toks.size(); ++j) {
    const uint8_t* vb = p->v_cache + toks[j].v_off;
    for (int d = 0; d < D; ++d) out[d] += w[j] * a[j] * std::fabs(p->v_scale * dec(p, vb, d) - o[d]);
  }
}

static void row_head(const orc_problem* p, int b, int r, int h, double* out) {
  const int D = p->D;
  std::vector<Tok> toks;
  visible(p, b, r, group_of(p, h), toks);
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (toks.empty()) return;  // dead row: +0.0
  std::vector<double> z;
  logits(p, b, r, h, toks, z);
  double M = -std::numeric_limits<double>::infinity();
  for (double v : z) M = std::max(M, v);
  double S = 0.0;
  for (double v : z) S += std::exp(v - M);
#if ORC_PLANT == 8
  S = 1.0 + 0.0 * S;  // planted: weights left unnormalised
#endif
  std::vector<double> acc(D, 0.0);
  for (size_t j = 0; j < toks.size(); ++j) {
    const double w = std::exp(z[j] - M) / S;
#if ORC_PLANT == 7
    const uint8_t* vb = p->k_cache + toks[j].k_off;  // planted: K read in place of V
#else
    const uint8_t* vb = p->v_cache + toks[j].v_off;
#endif
    for (int d = 0; d < D; ++d) acc[d] += w * dec(p, vb, d);
  }
  double vs = p->v_scale;
#if ORC_PLANT == 5
  vs = 1.0;  // planted: v_scale dropped
#endif
  for (int d = 0; d < D; ++d) out[d] = vs * acc[d];
}

// Split-KV in FP64: the visible sequence is cut into num_splits contiguous
// partitions; each stores an unnormalised numerator, its own max and its own
// sum; the combine rescales every partition to the global max and divides by
// the rescaled total.  Empty partitions hold (max=-inf, sum=0) and are skipped.
static void row_head_split(const orc_problem* p, int b, int r, int h, int S_, double* out) {
  const int D = p->D;
  std::vector<Tok> toks;
  visible(p, b, r, group_of(p, h), toks);
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  const int n = (int)toks.size();
  if (n == 0) return;
  std::vector<double> z;
  logits(p, b, r, h, toks, z);
  const int chunk = (n + S_ - 1) / S_;
  std::vector<double> m(S_, -std::numeric_limits<double>::infinity()), l(S_, 0.0);
  std::vector<double> num((size_t)S_ * D, 0.0);
  for (int s = 0; s < S_; ++s) {
    const int j0 = s * chunk, j1 = std::min(n, j0 + chunk);
    for (int j = j0; j < j1; ++j) m[s] = std::max(m[s], z[j]);
    for (int j = j0; j < j1; ++j) {
      const double e = std::exp(z[j] - m[s]);
      l[s] += e;
      const uint8_t* vb = p->v_cache + toks[j].v_off;
      for (int d = 0; d < D; ++d) num[(size_t)s * D + d] += e * dec(p, vb, d);
    }
  }
  double M = -std::numeric_limits<double>::infinity();
  for (int s = 0; s < S_; ++s) M = std::max(M, m[s]);
  double L = 0.0;
  std::vector<double> acc(D, 0.0);
  for (int s = 0; s < S_; ++s) {
    if (l[s] == 0.0) continue;
    const double w = std::exp(m[s] - M);
    L += w * l[s];
    for (int d = 0; d < D; ++d) acc[d] += w * num[(size_t)s * D + d];
  }
  for (int d = 0; d < D; ++d) out[d] = p->v_scale * acc[d] / L;
}

// ------------------------------------------------------------- drivers

static int check(const orc_problem* p) {
  if (!p || p->B < 0 || p->q < 1 || p->Hq < 1 || p->Hkv < 1 || p->D < 1) return -1;
  if (p->Hq % p->Hkv) return -1;
  if (p->mode == 1 && (p->q > 16 || (p->q > 8 && !p->entry_mask_hi))) return -1;
  if (p->kv_format < 0 || p->kv_format > 2) return -1;
  return 0;
}

template <class F>
static void parallel_items(int64_t n, int nthreads, F f) {
  if (nthreads <= 1 || n < 2) {
    for (int64_t i = 0; i < n; ++i) f(i);
    return;
  }
  nthreads = (int)std::min<int64_t>(nthreads, n);
  std::vector<std::thread> th;
  for (int t = 0; t < nthreads; ++t)
    th.emplace_back([=]() {
      for (int64_t i = t; i < n; i += nthreads) f(i);
    });
  for (auto& x : th) x.join();
}

// out: [B][q][Hq][D] doubles.
ORC_API int orc_attention(const orc_problem* p, double* out, int nthreads) {
  if (check(p)) return -1;
  const int64_t n = (int64_t)p->B * p->q * p->Hq;
  parallel_items(n, nthreads, [&](int64_t i) {
    const int h = (int)(i % p->Hq);
    const int r = (int)((i / p->Hq) % p->q);
    const int b = (int)(i / ((int64_t)p->Hq * p->q));
    row_head(p, b, r, h, out + i * p->D);
  });
  return 0;
}

// Only the listed (b, r, h) triples; out: [n_items][D].
ORC_API int orc_attention_items(const orc_problem* p, const int32_t* items, int n_items, double* out,
                        int nthreads) {
  if (check(p)) return -1;
  for (int i = 0; i < n_items; ++i) {
    const int b = items[3 * i], r = items[3 * i + 1], h = items[3 * i + 2];
    if (b < 0 || b >= p->B || r < 0 || r >= p->q || h < 0 || h >= p->Hq) return -1;
  }
  parallel_items(n_items, nthreads, [&](int64_t i) {
    row_head(p, items[3 * i], items[3 * i + 1], items[3 * i + 2], out + i * p->D);
  });
  return 0;
}

// out: [B][q][Hq][D] doubles, v_scale * sum_j w_j |dec(V_j[d])|.
ORC_API int orc_attention_abs(const orc_problem* p, double* out, int nthreads) {
  if (check(p)) return -1;
  const int64_t n = (int64_t)p->B * p->q * p->Hq;
  parallel_items(n, nthreads, [&](int64_t i) {
    const int h = (int)(i % p->Hq);
    const int r = (int)((i / p->Hq) % p->q);
    const int b = (int)(i / ((int64_t)p->Hq * p->q));
    row_head_abs(p, b, r, h, out + i * p->D);
  });
  return 0;
}

// out: [B][q][Hq][D] doubles, the logit condition of row_head_logit_cond.
ORC_API int orc_attention_logit_cond(const orc_problem* p, double* out, int nthreads) {
  if (check(p)) return -1;
  const int64_t n = (int64_t)p->B * p->q * p->Hq;
  parallel_items(n, nthreads, [&](int64_t i) {
    const int h = (int)(i % p->Hq);
    const int r = (int)((i / p->Hq) % p->q);
    const int b = (int)(i / ((int64_t)p->Hq * p->q));
    row_head_logit_cond(p, b, r, h, out + i * p->D);
  });
  return 0;
}

ORC_API int orc_attention_split(const orc_problem* p, int num_splits, double* out, int nthreads) {
  if (check(p) || num_splits < 1) return -1;
  const int64_t n = (int64_t)p->B * p->q * p->Hq;
  parallel_items(n, nthreads, [&](int64_t i) {
    const int h = (int)(i % p->Hq);
    const int r = (int)((i / p->Hq) % p->q);
    const int b = (int)(i / ((int64_t)p->Hq * p->q));
    row_head_split(p, b, r, h, num_splits, out + i * p->D);
  });
  return 0;
}

// ---------------------------------------------------- context-parallel merge

// Output and base-2 log-sum-exp of every query vector: out as orc_attention,
// lse = log2(sum_j 2^(log2(e) z_j)) over the visible tokens (-inf for a dead
// row).  A rank that holds a shard of the context emits this pair; merging
// the ranks' pairs gives the attention over the union ("Qualify calibrated
// E4M3 and disk PLE with QSA DCP2", commit exposing base-2 LSE and FP32
// partial output for cross-rank merging).
static void row_head_lse(const orc_problem* p, int b, int r, int h, double* out, double* lse) {
  row_head(p, b, r, h, out);
  std::vector<Tok> toks;
  visible(p, b, r, group_of(p, h), toks);
  if (toks.empty()) {
    *lse = -std::numeric_limits<double>::infinity();
    return;
  }
  std::vector<double> z;
  logits(p, b, r, h, toks, z);
  double M = -std::numeric_limits<double>::infinity();
  for (double v : z) M = std::max(M, v);
  double S = 0.0;
  for (double v : z) S += std::exp(v - M);
#if ORC_PLANT == 13
  S = 1.0;  // planted: the sum dropped from the log-sum-exp
#endif
  *lse = (M + std::log(S)) / std::log(2.0);
}

ORC_API int orc_attention_lse(const orc_problem* p, double* out, double* lse, int nthreads) {
  if (check(p)) return -1;
  const int64_t n = (int64_t)p->B * p->q * p->Hq;
  parallel_items(n, nthreads, [&](int64_t i) {
    const int h = (int)(i % p->Hq);
    const int r = (int)((i / p->Hq) % p->q);
    const int b = (int)(i / ((int64_t)p->Hq * p->q));
    row_head_lse(p, b, r, h, out + i * p->D, lse + i);
  });
  return 0;
}

// Merge R ranks' (out, lse) pairs of n vectors: L = log2(sum_r 2^lse_r),
// merged = sum_r 2^(lse_r - L) out_r (the softmax over the union of the
// shards, written per rank); a vector that no rank sees gets 0 and -inf.
ORC_API void orc_merge(int R, int64_t n, int D, const double* out, const double* lse, double* merged,
                       double* lse_merged) {
  for (int64_t i = 0; i < n; ++i) {
    double L = -std::numeric_limits<double>::infinity();
    for (int r = 0; r < R; ++r) L = std::max(L, lse[(int64_t)r * n + i]);
    double* m = merged + i * D;
    for (int d = 0; d < D; ++d) m[d] = 0.0;
    if (L == -std::numeric_limits<double>::infinity()) {
      lse_merged[i] = L;
      continue;
    }
    double W = 0.0;
    for (int r = 0; r < R; ++r) {
#if ORC_PLANT == 12
      W += std::exp(lse[(int64_t)r * n + i] - L);  // planted: natural base for base-2 LSEs
#else
      W += std::exp2(lse[(int64_t)r * n + i] - L);
#endif
    }
    for (int r = 0; r < R; ++r) {
#if ORC_PLANT == 12
      const double w = std::exp(lse[(int64_t)r * n + i] - L) / W;
#else
      const double w = std::exp2(lse[(int64_t)r * n + i] - L) / W;
#endif
      if (w == 0.0) continue;
      const double* o = out + ((int64_t)r * n + i) * D;
      for (int d = 0; d < D; ++d) m[d] += w * o[d];
    }
    lse_merged[i] = L + std::log2(W);
  }
}

ORC_API int orc_abi_version(void) { return 1; }

