// Tensor-core split kernel (tcgen05 + TMEM) for up to 64 query vectors per
// (request, KV head): the grouped-query rows of a verify or decode step.
// This header holds the kernel template and its helpers; split_tc.cu
// instantiates the variant whose MMA rows are the query vectors and
// split_tc_small.cu the transposed variant for small groups (SM).
//
// Per CTA: one partition (a contiguous token range, or entry range in the
// sparse microblock mode) of one (request, KV head, row chunk).  Warp roles:
//   warps 13, 14 producers (one thread each, K and V): bulk copies
//                (cp.async.bulk) of a tile's E4M3 K (V) rows from the paged
//                cache into that stream's raw shared-memory ring, completion
//                counted in bytes on an mbarrier; runs of tokens contiguous
//                in a page move as one copy, tokens no query row may see are
//                never copied, and the page walk of the next tile is loaded
//                while the current one waits for its stage;
//   warps 4-7    K decoders and
//   warps 8-11   V decoders: take a raw tile into registers and hand the raw
//                stage straight back, then convert E4M3 -> exact fp16 with the
//                hardware e4m3x2 -> f16x2 conversion into swizzled operand
//                tiles of the stream's ring (tokens that were not copied
//                become zeros).  K and V have separate rings because different
//                MMAs free them: a K pair once its QK is done, a V tile once
//                its PV is;
//   warp 12      TMEM allocation and UMMA issue (one thread), issuing
//                whichever of the next QK (per pair) and the next PV (per
//                tile) is ready;
//   warps 0-3    softmax: read S from TMEM, online softmax with FP32 state,
//                write P = P_hi + P_lo (two fp16 halves) back to TMEM in place
//                of S, rescale O when the running max moves, epilogue; Q is
//                staged by warps 0-11 after the setup barrier, so the
//                producers start without waiting for it.
// Per pair of 64-token tiles (2m, 2m+1):
//   QK:  S[64 x 128] = Q[64 x D] . [K(2m); K(2m+1)]^T  (one UMMA chain, M=64,
//        N=128: A = Q resident in shared memory, B = the pair's K tiles,
//        interleaved per column block, both K-major; N=64 for a last single
//        tile).  Query vector 16w+j (j < 16) lands in TMEM lane 32w+j.
// Per tile i:
//   PV:  O[128 x D] += P[128 x 64] . V[64 x D]  (M=128, A from TMEM, B = V
//        tile MN-major).  P_hi of vector 16w+j sits in lane 32w+j and its
//        P_lo twin in lane 32w+16+j, so one MMA accumulates both halves of
//        the probability split; the epilogue adds the two accumulator rows.
// TMEM: four S/P buffers of 64 columns (tile i uses buffer i % 4; P(i)
// overwrites S(i), hi in the lanes the M=64 QK writes, lo in the 16 lanes
// above) and O.  With four buffers the QK of pair m+2 is the first to wait
// for the PVs of pair m, so QK, softmax and PV of neighbouring tiles overlap.
// The hi/lo split keeps probabilities to ~22 bits ("compensated
// probabilities"); the FP32 partition numerator, max and sum follow the FP32
// state contract ("DFlash2 E4M3 attention with FP32 state", intro paragraph
// 4).  The running max is an integer (base-2 units) that only moves when a
// tile exceeds it by more than kTau, so P <= 2^kTau always fits fp16 and the
// rescale factor of O is an exact power of two.  The softmax first forms the
// exponents against the running max and takes a slow path (row maxima,
// possibly a rescale of O after the previous tile's PV) only when some
// exponent exceeds kTau, which in practice is a row's first visible tile.
//
// Every wait is bounded.  A wait that gives up sets a CTA-wide abort flag and
// FP8KV_STATUS_TIMEOUT; every role then stops issuing work, the producers wait
// for the bulk copies they already issued and the MMA thread for the UMMAs it
// already committed (both always complete), and only then is TMEM freed and
// the CTA allowed to exit (results of that launch are invalid).
//
// Non-finite V codes (E4M3 NaN, E5M2 infinities and NaNs): the P.V product
// runs over every token a tile copied, including tokens some rows do not see
// (their P is exactly 0), and 0 * NaN would reach those rows.  The V decoders
// therefore write such codes as 0 and flag the CTA; after the main loop a
// flagged CTA re-reads its partition's V bytes and sets the numerator element
// (vector, column) to NaN or +-infinity for exactly the vectors that see the
// token, as the exact softmax has it.  Unflagged CTAs (the normal case) only
// pay the byte test in the V decoders.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"
#include "new_tokens.cuh"
#include "tc_ptx.cuh"

namespace fp8kv {
namespace {

using namespace tc;

constexpr int kT = 64;              // tokens per tile (16 microblocks in sparse mode)
constexpr int kRows = 64;           // query vectors per CTA
constexpr int kE = kT / 4;          // sparse entries per tile
constexpr int kSoftmaxWarps = 4;
constexpr int kDecWarps = 4;        // per stream
constexpr int kDecThreads = 32 * kDecWarps;
constexpr int kKDecWarp0 = kSoftmaxWarps;              // 4
constexpr int kVDecWarp0 = kKDecWarp0 + kDecWarps;     // 8
constexpr int kMmaWarp = kVDecWarp0 + kDecWarps;       // 12
constexpr int kProdWarp = kMmaWarp + 1;                // 13 (K), 14 (V)
constexpr int kThreads = 32 * (kProdWarp + 2);        // 480
static_assert(kThreads == kTcThreads && kT == kTcTileTokens, "launch shape");
constexpr float kTau = 8.0f;        // lazy-rescale threshold (base-2 units)
// Probabilities go to the MMAs as two fp16 halves, P_hi = fp16(p') and
// P_lo = fp16((p' - P_hi) * 2^kLoBits), with p' = 2^kPShift * p: p' <= 2^(kTau +
// kPShift) = 2^15 still fits fp16, and neither half turns subnormal until p
// is 2^-21 of the running maximum (without the two factors a row whose
// maximum is an outlier far above its other tokens loses the low half of
// those tokens' probabilities).  P_lo accumulates in rows (or columns) of its
// own, so the epilogue undoes both factors exactly: O = (O_hi + O_lo *
// 2^-kLoBits) * 2^-kPShift, and the row sum is divided by 2^kPShift.
constexpr float kPShift = 7.0f;
constexpr float kLoScale = 2048.0f;        // 2^kLoBits
constexpr float kInvLoScale = 1.0f / 2048.0f;
constexpr float kInvPShift = 1.0f / 128.0f;
constexpr uint32_t kWaitLimit = 1u << 20;      // polls per wait (product path)
constexpr uint32_t kTestWaitLimit = 1u << 12;  // polls per wait under FP8KV_TEST_STALL_PIPELINE
constexpr uint32_t kDrainLimit = 1u << 20;     // polls for issued copies / UMMAs to complete
constexpr int kMaxStages = 4;
constexpr int kSBuf = 4;            // S/P buffers in TMEM (tile i uses buffer i % 4)

// SM (small-group kernel): the query vectors of a CTA (at most kN) form the N
// dimension of a transposed QK, S^T = K . Q^T (M = 128 tokens of a tile
// pair), and P^T (hi | lo, kNP columns) goes to shared memory as the B operand
// of O^T += V^T . P^T (M = 128 head-dim columns per block).
constexpr int kN = 16;
constexpr int kNP = 2 * kN;

template <int D, bool SM>
struct Cfg {
  static constexpr int kKStages = (D == 256) ? 2 : 4;      // fp16 K operand stages (pairs of tiles)
  static constexpr int kVStages = (D == 256) ? 2 : 4;      // fp16 V operand stages
  static constexpr int kRaw = (D == 256) ? 2 : 4;          // raw E4M3 stages per stream
  static constexpr int kQRows = SM ? kN : kRows;           // query vectors staged
  static constexpr int kQBytes = kQRows * D * 2;           // Q tile (fp16, swizzled)
  static constexpr int kOpBytes = kT * D * 2;              // one K or V operand tile (fp16)
  static constexpr int kRawBytes = kT * D;                 // raw K or V rows of a tile
  static constexpr int kPBytes = SM ? kT * kNP * 2 : 0;    // SM: one tile's P^T (64-byte rows, 64B swizzle)
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kKStages * kOpBytes;
  static constexpr int kOffRawK = kOffV + kVStages * kOpBytes;
  static constexpr int kOffRawV = kOffRawK + kRaw * kRawBytes;
  static constexpr int kOffP = kOffRawV + kRaw * kRawBytes;
  static constexpr int kOffRed = kOffP + kSBuf * kPBytes;   // SM: per-warp column maxima and sums
  static constexpr int kRedBytes = SM ? 2 * kSoftmaxWarps * kN * 4 : 0;
  static constexpr int kOffMeta = kOffRed + kRedBytes;
  static constexpr int kMetaBytes = 1024;
  static constexpr int kSmem = kOffMeta + kMetaBytes + 1024;  // + alignment slack
  // SM: the QK of a pair accumulates into kQKParts separate S^T buffers (an
  // equal share of the D/16 K16 steps each), added by the softmax with TwoSum
  static constexpr int kQKParts = SM ? 8 : 1;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;  // M64: kSBuf x 64 columns (P(i) overwrites S(i)); SM: 2 pairs x kQKParts x kN
  // M64: O at kColO (D columns).  SM: the PV of pair j goes to O^T region
  // j % 2 (D/128 blocks x kNP columns each, written fresh by the pair's first
  // MMA); the softmax warps drain each region into the compensated master sum
  // at kColM (per block: kN columns hi, then kN columns lo).
  static constexpr uint32_t kColO = SM ? 2 * kQKParts * kN : 256;
  static constexpr uint32_t kColM = kColO + 2 * (D / 128) * kNP;
  static_assert(kKStages <= kMaxStages && kVStages <= kMaxStages && kRaw <= kMaxStages, "ring sizes");
  static_assert(kKStages % 2 == 0, "the K ring holds pairs of tiles");
  static_assert(kQBytes % 1024 == 0 && kOffP % 1024 == 0, "operand alignment");
  static_assert(!SM || kColM + (D / 128) * 2 * kN <= kTmemCols, "TMEM columns");
  static_assert(kSmem <= 232448, "shared memory");
};

struct Meta {
  // K operand ring: one barrier pair per pair slot (a QK reads both tiles)
  uint64_t k_full[kMaxStages / 2], k_empty[kMaxStages / 2];
  // V operand ring: one barrier pair per tile stage (PVs run per tile)
  uint64_t v_full[kMaxStages], v_empty[kMaxStages];
  uint64_t rawk_full[kMaxStages], rawv_full[kMaxStages];
  uint64_t rawk_empty[kMaxStages], rawv_empty[kMaxStages];
  uint64_t s_full[2];                   // per pair of S buffers: the pair's QK done
  uint64_t p_ready[kSBuf];              // per tile buffer: its P written
  uint64_t pv_done[kSBuf];              // per tile buffer: its PV done
  uint32_t tmem;
  uint64_t validk[kMaxStages];          // per raw K stage: tokens that were copied
  uint64_t validv[kMaxStages];          // the same for the raw V stage
  int32_t nrow[kRows];                  // dense: live length of each query vector; sparse: its query row
  uint64_t drain;                       // the MMA thread's final commit (all its UMMAs done)
  uint64_t q_full;                      // the Q tile is in shared memory
  uint64_t s_empty[2];                  // SM: every softmax thread has read the pair's S^T
  int32_t pblk[2][32];                  // dense producers: block ids of the current tile's pages
  uint32_t abort;                       // a wait gave up: every role stops
  uint32_t vbad;                        // a V decoder met a non-finite code
};
static_assert(sizeof(Meta) <= 1024, "meta block");

// ---------------------------------------------------------------- TMEM 16xNb

// (Each wrapper waits for its own access, as those in tc_ptx.cuh do.)
// 16 lanes x 256 bits (8 columns) per repeat; thread t holds, per repeat g,
// lanes (t/4) and (t/4 + 8), columns 8g + 2*(t%4) + {0, 1}, registers in the
// order (lane t/4: col, col+1), (lane t/4+8: col, col+1).
__device__ __forceinline__ void ld_16x256b_x8(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float2 unpack_f16x2(uint32_t v) {
  return __half22float2(*reinterpret_cast<__half2*>(&v));
}

// Both halves of P (hi rows at taddr_hi, lo rows at taddr_lo), one wait.
// 16 lanes x 128 bits (4 columns) per repeat; thread t holds, per repeat g,
// lane (t/4) column 4g + t%4, then lane (t/4 + 8) column 4g + t%4.
__device__ __forceinline__ void st_16x128b_x8_pair(uint32_t taddr_hi, uint32_t taddr_lo, const uint32_t (&h)[16],
                                                   const uint32_t (&l)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x128b.x8.b32 [%0], "
      "{%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17};\n\t"
      "tcgen05.st.sync.aligned.16x128b.x8.b32 [%1], "
      "{%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr_hi),
      "r"(taddr_lo), "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3]), "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7]),
      "r"(h[8]), "r"(h[9]), "r"(h[10]), "r"(h[11]), "r"(h[12]), "r"(h[13]), "r"(h[14]), "r"(h[15]), "r"(l[0]),
      "r"(l[1]), "r"(l[2]), "r"(l[3]), "r"(l[4]), "r"(l[5]), "r"(l[6]), "r"(l[7]), "r"(l[8]), "r"(l[9]),
      "r"(l[10]), "r"(l[11]), "r"(l[12]), "r"(l[13]), "r"(l[14]), "r"(l[15])
      : "memory");
}

// Exact E4M3 -> fp16 for two bytes (hardware conversion): dec(b) itself;
// |dec| <= 448 and the subnormal quantum 2^-9 are both exact in fp16.
// Four E4M3 bytes (little-endian in w) -> two fp16 pairs (bytes 0,1 and 2,3).
template <int FMT>
__device__ __forceinline__ void cvt4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  if (FMT == FP8KV_KV_E5M2) {
    // E5M2 -> fp16 is exact too (the byte is the upper byte of the binary16)
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e5m2x2 %0, a;\n\tcvt.rn.f16x2.e5m2x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
  } else {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
  }
}
template <int FMT>
__device__ __forceinline__ uint4 dec8(uint32_t a, uint32_t b) {
  uint4 r;
  cvt4<FMT>(a, r.x, r.y);
  cvt4<FMT>(b, r.z, r.w);
  return r;
}

// Decoding one raw tile (kT rows of D E4M3 bytes) into a swizzled fp16
// operand tile with the kDecThreads threads of a stream: column block db =
// d/64 holds kT rows of 128 bytes, DBS bytes after the previous block; the
// 16-byte chunk c of row t sits at chunk position c ^ (t % 8).  Thread lt
// always takes raw chunk c = lt % (D/16) of rows lt / (D/16) + k * R (R =
// rows per pass of all threads), so every address is a per-thread base plus
// a compile-time offset.  It runs in two steps: load_raw brings the thread's
// raw chunks into registers (after which the raw stage may be refilled), and
// store_tile converts and stores them.  Rows whose bit in `valid` is clear
// were not copied and become zeros.  zap_nonfinite_tile (the V stream, in
// between) writes non-finite codes as 0 and sets `bad` (see the kernel's
// header).
template <int D>
struct DecShape {
  static constexpr int kChunks = D / 16;           // 16-byte raw chunks per row
  static constexpr int kR = kDecThreads / kChunks; // rows per pass
  static constexpr int kPer = kT / kR;             // chunks per thread
  static_assert(kDecThreads % kChunks == 0 && kT % kR == 0, "decoder shape");
};

template <int D>
__device__ __forceinline__ void load_raw(const uint8_t* raw, uint64_t valid, int lt, uint4 (&w)[DecShape<D>::kPer]) {
  using S = DecShape<D>;
  const int c = lt % S::kChunks, t0 = lt / S::kChunks;
  const uint8_t* src = raw + t0 * D + c * 16;
  const bool full = valid == ~0ull;
#pragma unroll
  for (int k = 0; k < S::kPer; ++k) {
    w[k] = (full || ((valid >> (t0 + k * S::kR)) & 1ull)) ? *reinterpret_cast<const uint4*>(src + k * S::kR * D)
                                                         : make_uint4(0, 0, 0, 0);
  }
}

// One test over the thread's chunks (no branch per chunk: on the V path a
// branch per chunk cost ~4 us of a 128K-token split), then the rare rewrite.
template <int D, int FMT>
__device__ __forceinline__ void zap_nonfinite_tile(uint4 (&w)[DecShape<D>::kPer], bool& bad) {
  using S = DecShape<D>;
  constexpr bool e5 = FMT == FP8KV_KV_E5M2;
  uint32_t any = 0u;
#pragma unroll
  for (int k = 0; k < S::kPer; ++k) any |= nonfinite_codes(w[k], e5);
  if (any != 0u) {
    bad = true;
#pragma unroll
    for (int k = 0; k < S::kPer; ++k) {
      w[k].x = zap_nonfinite(w[k].x, e5);
      w[k].y = zap_nonfinite(w[k].y, e5);
      w[k].z = zap_nonfinite(w[k].z, e5);
      w[k].w = zap_nonfinite(w[k].w, e5);
    }
  }
}

template <int D, int DBS, int FMT>
__device__ __forceinline__ void store_tile(uint8_t* op, const uint4 (&w)[DecShape<D>::kPer], int lt) {
  using S = DecShape<D>;
  const int c = lt % S::kChunks, t0 = lt / S::kChunks;
  const int db = c / 4;
  const int h0 = (c % 4) * 2;  // first of the two 16-byte fp16 chunks
  // alternate the order of the two stores between column blocks so the
  // eight threads of a store phase hit eight different bank groups
  const bool swap = (db & 1) != 0;
  const int first = swap ? h0 + 1 : h0;
  const int second = swap ? h0 : h0 + 1;
  uint8_t* dst = op + db * DBS + t0 * 128;
#pragma unroll
  for (int k = 0; k < S::kPer; ++k) {
    const int sw = (t0 + k * S::kR) & 7;
    uint8_t* row = dst + k * S::kR * 128;
    const uint4 x0 = dec8<FMT>(w[k].x, w[k].y), x1 = dec8<FMT>(w[k].z, w[k].w);
    *reinterpret_cast<uint4*>(row + ((first ^ sw) * 16)) = swap ? x1 : x0;
    *reinterpret_cast<uint4*>(row + ((second ^ sw) * 16)) = swap ? x0 : x1;
  }
}

// The block ids of the pages a dense tile touches, loaded by the producer
// warp one tile ahead of its copies (lane j: page page0 + j), so that the page
// walk does not wait for global loads between a raw stage becoming free and
// its refill.  A tile spans at most 32 pages for page sizes of 3 or more;
// smaller pages load the rest on the spot.
struct TilePages {
  int page0;
  int bid;  // this lane's page
};

// The page of token `tok` (0 <= tok < 2^31).
__device__ __forceinline__ int page_of(const Params& p, int tok) { return div_page(tok, p.page_size, p.page_div); }

__device__ __forceinline__ TilePages fetch_pages(const Params& p, int b, int u0, int u1, int i, int lane) {
  TilePages tp;
  const int tok0 = u0 + i * kT;
  tp.page0 = page_of(p, tok0);
  const int npages = tok0 < u1 ? page_of(p, min(u1, tok0 + kT) - 1) - tp.page0 + 1 : 0;
  tp.bid = lane < npages ? p.block_table[(int64_t)b * p.bt_stride + tp.page0 + lane] : -1;
  return tp;
}

// Dense: issue the bulk copies of one tile's K (or V) rows into a raw stage
// (one per run of tokens contiguous in a page) and return the set of token
// slots that were copied.
// `pblk` holds the tile's block ids (pblk[j]: page page0 + j, j < 32).  Lane
// 0 issues the runs (token rows adjacent in memory: token stride == D).
template <int D>
__device__ __forceinline__ uint64_t copy_rows_dense(const Params& p, const uint8_t* cache, int64_t sb, int64_t st,
                                                    int64_t sh, int b, int g, int u0, int u1, int i, uint8_t* dst,
                                                    uint64_t* bar, int page0, const int32_t* pblk, bool report) {
  uint64_t valid = 0ull;
  int t = 0;
  while (t < kT) {
    const int tok = u0 + i * kT + t;
    if (tok >= u1) break;
    const int page = page_of(p, tok), slot_in = tok - page * p.page_size;
    const int dp = page - page0;
    const int blk = dp < 32 ? pblk[dp] : p.block_table[(int64_t)b * p.bt_stride + page];
    const int run = min(kT - t, min(p.page_size - slot_in, u1 - tok));
    if (blk >= 0 && blk < p.num_kv_blocks) {
      mbar_expect_tx(bar, run * D);
      bulk_g2s(dst + t * D, cache + blk * sb + slot_in * st + g * sh, run * D, bar);
      valid |= ((run == 64) ? ~0ull : ((1ull << run) - 1ull)) << t;
    } else if (report) {
      set_status(p.status, FP8KV_STATUS_BAD_BLOCK);
    }
    t += run;
  }
  return valid;
}

// Gathers of single token rows (dense rows that are not adjacent in memory,
// e.g. several KV heads per slot; sparse microblock tokens), whole warp: lane
// l copies the rows of token slots l and l + 32 with 16-byte cp.async (one
// bulk copy per row costs the bulk-copy engine far more per byte for rows of
// 128 or 256 bytes); the caller then makes every lane arrive on the stage's
// barrier when its copies complete.  Returns the copied slots in every lane.
template <int D>
__device__ __forceinline__ void copy_row_async(uint8_t* dst, const uint8_t* src) {
#pragma unroll
  for (int c = 0; c < D / 16; ++c) cp_async16(dst + c * 16, src + c * 16);
}

template <int D>
__device__ __forceinline__ uint64_t copy_tokens_dense(const Params& p, const uint8_t* cache, int64_t sb, int64_t st,
                                                      int64_t sh, int b, int g, int u0, int u1, int i, uint8_t* dst,
                                                      int page0, const int32_t* pblk, bool report, int lane) {
  uint64_t valid = 0ull;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int t = lane + 32 * half;
    const int tok = u0 + i * kT + t;
    bool ok = false;
    if (tok < u1) {
      const int page = page_of(p, tok);
      const int dp = page - page0;
      const int blk = dp < 32 ? pblk[dp] : p.block_table[(int64_t)b * p.bt_stride + page];
      if (blk >= 0 && blk < p.num_kv_blocks) {
        ok = true;
        copy_row_async<D>(dst + t * D, cache + blk * sb + (tok - page * p.page_size) * st + g * sh);
      } else if (report) {
        set_status(p.status, FP8KV_STATUS_BAD_BLOCK);
      }
    }
    valid |= (uint64_t)__ballot_sync(0xffffffffu, ok) << (32 * half);
  }
  return valid;
}

// Sparse, whole warp: token slot t of the tile is token t % 4 of entry t / 4
// (whose checked mask and microblock id lane t / 4 holds); the slot is
// copied only if some query row attends it.
template <int D>
__device__ __forceinline__ uint64_t copy_tokens_sparse(const uint8_t* cache, int64_t sb, int64_t st, int64_t sh,
                                                       int g, uint8_t* dst, uint32_t mk, int bk, int lane) {
  uint64_t valid = 0ull;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int t = lane + 32 * half;
    const uint32_t m = __shfl_sync(0xffffffffu, mk, t >> 2);
    const int blk = __shfl_sync(0xffffffffu, bk, t >> 2);
    const bool seen = (m & (0x11111111u << (t & 3))) != 0u;
    if (seen) copy_row_async<D>(dst + t * D, cache + blk * sb + (t & 3) * st + g * sh);
    valid |= (uint64_t)__ballot_sync(0xffffffffu, seen) << (32 * half);
  }
  return valid;
}

// A CTA whose V decoders met a non-finite code (written as 0 in the operand)
// restores its effect on the partial numerators: every thread of the CTA
// re-reads the V bytes of the partition's tokens (the copied ones: dense all
// tokens below the longest row, sparse the tokens some row sees), and for
// each non-finite byte (token t, column d) marks every query vector i that
// sees t; then element (i, d) of the numerator becomes NaN (a NaN code, or
// infinities of both signs) or +-infinity.  `scratch` holds one byte per (vector, column):
// bit 0 NaN, bit 1 +inf, bit 2 -inf.
template <int D, int MODE, int FMT>
__device__ __noinline__ void patch_nonfinite_v(const Params& p, uint8_t* scratch, const int32_t* nrow, int b, int g,
                                               int u0, int u1, int RC, int64_t prow) {
  constexpr int kC = D / 16;  // 16-byte chunks per row
  uint32_t* kinds = reinterpret_cast<uint32_t*>(scratch);
  const int tid = threadIdx.x;
  for (int x = tid; x < kRows * D / 4; x += kThreads) kinds[x] = 0u;
  __syncthreads();
  const bool e5 = FMT == FP8KV_KV_E5M2;
  const int n_tok = (MODE == FP8KV_MODE_DENSE) ? (u1 - u0) : 4 * (u1 - u0);
  for (int x = tid; x < n_tok * kC; x += kThreads) {
    const int tu = x / kC, c = x % kC;
    const uint8_t* row;
    int tok = 0, tk = 0;
    uint32_t mk = 0u, mkh = 0u;
    if (MODE == FP8KV_MODE_DENSE) {
      tok = u0 + tu;
      const int blk = p.block_table[(int64_t)b * p.bt_stride + tok / p.page_size];
      if (blk < 0 || blk >= p.num_kv_blocks) continue;
      row = p.v_cache + blk * p.vsb + (tok % p.page_size) * p.vst + g * p.vsh;
    } else {
      const int e = u0 + tu / 4;
      tk = tu % 4;
      mk = p.entry_mask[(int64_t)b * p.entry_stride + e];
      mkh = mask_hi_of(p.entry_mask_hi, p.entry_stride, b, e);
      const int blk = p.entry_tbl[(int64_t)b * p.entry_stride + e];
      if (((mk | mkh) & (0x11111111u << tk)) == 0u || blk < 0 || blk >= p.num_kv_blocks) continue;
      row = p.v_cache + blk * p.vsb + tk * p.vst + g * p.vsh;
    }
    const uint4 w = *reinterpret_cast<const uint4*>(row + c * 16);
    if (nonfinite_codes(w, e5) == 0u) continue;
    const uint32_t wa[4] = {w.x, w.y, w.z, w.w};
    for (int j = 0; j < 16; ++j) {
      const uint32_t byte = (wa[j / 4] >> (8 * (j % 4))) & 0xFFu;
      const bool nf = e5 ? ((byte & 0x7Cu) == 0x7Cu) : ((byte & 0x7Fu) == 0x7Fu);
      if (!nf) continue;
      // E4M3: NaN; E5M2: mantissa bits set -> NaN, else an infinity of the byte's sign
      const uint32_t kind = (!e5 || (byte & 0x3u)) ? 1u : ((byte & 0x80u) ? 4u : 2u);
      const int d = c * 16 + j;
      for (int i = 0; i < RC; ++i) {
        const int n = nrow[i];
        const bool sees = (MODE == FP8KV_MODE_DENSE) ? (tok < n) : (n >= 0 && sparse_bit(mk, mkh, n, tk));
        if (sees) atomicOr(&kinds[i * (D / 4) + d / 4], kind << (8 * (d % 4)));
      }
    }
  }
  __syncthreads();
  for (int x = tid; x < RC * D; x += kThreads) {
    const int i = x / D, d = x % D;
    const uint32_t k = (kinds[i * (D / 4) + d / 4] >> (8 * (d % 4))) & 0xFFu;
    if (k == 0u) continue;
    const float v = ((k & 1u) || (k & 6u) == 6u) ? __uint_as_float(0x7FC00000u)
                                                  : ((k & 2u) ? INFINITY : -INFINITY);
    p.partial[(prow + i) * D + d] = v;
  }
}

// ---------------------------------------------------------------- the kernel

// NL (SM only): the query vectors the softmax handles per token (4, 8 or 16,
// at least the CTA's row chunk); the MMAs always use kN columns.
template <int D, int MODE, int FMT, bool SM, int NL>
__global__ void __launch_bounds__(kThreads, 1) split_tc(const Params p) {
  static_assert(NL == 4 || NL == 8 || NL == kN, "live columns");
  using C = Cfg<D, SM>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Meta& mt = *reinterpret_cast<Meta*>(smem + C::kOffMeta);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.x;
  const int g = blockIdx.y / p.n_row_chunks;
  const int chunk = blockIdx.y % p.n_row_chunks;
  const int b = blockIdx.z;
  const int row0 = chunk * p.row_chunk;
  const int RC = min(p.row_chunk, p.rows - row0);

  // ---------------------------------------------------------- loads
  // Everything the setup reads from global memory is requested up front,
  // so its latencies overlap: the Q tile (warps below the MMA warp, which
  // store it only after the barrier below: the producers need not wait for
  // it), the live length (or query row) of query vector tid, and the row
  // lengths that fix the partition range.
  constexpr int kQThreads = 32 * kMmaWarp;                      // warps 0..11
  constexpr int kQChunks = C::kQRows * (D / 8);                 // 16-byte Q chunks
  constexpr int kQPer = (kQChunks + kQThreads - 1) / kQThreads;
  uint4 qv[kQPer];
  if (tid < kQThreads) {
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int idx = tid + k * kQThreads;
      const int i = idx / (D / 8), c8 = idx % (D / 8);  // row, 8-element chunk
      qv[k] = make_uint4(0, 0, 0, 0);
      if (idx < kQChunks && i < RC) {
        const int rowi = row0 + i;
        const int r = rowi / p.G, h = g * p.G + rowi % p.G;
        qv[k] = *reinterpret_cast<const uint4*>(p.q + (((int64_t)b * p.q_max + r) * p.Hq + h) * D + c8 * 8);
      }
    }
  }
  // Dense producers: the block ids of the first tile, assuming that the
  // longest row has the planned maximum length (the usual case); checked
  // against the real range below and loaded again when it differs.
  TilePages tp_spec = {-1, -1};
  int u0_spec = 0, u1_spec = 0;
  if (MODE == FP8KV_MODE_DENSE && (warp == kProdWarp || warp == kProdWarp + 1)) {
    int per_s = max((p.max_kv_len + p.S - 1) / p.S, p.min_part);
    per_s = (per_s + kT - 1) / kT * kT;
    u0_spec = s * per_s;
    u1_spec = min(p.max_kv_len, u0_spec + per_s);
    if (u0_spec < u1_spec) tp_spec = fetch_pages(p, b, u0_spec, u1_spec, 0, lane);
  }
  int my_nrow = -1;
  if (tid < RC) {
    const int r = (row0 + tid) / p.G;
    my_nrow = (MODE == FP8KV_MODE_DENSE) ? min(max(p.row_len[(int64_t)b * p.q_max + r], 0), p.max_kv_len) : r;
  }

  // ---------------------------------------------------------- range
  int U;
  if (MODE == FP8KV_MODE_DENSE) {
    // the request's longest row: each warp loads the row lengths in
    // parallel (one per lane) and reduces them
    int n = 0;
    bool bad = false;
    for (int r = lane; r < p.q_max; r += 32) {
      const int v = p.row_len[(int64_t)b * p.q_max + r];
      bad |= (v < 0 || v > p.max_kv_len);
      n = max(n, min(max(v, 0), p.max_kv_len));
    }
    U = __reduce_max_sync(0xffffffffu, n);
    const bool any_bad = __any_sync(0xffffffffu, bad);
    if (tid == 0 && any_bad) set_status(p.status, FP8KV_STATUS_BAD_LEN);
  } else {
    U = p.n_entries[b];
    if (U < 0 || U > p.max_blocks) {
      if (tid == 0) set_status(p.status, FP8KV_STATUS_BAD_ENTRIES);
      U = min(max(U, 0), p.max_blocks);
    }
  }
  const int unit = (MODE == FP8KV_MODE_DENSE) ? kT : kE;
  int per = max((U + p.S - 1) / p.S, p.min_part);
  per = (per + unit - 1) / unit * unit;
  const int u0 = s * per;
  const int u1 = min(U, u0 + per);
  const int64_t prow = (((int64_t)b * p.Hkv + g) * p.S + s) * p.rows + row0;
  if (u0 >= u1) {
    for (int i = tid; i < RC; i += kThreads) p.ml[prow + i] = make_float2(-INFINITY, 0.f);
    return;
  }
  const int n_tiles = (u1 - u0 + unit - 1) / unit;

  // ---------------------------------------------------------- setup
  if (tid == 0) {
    for (int i = 0; i < C::kKStages / 2; ++i) {
      mbar_init(&mt.k_full[i], 2 * kDecThreads);  // every decoder thread, both tiles of the pair
      mbar_init(&mt.k_empty[i], 1);
    }
    for (int i = 0; i < C::kVStages; ++i) {
      mbar_init(&mt.v_full[i], kDecThreads);
      mbar_init(&mt.v_empty[i], 1);
    }
    for (int i = 0; i < C::kRaw; ++i) {
      mbar_init(&mt.rawk_full[i], 32);  // every lane of the producer warp
      mbar_init(&mt.rawv_full[i], 32);
      mbar_init(&mt.rawk_empty[i], kDecThreads);
      mbar_init(&mt.rawv_empty[i], kDecThreads);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&mt.s_full[i], 1);
    for (int i = 0; i < kSBuf; ++i) {
      mbar_init(&mt.pv_done[i], 1);
      // SM: a tile's P^T is written by the two softmax warps that hold its tokens
      mbar_init(&mt.p_ready[i], SM ? 64 : 32 * kSoftmaxWarps);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&mt.s_empty[i], 32 * kSoftmaxWarps);
    mbar_init(&mt.q_full, kQThreads);
    mbar_init(&mt.drain, 1);
    mt.abort = 0u;
    mt.vbad = 0u;
    mbar_init_fence();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&mt.tmem, C::kTmemCols);
    tmem_relinquish();
  }
  static_assert(kRows <= kThreads, "one query vector per thread");
  if (tid < kRows) mt.nrow[tid] = my_nrow;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = mt.tmem;
  if (MODE == FP8KV_MODE_DENSE && p.n_new > 0) {
    // a verify step's new tokens in this partition: written by every thread
    // before any copy of the pipeline can read them
    if (u1 > U - p.n_new) write_new_tokens_and_fence<FMT>(p, b, g, U, u0, u1, tid, kThreads);
    __syncthreads();
  }
  volatile uint32_t* const abort_flag = &mt.abort;
  const uint32_t wlim = (p.test_flags & FP8KV_TEST_STALL_PIPELINE) ? kTestWaitLimit : kWaitLimit;

  if (tid < kQThreads) {
    // Q rows -> swizzled K-major tile in shared memory (rows >= RC are zero);
    // the MMA thread waits for q_full before the first QK
    uint8_t* sQ = smem + C::kOffQ;
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int idx = tid + k * kQThreads;
      if (idx < kQChunks) {
        const int i = idx / (D / 8), c8 = idx % (D / 8);
        const int db = c8 / 8, ch = c8 % 8;
        *reinterpret_cast<uint4*>(sQ + db * (C::kQRows * 128) + i * 128 + ((ch ^ (i & 7)) * 16)) = qv[k];
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(&mt.q_full);
  }

  if (warp == kProdWarp || warp == kProdWarp + 1) {
    // ======================================================== producers
    // Dense: lane 0 walks the pages and issues one copy per run of tokens.
    // Sparse: lane e holds entry e of the tile (mask and microblock id, loaded
    // one tile ahead) and every lane issues the copies of two token slots.
    const bool is_k = warp == kProdWarp;
    uint64_t* raw_full = is_k ? mt.rawk_full : mt.rawv_full;
    uint64_t* raw_empty = is_k ? mt.rawk_empty : mt.rawv_empty;
    uint64_t* valid = is_k ? mt.validk : mt.validv;
    const uint8_t* cache = is_k ? p.k_cache : p.v_cache;
    const int64_t csb = is_k ? p.ksb : p.vsb, cst = is_k ? p.kst : p.vst, csh = is_k ? p.ksh : p.vsh;
    uint8_t* raw_base = smem + (is_k ? C::kOffRawK : C::kOffRawV);
    const bool stall_test = is_k && (p.test_flags & FP8KV_TEST_STALL_PIPELINE);
    bool ok = true;
    int issued = 0;  // tiles whose copies were issued
    // the page walk of tile i + 1 (block ids, or sparse entries) is loaded
    // while tile i waits for its stage
    TilePages tp = {0, -1};
    uint32_t mk = 0u;
    int bk = 0;
    auto fetch = [&](int i, TilePages& t, uint32_t& m, int& k) {
      if (MODE == FP8KV_MODE_DENSE) {
        t = fetch_pages(p, b, u0, u1, i, lane);
      } else {
        const int e = u0 + i * kE + lane;
        const bool in = lane < kE && e < u1;
        // the copies only ask whether some row sees a token: both words folded
        m = in ? (p.entry_mask[(int64_t)b * p.entry_stride + e] | mask_hi_of(p.entry_mask_hi, p.entry_stride, b, e))
               : 0u;
        k = in ? p.entry_tbl[(int64_t)b * p.entry_stride + e] : 0;
      }
    };
    if (MODE == FP8KV_MODE_DENSE && u0 == u0_spec && u1 == u1_spec)
      tp = tp_spec;
    else
      fetch(0, tp, mk, bk);
    for (int i = 0; i < n_tiles; ++i) {
      const int slot = i % C::kRaw;
      TilePages tp_next = {0, -1};
      uint32_t mk_next = 0u;
      int bk_next = 0;
      if (i + 1 < n_tiles) fetch(i + 1, tp_next, mk_next, bk_next);
      if (MODE == FP8KV_MODE_SPARSE_PAGE4 && mk != 0u && (bk < 0 || bk >= p.num_kv_blocks)) {
        // an entry with a bad block contributes nothing
        if (is_k) set_status(p.status, FP8KV_STATUS_BAD_BLOCK);
        mk = 0u;
      }
      // the raw stage is free once the decoders loaded its previous tile
      bool got = true;
      if (lane == 0 && i >= C::kRaw) got = mbar_wait(&raw_empty[slot], ((i / C::kRaw) - 1) & 1, wlim, abort_flag);
      if (!__shfl_sync(0xffffffffu, got, 0)) {
        ok = false;
        break;
      }
      uint64_t v = 0ull;
      if (MODE == FP8KV_MODE_DENSE) {
        int32_t* pblk = mt.pblk[is_k ? 0 : 1];
        pblk[lane] = tp.bid;
        __syncwarp();
        if (cst == D) {
          if (lane == 0)
            v = copy_rows_dense<D>(p, cache, csb, cst, csh, b, g, u0, u1, i, raw_base + slot * C::kRawBytes,
                                   &raw_full[slot], tp.page0, pblk, is_k);
        } else {
          v = copy_tokens_dense<D>(p, cache, csb, cst, csh, b, g, u0, u1, i, raw_base + slot * C::kRawBytes,
                                   tp.page0, pblk, is_k, lane);
        }
        __syncwarp();  // pblk is rewritten for the next tile only after every lane used it
      } else {
        v = copy_tokens_sparse<D>(cache, csb, cst, csh, g, raw_base + slot * C::kRawBytes, mk, bk, lane);
      }
      if (lane == 0) valid[slot] = v;
      __syncwarp();  // the bulk copies' expected bytes and the valid bits precede every arrival
      issued = i + 1;
      if (stall_test && i == 0) {
        // test only: hold back the arrivals until a waiting warp has given
        // up, so that the timeout path runs; then stop issuing
        for (uint32_t k = 0; k < kDrainLimit && *abort_flag == 0u; ++k) __nanosleep(256);
      }
      // every lane arrives: a gathering lane once its own cp.async copies
      // have landed, a lane of a bulk-copy tile at once (the barrier then
      // also waits for the bulk copies' bytes)
      if (MODE == FP8KV_MODE_SPARSE_PAGE4 || cst != D)
        cp_async_arrive(&raw_full[slot]);
      else
        mbar_arrive(&raw_full[slot]);
      if (stall_test && i == 0) break;
      tp = tp_next;
      mk = mk_next;
      bk = bk_next;
    }
    if (lane == 0) {
      // Drain: the copies of the last tile of every stage must have landed
      // before the CTA may exit (the decoders normally consumed them already;
      // after a give-up they may not have).  Nobody else arms these barriers,
      // so each last phase completes once its bytes arrive.
      for (int i = max(0, issued - C::kRaw); i < issued; ++i)
        mbar_wait_plain(&raw_full[i % C::kRaw], (i / C::kRaw) & 1, kDrainLimit);
      if (!ok) set_status(p.status, FP8KV_STATUS_TIMEOUT);
    }
    __syncwarp();
  } else if (warp >= kKDecWarp0 && warp < kMmaWarp) {
    // ======================================================== decoders
    const bool is_k = warp < kVDecWarp0;
    const int lt = tid - 32 * (is_k ? kKDecWarp0 : kVDecWarp0);
    const int n_stages = is_k ? C::kKStages : C::kVStages;
    uint64_t* raw_full = is_k ? mt.rawk_full : mt.rawv_full;
    uint64_t* raw_empty = is_k ? mt.rawk_empty : mt.rawv_empty;
    const uint64_t* valid = is_k ? mt.validk : mt.validv;
    const uint8_t* raw_base = smem + (is_k ? C::kOffRawK : C::kOffRawV);
    uint8_t* op_base = smem + (is_k ? C::kOffK : C::kOffV);
    bool ok = true, bad = false;
    for (int i = 0; i < n_tiles; ++i) {
      const int slot = i % C::kRaw;
      const int st = i % n_stages;
      // raw rows arrived: take them into registers and hand the raw stage
      // back to the producer at once, so its refill overlaps the wait for
      // the operand stage and the conversion
      if (!mbar_wait(&raw_full[slot], (i / C::kRaw) & 1, wlim, abort_flag)) {
        ok = false;
        break;
      }
      uint4 w[DecShape<D>::kPer];
      load_raw<D>(raw_base + slot * C::kRawBytes, valid[slot], lt, w);
      mbar_arrive(&raw_empty[slot]);
      // V: the check runs after the raw stage is handed back, off the paths
      // of both the refill and the PV (placed before the hand-back it cost
      // ~1.5 us more, after the wait for the operand stage ~3 us more)
      if (!is_k) zap_nonfinite_tile<D, FMT>(w, bad);
      if (is_k) {
        // K stages hold pairs of tiles interleaved per 64-column block, so
        // that two consecutive tiles form one 128-row operand of the pair's
        // QK; the slot is free once the previous QK that read it is done.
        // (Waiting per 64-column block instead was measured slower: every
        // decoder warp holds chunks of all blocks, so its lanes diverge.)
        const int m = i >> 1, slot = m % (C::kKStages / 2);
        if (m >= C::kKStages / 2 &&
            !mbar_wait(&mt.k_empty[slot], ((m / (C::kKStages / 2)) - 1) & 1, wlim, abort_flag)) {
          ok = false;
          break;
        }
        store_tile<D, 2 * kT * 128, FMT>(op_base + slot * (2 * C::kOpBytes) + (i & 1) * (kT * 128), w, lt);
        fence_proxy_async_smem();
        mbar_arrive(&mt.k_full[slot]);
        if ((i & 1) == 0 && i + 1 == n_tiles) mbar_arrive(&mt.k_full[slot]);  // a last tile without partner
      } else {
        // the V stage is free once the PV of its previous tile is done
        if (i >= n_stages && !mbar_wait(&mt.v_empty[st], ((i / n_stages) - 1) & 1, wlim, abort_flag)) {
          ok = false;
          break;
        }
        store_tile<D, kT * 128, FMT>(op_base + st * C::kOpBytes, w, lt);
        fence_proxy_async_smem();
        mbar_arrive(&mt.v_full[st]);
      }
    }
    if (bad) mt.vbad = 1u;
    if (!ok) set_status(p.status, FP8KV_STATUS_TIMEOUT);
  } else if (warp == kMmaWarp) {
    // ======================================================== MMA issuer
    if constexpr (SM) {
      // Small group: QK of pair m is S^T[128 x kN] = [K(2m); K(2m+1)] . Q^T
      // (A = the pair's K tiles, K-major; B = Q^T, K-major) into S^T buffer
      // m % 2; PV of tile i is O^T[128 x kNP] (+)= V(i)^T . P^T(i) per block
      // of 128 head-dim columns into the region of its pair (i / 2) % 2, the
      // pair's first MMA overwriting it (A = the V tile read MN-major, B = P^T
      // from shared memory, MN-major, 64B swizzle).  A region therefore sums
      // 128 tokens at most: the tensor core's FP32 accumulation is not
      // correctly rounded, and its error grows with the number of MMAs that
      // accumulate into one place.  Same issue rule as below:
      // whichever of the next QK (block 0 decoded, its S^T buffer read by
      // every softmax thread) and the next PV (P^T written, V decoded) is
      // ready, QK first.
      if (lane == 0) {
        const uint32_t idesc_qk = idesc_f16_f32(128, kN, false, false);
        const uint32_t idesc_pv = idesc_f16_f32(128, kNP, true, true);
        const uint64_t qdesc = smem_desc(smem_u32(smem + C::kOffQ), 16, 1024, kSw128);
        const uint64_t kdesc = smem_desc(smem_u32(smem + C::kOffK), 16, 1024, kSw128);
        const uint64_t vdesc = smem_desc(smem_u32(smem + C::kOffV), kT * 128, 1024, kSw128);
        const uint64_t pdesc = smem_desc(smem_u32(smem + C::kOffP), kT * 64, 512, kSw64);
        constexpr int kPairSlots = C::kKStages / 2;
        const int n_pairs = (n_tiles + 1) / 2;
        bool ok = mbar_wait(&mt.q_full, 0, wlim, abort_flag);
        tc_fence_after();
        auto issue_qk = [&](int m) {
          const int slot = m % kPairSlots;
          if (!mbar_wait(&mt.k_full[slot], (m / kPairSlots) & 1, wlim, abort_flag)) {
            ok = false;
            return;
          }
          tc_fence_after();
          // K16 step kk accumulates into part kk / kSteps of the pair's buffer
          constexpr int kSteps = D / 16 / C::kQKParts;
          const uint32_t dcol = tmem + C::kColS + (m & 1) * (C::kQKParts * kN);
          const uint64_t kb = kdesc + (uint64_t)((slot * 2 * C::kOpBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(dcol + (kk / kSteps) * kN, kb + (uint64_t)(((kk / 4) * (2 * kT * 128) + (kk % 4) * 32) >> 4),
                   qdesc + (uint64_t)(((kk / 4) * (kN * 128) + (kk % 4) * 32) >> 4), idesc_qk, (kk % kSteps) > 0);
          mma_commit(&mt.k_empty[slot]);
          mma_commit(&mt.s_full[m & 1]);
        };
        auto issue_pv = [&](int i) {
          const int st = i % C::kVStages, pb = i % kSBuf;
          tc_fence_after();
#pragma unroll
          for (int db2 = 0; db2 < D / 128; ++db2)
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk)
              mma_ss(tmem + C::kColO + (((i >> 1) & 1) * (D / 128) + db2) * kNP,
                     vdesc + (uint64_t)((st * C::kOpBytes + 2 * db2 * (kT * 128) + kk * 16 * 128) >> 4),
                     pdesc + (uint64_t)((pb * C::kPBytes + kk * 16 * 64) >> 4), idesc_pv,
                     ((i & 1) || kk > 0) ? 1u : 0u);
          mma_commit(&mt.v_empty[st]);
          mma_commit(&mt.pv_done[pb]);
        };
        int qn = 0, pn = 0;
        uint32_t idle = 0;
        while (ok && pn < n_tiles) {
          if (qn < n_pairs && mbar_test(&mt.k_full[qn % kPairSlots], (qn / kPairSlots) & 1) &&
              (qn < 2 || mbar_test(&mt.s_empty[qn & 1], ((qn >> 1) - 1) & 1))) {
            issue_qk(qn++);
            idle = 0;
            continue;
          }
          if (pn < 2 * qn && mbar_test(&mt.p_ready[pn % kSBuf], (pn / kSBuf) & 1) &&
              mbar_test(&mt.v_full[pn % C::kVStages], (pn / C::kVStages) & 1)) {
            issue_pv(pn++);
            idle = 0;
            continue;
          }
          if (*abort_flag || ++idle > wlim) {
            *abort_flag = 1u;
            ok = false;
            break;
          }
          __nanosleep(32);
        }
        mma_commit(&mt.drain);
        mbar_wait_plain(&mt.drain, 0, kDrainLimit);
        if (!ok) set_status(p.status, FP8KV_STATUS_TIMEOUT);
      }
      __syncwarp();
    } else {
    // One thread issues every UMMA.  QK of pair m: once both K tiles are
    // decoded, the D/16 K16 steps of one chain, then commits that free the K
    // slot and mark S full.  PV of tile i: once its P is written and its V
    // tile decoded, four K16 steps into O, then commits that free the V stage
    // and mark the tile's PV done.  The thread issues whichever of the next
    // QK and the next PV is ready (the QK first when both are): every
    // operation depends only on operations issued before it, so no order can
    // deadlock.  Descriptors are built once; a step only adds its offset to
    // the start-address field (shared-memory offsets stay below 2^18).
    if (lane == 0) {
      const uint32_t idesc_qk1 = idesc_f16_f32(64, kT, false, false);
      const uint32_t idesc_qk2 = idesc_f16_f32(64, 2 * kT, false, false);
      const uint32_t idesc_pv = idesc_f16_f32(128, D, false, true);
      const uint64_t qdesc = smem_desc(smem_u32(smem + C::kOffQ), 16, 1024, kSw128);
      const uint64_t kdesc = smem_desc(smem_u32(smem + C::kOffK), 16, 1024, kSw128);
      const uint64_t vdesc = smem_desc(smem_u32(smem + C::kOffV), kT * 128, 1024, kSw128);
      constexpr int kPairSlots = C::kKStages / 2;
      const int n_pairs = (n_tiles + 1) / 2;
      bool ok = mbar_wait(&mt.q_full, 0, wlim, abort_flag);
      tc_fence_after();
      // S = Q . [K(2m); K(2m+1)]^T: one N=128 chain (N=64 for a last single tile)
      auto issue_qk = [&](int m) {
        const int slot = m % kPairSlots;
        const uint32_t par = (m / kPairSlots) & 1;
        const uint32_t idesc = (2 * m + 1 < n_tiles) ? idesc_qk2 : idesc_qk1;
        const uint32_t dcol = tmem + C::kColS + ((2 * m) % kSBuf) * kT;
        const uint64_t kb = kdesc + (uint64_t)((slot * 2 * C::kOpBytes) >> 4);
        if (!mbar_wait(&mt.k_full[slot], par, wlim, abort_flag)) {
          ok = false;
          return;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(dcol, qdesc + (uint64_t)(((kk / 4) * (kRows * 128) + (kk % 4) * 32) >> 4),
                 kb + (uint64_t)(((kk / 4) * (2 * kT * 128) + (kk % 4) * 32) >> 4), idesc, kk > 0);
        mma_commit(&mt.k_empty[slot]);
        mma_commit(&mt.s_full[m & 1]);
      };
      // O += P(i) . V(i): A = P from TMEM (hi rows and their lo twins), B = V
      auto issue_pv = [&](int i) {
        const int st = i % C::kVStages;
        tc_fence_after();
        const uint64_t vb = vdesc + (uint64_t)((st * C::kOpBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)
          mma_ts(tmem + C::kColO, tmem + C::kColS + (i % kSBuf) * kT + kk * 8,
                 vb + (uint64_t)((kk * 16 * 128) >> 4), idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&mt.v_empty[st]);
        mma_commit(&mt.pv_done[i % kSBuf]);
      };
      int qn = 0, pn = 0;  // next QK pair, next PV tile
      uint32_t idle = 0;
      while (ok && pn < n_tiles) {
        // QK(qn) may start once block 0 of its pair is decoded and its S
        // buffers are free (the PVs of tiles 2qn-4 and 2qn-3 are done)
        if (qn < n_pairs && mbar_test(&mt.k_full[qn % kPairSlots], (qn / kPairSlots) & 1) &&
            (qn < 2 || mbar_test(&mt.pv_done[(2 * qn - 3) % kSBuf], ((2 * qn - 3) / kSBuf) & 1))) {
          issue_qk(qn++);
          idle = 0;
          continue;
        }
        // PV(pn) once its P is written and its V decoded
        if (pn < 2 * qn && mbar_test(&mt.p_ready[pn % kSBuf], (pn / kSBuf) & 1) &&
            mbar_test(&mt.v_full[pn % C::kVStages], (pn / C::kVStages) & 1)) {
          issue_pv(pn++);
          idle = 0;
          continue;
        }
        if (*abort_flag || ++idle > wlim) {
          *abort_flag = 1u;
          ok = false;
          break;
        }
        __nanosleep(32);
      }
      // Drain: every UMMA this thread issued must be done before TMEM is
      // freed (normally the softmax warps already waited for the last PV).
      mma_commit(&mt.drain);
      mbar_wait_plain(&mt.drain, 0, kDrainLimit);
      if (!ok) set_status(p.status, FP8KV_STATUS_TIMEOUT);
    }
    __syncwarp();
    }
  } else if constexpr (SM) {
    // ======================================================== softmax warps (small group)
    // Thread = one token of the tile pair (warp w holds TMEM lanes 32w..32w+31
    // = tokens 32w.. of the pair), kN columns = query vectors.  The running
    // maxima are per column and identical in every thread; each thread keeps
    // partial sums of its own tokens, reduced once at the end.  Exponents are
    // formed against the running maxima; only when one exceeds kTau anywhere
    // (a vote over the four warps) do the warps exchange column maxima.
    const float ks = p.k_scale_dev ? *p.k_scale_dev : p.k_scale;
    const LogitScale cs = logit_scale(p.softmax_scale, ks);
    // columns NL.. of S^T, P^T and O^T belong to no query vector of the CTA
    float mrow[NL], lpart[NL];
#pragma unroll
    for (int n = 0; n < NL; ++n) {
      mrow[n] = -INFINITY;
      lpart[n] = 0.f;
    }
    const int tl = 32 * warp + lane;          // token of the pair
    const int h = tl >> 6, r = tl & 63;       // tile of the pair, row in the tile
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    float* red_max = reinterpret_cast<float*>(smem + C::kOffRed);  // [warp][kN]
    float* red_l = red_max + kSoftmaxWarps * kN;
    const int n_pairs = (n_tiles + 1) / 2;
    bool ok = true;
    // Master sum of O^T (thread = head-dim lane 32w + lane of each 128-column
    // block): hi + lo per vector, the PV of every drained pair added with
    // TwoSum (P_hi part) and into lo (P_lo part, 2^-11 below it).  The last
    // pair is not drained: the epilogue adds it on the way out.
    auto drain = [&](int j, bool last) {
      constexpr int CW = NL < 8 ? NL : 8;  // columns per step (bounds the live registers)
      tc_fence_after();
#pragma unroll
      for (int db2 = 0; db2 < D / 128; ++db2) {
#pragma unroll 1
        for (int c0 = 0; c0 < NL; c0 += CW) {
          uint32_t oh[CW], ol[CW], mh[CW], ml[CW];
          const uint32_t rb = tmem + C::kColO + ((j & 1) * (D / 128) + db2) * kNP + c0 + lane_off;
          const uint32_t mb = tmem + C::kColM + db2 * (2 * kN) + c0 + lane_off;
          tmem_ld_cols<CW>(rb, oh);
          tmem_ld_cols<CW>(rb + kN, ol);
          if (j > 0) {
            tmem_ld_cols<CW>(mb, mh);
            tmem_ld_cols<CW>(mb + kN, ml);
          }
#pragma unroll
          for (int n = 0; n < CW; ++n) {
            float hi = j > 0 ? __uint_as_float(mh[n]) : 0.f, lo = j > 0 ? __uint_as_float(ml[n]) : 0.f;
            two_sum_acc(hi, lo, __uint_as_float(oh[n]));
            lo = fmaf(__uint_as_float(ol[n]), kInvLoScale, lo);
            mh[n] = __float_as_uint(hi);
            ml[n] = __float_as_uint(lo);
          }
          if (last) {
            const int d = 128 * db2 + 32 * warp + lane;
#pragma unroll
            for (int n = 0; n < CW; ++n)
              if (c0 + n < RC)
                p.partial[(prow + c0 + n) * D + d] = (__uint_as_float(mh[n]) + __uint_as_float(ml[n])) * kInvPShift;
          } else {
            tmem_st_cols<CW>(mb, mh);
            tmem_st_cols<CW>(mb + kN, ml);
          }
        }
      }
      tc_fence_before();
    };
    for (int m2 = 0; m2 < n_pairs; ++m2) {
      // Named barriers below need all four warps: the decision to stop (a
      // bounded wait gave up, here or in the previous pair) is taken jointly.
      if (ok && !mbar_wait(&mt.s_full[m2 & 1], (m2 >> 1) & 1, wlim, abort_flag)) ok = false;
      if (named_bar_or(1, 32 * kSoftmaxWarps, !ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // compensated QK: the parts of S^T (each an exact-product sum over a
      // share of D) added with TwoSum into hi + lo
      float shi[NL], slo[NL];
      {
        const uint32_t sb = tmem + C::kColS + (m2 & 1) * (C::kQKParts * kN) + lane_off;
#pragma unroll
        for (int part = 0; part < C::kQKParts; ++part) {
          uint32_t sr[NL];
          tmem_ld_cols<NL>(sb + part * kN, sr);
#pragma unroll
          for (int n = 0; n < NL; ++n) {
            if (part == 0) {
              shi[n] = __uint_as_float(sr[n]);
              slo[n] = 0.f;
            } else {
              two_sum_acc(shi[n], slo[n], __uint_as_float(sr[n]));
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&mt.s_empty[m2 & 1]);
      bool drained = m2 == 0;    // the previous pair is in the master sum
      const int i = 2 * m2 + h;  // this thread's tile
      // bit n: query vector n sees this token
      uint32_t vis = 0u;
      if (i < n_tiles) {
        if (MODE == FP8KV_MODE_DENSE) {
          const int tok = u0 + i * kT + r;
          if (tok < u1) {
#pragma unroll
            for (int n = 0; n < NL; ++n) vis |= (tok < mt.nrow[n] ? 1u : 0u) << n;
          }
        } else {
          const int e = u0 + i * kE + (r >> 2), tk = r & 3;
          if (e < u1) {
            uint32_t mk = p.entry_mask[(int64_t)b * p.entry_stride + e];
            uint32_t mkh = mask_hi_of(p.entry_mask_hi, p.entry_stride, b, e);
            const int blk = p.entry_tbl[(int64_t)b * p.entry_stride + e];
            if (blk < 0 || blk >= p.num_kv_blocks) mk = mkh = 0u;
#pragma unroll
            for (int n = 0; n < NL; ++n) {
              const int qr = mt.nrow[n];
              vis |= ((qr >= 0) ? sparse_bit(mk, mkh, qr, tk) : 0u) << n;
            }
          }
        }
      }
      float e[NL];
      auto exps = [&]() {
#pragma unroll
        for (int n = 0; n < NL; ++n) {
          const float mu = mrow[n] == -INFINITY ? -3.0e38f : mrow[n];
          const float x = fmaf(shi[n], cs.hi, -mu) + fmaf(slo[n], cs.hi, shi[n] * cs.lo);
          e[n] = ((vis >> n) & 1u) ? x : -INFINITY;
        }
      };
      exps();
      bool need = false;
#pragma unroll
      for (int n = 0; n < NL; ++n) need |= e[n] > kTau;
      if (named_bar_or(1, 32 * kSoftmaxWarps, need)) {
        // Slow path (always on the first pair): column maxima of the visible
        // logits over the pair's 128 tokens, lazy integer maxima, rescale.
#pragma unroll
        for (int n = 0; n < NL; ++n) {
          float x = ((vis >> n) & 1u) ? shi[n] * cs.hi : -INFINITY;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
          if (lane == 0) red_max[warp * kN + n] = x;
        }
        named_bar_sync(1, 32 * kSoftmaxWarps);
        float alpha[NL];
        bool resc = false;
#pragma unroll
        for (int n = 0; n < NL; ++n) {
          float mx = red_max[n];
#pragma unroll
          for (int w = 1; w < kSoftmaxWarps; ++w) mx = fmaxf(mx, red_max[w * kN + n]);
          const float mo = mrow[n];
          const float mn = (mx > mo + kTau || mo == -INFINITY) ? fmaxf(mo, ceilf(mx)) : mo;
          alpha[n] = (mo != -INFINITY && mn != mo) ? exp2_int(mo - mn) : 1.f;
          resc |= alpha[n] != 1.f;
          mrow[n] = mn;
          lpart[n] *= alpha[n];
        }
        named_bar_sync(1, 32 * kSoftmaxWarps);  // the maxima are read before any later exchange
        exps();
        if (resc && m2 > 0) {
          // everything before this pair was made under the old maxima: drain
          // the previous pair now, then scale the master's column n (hi and
          // lo) by the exact power of two alpha[n]
          if (ok && mbar_wait(&mt.pv_done[(2 * m2 - 1) % kSBuf], ((2 * m2 - 1) / kSBuf) & 1, wlim, abort_flag)) {
            drain(m2 - 1, false);
            drained = true;
#pragma unroll
            for (int db2 = 0; db2 < D / 128; ++db2) {
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                uint32_t o[NL];
                const uint32_t ta = tmem + C::kColM + db2 * (2 * kN) + half * kN + lane_off;
                tmem_ld_cols<NL>(ta, o);
#pragma unroll
                for (int n = 0; n < NL; ++n) o[n] = __float_as_uint(__uint_as_float(o[n]) * alpha[n]);
                tmem_st_cols<NL>(ta, o);
              }
            }
            tc_fence_before();
          } else {
            ok = false;
          }
        }
      }
      // P = P_hi + P_lo: this token's row of P^T (kN hi columns, then kN lo;
      // only the first NL of each are written)
      uint32_t ph[NL / 2], pl[NL / 2];
#pragma unroll
      for (int n = 0; n < NL; n += 2) {
        const float p0 = fast_exp2(e[n] + kPShift), p1 = fast_exp2(e[n + 1] + kPShift);
        lpart[n] += p0;
        lpart[n + 1] += p1;
        const uint32_t hh = pack_f16x2(p0, p1);
        const float2 f = unpack_f16x2(hh);
        ph[n / 2] = hh;
        pl[n / 2] = pack_f16x2((p0 - f.x) * kLoScale, (p1 - f.y) * kLoScale);
      }
      if (i < n_tiles) {
        // the tile's P^T buffer is free once the PV of tile i - kSBuf is done
        const int pb = i % kSBuf;
        if (i >= kSBuf && !mbar_wait(&mt.pv_done[pb], ((i / kSBuf) - 1) & 1, wlim, abort_flag)) {
          ok = false;
        } else {
          uint8_t* row = smem + C::kOffP + pb * C::kPBytes + r * (kNP * 2);
          const int sw = (r >> 1) & 3;  // 64-byte swizzle: 16-byte chunk c at c ^ ((row / 2) % 4)
          // chunks 1 and 3 (columns 8..15 of each half) feed only O^T columns
          // that no vector reads when NL <= 8, so they are left unwritten
          if constexpr (NL == 4) {
            *reinterpret_cast<uint4*>(row + ((0 ^ sw) * 16)) = make_uint4(ph[0], ph[1], 0u, 0u);
            *reinterpret_cast<uint4*>(row + ((2 ^ sw) * 16)) = make_uint4(pl[0], pl[1], 0u, 0u);
          } else {
            *reinterpret_cast<uint4*>(row + ((0 ^ sw) * 16)) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
            *reinterpret_cast<uint4*>(row + ((2 ^ sw) * 16)) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
          }
          if constexpr (NL == kN) {
            *reinterpret_cast<uint4*>(row + ((1 ^ sw) * 16)) = make_uint4(ph[4], ph[5], ph[6], ph[7]);
            *reinterpret_cast<uint4*>(row + ((3 ^ sw) * 16)) = make_uint4(pl[4], pl[5], pl[6], pl[7]);
          }
          fence_proxy_async_smem();
          mbar_arrive(&mt.p_ready[pb]);
        }
      }
      // the previous pair's PV ran while this pair's softmax did
      if (!drained) {
        if (ok && mbar_wait(&mt.pv_done[(2 * m2 - 1) % kSBuf], ((2 * m2 - 1) / kSBuf) & 1, wlim, abort_flag))
          drain(m2 - 1, false);
        else
          ok = false;
      }
    }
    // ------------------------------------------------------ epilogue (small group)
    if (!ok || !mbar_wait(&mt.pv_done[(n_tiles - 1) % kSBuf], ((n_tiles - 1) / kSBuf) & 1, wlim, abort_flag))
      ok = false;
    tc_fence_after();
    if (!ok) set_status(p.status, FP8KV_STATUS_TIMEOUT);
    // row sums: each thread's partial sums over its tokens, reduced across the
    // 128 softmax threads in a fixed order
#pragma unroll
    for (int n = 0; n < NL; ++n) {
      float x = lpart[n];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      if (lane == 0) red_l[warp * kN + n] = x;
    }
    named_bar_sync(1, 32 * kSoftmaxWarps);
    if (tid < RC) {
      float l = red_l[tid];
#pragma unroll
      for (int w = 1; w < kSoftmaxWarps; ++w) l += red_l[w * kN + tid];
      float m = -INFINITY;
#pragma unroll
      for (int n = 0; n < NL; ++n) m = (n == tid) ? mrow[n] : m;
      p.ml[prow + tid] = make_float2(m, l * kInvPShift);
    }
    // numerators: the master sum plus the last pair (thread = head-dim
    // column 128 * db2 + 32w + lane)
    drain(n_pairs - 1, true);
  } else {
    // ======================================================== softmax warps
    const float ks = p.k_scale_dev ? *p.k_scale_dev : p.k_scale;
    // base-2 logit factor (K is decoded to its exact value)
    const float c = p.softmax_scale * ks * kLog2e;
    const int ra = 16 * warp + (lane >> 2);  // this thread's two rows: ra and ra + 8
    const int rb = ra + 8;
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    const bool warp_live = 16 * warp < RC;   // warps without query vectors only keep the barriers
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
    const int n_a = mt.nrow[ra], n_b = mt.nrow[rb];
    bool ok = true;
    for (int i = 0; i < n_tiles && ok; ++i) {
      if (!mbar_wait(&mt.s_full[(i >> 1) & 1], (i >> 2) & 1, wlim, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (warp_live) {
        uint32_t sr[32];
        ld_16x256b_x8(tmem + C::kColS + (i % kSBuf) * kT + lane_off, sr);
        // visibility of this thread's 16 columns for rows ra (bits 0..15) and rb (16..31)
        uint32_t vis;
        if (MODE == FP8KV_MODE_DENSE) {
          const int t0 = u0 + i * kT;
          const int lim_a = min(u1, n_a) - t0, lim_b = min(u1, n_b) - t0;
          if (lim_a >= kT && lim_b >= kT) {
            vis = 0xFFFFFFFFu;
          } else {
            vis = 0;
#pragma unroll
            for (int gq = 0; gq < 8; ++gq)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int col = 8 * gq + 2 * (lane & 3) + e;
                vis |= (col < lim_a ? 1u : 0u) << (2 * gq + e);
                vis |= (col < lim_b ? 1u : 0u) << (16 + 2 * gq + e);
              }
          }
        } else {
          // columns 8gq + 2(lane%4) + {0,1} lie in entry 2gq + (lane%4)/2 of
          // the tile; an entry whose block is out of range attends nothing
          vis = 0;
#pragma unroll
          for (int gq = 0; gq < 8; ++gq) {
            const int ent = u0 + i * kE + 2 * gq + ((lane & 3) >> 1);
            uint32_t mk = 0u, mkh = 0u;
            if (ent < u1) {
              mk = p.entry_mask[(int64_t)b * p.entry_stride + ent];
              mkh = mask_hi_of(p.entry_mask_hi, p.entry_stride, b, ent);
              const int blk = p.entry_tbl[(int64_t)b * p.entry_stride + ent];
              if (blk < 0 || blk >= p.num_kv_blocks) mk = mkh = 0u;
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int pos = (2 * (lane & 3) + e) & 3;
              vis |= ((n_a >= 0) ? sparse_bit(mk, mkh, n_a, pos) : 0u) << (2 * gq + e);
              vis |= ((n_b >= 0) ? sparse_bit(mk, mkh, n_b, pos) : 0u) << (16 + 2 * gq + e);
            }
          }
        }
        // a tile every column of which both rows see skips the selects
        const bool full = __all_sync(0xffffffffu, vis == 0xFFFFFFFFu);
        // Exponents against the running maximum (a row that has seen nothing
        // yet uses a huge negative stand-in, so any visible element forces
        // the slow path below); masked elements get -inf by selection, so
        // their p is exactly 0 and a NaN logit of an unseen token is dropped.
        float ea[16], eb[16];
        auto exps = [&](float mua, float mub) {
#pragma unroll
          for (int q2 = 0; q2 < 8; ++q2)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float xa = fmaf(__uint_as_float(sr[4 * q2 + e]), c, -mua);
              const float xb = fmaf(__uint_as_float(sr[4 * q2 + 2 + e]), c, -mub);
              ea[2 * q2 + e] = (full || ((vis >> (2 * q2 + e)) & 1u)) ? xa : -INFINITY;
              eb[2 * q2 + e] = (full || ((vis >> (16 + 2 * q2 + e)) & 1u)) ? xb : -INFINITY;
            }
        };
        exps(m_a == -INFINITY ? -3.0e38f : m_a, m_b == -INFINITY ? -3.0e38f : m_b);
        float xa = ea[0], xb = eb[0];
#pragma unroll
        for (int j = 1; j < 16; ++j) {
          xa = fmaxf(xa, ea[j]);
          xb = fmaxf(xb, eb[j]);
        }
        float alpha_a = 1.f, alpha_b = 1.f;
        if (__any_sync(0xffffffffu, xa > kTau || xb > kTau)) {
          // Slow path: some row's lazy integer maximum must move (always on
          // a row's first visible tile).  Row maxima over the visible logits.
          float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
          for (int q2 = 0; q2 < 8; ++q2)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              if (full || ((vis >> (2 * q2 + e)) & 1u)) mx_a = fmaxf(mx_a, __uint_as_float(sr[4 * q2 + e]) * c);
              if (full || ((vis >> (16 + 2 * q2 + e)) & 1u))
                mx_b = fmaxf(mx_b, __uint_as_float(sr[4 * q2 + 2 + e]) * c);
            }
          mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
          mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
          mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
          mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
          const float mn_a = (mx_a > m_a + kTau || m_a == -INFINITY) ? fmaxf(m_a, ceilf(mx_a)) : m_a;
          const float mn_b = (mx_b > m_b + kTau || m_b == -INFINITY) ? fmaxf(m_b, ceilf(mx_b)) : m_b;
          const bool resc_a = (m_a != -INFINITY) && (mn_a != m_a);
          const bool resc_b = (m_b != -INFINITY) && (mn_b != m_b);
          alpha_a = resc_a ? exp2_int(m_a - mn_a) : 1.f;
          alpha_b = resc_b ? exp2_int(m_b - mn_b) : 1.f;
          m_a = mn_a;
          m_b = mn_b;
          exps(m_a == -INFINITY ? -3.0e38f : m_a, m_b == -INFINITY ? -3.0e38f : m_b);
          if (__any_sync(0xffffffffu, resc_a || resc_b) && i > 0 &&
              mbar_wait(&mt.pv_done[(i - 1) % kSBuf], ((i - 1) / kSBuf) & 1, wlim, abort_flag)) {
            // O holds exactly the PVs of the tiles before this one (all made
            // under the old maxima): scale it by the exact power of two.
            // Thread `lane` owns TMEM lane 32w + lane = vector 16w + lane%16
            // (the P_hi row for lane < 16, its P_lo twin above); the alpha of
            // vector 16w + x lives in thread 4*(x%8), as its a (x < 8) or b value.
            tc_fence_after();
            const int x = lane & 15;
            const float al_a = __shfl_sync(0xffffffffu, alpha_a, 4 * (x & 7));
            const float al_b = __shfl_sync(0xffffffffu, alpha_b, 4 * (x & 7));
            const float al = (x < 8) ? al_a : al_b;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 16) {
              uint32_t o[16];
              tmem_ld16(tmem + C::kColO + lane_off + c0, o);
#pragma unroll
              for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * al);
              tmem_st16(tmem + C::kColO + lane_off + c0, o);
            }
          }
        }
        // P = P_hi + P_lo (two fp16 halves) replaces S in the tile's buffer:
        // hi in lanes 32w+0..15, lo 16 above
        uint32_t ph[16], pl[16];
        float sum_a = 0.f, sum_b = 0.f;
#pragma unroll
        for (int q2 = 0; q2 < 8; ++q2) {
          const float pa0 = fast_exp2(ea[2 * q2] + kPShift), pa1 = fast_exp2(ea[2 * q2 + 1] + kPShift);
          const float pb0 = fast_exp2(eb[2 * q2] + kPShift), pb1 = fast_exp2(eb[2 * q2 + 1] + kPShift);
          sum_a += pa0 + pa1;
          sum_b += pb0 + pb1;
          const uint32_t ha = pack_f16x2(pa0, pa1), hb = pack_f16x2(pb0, pb1);
          const float2 fa = unpack_f16x2(ha), fb = unpack_f16x2(hb);
          ph[2 * q2] = ha;
          ph[2 * q2 + 1] = hb;
          pl[2 * q2] = pack_f16x2((pa0 - fa.x) * kLoScale, (pa1 - fa.y) * kLoScale);
          pl[2 * q2 + 1] = pack_f16x2((pb0 - fb.x) * kLoScale, (pb1 - fb.y) * kLoScale);
        }
        sum_a += __shfl_xor_sync(0xffffffffu, sum_a, 1);
        sum_a += __shfl_xor_sync(0xffffffffu, sum_a, 2);
        sum_b += __shfl_xor_sync(0xffffffffu, sum_b, 1);
        sum_b += __shfl_xor_sync(0xffffffffu, sum_b, 2);
        l_a = l_a * alpha_a + sum_a;
        l_b = l_b * alpha_b + sum_b;
        const uint32_t pcol = tmem + C::kColS + (i % kSBuf) * kT + lane_off;
        st_16x128b_x8_pair(pcol, pcol + (16u << 16), ph, pl);
      }
      tc_fence_before();
      mbar_arrive(&mt.p_ready[i % kSBuf]);
    }
    // ------------------------------------------------------ epilogue
    if (!ok || !mbar_wait(&mt.pv_done[(n_tiles - 1) % kSBuf], ((n_tiles - 1) / kSBuf) & 1, wlim, abort_flag))
      ok = false;
    tc_fence_after();
    if (!ok) set_status(p.status, FP8KV_STATUS_TIMEOUT);
    if (warp_live) {
      const int myrow = 16 * warp + (lane & 15);
      const bool up = lane >= 16;
      const float own = up ? kInvLoScale : 1.f;  // this lane's rows hold P_lo (scaled) or P_hi sums
      float* dst = p.partial + (prow + myrow) * D + (up ? 32 : 0);
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 64) {
        uint32_t o[64];
        tmem_ld64(tmem + C::kColO + lane_off + c0, o);
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float keep = __uint_as_float(up ? o[j + 32] : o[j]) * own;
          const float give = __uint_as_float(up ? o[j] : o[j + 32]) * own;
          v[j] = (keep + __shfl_xor_sync(0xffffffffu, give, 16)) * kInvPShift;
        }
        if (myrow < RC) {
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(dst + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
      }
      if ((lane & 3) == 0) {
        if (ra < RC) p.ml[prow + ra] = make_float2(m_a, l_a * kInvPShift);
        if (rb < RC) p.ml[prow + rb] = make_float2(m_b, l_b * kInvPShift);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (mt.vbad) patch_nonfinite_v<D, MODE, FMT>(p, smem + C::kOffRawK, mt.nrow, b, g, u0, u1, RC, prow);
}

template <int D, int MODE, int FMT, bool SM, int NL>
cudaError_t launch(const fp8kv_attn_plan_t* plan, const Params& p, cudaStream_t st) {
  auto fn = split_tc<D, MODE, FMT, SM, NL>;
  static DeviceOnce once;
  cudaError_t e = once.run([&] {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D, SM>::kSmem);
  });
  if (e != cudaSuccess) return e;
  dim3 grid(plan->grid[0], plan->grid[1], plan->grid[2]);
  fn<<<grid, kThreads, Cfg<D, SM>::kSmem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace
}  // namespace fp8kv
