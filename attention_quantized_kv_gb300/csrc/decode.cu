// decode.cu -- split-K flash-decoding over a block-quantized KV cache.
//
// Computes, for every (sequence, query head), o = softmax(scale * q K^T) V
// over all cached keys, with K and V dequantized from f16 / q8_0 / q4_0 blocks
// or turbo4 rotated rows (the codecs of the "Codecs" table of the
// buun-llama-cpp listing; the K and V sides are typed independently, as in
// its VBR section's per-(layer, side) ladder).  turbo4 is never un-rotated
// per token: the query is rotated once (q . x^ = (H s q / 16) . y^), V is
// accumulated in the rotated space and the merged output is rotated back.
// Work is cut along the token axis; each piece produces a partial (running
// max m, running sum l, unnormalised o), and a second kernel, launched right
// behind the first (programmatic dependent launch), merges the partials of
// each (sequence, head) with the log-sum-exp identity and writes the output
// rows: one CTA per stream, every partial requested at once.
//
// Work partition.  A "stream" is one (sequence, kv head, group of up to 8
// query heads); its keys are 16-token units.  All units of all streams are
// laid end to end and the grid (about two CTAs per SM, all resident) takes
// equal contiguous slices, so ragged lengths cost no imbalance.  A CTA's slice
// crosses at most a few stream boundaries; at each one its warps merge their
// partials and the CTA writes one partial for that stream.
//
// Inside a CTA (8 warps):
//  * A ring of shared-memory stages, one 16-token unit of K and V per stage,
//    filled with 1-D bulk async copies (TMA engine) on mbarriers.  Unit k
//    goes to stage k % NS and is consumed by warp k % 8 (NS is a multiple of
//    8, so every stage has one owner warp); after consuming unit k the owner
//    refills the stage with unit k + NS, so ~80 KB per CTA stay in flight.
//  * The cache layout (include/kvq.h) stores each unit so that every thread
//    fetches exactly its tensor-core operand bytes with aligned 16-byte
//    shared loads (a warp reads 512 contiguous bytes: conflict-free).
//  * Quants become exact fp16 integers in registers (bias-and-subtract on
//    the fp16 mantissa).  S = K Q^T runs on mma.sync m16n8k16 with the 16
//    tokens as M and the query heads of the group as N.  Block scales are
//    factored out of the 32-value sums (two MMAs per block into a fresh
//    accumulator, then s += d * partial), so K dequantization is exact.
//  * Online softmax in the log2 domain per head with xor-shuffle maxima; P is
//    transposed in registers (movmatrix) into the B operand of O^T = V^T P^T
//    (M = 16 head dims); the V block scale is folded into P.
//
// The fused decode step (attn_decode_append) is a second instantiation of
// the same kernel (FUSED): each sequence's new token is encoded into the
// cache by the warp that consumes the item holding it, before that warp
// issues any copy (so its small loads and stores go out ahead of the copy
// flood), and the lengths advance once every CTA has read them.
#include <cuda_runtime.h>

#include <math.h>

#include "kvq_device.cuh"
#include "kvq_encode.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRingBytes = 84 * 1024;
constexpr int kMaxSeqs = kDecodeMaxSeqs;
constexpr int kRedFloats = 36;  // per lane: o[8][4], m0, m1, l0, l1

struct DecodeParams {
  const uint8_t *k_cache;
  const uint8_t *v_cache;
  const int32_t *seq_lens;
  const __half *q;
  // Fused decode step (k_new != nullptr): one new token per sequence,
  // fp16 rows [n_seqs][n_kv][128], encoded into the cache at position
  // seq_lens[s] by the warp that consumes the item holding it; lens_rw
  // (= seq_lens) is advanced by the last CTA to finish reading the lengths,
  // counted in rd_ctr (zero between calls).
  const __half *k_new;
  const __half *v_new;
  int32_t *lens_rw;
  unsigned *rd_ctr;
  float *part_o;    // [slots][8][128]
  float2 *part_ml;  // [slots][8]: (max in log2 units, sum)
  __half *out;      // [n_seqs][n_q][128]
  float *lse;       // [n_seqs][n_q] or null
  int32_t *err;
  const int32_t *table;  // paged layers: block table; nullptr: contiguous
  int n_seqs, n_kv, n_q, G, n_hg, capacity, max_len, pages_per_seq, n_pages;
  float scale_log2;
};

// Units per work item: nibble codecs (q4_0, turbo4) on both sides move two
// consecutive units (32 tokens) of each side per stage, so that every bulk
// copy carries over 2 KB (the copy engine's per-copy cost shows below a few
// KB); wider codecs keep one unit per stage and more stages per warp.
// (Four units per item measured no faster than two.)
constexpr int kNibbleItemUnits = 2;
__host__ __device__ constexpr int items_units(int ck, int cv) {
  return (nibble_codec(ck) && nibble_codec(cv)) ? kNibbleItemUnits : 1;
}

template <int CK, int CV>
struct DecodeCfg {
  static constexpr int UK = unit_bytes(CK);
  static constexpr int UV = unit_bytes(CV);
  static constexpr int UPS = items_units(CK, CV);  // units per item (and stage)
  static constexpr int STAGE = UPS * (UK + UV);    // [UPS K units][UPS V units]
  // Stage s always belongs to warp s % kWarps (NS is a multiple of kWarps):
  // the warp that consumes item k also refills its stage with item k + NS
  // and is the only waiter on that stage's mbarrier, so phase waits are
  // strictly sequential per barrier.
  static constexpr int NS_RAW = kRingBytes / STAGE / kWarps * kWarps;
  static constexpr int NS = NS_RAW > 32 ? 32 : (NS_RAW < kWarps ? kWarps : NS_RAW);
  static constexpr int RING = NS * STAGE;
  static constexpr int RED = 4 * 32 * kRedFloats * 4;  // tree-merge slots
  static constexpr int SMEM = RING + RED;
  static_assert(NS % kWarps == 0, "stage ownership needs NS % warps == 0");
  // Two one-unit items per warp step when each warp owns at least four stages.
  static constexpr bool PAIR = UPS == 1 && NS / kWarps >= 4;
};

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
}

// Head-dim index of accumulator row (m-row) of m-tile mt for the V codec.
template <int CV>
__device__ __forceinline__ int v_dim(int mt, int mrow) {
  if (nibble_codec(CV)) {
    const int b = mt >> 1, hh = mt & 1;
    return 32 * b + 8 * hh + (mrow & 7) + (mrow >> 3) * 16;
  }
  return 16 * mt + 2 * (mrow & 7) + (mrow >> 3);
}

// S (16 tokens x 8 heads) of one unit, multiplied by scale*log2(e).
template <int CK>
__device__ __forceinline__ void unit_scores(const uint8_t *ku, int lane, const uint32_t (&qb)[8][2],
                                            const uint2 *qlo, float scale_log2, float (&s)[4]) {
  const int g = lane >> 2;
  s[0] = s[1] = s[2] = s[3] = 0.0f;
  if (CK == KVQ_F16) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint4 r0 = lds128(ku + (2 * b) * 512 + lane * 16);
      const uint4 r1 = lds128(ku + (2 * b + 1) * 512 + lane * 16);
      const uint32_t a0[4] = {r0.x, r1.x, r0.y, r1.y};
      const uint32_t a1[4] = {r0.z, r1.z, r0.w, r1.w};
      mma16816(s, a0, qb[2 * b][0], qb[2 * b][1]);
      mma16816(s, a1, qb[2 * b + 1][0], qb[2 * b + 1][1]);
    }
  } else if (CK == KVQ_TURBO4) {
    // one scale per row: the four 32-dim groups share one accumulator; the
    // rotated query is the fp16 pair qb + qlo (qlo[c * 32]: this lane's low
    // halves of k-step c, in shared memory), both against the same operands
    const uint32_t sc = *reinterpret_cast<const uint32_t *>(ku + 1024 + g * 4);
    float sb[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int jv = 0; jv < 2; ++jv) {
      const uint4 w = lds128(ku + jv * 512 + lane * 16);
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        const int b = 2 * jv + hb;
        const uint32_t W0 = hb ? w.z : w.x, W1 = hb ? w.w : w.y;
        const uint32_t X0 = W0 >> 8, X1 = W1 >> 8;
        const uint32_t a0[4] = {u4_pair_minus8(W0), u4_pair_minus8(W1), u4_pair_minus8(X0),
                                u4_pair_minus8(X1)};
        const uint32_t a1[4] = {u4_pair_minus8_hi(W0), u4_pair_minus8_hi(W1),
                                u4_pair_minus8_hi(X0), u4_pair_minus8_hi(X1)};
        mma16816(sb, a0, qb[2 * b][0], qb[2 * b][1]);
        mma16816(sb, a1, qb[2 * b + 1][0], qb[2 * b + 1][1]);
        const uint2 l0 = qlo[(2 * b) * 32], l1 = qlo[(2 * b + 1) * 32];
        mma16816(sb, a0, l0.x, l0.y);
        mma16816(sb, a1, l1.x, l1.y);
      }
    }
    const float dlo = half_bits_to_float(sc & 0xffffu), dhi = half_bits_to_float(sc >> 16);
    s[0] = dlo * sb[0];
    s[1] = dlo * sb[1];
    s[2] = dhi * sb[2];
    s[3] = dhi * sb[3];
  } else {
    const uint4 sc = lds128(ku + unit_scale_offset(CK) + g * 16);
    const uint32_t dl[2] = {sc.x, sc.y}, dh[2] = {sc.z, sc.w};
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float sb[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (CK == KVQ_Q8_0) {
        const uint4 w = lds128(ku + b * 512 + lane * 16);
        const uint32_t a0[4] = {s8_pair_02(w.x), s8_pair_02(w.z), s8_pair_13(w.x), s8_pair_13(w.z)};
        const uint32_t a1[4] = {s8_pair_02(w.y), s8_pair_02(w.w), s8_pair_13(w.y), s8_pair_13(w.w)};
        mma16816(sb, a0, qb[2 * b][0], qb[2 * b][1]);
        mma16816(sb, a1, qb[2 * b + 1][0], qb[2 * b + 1][1]);
      } else {
        const uint4 w = lds128(ku + (b >> 1) * 512 + lane * 16);
        const uint32_t W0 = (b & 1) ? w.z : w.x, W1 = (b & 1) ? w.w : w.y;
        const uint32_t X0 = W0 >> 8, X1 = W1 >> 8;
        const uint32_t a0[4] = {u4_pair_minus8(W0), u4_pair_minus8(W1), u4_pair_minus8(X0),
                                u4_pair_minus8(X1)};
        const uint32_t a1[4] = {u4_pair_minus8_hi(W0), u4_pair_minus8_hi(W1),
                                u4_pair_minus8_hi(X0), u4_pair_minus8_hi(X1)};
        mma16816(sb, a0, qb[2 * b][0], qb[2 * b][1]);
        mma16816(sb, a1, qb[2 * b + 1][0], qb[2 * b + 1][1]);
      }
      const float dlo = half_bits_to_float(dl[b >> 1] >> (16 * (b & 1)));
      const float dhi = half_bits_to_float(dh[b >> 1] >> (16 * (b & 1)));
      s[0] = fmaf(dlo, sb[0], s[0]);
      s[1] = fmaf(dlo, sb[1], s[1]);
      s[2] = fmaf(dhi, sb[2], s[2]);
      s[3] = fmaf(dhi, sb[3], s[3]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) s[i] *= scale_log2;
}

// O^T (128 dims x 8 heads) += V^T (dims x 16 tokens) * P^T (16 tokens x heads).
// FULL: all 16 tokens of the unit are valid (no masking needed).
//
// q4_0 V takes the nibbles n as fp16 subnormals, one AND each: rows g of an
// m-tile get n * 2^-24 (low nibbles), rows g+8 get 16n * 2^-24 (high nibbles
// masked in place).  Every product with the folded P (an fp16 number) is
// still exact in fp32.  The offset of the codec, -8 per value, is restored
// at the end of the segment from corr, whose rows r collect
// C_b = sum over tokens of d_b(t) p(t, h) for block b = r & 3: one MMA with
// A rows r holding the scales d_{r&3} of the unit's tokens and B = P^T.
template <int CV, bool FULL>
__device__ __forceinline__ void unit_pv(const uint8_t *vu, int lane, uint32_t B0, uint32_t B1,
                                        int nvalid, float (&o)[8][4], float (&corr)[4]) {
  const int tig = lane & 3;
  // token validity of the halves this thread holds: (2tig, 2tig+1) and (+8, +9)
  uint32_t m01 = 0xffffffffu, m23 = 0xffffffffu;
  if (!FULL) {
    m01 = (2 * tig < nvalid ? 0x0000ffffu : 0u) | (2 * tig + 1 < nvalid ? 0xffff0000u : 0u);
    m23 = (2 * tig + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * tig + 9 < nvalid ? 0xffff0000u : 0u);
  }
  if (CV == KVQ_F16) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const uint4 r = lds128(vu + mt * 512 + lane * 16);
      uint32_t a[4] = {r.x, r.y, r.z, r.w};
      if (!FULL) { a[0] &= m01; a[1] &= m01; a[2] &= m23; a[3] &= m23; }
      mma16816(o[mt], a, B0, B1);
    }
  } else {
    uint32_t dp01[4], dp23[4];
    if (CV == KVQ_TURBO4) {  // one scale per token: (2tig, 2tig+1), (2tig+8, 2tig+9)
      const uint2 sv = lds64(vu + 1024 + tig * 8);
#pragma unroll
      for (int b = 0; b < 4; ++b) { dp01[b] = sv.x; dp23[b] = sv.y; }
    } else {
      const uint4 s01 = lds128(vu + unit_scale_offset(CV) + tig * 32);
      const uint4 s23 = lds128(vu + unit_scale_offset(CV) + tig * 32 + 16);
      dp01[0] = s01.x; dp01[1] = s01.z; dp01[2] = s23.x; dp01[3] = s23.z;
      dp23[0] = s01.y; dp23[1] = s01.w; dp23[2] = s23.y; dp23[3] = s23.w;
    }
    if (!FULL) {
#pragma unroll
      for (int b = 0; b < 4; ++b) { dp01[b] &= m01; dp23[b] &= m23; }
    }
    // P^T with the V block scale folded in, one pair of B registers per block
    uint32_t bp0[4], bp1[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      bp0[b] = hmul2_bits(B0, dp01[b]);
      bp1[b] = hmul2_bits(B1, dp23[b]);
    }
    if (CV == KVQ_Q8_0) {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint4 w = lds128(vu + b * 512 + lane * 16);
        const uint32_t a0[4] = {s8_pair_02(w.x), s8_pair_13(w.x), s8_pair_02(w.y), s8_pair_13(w.y)};
        const uint32_t a1[4] = {s8_pair_02(w.z), s8_pair_13(w.z), s8_pair_02(w.w), s8_pair_13(w.w)};
        mma16816(o[2 * b], a0, bp0[b], bp1[b]);
        mma16816(o[2 * b + 1], a1, bp0[b], bp1[b]);
      }
    } else {
#pragma unroll
      for (int jv = 0; jv < 2; ++jv) {
        const uint4 w = lds128(vu + jv * 512 + lane * 16);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const int mt = 4 * jv + qq, b = mt >> 1;
          const uint32_t W = ws[qq], X = W >> 8;
          const uint32_t a[4] = {W & 0x000f000fu, W & 0x00f000f0u, X & 0x000f000fu,
                                 X & 0x00f000f0u};
          mma16816(o[mt], a, bp0[b], bp1[b]);
        }
      }
      const int g = lane >> 2;
      // scales of block g & 3 for tokens (2tig, 2tig+1) and (2tig+8, 2tig+9)
      uint2 dg = CV == KVQ_TURBO4 ? lds64(vu + 1024 + tig * 8)
                                  : lds64(vu + unit_scale_offset(CV) + tig * 32 + (g & 3) * 8);
      if (!FULL) { dg.x &= m01; dg.y &= m23; }
      const uint32_t a[4] = {dg.x, dg.x, dg.y, dg.y};
      mma16816(corr, a, B0, B1);
    }
  }
}

// Position in the flattened unit space: sequence, stream within the
// sequence (kv head * n_hg + head group), unit within the stream, and the
// unit's index in the cache (for the bulk copy).
struct Cursor {
  int seq, sl, j, n_s;  // j, n_s: items of the stream
  int64_t unit;   // contiguous layers: the index of the item's first unit in the cache
  int pg0, pg1;   // paged layers: pool pages of the item's page and the next one
};

struct Geo {
  const int32_t *pfx;    // items per stream, prefix-summed over the sequences
  int n_seqs, n_kv, n_hg, KH;
  int64_t upst;          // units per (seq, kv head) stream of the cache
  int upi, ipp;          // units per item; items per page
  const int32_t *table;  // paged layers: block table; nullptr: contiguous
  int pps, n_pages;
};

// Paged layers: the cursor's pool pages, this page and the next one of the
// stream (-1 past the stream or for an entry outside the pool); the next
// page's entry is requested a whole page ahead of its first use.
__device__ __forceinline__ void cursor_pages(const Geo &q, Cursor &c) {
  const int pj = c.j / q.ipp;
  c.pg0 = page_of(q.table, q.pps, q.n_pages, c.seq, pj);
  c.pg1 = (pj + 1) * q.ipp < c.n_s ? page_of(q.table, q.pps, q.n_pages, c.seq, pj + 1) : -1;
}

__device__ __forceinline__ int64_t cache_unit(const Geo &q, int seq, int sl, int j) {
  return (static_cast<int64_t>(seq) * q.n_kv + sl / q.n_hg) * q.upst +
         static_cast<int64_t>(j) * q.upi;
}

// Largest s with pfx[s] * KH <= u (pfx non-decreasing, pfx[0] = 0).
__device__ __forceinline__ int find_seq(const Geo &q, int64_t u) {
  int lo = 0, hi = q.n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(q.pfx[mid]) * q.KH <= u) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ Cursor cursor_at(const Geo &q, int64_t u) {
  Cursor c;
  if (u >= static_cast<int64_t>(q.pfx[q.n_seqs]) * q.KH) {  // past the end: inert
    c.seq = q.n_seqs;
    c.sl = c.j = 0;
    c.n_s = 1;
    c.unit = 0;
    return c;
  }
  c.seq = find_seq(q, u);
  c.n_s = q.pfx[c.seq + 1] - q.pfx[c.seq];
  const int64_t within = u - static_cast<int64_t>(q.pfx[c.seq]) * q.KH;
  const int64_t sl = within / c.n_s;
  c.sl = static_cast<int>(sl);
  c.j = static_cast<int>(within - sl * c.n_s);
  c.unit = cache_unit(q, c.seq, c.sl, c.j);
  if (q.table) cursor_pages(q, c);
  return c;
}

// Advance a cursor by `step` items (stops being meaningful past the end).
__device__ __forceinline__ void cursor_advance(Cursor &c, int step, const Geo &q) {
  const int old_page = c.j / q.ipp;
  c.j += step;
  if (c.j < c.n_s) {
    c.unit += static_cast<int64_t>(step) * q.upi;
    if (q.table) {
      const int pj = c.j / q.ipp;
      if (pj == old_page + 1) {  // the common crossing: shift, request the next entry
        c.pg0 = c.pg1;
        c.pg1 = (pj + 1) * q.ipp < c.n_s
                    ? page_of(q.table, q.pps, q.n_pages, c.seq, pj + 1) : -1;
      } else if (pj != old_page) {
        cursor_pages(q, c);
      }
    }
    return;
  }
  do {
    c.j -= c.n_s;
    if (++c.sl == q.KH) {
      c.sl = 0;
      do {
        ++c.seq;
      } while (c.seq < q.n_seqs && q.pfx[c.seq + 1] == q.pfx[c.seq]);
      if (c.seq >= q.n_seqs) return;
      c.n_s = q.pfx[c.seq + 1] - q.pfx[c.seq];
    }
  } while (c.j >= c.n_s);
  c.unit = cache_unit(q, c.seq, c.sl, c.j);
  if (q.table) cursor_pages(q, c);
}

// Index of the cursor's item's first unit in the cache (contiguous) or the
// pool (paged; an entry outside the pool reads pool page 0, flagged by the
// caller).  An item's units are consecutive there: an item never straddles
// a page (items per page = 16 / units per item).
__device__ __forceinline__ int64_t cursor_unit(const Geo &q, const Cursor &c) {
  if (!q.table) return c.unit;
  const int pg = c.pg0 < 0 ? 0 : c.pg0;
  return (static_cast<int64_t>(pg) * q.n_kv + c.sl / q.n_hg) * kPageUnits +
         (c.j % q.ipp) * q.upi;
}

// Merge partial b into a (per lane; m uniform across the lanes of a head).
__device__ __forceinline__ void merge_into(float (&o)[8][4], float &m0, float &m1, float &l0,
                                           float &l1, const float *r) {
  const float bm0 = r[32], bm1 = r[33], bl0 = r[34], bl1 = r[35];
  const float M0 = fmaxf(m0, bm0), M1 = fmaxf(m1, bm1);
  const float sa0 = m0 == -INFINITY ? 0.0f : fast_exp2(m0 - M0);
  const float sb0 = bm0 == -INFINITY ? 0.0f : fast_exp2(bm0 - M0);
  const float sa1 = m1 == -INFINITY ? 0.0f : fast_exp2(m1 - M1);
  const float sb1 = bm1 == -INFINITY ? 0.0f : fast_exp2(bm1 - M1);
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    o[mt][0] = o[mt][0] * sa0 + r[4 * mt + 0] * sb0;
    o[mt][1] = o[mt][1] * sa1 + r[4 * mt + 1] * sb1;
    o[mt][2] = o[mt][2] * sa0 + r[4 * mt + 2] * sb0;
    o[mt][3] = o[mt][3] * sa1 + r[4 * mt + 3] * sb1;
  }
  l0 = l0 * sa0 + bl0 * sb0;
  l1 = l1 * sa1 + bl1 * sb1;
  m0 = M0;
  m1 = M1;
}

__device__ __forceinline__ void store_red(float *r, const float (&o)[8][4], float m0, float m1,
                                          float l0, float l1) {
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
    reinterpret_cast<float4 *>(r)[mt] = make_float4(o[mt][0], o[mt][1], o[mt][2], o[mt][3]);
  reinterpret_cast<float4 *>(r)[8] = make_float4(m0, m1, l0, l1);
}

__device__ __forceinline__ void cta_bar() {
  asm volatile("bar.sync 1, %0;\n" ::"n"(kThreads) : "memory");
}
__device__ __forceinline__ void half_bar() {  // warps 0 .. kWarps/2 - 1
  asm volatile("bar.sync 2, %0;\n" ::"n"(kThreads / 2) : "memory");
}

// Online softmax + PV for N units at once (N = 1, 2 or 4): one max reduction and
// at most one rescale per call.  A unit may have no valid token at all (the
// second unit of a two-unit item past the length): it is fully masked.
template <int CK, int CV, int N>
__device__ __forceinline__ void process_units(const uint8_t *const (&ku)[N],
                                              const uint8_t *const (&vus)[N],
                                              const int (&nvalid)[N], int lane,
                                              const uint32_t (&qb)[8][2], const uint2 *qlo,
                                              float scale_log2,
                                              float (&o)[8][4], float (&corr)[4],
                                              float &m0, float &m1, float &l0, float &l1) {
  const int g = lane >> 2;
  float sc[N][4];
#pragma unroll
  for (int u = 0; u < N; ++u) {
    unit_scores<CK>(ku[u], lane, qb, qlo, scale_log2, sc[u]);
    if (nvalid[u] < kUnitTokens) {
      if (g >= nvalid[u]) sc[u][0] = sc[u][1] = -INFINITY;
      if (g + 8 >= nvalid[u]) sc[u][2] = sc[u][3] = -INFINITY;
    }
  }
  float mx0 = fmaxf(sc[0][0], sc[0][2]), mx1 = fmaxf(sc[0][1], sc[0][3]);
#pragma unroll
  for (int u = 1; u < N; ++u) {
    mx0 = fmaxf(mx0, fmaxf(sc[u][0], sc[u][2]));
    mx1 = fmaxf(mx1, fmaxf(sc[u][1], sc[u][3]));
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
  }
  const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
  if (__any_sync(0xffffffffu, mn0 > m0 || mn1 > m1)) {
    const float a0 = fast_exp2(m0 - mn0), a1 = fast_exp2(m1 - mn1);
    l0 *= a0;
    l1 *= a1;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      o[mt][0] *= a0; o[mt][1] *= a1; o[mt][2] *= a0; o[mt][3] *= a1;
    }
    if (nibble_codec(CV)) { corr[0] *= a0; corr[1] *= a1; corr[2] *= a0; corr[3] *= a1; }
    m0 = mn0;
    m1 = mn1;
  }
#pragma unroll
  for (int u = 0; u < N; ++u) {
    const float p0 = fast_exp2(sc[u][0] - m0), p1 = fast_exp2(sc[u][1] - m1);
    const float p2 = fast_exp2(sc[u][2] - m0), p3 = fast_exp2(sc[u][3] - m1);
    l0 += p0 + p2;
    l1 += p1 + p3;
    const uint32_t B0 = movmatrix_trans(pack_half2(p0, p1));
    const uint32_t B1 = movmatrix_trans(pack_half2(p2, p3));
    const uint8_t *vu = vus[u];
    if (nvalid[u] == kUnitTokens) unit_pv<CV, true>(vu, lane, B0, B1, nvalid[u], o, corr);
    else unit_pv<CV, false>(vu, lane, B0, B1, nvalid[u], o, corr);
  }
}

// B fragments of Q for query head g of head group hg (zero beyond the
// group), with the per-codec order of the k (head-dim) index that matches the
// K unit layout.
template <int CK>
__device__ __forceinline__ void load_q_frags(const __half *q, int64_t qrow0, int n_q, int G, int hg,
                                             int lane, uint32_t (&qb)[8][2],
                                             uint32_t (&qlo)[8][2]) {
  const int g = lane >> 2, tig = lane & 3;
  const int hq = hg * 8 + g;
  const bool hvalid = hq < G;
  const __half *qrow = q + (qrow0 + (hvalid ? hq : 0)) * kD;
  if (CK == KVQ_TURBO4) {
    rotated_q_frags(qrow, hvalid, tig, qb, qlo, [](const __half *p) {
      return *reinterpret_cast<const uint2 *>(p);
    });
  } else {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int base = 32 * (c >> 1) + 16 * (c & 1) + 4 * tig;
      uint2 v = make_uint2(0u, 0u);
      if (hvalid) v = *reinterpret_cast<const uint2 *>(qrow + base);
      if (CK == KVQ_F16) {
        qb[c][0] = v.x;
        qb[c][1] = v.y;
      } else {
        qb[c][0] = __byte_perm(v.x, v.y, 0x5410);
        qb[c][1] = __byte_perm(v.x, v.y, 0x7632);
      }
    }
  }
}

// The same fragments from a copy of the group's query rows in shared memory
// (nh = rows present; row r is query head hg * 8 + r).
template <int CK>
__device__ __forceinline__ void load_q_frags_smem(const __half *qs, int nh, int lane,
                                                  uint32_t (&qb)[8][2], uint32_t (&qlo)[8][2]) {
  const int g = lane >> 2, tig = lane & 3;
  const bool hvalid = g < nh;
  const __half *qrow = qs + (hvalid ? g : 0) * kD;
  if (CK == KVQ_TURBO4) {
    rotated_q_frags(qrow, hvalid, tig, qb, qlo, [](const __half *p) { return lds64(p); });
  } else {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int base = 32 * (c >> 1) + 16 * (c & 1) + 4 * tig;
      uint2 v = make_uint2(0u, 0u);
      if (hvalid) v = lds64(qrow + base);
      if (CK == KVQ_F16) {
        qb[c][0] = v.x;
        qb[c][1] = v.y;
      } else {
        qb[c][0] = __byte_perm(v.x, v.y, 0x5410);
        qb[c][1] = __byte_perm(v.x, v.y, 0x7632);
      }
    }
  }
}

// Where a merged row goes: out [n_seqs][n_q][128] fp16, lse [n_seqs][n_q].
struct MergeArgs {
  const float2 *part_ml;
  const float *part_o;
  __half *out;
  float *lse;
  int n_q, G;
};

// One head's merged row: o = acc / L (rotated back for turbo4 V), fp16, and
// its natural-log lse (M is in log2 units).
template <bool ROT>
__device__ __forceinline__ void merge_write(const MergeArgs &p, int seq, int kvh, int hg, int h,
                                            int lane, float4 acc, float M, float L,
                                            bool dry = false) {
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  const int64_t row = static_cast<int64_t>(seq) * p.n_q + kvh * p.G + hg * 8 + h;
  float ov[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
  if (ROT) turbo_unrotate_lane(ov, lane);  // turbo4 V: back from the rotated space
  const __half2 o01 = __floats2half2_rn(ov[0], ov[1]), o23 = __floats2half2_rn(ov[2], ov[3]);
  const float lse = L > 0.0f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
  if (dry) return;
  __half2 *dst = reinterpret_cast<__half2 *>(p.out + row * kD) + lane * 2;
  dst[0] = o01;
  dst[1] = o23;
  if (p.lse && lane == 0) p.lse[row] = lse;
}

// Keys sequence s attends: its length, plus the token a fused decode step
// appends when it fits the capacity.
__device__ __forceinline__ int attended_len(const DecodeParams &p, int s) {
  int len = p.seq_lens[s];
  if (p.k_new && len >= 0 && len < p.capacity) ++len;
  return len;
}

// Fused decode step, one thread per CTA after the CTA's last read of the
// lengths: the last CTA to get here advances them (each CTA counts itself
// only after all its reads, so no CTA sees a new length).
__device__ __noinline__ void lengths_read(const DecodeParams &p) {
  __threadfence();
  const unsigned old = atomicInc(p.rd_ctr, gridDim.x - 1);
  if (old != gridDim.x - 1) return;
  __threadfence();
  for (int s = 0; s < p.n_seqs; ++s) {
    const int len = p.seq_lens[s];
    if (len >= 0 && len < p.capacity) p.lens_rw[s] = len + 1;
  }
}

// Fused decode step: the appended token of sequence seq exists (its length
// is in [0, capacity)).
__device__ __forceinline__ bool appends(const DecodeParams &p, int seq) {
  const int len = p.seq_lens[seq];
  return p.k_new && len >= 0 && len < p.capacity;
}

// Fused decode step: write sequence seq's new K and V rows of kv head kvh
// (fp16 from k_new / v_new; all 32 lanes) into the cache at position
// pos = seq_lens[seq] (the old length).
template <int CK, int CV>
__device__ __forceinline__ void write_new_rows(const DecodeParams &p, int seq, int kvh, int lane) {
  const int pos = p.seq_lens[seq];
  const int64_t row = static_cast<int64_t>(seq) * p.n_kv + kvh;
  const uint2 rk = reinterpret_cast<const uint2 *>(p.k_new + row * kD)[lane];
  const uint2 rv = reinterpret_cast<const uint2 *>(p.v_new + row * kD)[lane];
  int64_t unit;
  if (p.table) {
    const int pg =
        page_of(p.table, p.pages_per_seq, p.n_pages, seq, pos / (kUnitTokens * kPageUnits));
    if (pg < 0) {
      if (lane == 0) set_err(p.err, KVQ_DEVERR_PAGE);
      return;
    }
    unit = (static_cast<int64_t>(pg) * p.n_kv + kvh) * kPageUnits + (pos / kUnitTokens) % kPageUnits;
  } else {
    unit = row * (p.capacity / kUnitTokens) + pos / kUnitTokens;
  }
  const int r = pos % kUnitTokens;
  encode_row_into<0>(CK, rk, const_cast<uint8_t *>(p.k_cache) + unit * unit_bytes(CK), r, lane);
  encode_row_into<1>(CV, rv, const_cast<uint8_t *>(p.v_cache) + unit * unit_bytes(CV), r, lane);
}

__device__ __forceinline__ Geo make_geo(const DecodeParams &p, const int32_t *pfx, int ups) {
  Geo geo;
  geo.pfx = pfx;
  geo.n_seqs = p.n_seqs;
  geo.n_kv = p.n_kv;
  geo.n_hg = p.n_hg;
  geo.KH = p.n_kv * p.n_hg;
  geo.upst = p.capacity / kUnitTokens;
  geo.upi = ups;
  geo.ipp = kPageUnits / ups;
  geo.table = p.table;
  geo.pps = p.pages_per_seq;
  geo.n_pages = p.n_pages;
  return geo;
}

// FUSED: the fused decode step (p.k_new set); a separate instantiation, so
// that the plain decode loop carries none of its state.
template <int CK, int CV, bool FUSED>
__global__ void __launch_bounds__(kThreads, 2) decode_split_kernel(const DecodeParams p) {
  using C = DecodeCfg<CK, CV>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full[C::NS];
  __shared__ int32_t pfx[kMaxSeqs + 1];
  __shared__ int abort_flag;
  // query rows of the current and the next segment (bulk copies, one
  // segment ahead; the first is requested before the ring's copies)
  __shared__ __align__(128) __half q_s[2][8 * kD];
  __shared__ uint64_t q_bar[2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;

  // The previous kernel on the stream (the append) must be complete before
  // the lengths and the cache are read.
  grid_dependency_wait();

  // Units per stream of each sequence, prefix-summed (one warp).
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < p.n_seqs; base += 32) {
      const int s = base + lane;
      int n = 0;
      if (s < p.n_seqs) {
        if (p.k_new && blockIdx.x == 0) {
          const int old = p.seq_lens[s];
          if (old < 0 || old >= p.capacity) set_err(p.err, KVQ_DEVERR_CAPACITY);
        }
        int len = attended_len(p, s);
        if (len > p.max_len) {
          if (blockIdx.x == 0) set_err(p.err, KVQ_DEVERR_MAXLEN);
          len = p.max_len;
        }
        n = len > 0 ? (len + C::UPS * kUnitTokens - 1) / (C::UPS * kUnitTokens) : 0;
      }
      int incl = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
      }
      if (s < p.n_seqs) pfx[s + 1] = carry + incl;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      pfx[0] = 0;
      abort_flag = 0;
    }
    for (int s = lane; s < C::NS; s += 32) mbar_init(&full[s], 1);
    if (lane < 2) mbar_init(&q_bar[lane], 1);
    fence_mbar_init();
  }
  __syncthreads();
  grid_launch_dependents();

  // Sequences with no keys get no unit, hence no partial: CTA 0 writes their
  // rows (out = 0, lse = -inf).
  if (blockIdx.x == 0) {
    for (int row = warp; row < p.n_seqs * p.n_q; row += kWarps) {
      const int s = row / p.n_q;
      if (pfx[s + 1] != pfx[s]) continue;
      reinterpret_cast<uint2 *>(p.out + static_cast<int64_t>(row) * kD)[lane] = make_uint2(0u, 0u);
      if (p.lse && lane == 0) p.lse[row] = -INFINITY;
    }
  }

  const Geo geo = make_geo(p, pfx, C::UPS);
  const int64_t U = static_cast<int64_t>(pfx[p.n_seqs]) * geo.KH;
  const int P = gridDim.x;
  const int64_t u0 = U * blockIdx.x / P;
  const int64_t u1 = U * (blockIdx.x + 1) / P;
  const int R = static_cast<int>(u1 - u0);
  if (R <= 0) {  // whole CTA: nothing to do
    if (FUSED && threadIdx.x == 0) lengths_read(p);
    return;
  }

  uint8_t *ring = smem;
  float *red = reinterpret_cast<float *>(smem + C::RING);
  // turbo4 keys: this lane's slots for the low halves of the rotated query
  // (8 per lane, 2 KB per warp) at the start of the reduction slots
  uint2 *const qlo = reinterpret_cast<uint2 *>(red) + warp * 8 * 32 + lane;

  // Issue unit k of this CTA's slice into stage k % NS (lane 0 of its owner).
  auto issue = [&](int k, const Cursor &c) {
    const int s = k % C::NS;
    uint8_t *dst = ring + s * C::STAGE;
    const int64_t unit = cursor_unit(geo, c);
    if (geo.table && c.pg0 < 0) set_err(p.err, KVQ_DEVERR_PAGE);
    mbar_arrive_expect_tx(&full[s], C::STAGE);
    bulk_copy_g2s(dst, p.k_cache + unit * C::UK, C::UPS * C::UK, &full[s]);
    bulk_copy_g2s(dst + C::UPS * C::UK, p.v_cache + unit * C::UV, C::UPS * C::UV, &full[s]);
  };

  // Query rows of the segment at cursor c into q_s[buf] (thread 0).
  const bool q_bulk = (reinterpret_cast<uintptr_t>(p.q) & 15) == 0;
  auto issue_q = [&](int buf, const Cursor &c) {
    const int hgc = c.sl % p.n_hg;
    const uint32_t bytes = static_cast<uint32_t>(min(8, p.G - hgc * 8)) * kD * 2;
    const __half *src =
        p.q + (static_cast<int64_t>(c.seq) * p.n_q + (c.sl / p.n_hg) * p.G + hgc * 8) * kD;
    mbar_arrive_expect_tx(&q_bar[buf], bytes);
    bulk_copy_g2s(q_s[buf], src, bytes, &q_bar[buf]);
  };

  Cursor seg = cursor_at(geo, u0);
  int q_iss = 0;  // query-row copies issued (thread 0: segments 0 .. q_iss - 1)
  if (q_bulk && threadIdx.x == 0) {
    issue_q(0, seg);
    q_iss = 1;
  }
  // Fused decode step: a stream's new token lies in its last item.  For
  // every stream that ends inside this slice, the warp that consumes that
  // item writes the new rows into the cache before it issues any copy, and
  // orders those writes before its copies (with several head groups per kv
  // head each group's stream writes the same bytes).
  if (FUSED) {
    bool wrote = false;
    int64_t u = u0;
    while (u < u1) {
      const Cursor c = cursor_at(geo, u);
      const int64_t send = u + (c.n_s - c.j);
      if (send <= u1 && static_cast<int>(send - 1 - u0) % kWarps == warp && appends(p, c.seq)) {
        write_new_rows<CK, CV>(p, c.seq, c.sl / p.n_hg, lane);
        wrote = true;
      }
      u = send;
    }
    if (wrote) asm volatile("fence.proxy.async.global;\n" ::: "memory");
    __syncwarp();
  }

  // Prologue: each warp issues its own first stages (k = warp, warp + 8, ...
  // below NS).  Afterwards the producer cursor pc sits at unit k + NS for the
  // warp's next unit k.
  Cursor pc = cursor_at(geo, u0 + warp);
  if (lane == 0) {
    Cursor c = pc;
    for (int k = warp; k < C::NS && k < R; k += kWarps) {
      issue(k, c);
      cursor_advance(c, kWarps, geo);
    }
  }
  cursor_advance(pc, C::NS, geo);

  // Walk the segments (stream pieces) of this slice.
  int64_t useg = u0;
  int k_next = warp;  // next unit index (CTA-local) this warp consumes
  bool ok = true;
  int k_fail = -1;    // first unit not consumed after an abort
  int si = 0;         // segment index (its query rows are in q_s[si & 1])
  while (useg < u1) {
    const int64_t seg_end = min(u1, useg + (seg.n_s - seg.j));
    const int k0 = static_cast<int>(useg - u0), k1 = static_cast<int>(seg_end - u0);
    const int seq = seg.seq, kvh = seg.sl / p.n_hg, hg = seg.sl % p.n_hg;
    int len = attended_len(p, seq);
    len = len < p.max_len ? len : p.max_len;

    uint32_t qb[8][2], qlo_r[8][2];
    if (q_bulk) {
      const int buf = si & 1;
      bool got_q =
          ok && mbar_wait_bounded(&q_bar[buf], static_cast<uint32_t>(si >> 1) & 1u, &abort_flag);
      got_q = __all_sync(0xffffffffu, got_q);
      if (!got_q && ok) {
        if (lane == 0) {
          set_err(p.err, KVQ_DEVERR_TIMEOUT);
          atomicExch(&abort_flag, 1);
        }
        ok = false;
        k_fail = k_next;
      }
      load_q_frags_smem<CK>(q_s[buf], min(8, p.G - hg * 8), lane, qb, qlo_r);
      // The next segment's rows go out now, a whole segment ahead of their
      // use (q_s[buf ^ 1] was last read before the previous segment's
      // barriers).
      if (threadIdx.x == 0 && seg_end < u1 && ok) {
        fence_proxy_async_smem();
        issue_q(buf ^ 1, cursor_at(geo, seg_end));
        ++q_iss;
      }
    } else {
      load_q_frags<CK>(p.q, static_cast<int64_t>(seq) * p.n_q + kvh * p.G, p.n_q, p.G, hg, lane,
                       qb, qlo_r);
    }
    // turbo4 keys: the query's low halves wait in this warp's part of the
    // reduction slots (free until the segment ends) rather than in registers
    if (CK == KVQ_TURBO4) {
#pragma unroll
      for (int c = 0; c < 8; ++c) qlo[c * 32] = make_uint2(qlo_r[c][0], qlo_r[c][1]);
      __syncwarp();
    }
    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.0f;
    float corr[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // q4_0 V: per-block sums of the folded P
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;

    while (k_next < k1) {
      const int k = k_next;
      const bool two = C::PAIR && k + kWarps < k1;
      const int s0 = k % C::NS;
      const int s1 = (k + kWarps) % C::NS;
      bool got = ok && mbar_wait_bounded(&full[s0], static_cast<uint32_t>(k / C::NS) & 1u,
                                         &abort_flag);
      if (two)
        got = got && mbar_wait_bounded(&full[s1],
                                       static_cast<uint32_t>((k + kWarps) / C::NS) & 1u,
                                       &abort_flag);
      got = __all_sync(0xffffffffu, got);
      if (!got) {
        if (ok && lane == 0) {
          set_err(p.err, KVQ_DEVERR_TIMEOUT);
          atomicExch(&abort_flag, 1);
        }
        if (ok) k_fail = k;
        ok = false;
        k_next += two ? 2 * kWarps : kWarps;
        continue;
      }
      const int j = seg.j + (k - k0);
      if (C::UPS > 1) {  // one item: UPS consecutive units of each side
        const uint8_t *st = ring + s0 * C::STAGE;
        const uint8_t *ku[C::UPS];
        const uint8_t *vu[C::UPS];
        int nv[C::UPS];
#pragma unroll
        for (int u = 0; u < C::UPS; ++u) {
          ku[u] = st + u * C::UK;
          vu[u] = st + C::UPS * C::UK + u * C::UV;
          nv[u] = min(kUnitTokens, len - (C::UPS * j + u) * kUnitTokens);
        }
        process_units<CK, CV, C::UPS>(ku, vu, nv, lane, qb, qlo, p.scale_log2, o, corr, m0, m1, l0,
                                      l1);
      } else if (two) {
        const uint8_t *ku[2] = {ring + s0 * C::STAGE, ring + s1 * C::STAGE};
        const uint8_t *vu[2] = {ku[0] + C::UK, ku[1] + C::UK};
        const int nv[2] = {min(kUnitTokens, len - j * kUnitTokens),
                           min(kUnitTokens, len - (j + kWarps) * kUnitTokens)};
        process_units<CK, CV, 2>(ku, vu, nv, lane, qb, qlo, p.scale_log2, o, corr, m0, m1, l0, l1);
      } else {
        const uint8_t *ku[1] = {ring + s0 * C::STAGE};
        const uint8_t *vu[1] = {ku[0] + C::UK};
        const int nv[1] = {min(kUnitTokens, len - j * kUnitTokens)};
        process_units<CK, CV, 1>(ku, vu, nv, lane, qb, qlo, p.scale_log2, o, corr, m0, m1, l0, l1);
      }
      // The consumed stages are free: refill them with units k + NS (+ 8).
      __syncwarp();
      if (lane == 0) {
        fence_proxy_async_smem();
        if (k + C::NS < R) issue(k + C::NS, pc);
      }
      cursor_advance(pc, kWarps, geo);
      if (two) {
        if (lane == 0 && k + kWarps + C::NS < R) issue(k + kWarps + C::NS, pc);
        cursor_advance(pc, kWarps, geo);
      }
      k_next += two ? 2 * kWarps : kWarps;
    }

    if (nibble_codec(CV)) {
      // Restore the codec offset: o = 2^24 o - 8 C_b (rows g) and
      // 2^20 o - 8 C_b (rows g+8), C_b from lane 4b + tig of corr.
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float c0 = -8.0f * __shfl_sync(0xffffffffu, corr[0], 4 * b + tig);
        const float c1 = -8.0f * __shfl_sync(0xffffffffu, corr[1], 4 * b + tig);
#pragma unroll
        for (int mt = 2 * b; mt < 2 * b + 2; ++mt) {
          o[mt][0] = fmaf(0x1p24f, o[mt][0], c0);
          o[mt][1] = fmaf(0x1p24f, o[mt][1], c1);
          o[mt][2] = fmaf(0x1p20f, o[mt][2], c0);
          o[mt][3] = fmaf(0x1p20f, o[mt][3], c1);
        }
      }
    }

    // Merge the 8 warps' partials for this segment: 8 -> 4 in pairs, then
    // warp 0 takes in warps 1..3.  Four shared slots, three barriers (turbo4
    // keys: one more first, as the slots hold the query's low halves until
    // every warp has left the unit loop).
    if (CK == KVQ_TURBO4) cta_bar();
    float *rs = red + lane * kRedFloats;
    if (warp >= 4) store_red(rs + (warp - 4) * 32 * kRedFloats, o, m0, m1, l0, l1);
    cta_bar();
    // (every thread has read this segment's length: after the last segment
    // the fused step's lengths may advance)
    if (FUSED && seg_end == u1 && threadIdx.x == kThreads - 1) lengths_read(p);
    if (warp < 4) {
      merge_into(o, m0, m1, l0, l1, rs + warp * 32 * kRedFloats);
      if (warp >= 1) store_red(rs + warp * 32 * kRedFloats, o, m0, m1, l0, l1);
      half_bar();  // warps 0-3 only
    }
    const int stream = seq * geo.KH + seg.sl;
    if (warp == 0) {
#pragma unroll 1
      for (int w = 1; w < 4; ++w) merge_into(o, m0, m1, l0, l1, rs + w * 32 * kRedFloats);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
      }
      // The CTA's partial of this stream, in slot blockIdx.x + stream (a
      // CTA's slice covers consecutive streams, so the slots of all (CTA,
      // stream) pairs are distinct); the merge kernel reads it after this
      // kernel has completed.
      const int64_t slot = static_cast<int64_t>(blockIdx.x) + stream;
      float *po = p.part_o + slot * 8 * kD;
      const int h0 = 2 * tig, h1 = 2 * tig + 1;
      const bool v0 = hg * 8 + h0 < p.G, v1 = hg * 8 + h1 < p.G;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int dlo = v_dim<CV>(mt, g), dhi = v_dim<CV>(mt, g + 8);
        if (v0) { po[h0 * kD + dlo] = o[mt][0]; po[h0 * kD + dhi] = o[mt][2]; }
        if (v1) { po[h1 * kD + dlo] = o[mt][1]; po[h1 * kD + dhi] = o[mt][3]; }
      }
      if (g == 0) {
        if (v0) p.part_ml[slot * 8 + h0] = make_float2(ok ? m0 : -INFINITY, ok ? l0 : 0.0f);
        if (v1) p.part_ml[slot * 8 + h1] = make_float2(ok ? m1 : -INFINITY, ok ? l1 : 0.0f);
      }
    }
    cta_bar();  // the reduction slots are free again

    useg = seg_end;
    ++si;
    if (useg < u1) seg = cursor_at(geo, useg);
  }

  // Query-row copies: segment i's copy is phase i >> 1 of q_bar[i & 1].
  // Wait (bounded) for the last one issued into each buffer, which has
  // already completed unless the run was aborted.
  if (threadIdx.x == 0) {
    for (int i = q_iss - 1; i >= 0 && i >= q_iss - 2; --i)
      mbar_wait_bounded(&q_bar[i & 1], static_cast<uint32_t>(i >> 1) & 1u, nullptr, 100000000ull);
  }

  // After an aborted run, wait (bounded) for this warp's copies still in
  // flight: the units k_fail, k_fail + 8, ... below k_fail + NS were issued
  // (each after the unit NS before it was consumed) but never consumed.
  if (k_fail >= 0 && lane == 0) {
    for (int k = k_fail; k < R && k < k_fail + C::NS; k += kWarps)
      mbar_wait_bounded(&full[k % C::NS], static_cast<uint32_t>(k / C::NS) & 1u, nullptr,
                        100000000ull);
  }
}

// ------------------------------------------------------------------ merge

struct MergeParams {
  MergeArgs a;
  const int32_t *seq_lens;  // after the decode kernel (a fused step has advanced them)
  int n_seqs, n_kv, n_hg, max_len;
  int ups;    // units per work item of the decode kernel's codec pair
  int grid;   // the decode kernel's CTAs
  int fused;  // the decode kernel advances the lengths (a fused decode step)
};

// The log-sum-exp merge of every stream's partials (the second kernel of a
// decode call), one 4-warp CTA per (stream, query head of its group):
// o = sum_j 2^(m_j - M) o_j / L with M = max_j m_j and
// L = sum_j 2^(m_j - M) l_j over the stream's parts j (the partials of the
// CTAs whose slices overlap the stream, in CTA order).  Parts go in windows
// of 64: every lane fetches the (max, sum) of parts base + lane and base +
// 32 + lane, and warp w requests the rows of its parts j = w (mod 4) of the
// window all at once (one round trip for up to 64 parts; the head's 512-byte
// rows come from one SM each, so a stream's merge is spread over as many SMs
// as the group has heads).  Every sum runs in a fixed order (warp w's parts
// in increasing j, then warps 0..3; the sum L lane-strided in warp 0), so the
// output does not depend on timing.  The partition is recomputed from the
// lengths exactly as the decode kernel computed it (a fused step's lengths
// are already advanced, which is the count it attended).
constexpr int kMergeWarps = 4;
constexpr int kMergeRows = 64 / kMergeWarps;  // rows of a warp per window

template <bool ROT>
__global__ void __launch_bounds__(kMergeWarps * 32) decode_merge_kernel(const MergeParams p) {
  __shared__ int32_t pfx[kMaxSeqs + 1];
  __shared__ float4 accs[kMergeWarps][32];
  // The lengths are final once the decode kernel has started (this grid
  // launches after every one of its CTAs passed its own dependency wait), and
  // only a fused step changes them after that: a plain decode's partition is
  // rebuilt while the decode kernel still runs, a fused step's after it.
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (p.fused) grid_dependency_wait();
  if (warp == 0) {
    const int item_tok = p.ups * kUnitTokens;
    int carry = 0;
    for (int base = 0; base < p.n_seqs; base += 32) {
      const int s = base + lane;
      int n = 0;
      if (s < p.n_seqs) {
        int len = p.seq_lens[s];
        len = len < p.max_len ? len : p.max_len;
        n = len > 0 ? (len + item_tok - 1) / item_tok : 0;
      }
      int incl = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
      }
      if (s < p.n_seqs) pfx[s + 1] = carry + incl;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) pfx[0] = 0;
  }
  if (!p.fused) grid_dependency_wait();  // the partials are complete
  grid_launch_dependents();
  __syncthreads();
  const int KH = p.n_kv * p.n_hg;
  const int stream = blockIdx.x, seq = stream / KH, sl = stream % KH;
  const int kvh = sl / p.n_hg, hg = sl % p.n_hg, h = blockIdx.y;
  const int n_s = pfx[seq + 1] - pfx[seq];
  // no keys: the decode kernel wrote the rows; heads past the group: nothing
  if (n_s == 0 || h >= min(8, p.a.G - hg * 8)) return;
  const int64_t U = static_cast<int64_t>(pfx[p.n_seqs]) * KH;
  const int64_t P = p.grid;
  const int64_t S = static_cast<int64_t>(pfx[seq]) * KH + static_cast<int64_t>(sl) * n_s;
  // Part j: with at least one item per CTA (U >= P) the partial of CTA
  // c_first + j; otherwise CTAs hold at most one item and part j is the
  // partial of the owner of item S + j (the owner of item u is
  // floor(((u + 1) P - 1) / U)).
  const bool sparse = U < P;
  const int64_t c_first = ((S + 1) * P - 1) / U;
  const int n_live = sparse ? n_s : static_cast<int>(((S + n_s) * P - 1) / U - c_first + 1);
  auto slot_of = [&](int j) -> int64_t {
    return (sparse ? ((S + j + 1) * P - 1) / U : c_first + j) + stream;
  };
  const float2 *ml = p.a.part_ml + h;                                           // + slot * 8
  const float4 *rows = reinterpret_cast<const float4 *>(p.a.part_o + h * kD) + lane;  // + slot * 256
  // window `base`: (max, sum) of parts base + lane and base + 32 + lane, and
  // this warp's rows of the window (parts base + warp + 4 t), all in flight
  int64_t sa = 0, sb = 0;
  float2 mla, mlb;
  float4 x[kMergeRows];
  auto load_window = [&](int base) {
    sa = base + lane < n_live ? slot_of(base + lane) : 0;
    sb = base + 32 + lane < n_live ? slot_of(base + 32 + lane) : 0;
    mla = base + lane < n_live ? __ldcg(ml + sa * 8) : make_float2(-INFINITY, 0.0f);
    mlb = base + 32 + lane < n_live ? __ldcg(ml + sb * 8) : make_float2(-INFINITY, 0.0f);
#pragma unroll
    for (int t = 0; t < kMergeRows; ++t) {
      const int jr = warp + kMergeWarps * t;  // window-relative part
      const int64_t st = __shfl_sync(0xffffffffu, jr < 32 ? sa : sb, jr & 31);
      x[t] = base + jr < n_live ? __ldcg(rows + st * (8 * kD / 4))
                                : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
  };
  load_window(0);
  float M = fmaxf(mla.x, mlb.x);
  for (int j = 64 + lane; j < n_live; j += 32) M = fmaxf(M, __ldcg(ml + slot_of(j) * 8).x);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float L = 0.0f;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (M != -INFINITY) {
    for (int base = 0;;) {
      const float wa = mla.x == -INFINITY ? 0.0f : fast_exp2(mla.x - M);
      const float wb = mlb.x == -INFINITY ? 0.0f : fast_exp2(mlb.x - M);
      L = fmaf(wa, mla.y, L);  // lane l: parts l, l + 32, l + 64, ... in order
      L = fmaf(wb, mlb.y, L);
#pragma unroll
      for (int t = 0; t < kMergeRows; ++t) {
        const int jr = warp + kMergeWarps * t;
        const float w = __shfl_sync(0xffffffffu, jr < 32 ? wa : wb, jr & 31);
        if (base + jr < n_live) {
          acc.x = fmaf(w, x[t].x, acc.x);
          acc.y = fmaf(w, x[t].y, acc.y);
          acc.z = fmaf(w, x[t].z, acc.z);
          acc.w = fmaf(w, x[t].w, acc.w);
        }
      }
      base += 64;
      if (base >= n_live) break;
      load_window(base);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  }
  accs[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int w = 1; w < kMergeWarps; ++w) {
      const float4 y = accs[w][lane];
      acc.x += y.x; acc.y += y.y; acc.z += y.z; acc.w += y.w;
    }
    merge_write<ROT>(p.a, seq, kvh, hg, h, lane, acc, M, L);
  }
}

template <int CK, int CV, bool FUSED>
cudaError_t launch_split_f(const DecodeParams &p, int grid, cudaStream_t stream) {
  using C = DecodeCfg<CK, CV>;
  static std::atomic<uint64_t> optin{0};
  const cudaError_t e = smem_optin(decode_split_kernel<CK, CV, FUSED>, C::SMEM, optin);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_split_kernel<CK, CV, FUSED>, dim3(grid), dim3(kThreads), C::SMEM,
                    stream, p);
}

template <int CK, int CV>
cudaError_t launch_split(const DecodeParams &p, int grid, cudaStream_t stream) {
  return p.k_new ? launch_split_f<CK, CV, true>(p, grid, stream)
                 : launch_split_f<CK, CV, false>(p, grid, stream);
}

template <int CK>
cudaError_t launch_split_v(int cv, const DecodeParams &p, int grid, cudaStream_t stream) {
  switch (cv) {
    case KVQ_F16: return launch_split<CK, KVQ_F16>(p, grid, stream);
    case KVQ_Q8_0: return launch_split<CK, KVQ_Q8_0>(p, grid, stream);
    case KVQ_Q4_0: return launch_split<CK, KVQ_Q4_0>(p, grid, stream);
    default: return launch_split<CK, KVQ_TURBO4>(p, grid, stream);
  }
}

}  // namespace

DecodePlan plan_decode(const kvq_layer &L, int max_len, int num_sms) {
  DecodePlan pl;
  const int G = L.n_q_heads / L.n_kv_heads;
  pl.n_hgroups = (G + 7) / 8;
  const int64_t streams = static_cast<int64_t>(L.n_seqs) * L.n_kv_heads * pl.n_hgroups;
  const int upi = items_units(L.codec_k, L.codec_v);
  const int64_t item_tok = static_cast<int64_t>(kUnitTokens) * upi;
  const int64_t max_items = streams * ((max_len + item_tok - 1) / item_tok);
  // Two resident CTAs per SM, but at least ~8 units (one per warp) per CTA:
  // short contexts spread over enough CTAs that each warp has about one
  // unit (a 4096-key layer: 16.9 -> 14.9 us against 32 units per CTA),
  // without splitting into partials that hold less than a unit per warp.
  int64_t grid = static_cast<int64_t>(num_sms > 0 ? num_sms : 148) * 2;
  const int64_t by_work = (max_items * upi + 7) / 8;
  if (grid > by_work) grid = by_work;
  if (grid < 1) grid = 1;
  pl.grid = static_cast<int>(grid);
  pl.slots = grid + streams;
  pl.ticket_bytes = kDecodeTicketBytes;  // fixed region: never overlaps another plan's partials
  pl.ml_bytes = pl.slots * 8 * 8;
  pl.o_bytes = pl.slots * 8 * kD * 4;
  pl.ws_bytes = pl.ticket_bytes + pl.ml_bytes + pl.o_bytes;
  return pl;
}

cudaError_t launch_decode(const kvq_layer &L, const DecodePlan &pl, const void *q, float scale,
                          void *out, float *lse, int max_len, void *workspace,
                          cudaStream_t stream, const void *k_new, const void *v_new) {
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  DecodeParams p;
  p.k_cache = static_cast<const uint8_t *>(L.k_cache);
  p.v_cache = static_cast<const uint8_t *>(L.v_cache);
  p.seq_lens = L.seq_lens;
  p.k_new = static_cast<const __half *>(k_new);
  p.v_new = static_cast<const __half *>(v_new);
  p.lens_rw = L.seq_lens;
  p.rd_ctr = reinterpret_cast<unsigned *>(ws) + (kDecodeTicketBytes / 4 - 1);
  p.q = static_cast<const __half *>(q);
  p.part_ml = reinterpret_cast<float2 *>(ws + pl.ticket_bytes);
  p.part_o = reinterpret_cast<float *>(ws + pl.ticket_bytes + pl.ml_bytes);
  p.out = static_cast<__half *>(out);
  p.lse = lse;
  p.err = L.err;
  p.table = L.pages_per_seq > 0 ? L.block_table : nullptr;
  p.pages_per_seq = L.pages_per_seq;
  p.n_pages = L.n_pages;
  p.n_seqs = L.n_seqs;
  p.n_kv = L.n_kv_heads;
  p.n_q = L.n_q_heads;
  p.G = L.n_q_heads / L.n_kv_heads;
  p.n_hg = pl.n_hgroups;
  p.capacity = L.capacity;
  p.max_len = max_len;
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaError_t e;
  switch (L.codec_k) {
    case KVQ_F16: e = launch_split_v<KVQ_F16>(L.codec_v, p, pl.grid, stream); break;
    case KVQ_Q8_0: e = launch_split_v<KVQ_Q8_0>(L.codec_v, p, pl.grid, stream); break;
    case KVQ_Q4_0: e = launch_split_v<KVQ_Q4_0>(L.codec_v, p, pl.grid, stream); break;
    default: e = launch_split_v<KVQ_TURBO4>(L.codec_v, p, pl.grid, stream); break;
  }
  if (e != cudaSuccess) return e;
  MergeParams mp;
  mp.a = {p.part_ml, p.part_o, p.out, p.lse, p.n_q, p.G};
  mp.seq_lens = L.seq_lens;
  mp.n_seqs = p.n_seqs;
  mp.n_kv = p.n_kv;
  mp.n_hg = p.n_hg;
  mp.max_len = max_len;
  mp.ups = items_units(L.codec_k, L.codec_v);
  mp.grid = pl.grid;
  mp.fused = k_new != nullptr;
  const dim3 mgrid(static_cast<unsigned>(p.n_seqs * p.n_kv * p.n_hg),
                   static_cast<unsigned>(p.G < 8 ? p.G : 8));
  const dim3 mblock(kMergeWarps * 32);
  return L.codec_v == KVQ_TURBO4
             ? launch_pdl(decode_merge_kernel<true>, mgrid, mblock, 0, stream, mp)
             : launch_pdl(decode_merge_kernel<false>, mgrid, mblock, 0, stream, mp);
}

}  // namespace kvq
