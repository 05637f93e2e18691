// evict.cu -- probe-scored eviction over a block-quantized KV cache.
//
// The "Sparse KV eviction" item of the "How It Works" section of the GitHot
// listing of VITRIOL: an attention probe (q.K softmax with exponential decay)
// scores the cache cells, the lowest-scored middle cells are evicted first,
// and the attention sinks (first cells) and the recent cells are protected.
// Three kernels:
//
//  * probe_kernel: for every token t below a sequence's length, the softmax
//    weight that the decode query of every query head puts on t, summed over
//    the query heads (the probe mass), folded into the running score:
//    score = decay * score + mass.  The softmax normaliser of each head is the
//    log-sum-exp that attn_decode returns for the same query, so the probe is
//    one more pass over K only.  One CTA per (sequence, page of 256 tokens):
//    warp w takes units w and w + 8 of the page for every (kv head, group of
//    up to 8 query heads) in a fixed order, so the sums are deterministic and
//    need no atomics; S = K Q^T runs on mma.sync with the K bytes loaded
//    straight into the operand registers (the fragment-native unit layout).
//  * select_kernel: per sequence, the n smallest (score, t) pairs among the
//    middle positions [n_sink, len - n_recent): a radix select over the
//    order-preserving bits of the fp32 scores (digits of 11, 11 and 10 bits)
//    finds the threshold key; every key below it is taken and the keys equal
//    to it are taken in position order; the positions are written in
//    increasing order by one block-wide scan per 8192 positions.
//  * compact_kernel: the kept tokens move down in order, bytes unchanged,
//    into a second cache of the same layout.  A row's bytes sit inside its
//    16-token unit at offsets whose row-dependent bits are fixed per codec and
//    side (RowBits), so each destination 16-byte chunk is gathered from the
//    source units (staged in shared memory) piece by piece, with the source
//    row of every destination row found by a binary search of the sorted
//    eviction list.
#include <cuda_runtime.h>

#include <limits.h>
#include <math.h>

#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

// ------------------------------------------------------------------ probe

constexpr int kProbeWarps = 8;
constexpr int kProbeUnits = 2 * kProbeWarps;  // units per CTA: one page
static_assert(kProbeUnits == kPageUnits, "a probe CTA covers exactly one page");

struct ProbeParams {
  const uint8_t *k_cache;
  const int32_t *seq_lens;
  const __half *q;     // [n_seqs][n_q][128]
  const float *lse;    // [n_seqs][n_q], natural log
  float *scores;       // [n_seqs][capacity]
  int32_t *err;
  const int32_t *table;
  int n_kv, n_q, G, n_hg, capacity, pages_per_seq, n_pages;
  float scale_log2, decay;
};

// The K operand bytes one lane needs from one unit: the 16-byte pieces at
// c * 512 + lane * 16 and, for block codecs, the scales of rows g and g + 8.
template <int CK>
struct KFrag {
  static constexpr int NW = CK == KVQ_F16 ? 8 : (CK == KVQ_Q8_0 ? 4 : 2);
  uint4 w[NW];
  uint4 sc;  // turbo4: .x = scales of rows g and g + 8
};

template <int CK>
__device__ __forceinline__ void kfrag_load(const uint8_t *ku, int lane, KFrag<CK> &f) {
#pragma unroll
  for (int c = 0; c < KFrag<CK>::NW; ++c)
    f.w[c] = __ldcs(reinterpret_cast<const uint4 *>(ku + c * 512 + lane * 16));
  if (CK == KVQ_TURBO4)
    f.sc.x = __ldcs(reinterpret_cast<const unsigned int *>(ku + 1024 + (lane >> 2) * 4));
  else if (CK != KVQ_F16)
    f.sc = __ldcs(reinterpret_cast<const uint4 *>(ku + unit_scale_offset(CK) + (lane >> 2) * 16));
}

// S (16 tokens x 8 heads) of one unit from its fragments, unscaled: exact
// block dequantization (two MMAs per 32-value block into a fresh
// accumulator, then s += d * partial), fp32 accumulation.
template <int CK>
__device__ __forceinline__ void kfrag_scores(const KFrag<CK> &f, const uint32_t (&qb)[8][2],
                                             const uint32_t (&qlo)[8][2], float (&s)[4]) {
  s[0] = s[1] = s[2] = s[3] = 0.0f;
  if (CK == KVQ_F16) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint4 r0 = f.w[2 * b], r1 = f.w[2 * b + 1];
      const uint32_t a0[4] = {r0.x, r1.x, r0.y, r1.y};
      const uint32_t a1[4] = {r0.z, r1.z, r0.w, r1.w};
      mma16816(s, a0, qb[2 * b][0], qb[2 * b][1]);
      mma16816(s, a1, qb[2 * b + 1][0], qb[2 * b + 1][1]);
    }
    return;
  }
  if (CK == KVQ_TURBO4) {  // one scale per row: one accumulator for the four groups
    // the rotated query as the fp16 pair qb + qlo: both halves multiply the
    // same (exact) nibble operands
    float sb[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint4 w = f.w[b >> 1];
      const uint32_t W0 = (b & 1) ? w.z : w.x, W1 = (b & 1) ? w.w : w.y;
      const uint32_t X0 = W0 >> 8, X1 = W1 >> 8;
      const uint32_t a0[4] = {u4_pair_minus8(W0), u4_pair_minus8(W1), u4_pair_minus8(X0),
                              u4_pair_minus8(X1)};
      const uint32_t a1[4] = {u4_pair_minus8_hi(W0), u4_pair_minus8_hi(W1),
                              u4_pair_minus8_hi(X0), u4_pair_minus8_hi(X1)};
      mma16816(sb, a0, qb[2 * b][0], qb[2 * b][1]);
      mma16816(sb, a1, qb[2 * b + 1][0], qb[2 * b + 1][1]);
      mma16816(sb, a0, qlo[2 * b][0], qlo[2 * b][1]);
      mma16816(sb, a1, qlo[2 * b + 1][0], qlo[2 * b + 1][1]);
    }
    const float dlo = __half2float(__ushort_as_half(static_cast<unsigned short>(f.sc.x)));
    const float dhi = __half2float(__ushort_as_half(static_cast<unsigned short>(f.sc.x >> 16)));
    s[0] = dlo * sb[0];
    s[1] = dlo * sb[1];
    s[2] = dhi * sb[2];
    s[3] = dhi * sb[3];
    return;
  }
  const uint32_t dl[2] = {f.sc.x, f.sc.y}, dh[2] = {f.sc.z, f.sc.w};
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    float sb[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (CK == KVQ_Q8_0) {
      const uint4 w = f.w[b];
      const uint32_t a0[4] = {s8_pair_02(w.x), s8_pair_02(w.z), s8_pair_13(w.x), s8_pair_13(w.z)};
      const uint32_t a1[4] = {s8_pair_02(w.y), s8_pair_02(w.w), s8_pair_13(w.y), s8_pair_13(w.w)};
      mma16816(sb, a0, qb[2 * b][0], qb[2 * b][1]);
      mma16816(sb, a1, qb[2 * b + 1][0], qb[2 * b + 1][1]);
    } else {
      const uint4 w = f.w[b >> 1];
      const uint32_t W0 = (b & 1) ? w.z : w.x, W1 = (b & 1) ? w.w : w.y;
      const uint32_t X0 = W0 >> 8, X1 = W1 >> 8;
      const uint32_t a0[4] = {u4_pair_minus8(W0), u4_pair_minus8(W1), u4_pair_minus8(X0),
                              u4_pair_minus8(X1)};
      const uint32_t a1[4] = {u4_pair_minus8_hi(W0), u4_pair_minus8_hi(W1),
                              u4_pair_minus8_hi(X0), u4_pair_minus8_hi(X1)};
      mma16816(sb, a0, qb[2 * b][0], qb[2 * b][1]);
      mma16816(sb, a1, qb[2 * b + 1][0], qb[2 * b + 1][1]);
    }
    const float dlo =
        __half2float(__ushort_as_half(static_cast<unsigned short>(dl[b >> 1] >> (16 * (b & 1)))));
    const float dhi =
        __half2float(__ushort_as_half(static_cast<unsigned short>(dh[b >> 1] >> (16 * (b & 1)))));
    s[0] = fmaf(dlo, sb[0], s[0]);
    s[1] = fmaf(dlo, sb[1], s[1]);
    s[2] = fmaf(dhi, sb[2], s[2]);
    s[3] = fmaf(dhi, sb[3], s[3]);
  }
}

// B fragments of Q (query head g of the group; zero past the group) in the
// head-dim order of the codec's K unit layout.
template <int CK>
__device__ __forceinline__ void probe_q_frags(const __half *qrow0, int nh, int lane,
                                              uint32_t (&qb)[8][2], uint32_t (&qlo)[8][2]) {
  const int g = lane >> 2, tig = lane & 3;
  const bool hvalid = g < nh;
  const __half *qrow = qrow0 + (hvalid ? g : 0) * kD;
  if (CK == KVQ_TURBO4) {  // turbo4 keys: the rotated query (fp16 pair)
    rotated_q_frags(qrow, hvalid, tig, qb, qlo,
                    [](const __half *p) { return __ldg(reinterpret_cast<const uint2 *>(p)); });
  } else {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int base = 32 * (c >> 1) + 16 * (c & 1) + 4 * tig;
      uint2 v = make_uint2(0u, 0u);
      if (hvalid) v = __ldg(reinterpret_cast<const uint2 *>(qrow + base));
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

template <int CK>
__global__ void __launch_bounds__(kProbeWarps * 32) probe_kernel(const ProbeParams p) {
  grid_dependency_wait();
  const int s = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
  const int len = min(p.seq_lens[s], p.capacity);
  const int u_base = blockIdx.x * kProbeUnits;
  if (u_base * kUnitTokens >= len) {
    grid_launch_dependents();
    return;
  }
  constexpr int UB = unit_bytes(CK);
  int64_t unit0, stride_h;  // unit u_base of kv head 0; kv head step
  if (p.table) {
    const int pg = page_of(p.table, p.pages_per_seq, p.n_pages, s, blockIdx.x);
    if (pg < 0) {
      if (threadIdx.x == 0) set_err(p.err, KVQ_DEVERR_PAGE);
      return;
    }
    unit0 = static_cast<int64_t>(pg) * p.n_kv * kPageUnits;
    stride_h = kPageUnits;
  } else {
    stride_h = p.capacity / kUnitTokens;
    unit0 = static_cast<int64_t>(s) * p.n_kv * stride_h + u_base;
  }
  int nvalid[2];
#pragma unroll
  for (int i = 0; i < 2; ++i)
    nvalid[i] = min(kUnitTokens, len - (u_base + warp + i * kProbeWarps) * kUnitTokens);
  float acc[2][2] = {{0.0f, 0.0f}, {0.0f, 0.0f}};  // [unit][token g, g + 8]
  const float *lse_s = p.lse + static_cast<int64_t>(s) * p.n_q;
  const __half *q_s = p.q + static_cast<int64_t>(s) * p.n_q * kD;
  const int n_streams = p.n_kv * p.n_hg;
  for (int st = 0; st < n_streams; ++st) {
    const int kvh = st / p.n_hg, hg = st - kvh * p.n_hg;
    KFrag<CK> f[2];
#pragma unroll
    for (int i = 0; i < 2; ++i)
      if (nvalid[i] > 0)
        kfrag_load<CK>(p.k_cache + (unit0 + kvh * stride_h + warp + i * kProbeWarps) * UB, lane,
                       f[i]);
    const int nh = min(8, p.G - hg * 8);
    uint32_t qb[8][2], qlo[8][2];
    probe_q_frags<CK>(q_s + (static_cast<int64_t>(kvh) * p.G + hg * 8) * kD, nh, lane, qb, qlo);
    // log2-domain normalisers of the two heads in this lane's columns
    const int h0 = 2 * tig, h1 = 2 * tig + 1;
    const int64_t hrow = static_cast<int64_t>(kvh) * p.G + hg * 8;
    const float n0 = h0 < nh ? lse_s[hrow + h0] * 1.4426950408889634f : INFINITY;
    const float n1 = h1 < nh ? lse_s[hrow + h1] * 1.4426950408889634f : INFINITY;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (nvalid[i] <= 0) continue;  // warp-uniform
      float sc[4];
      kfrag_scores<CK>(f[i], qb, qlo, sc);
      const float p0 = fast_exp2(fmaf(sc[0], p.scale_log2, -n0));
      const float p1 = fast_exp2(fmaf(sc[1], p.scale_log2, -n1));
      const float p2 = fast_exp2(fmaf(sc[2], p.scale_log2, -n0));
      const float p3 = fast_exp2(fmaf(sc[3], p.scale_log2, -n1));
      float t0 = g < nvalid[i] ? p0 + p1 : 0.0f;
      float t1 = g + 8 < nvalid[i] ? p2 + p3 : 0.0f;
      t0 += __shfl_xor_sync(0xffffffffu, t0, 1);
      t1 += __shfl_xor_sync(0xffffffffu, t1, 1);
      t0 += __shfl_xor_sync(0xffffffffu, t0, 2);
      t1 += __shfl_xor_sync(0xffffffffu, t1, 2);
      acc[i][0] += t0;
      acc[i][1] += t1;
    }
  }
  // lane l updates token l & 15 of unit (l >> 4 ? second : first); the sums
  // of token r sit in lane 4 * (r & 7), slot r >> 3.
  const int r = lane & 15, src = 4 * (r & 7);
  const float a00 = __shfl_sync(0xffffffffu, acc[0][0], src);
  const float a01 = __shfl_sync(0xffffffffu, acc[0][1], src);
  const float a10 = __shfl_sync(0xffffffffu, acc[1][0], src);
  const float a11 = __shfl_sync(0xffffffffu, acc[1][1], src);
  const int i = lane >> 4;
  const float mass = i == 0 ? (r < 8 ? a00 : a01) : (r < 8 ? a10 : a11);
  const int t = (u_base + warp + i * kProbeWarps) * kUnitTokens + r;
  if (t < len) {
    float *sp = p.scores + static_cast<int64_t>(s) * p.capacity + t;
    *sp = fmaf(p.decay, *sp, mass);
  }
  grid_launch_dependents();
}

// ------------------------------------------------------------------ select

constexpr int kSelThreads = 1024;
constexpr int kSelItems = 8;  // consecutive positions per thread in the output pass
constexpr int kSelBins = 2048;

struct SelectParams {
  const float *scores;
  const int32_t *seq_lens;
  int32_t *evict;    // [n_seqs][n_evict]
  int32_t *n_out;    // [n_seqs]
  int capacity, n_sink, n_recent, n_evict;
};

// Order-preserving unsigned key of an fp32 score: -0 ties with +0 (as the
// float comparison does), NaN orders after every number.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7fffffffu) > 0x7f800000u) b = 0x7fffffffu;
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Inclusive sum over the CTA's threads (thread order); `red` holds 32 words.
__device__ __forceinline__ uint32_t block_scan_incl(uint32_t v, uint32_t *red, uint32_t *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = red[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    red[lane] = w;
  }
  __syncthreads();
  const uint32_t r = v + (warp > 0 ? red[warp - 1] : 0u);
  *total = red[31];
  __syncthreads();  // red is reused by the next call
  return r;
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(const SelectParams p) {
  __shared__ uint32_t hist[kSelBins];
  __shared__ uint32_t red[32];
  __shared__ uint32_t sel_digit, sel_below;
  grid_dependency_wait();
  const int s = blockIdx.x;
  const int len = min(max(p.seq_lens[s], 0), p.capacity);
  const int lo = p.n_sink, hi = len - p.n_recent;
  const int n = hi - lo;
  const int k = n > 0 ? min(p.n_evict, n) : 0;
  if (k <= 0) {
    if (threadIdx.x == 0) p.n_out[s] = 0;
    grid_launch_dependents();
    return;
  }
  const float *sc = p.scores + static_cast<int64_t>(s) * p.capacity;
  // radix select of the k-th smallest key, most significant digit first
  uint32_t prefix = 0u, pmask = 0u, kk = static_cast<uint32_t>(k);
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t dmask = pass == 2 ? 0x3ffu : 0x7ffu;
    for (int i = threadIdx.x; i < kSelBins; i += kSelThreads) hist[i] = 0u;
    __syncthreads();
    for (int t = lo + threadIdx.x; t < hi; t += kSelThreads) {
      const uint32_t key = order_key(sc[t]);
      if ((key & pmask) == prefix) atomicAdd(&hist[(key >> sh) & dmask], 1u);
    }
    __syncthreads();
    const uint32_t a = hist[2 * threadIdx.x], b = hist[2 * threadIdx.x + 1];
    uint32_t tot;
    const uint32_t incl = block_scan_incl(a + b, red, &tot);
    const uint32_t excl = incl - a - b;
    if (excl < kk && kk <= excl + a) {
      sel_digit = 2 * threadIdx.x;
      sel_below = excl;
    } else if (excl + a < kk && kk <= incl) {
      sel_digit = 2 * threadIdx.x + 1;
      sel_below = excl + a;
    }
    __syncthreads();
    prefix |= sel_digit << sh;
    pmask |= dmask << sh;
    kk -= sel_below;
    __syncthreads();
  }
  // every key below the threshold, and the first kk keys equal to it
  const uint32_t T = prefix;
  uint32_t out_base = 0u, eq_base = 0u;
  int32_t *ev = p.evict + static_cast<int64_t>(s) * p.n_evict;
#pragma unroll 1
  for (int c0 = lo; c0 < hi; c0 += kSelThreads * kSelItems) {
    const int t0 = c0 + threadIdx.x * kSelItems;
    uint32_t key[kSelItems];
    uint32_t lt = 0u, eq = 0u;
#pragma unroll
    for (int j = 0; j < kSelItems; ++j) {
      key[j] = t0 + j < hi ? order_key(sc[t0 + j]) : 0xffffffffu;
      lt += key[j] < T;
      eq += t0 + j < hi && key[j] == T;
    }
    const uint32_t packed = lt | (eq << 16);
    uint32_t tot;
    const uint32_t incl = block_scan_incl(packed, red, &tot);
    const uint32_t excl = incl - packed;
    uint32_t eq_seen = eq_base + (excl >> 16);
    uint32_t o = out_base + (excl & 0xffffu) + min(eq_seen, kk) - min(eq_base, kk);
#pragma unroll
    for (int j = 0; j < kSelItems; ++j) {
      if (t0 + j >= hi) break;
      const bool take = key[j] < T || (key[j] == T && eq_seen < kk);
      eq_seen += key[j] == T;
      if (take) {
        if (o < static_cast<uint32_t>(k)) ev[o] = t0 + j;  // o < k always; kept as a guard
        ++o;
      }
    }
    const uint32_t tot_lt = tot & 0xffffu, tot_eq = tot >> 16;
    out_base += tot_lt + min(eq_base + tot_eq, kk) - min(eq_base, kk);
    eq_base += tot_eq;
  }
  if (threadIdx.x == 0) p.n_out[s] = k;
  grid_launch_dependents();
}

// ------------------------------------------------------------------ compact

// One region of the unit layout (the values, or the 128 bytes of block
// scales): its byte offset x inside the region holds bit i of the token row
// at bit Pi, and every other bit of x is the same for all rows.  A row's
// bytes inside the region are the runs of 2^min(Pi) bytes between the row
// bits.
template <int BASE, int SIZE, int P0, int P1, int P2, int P3>
struct RowBits {
  static constexpr int kBase = BASE;
  static constexpr uint32_t kMask = (1u << P0) | (1u << P1) | (1u << P2) | (1u << P3);
  static constexpr int kMinBit = P0 < P1 ? (P0 < P2 ? (P0 < P3 ? P0 : P3) : (P2 < P3 ? P2 : P3))
                                         : (P1 < P2 ? (P1 < P3 ? P1 : P3) : (P2 < P3 ? P2 : P3));
  static constexpr int kPiece = kMinBit >= 4 ? 16 : (1 << kMinBit);  // bytes per gather
  __host__ __device__ static constexpr int row_of(uint32_t x) {
    return static_cast<int>(((x >> P0) & 1u) | (((x >> P1) & 1u) << 1) | (((x >> P2) & 1u) << 2) |
                            (((x >> P3) & 1u) << 3));
  }
  __device__ static __forceinline__ uint32_t dep(int r) {
    return ((static_cast<uint32_t>(r) & 1u) << P0) | (((static_cast<uint32_t>(r) >> 1) & 1u) << P1) |
           (((static_cast<uint32_t>(r) >> 2) & 1u) << P2) |
           (((static_cast<uint32_t>(r) >> 3) & 1u) << P3);
  }
};

// Row bit positions of each (codec, side): the unit layout of include/kvq.h
// (K side rows g = r & 7 and rh = r >> 3 of the A operand; V side rows
// par = r & 1, tig = (r >> 1) & 3 and rh = r >> 3 of the B operand).
template <int CODEC, int SIDE>
struct UnitRows;
template <> struct UnitRows<KVQ_F16, 0> {
  using D = RowBits<0, 4096, 6, 7, 8, 9>;
  using S = D;
  static constexpr bool kScales = false;
};
template <> struct UnitRows<KVQ_Q8_0, 0> {
  using D = RowBits<0, 2048, 6, 7, 8, 3>;
  using S = RowBits<2048, 128, 4, 5, 6, 3>;
  static constexpr bool kScales = true;
};
template <> struct UnitRows<KVQ_Q4_0, 0> {
  using D = RowBits<0, 1024, 6, 7, 8, 2>;
  using S = RowBits<1024, 128, 4, 5, 6, 3>;
  static constexpr bool kScales = true;
};
template <> struct UnitRows<KVQ_TURBO4, 0> {
  using D = RowBits<0, 1024, 6, 7, 8, 2>;
  using S = RowBits<1024, 32, 2, 3, 4, 1>;
  static constexpr bool kScales = true;
};
template <> struct UnitRows<KVQ_F16, 1> {
  using D = RowBits<0, 4096, 1, 4, 5, 3>;
  using S = D;
  static constexpr bool kScales = false;
};
template <> struct UnitRows<KVQ_Q8_0, 1> {
  using D = RowBits<0, 2048, 1, 4, 5, 2>;
  using S = RowBits<2048, 128, 1, 5, 6, 2>;
  static constexpr bool kScales = true;
};
template <> struct UnitRows<KVQ_Q4_0, 1> {
  using D = RowBits<0, 1024, 1, 4, 5, 0>;
  using S = RowBits<1024, 128, 1, 5, 6, 2>;
  static constexpr bool kScales = true;
};
template <> struct UnitRows<KVQ_TURBO4, 1> {
  using D = RowBits<0, 1024, 1, 4, 5, 0>;
  using S = RowBits<1024, 32, 1, 3, 4, 2>;
  static constexpr bool kScales = true;
};

constexpr int kCpThreads = 256;
constexpr int kCpUnits = 8;                    // destination units per CTA
constexpr int kCpRows = kCpUnits * kUnitTokens;  // 128 destination rows
constexpr int kCpSlots = 10;                   // source units staged at a time
static_assert(kPageUnits % kCpUnits == 0, "a destination run lies inside one page");

struct CompactParams {
  const uint8_t *src[2];  // K, V caches (or pools)
  uint8_t *dst[2];
  const int32_t *seq_lens;
  const int32_t *evict;   // [n_seqs][max_evict], increasing
  const int32_t *n_ev;    // [n_seqs]
  const float *scores;    // [n_seqs][capacity] or null
  float *scores_dst;
  int32_t *lens_dst;      // [n_seqs] or null
  int32_t *err;
  const int32_t *table;
  int max_evict, n_kv, capacity, pages_per_seq, n_pages;
};

struct CompactSmem {
  int32_t srcpos[kCpRows];   // source token of each destination row of the run
  int32_t slot[kCpRows];     // staging slot (distinct source units, in row order)
  int32_t offd[kCpRows];     // shared-memory offset of the row in the values region
  int32_t offs[kCpRows];     // ... in the scales region
  int32_t slot_unit[kCpRows];  // source unit of each slot
  int32_t red[kCpThreads / 32];
  int32_t win[kCpThreads];   // a window of c_j = e[j] - j of the eviction list
  int64_t offgd[kUnitTokens];  // a unit gathered from global memory: row offsets
  int64_t offgs[kUnitTokens];
  uint64_t bar;              // completion of the round's bulk copies
};

__device__ __forceinline__ int64_t unit_index(const CompactParams &p, int s, int kvh, int u) {
  if (!p.table)
    return (static_cast<int64_t>(s) * p.n_kv + kvh) * (p.capacity / kUnitTokens) + u;
  const int pg = page_of(p.table, p.pages_per_seq, p.n_pages, s, u / kPageUnits);
  if (pg < 0) return -1;
  return (static_cast<int64_t>(pg) * p.n_kv + kvh) * kPageUnits + u % kPageUnits;
}

// Gather one 16-byte chunk (offset x0 inside region R of destination unit
// ud of the run) from the source units: staged in shared memory (off: int32
// offsets into the stage) or, for a unit with too many source units, read
// straight from the cache (off: int64 offsets into it).
template <typename R, typename OffT>
__device__ __forceinline__ uint4 gather_chunk(const uint8_t *stage, const OffT *off, int ud,
                                              int rows_valid, uint32_t x0) {
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  constexpr int P = R::kPiece;
  // x0 is 16-aligned, so x0 + j (j < 16) has x0's bits above bit 3 and j's
  // below: the row and the row-free offset split into a per-chunk part and
  // a compile-time part.
  const int rbase = ud * kUnitTokens + R::row_of(x0);
  const uint8_t *cbase = stage + (x0 & ~R::kMask);
#pragma unroll
  for (int j = 0; j < 16; j += P) {
    const int i = rbase + R::row_of(static_cast<uint32_t>(j));
    if (i >= rows_valid) continue;  // rows past the new length stay zero
    const uint8_t *src = cbase + off[i] + (static_cast<uint32_t>(j) & ~R::kMask);
    if (P == 16) {
      const uint4 v = *reinterpret_cast<const uint4 *>(src);
      w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if (P == 8) {
      const uint2 v = *reinterpret_cast<const uint2 *>(src);
      w[j / 4] = v.x;
      w[j / 4 + 1] = v.y;
    } else if (P == 4) {
      w[j / 4] = *reinterpret_cast<const uint32_t *>(src);
    } else if (P == 2) {
      w[j / 4] |= static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(src)) << (8 * (j & 3));
    } else {
      w[j / 4] |= static_cast<uint32_t>(*src) << (8 * (j & 3));
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// One CTA's run of kCpUnits destination units of one (sequence, kv head,
// side): source rows by binary search, distinct source units in slots,
// rounds of destination units whose sources fit kCpSlots slots.  Each round's
// source units arrive by bulk async copies on one mbarrier (all of them in
// flight together), then every thread gathers 16-byte destination chunks and
// stores them straight to global memory.  A destination unit whose rows come
// from more than kCpSlots source units (many evictions inside 16 kept rows)
// is gathered from global memory directly.
template <int CODEC, int SIDE>
__device__ __forceinline__ void compact_run(const CompactParams &p, CompactSmem &sm,
                                            uint8_t *stage, int s, int kvh, int u0, int len,
                                            int n, int rows) {
  using L = UnitRows<CODEC, SIDE>;
  using D = typename L::D;
  using S = typename L::S;
  constexpr int UB = unit_bytes(CODEC);
  constexpr int CH = UB / 16;  // 16-byte chunks per unit
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t *ev = p.evict + static_cast<int64_t>(s) * p.max_evict;
  // Source token of destination row w: w plus the number of evicted
  // positions e[j] with c_j = e[j] - j <= w (c is non-decreasing).  The count
  // at the run's first row comes from a parallel search (each round tests
  // kCpThreads evenly spaced candidates: two rounds for 65536 entries); the
  // rows then count inside windows of the list staged in shared memory.
  const int w0 = u0 * kUnitTokens;
  int lo = 0, hi = n;  // the count a0 lies in [lo, hi]
  while (lo < hi) {
    const int step = (hi - lo + kCpThreads - 1) / kCpThreads;
    const int j = lo + tid * step;
    const bool le = j < hi && ev[j] - j <= w0;
    const int m = __syncthreads_count(le);  // le holds for a prefix of the candidates
    if (m == 0) {
      hi = lo;
    } else {
      const int last = lo + (m - 1) * step;
      hi = min(hi, lo + m * step);
      lo = last + 1;
    }
  }
  int cnt = -1;  // this row's count once its window held it
  for (int base = lo;; base += kCpThreads) {
    sm.win[tid] = base + tid < n ? ev[base + tid] - (base + tid) : INT_MAX;
    __syncthreads();
    bool open = false;
    if (tid < rows && cnt < 0) {
      const int w = w0 + tid;
      int a = 0, b = kCpThreads;  // entries of the window with c <= w
      while (a < b) {
        const int mid = (a + b) >> 1;
        if (sm.win[mid] <= w) a = mid + 1;
        else b = mid;
      }
      if (a < kCpThreads || base + kCpThreads >= n) cnt = base + a;
      else open = true;  // every entry of the window counts: look further
    }
    if (!__syncthreads_or(open)) break;
  }
  if (tid < kCpRows) sm.srcpos[tid] = tid < rows ? min(max(w0 + tid + cnt, 0), len - 1) : 0;
  __syncthreads();
  if (SIDE == 0 && kvh == 0 && p.scores && tid < rows) {
    const int64_t base = static_cast<int64_t>(s) * p.capacity;
    p.scores_dst[base + u0 * kUnitTokens + tid] = p.scores[base + sm.srcpos[tid]];
  }
  // staging slots: one per run of rows with the same source unit
  int su = 0, before = 0;
  bool head = false;
  if (tid < kCpRows) {  // warps 0..3, whole warps
    su = sm.srcpos[tid] / kUnitTokens;
    head = tid < rows && (tid == 0 || sm.srcpos[tid - 1] / kUnitTokens != su);
    const uint32_t bal = __ballot_sync(0xffffffffu, head);
    before = __popc(bal & ((1u << lane) - 1u));
    if (lane == 31) sm.red[warp] = before + (head ? 1 : 0);
  }
  __syncthreads();
  if (tid < kCpRows) {
    int wofs = 0;
    for (int k = 0; k < warp; ++k) wofs += sm.red[k];
    const int slot = wofs + before + (head ? 1 : 0) - 1;
    sm.slot[tid] = slot;
    if (head) sm.slot_unit[slot] = su;
  }
  __syncthreads();
  const int n_units = (rows + kUnitTokens - 1) / kUnitTokens;
  const int64_t d_unit0 = unit_index(p, s, kvh, u0);
  if (d_unit0 < 0) {
    if (tid == 0) set_err(p.err, KVQ_DEVERR_PAGE);
    return;
  }
  const uint8_t *src = p.src[SIDE];
  uint8_t *dst = p.dst[SIDE];
  uint32_t phase = 0;
  int ua = 0;
  while (ua < n_units) {  // rounds of destination units whose sources fit the slots
    const int s_first = sm.slot[ua * kUnitTokens];
    if (sm.slot[min((ua + 1) * kUnitTokens, rows) - 1] - s_first >= kCpSlots) {
      // this unit's rows come from more source units than the stage holds:
      // gather it straight from global memory
      const int r0 = ua * kUnitTokens, r1 = min(r0 + kUnitTokens, rows);
      if (tid >= r0 && tid < r1) {
        int64_t gi = unit_index(p, s, kvh, sm.srcpos[tid] / kUnitTokens);
        if (gi < 0) {
          set_err(p.err, KVQ_DEVERR_PAGE);
          gi = 0;
        }
        const int rs = sm.srcpos[tid] % kUnitTokens;
        sm.offgd[tid - r0] = gi * UB + D::kBase + D::dep(rs);
        sm.offgs[tid - r0] = gi * UB + S::kBase + S::dep(rs);
      }
      __syncthreads();
      for (int c = tid; c < CH; c += kCpThreads) {
        const uint32_t x = static_cast<uint32_t>(c) * 16u;
        uint4 v;
        if (!L::kScales || x < static_cast<uint32_t>(S::kBase))
          v = gather_chunk<D>(src, sm.offgd, 0, r1 - r0, x - D::kBase);
        else
          v = gather_chunk<S>(src, sm.offgs, 0, r1 - r0, x - S::kBase);
        reinterpret_cast<uint4 *>(dst + (d_unit0 + ua) * UB)[c] = v;
      }
      __syncthreads();
      ++ua;
      continue;
    }
    int ub = ua + 1;
    while (ub < n_units && sm.slot[min((ub + 1) * kUnitTokens, rows) - 1] - s_first < kCpSlots)
      ++ub;
    const int n_sl = sm.slot[min(ub * kUnitTokens, rows) - 1] - s_first + 1;
    if (tid == 0) {
      // the previous round's reads of the stage are ordered before these
      // async writes by the barrier that ended the round and this fence
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&sm.bar, static_cast<uint32_t>(n_sl * UB));
      for (int k = 0; k < n_sl; ++k) {
        int64_t gi = unit_index(p, s, kvh, sm.slot_unit[s_first + k]);
        if (gi < 0) {
          set_err(p.err, KVQ_DEVERR_PAGE);
          gi = 0;
        }
        bulk_copy_g2s(stage + k * UB, src + gi * UB, UB, &sm.bar);
      }
    }
    if (tid < kCpRows && tid >= ua * kUnitTokens && tid < min(ub * kUnitTokens, rows)) {
      const int rel = sm.slot[tid] - s_first, rs = sm.srcpos[tid] % kUnitTokens;
      sm.offd[tid] = rel * UB + D::kBase + static_cast<int>(D::dep(rs));
      sm.offs[tid] = rel * UB + S::kBase + static_cast<int>(S::dep(rs));
    }
    __syncthreads();
    const bool ok = mbar_wait_bounded(&sm.bar, phase);
    if (__syncthreads_or(!ok)) {
      // copies still in flight after the limit: flag, wait once more, leave
      if (tid == 0) set_err(p.err, KVQ_DEVERR_TIMEOUT);
      mbar_wait_bounded(&sm.bar, phase);
      return;
    }
    phase ^= 1u;
    for (int c = tid; c < (ub - ua) * CH; c += kCpThreads) {
      const int ud = ua + c / CH;
      const uint32_t x = static_cast<uint32_t>(c % CH) * 16u;
      uint4 v;
      if (!L::kScales || x < static_cast<uint32_t>(S::kBase))
        v = gather_chunk<D>(stage, sm.offd, ud, rows, x - D::kBase);
      else
        v = gather_chunk<S>(stage, sm.offs, ud, rows, x - S::kBase);
      reinterpret_cast<uint4 *>(dst + (d_unit0 + ud) * UB)[x / 16] = v;
    }
    __syncthreads();
    ua = ub;
  }
}

// blockIdx = (run of kCpUnits destination units, kv head * 2 + side, sequence):
// both sides in one launch, so that the K and V runs are in flight together.
template <int CK, int CV>
__global__ void __launch_bounds__(kCpThreads) compact_kernel(const CompactParams p) {
  extern __shared__ __align__(128) uint8_t cp_stage[];
  __shared__ CompactSmem sm;
  const int s = blockIdx.z, kvh = blockIdx.y >> 1, side = blockIdx.y & 1;
  const int u0 = blockIdx.x * kCpUnits, tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    fence_mbar_init();
  }
  grid_dependency_wait();
  const int len = min(max(p.seq_lens[s], 0), p.capacity);
  const int n = min(max(p.n_ev[s], 0), min(p.max_evict, len));
  const int new_len = len - n;
  if (side == 0 && kvh == 0 && blockIdx.x == 0) {
    // the list must hold increasing positions below the length
    const int32_t *ev = p.evict + static_cast<int64_t>(s) * p.max_evict;
    bool bad = p.n_ev[s] < 0 || p.n_ev[s] > min(p.max_evict, len);
    for (int j = tid; j < n && !bad; j += kCpThreads)
      bad = ev[j] < 0 || ev[j] >= len || (j > 0 && ev[j] <= ev[j - 1]);
    if (bad) set_err(p.err, KVQ_DEVERR_EVICT);
    if (tid == 0 && p.lens_dst) p.lens_dst[s] = new_len;
  }
  const int rows = min(kCpRows, new_len - u0 * kUnitTokens);
  if (rows > 0) {
    __syncthreads();  // the mbarrier's initialisation is visible to every thread
    if (side == 0) compact_run<CK, 0>(p, sm, cp_stage, s, kvh, u0, len, n, rows);
    else compact_run<CV, 1>(p, sm, cp_stage, s, kvh, u0, len, n, rows);
  }
  grid_launch_dependents();
}

template <int CK, int CV>
cudaError_t launch_compact_t(const CompactParams &p, dim3 grid, cudaStream_t stream) {
  constexpr int ub = unit_bytes(CK) > unit_bytes(CV) ? unit_bytes(CK) : unit_bytes(CV);
  constexpr int smem = kCpSlots * ub;
  static std::atomic<uint64_t> optin{0};
  const cudaError_t e = smem_optin(compact_kernel<CK, CV>, smem, optin);
  if (e != cudaSuccess) return e;
  return launch_pdl(compact_kernel<CK, CV>, grid, dim3(kCpThreads), smem, stream, p);
}

template <int CK>
cudaError_t launch_compact_v(int cv, const CompactParams &p, dim3 grid, cudaStream_t stream) {
  switch (cv) {
    case KVQ_F16: return launch_compact_t<CK, KVQ_F16>(p, grid, stream);
    case KVQ_Q8_0: return launch_compact_t<CK, KVQ_Q8_0>(p, grid, stream);
    case KVQ_Q4_0: return launch_compact_t<CK, KVQ_Q4_0>(p, grid, stream);
    default: return launch_compact_t<CK, KVQ_TURBO4>(p, grid, stream);
  }
}

}  // namespace

cudaError_t launch_probe(const kvq_layer &L, const void *q, float scale, const float *lse,
                         float decay, float *scores, cudaStream_t stream) {
  ProbeParams p;
  p.k_cache = static_cast<const uint8_t *>(L.k_cache);
  p.seq_lens = L.seq_lens;
  p.q = static_cast<const __half *>(q);
  p.lse = lse;
  p.scores = scores;
  p.err = L.err;
  p.table = L.pages_per_seq > 0 ? L.block_table : nullptr;
  p.n_kv = L.n_kv_heads;
  p.n_q = L.n_q_heads;
  p.G = L.n_q_heads / L.n_kv_heads;
  p.n_hg = (p.G + 7) / 8;
  p.capacity = L.capacity;
  p.pages_per_seq = L.pages_per_seq;
  p.n_pages = L.n_pages;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.decay = decay;
  const dim3 grid(L.capacity / (kProbeUnits * kUnitTokens), L.n_seqs);
  switch (L.codec_k) {
    case KVQ_F16: return launch_pdl(probe_kernel<KVQ_F16>, grid, dim3(kProbeWarps * 32), 0, stream, p);
    case KVQ_Q8_0: return launch_pdl(probe_kernel<KVQ_Q8_0>, grid, dim3(kProbeWarps * 32), 0, stream, p);
    case KVQ_Q4_0: return launch_pdl(probe_kernel<KVQ_Q4_0>, grid, dim3(kProbeWarps * 32), 0, stream, p);
    default: return launch_pdl(probe_kernel<KVQ_TURBO4>, grid, dim3(kProbeWarps * 32), 0, stream, p);
  }
}

cudaError_t launch_evict_select(const kvq_layer &L, const float *scores, int n_sink,
                                int n_recent, int n_evict, int32_t *evict, int32_t *n_evicted,
                                cudaStream_t stream) {
  SelectParams p;
  p.scores = scores;
  p.seq_lens = L.seq_lens;
  p.evict = evict;
  p.n_out = n_evicted;
  p.capacity = L.capacity;
  p.n_sink = n_sink;
  p.n_recent = n_recent;
  p.n_evict = n_evict;
  return launch_pdl(select_kernel, dim3(L.n_seqs), dim3(kSelThreads), 0, stream, p);
}

cudaError_t launch_compact(const kvq_layer &L, const int32_t *evict, const int32_t *n_evicted,
                           int max_evict, void *k_dst, void *v_dst, const float *scores,
                           float *scores_dst, int32_t *lens_dst, cudaStream_t stream) {
  CompactParams p;
  p.src[0] = static_cast<const uint8_t *>(L.k_cache);
  p.src[1] = static_cast<const uint8_t *>(L.v_cache);
  p.dst[0] = static_cast<uint8_t *>(k_dst);
  p.dst[1] = static_cast<uint8_t *>(v_dst);
  p.seq_lens = L.seq_lens;
  p.evict = evict;
  p.n_ev = n_evicted;
  p.scores = scores;
  p.scores_dst = scores_dst;
  p.lens_dst = lens_dst;
  p.err = L.err;
  p.table = L.pages_per_seq > 0 ? L.block_table : nullptr;
  p.max_evict = max_evict;
  p.n_kv = L.n_kv_heads;
  p.capacity = L.capacity;
  p.pages_per_seq = L.pages_per_seq;
  p.n_pages = L.n_pages;
  const dim3 grid(L.capacity / kCpRows, 2 * L.n_kv_heads, L.n_seqs);
  switch (L.codec_k) {
    case KVQ_F16: return launch_compact_v<KVQ_F16>(L.codec_v, p, grid, stream);
    case KVQ_Q8_0: return launch_compact_v<KVQ_Q8_0>(L.codec_v, p, grid, stream);
    case KVQ_Q4_0: return launch_compact_v<KVQ_Q4_0>(L.codec_v, p, grid, stream);
    default: return launch_compact_v<KVQ_TURBO4>(L.codec_v, p, grid, stream);
  }
}

}  // namespace kvq
