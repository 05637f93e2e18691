// decode.cu -- split-K flash-decoding over a block-quantized KV cache.
//
// Computes, for every (sequence, query head), o = softmax(scale * q K^T) V
// over all cached keys, with K and V dequantized from f16 / q8_0 / q4_0 blocks
// (the codecs of the "Codecs" table of the buun-llama-cpp listing; the K and
// V sides are typed independently, as in its VBR section's per-(layer, side)
// ladder).  The token axis is cut into splits; each split produces a partial
// (running max m, running sum l, unnormalised o) and a second kernel merges
// the partials with the log-sum-exp identity.
//
// Design (one CTA = 4 warps = one split of one (sequence, kv head, group of
// up to 8 query heads)):
//  * Each warp owns a ring of shared-memory stages; lane 0 streams 16-token
//    units of K and V into it with 1-D bulk async copies (TMA engine) tracked
//    by mbarriers, so that many KB per SM are in flight without registers.
//  * The cache layout (include/kvq.h) stores each unit so that every thread
//    fetches exactly its tensor-core operand bytes with aligned 16-byte
//    shared loads (conflict-free: a warp reads 512 contiguous bytes).
//  * Quants become exact fp16 integers in registers (bias-and-subtract on
//    the fp16 mantissa).  S = K Q^T runs on mma.sync m16n8k16 with the 16
//    tokens of a unit as M and the query heads of the group as N.  Per-block
//    scales are factored out of the 32-value sums (two MMAs per block into a
//    fresh accumulator, then s += d * partial), so dequantization is exact.
//  * Online softmax in the log2 domain, per head, with xor-shuffle maxima;
//    P is transposed in registers (movmatrix) into the B operand of O^T = V^T
//    P^T, whose M is 16 head dims; the V block scale is folded into P.
#include <cuda_runtime.h>

#include <math.h>

#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kDecodeWarps = 4;
constexpr int kWarpSmemBudget = 24576;

struct DecodeParams {
  const uint8_t *k_cache;
  const uint8_t *v_cache;
  const int32_t *seq_lens;
  const __half *q;
  float *part_o;   // [n_seqs][n_q][n_splits][128]
  float2 *part_ml; // [n_seqs][n_q][n_splits]: (max in log2 units, sum)
  int32_t *err;
  int n_seqs, n_kv, n_q, G, n_hgroups, capacity, max_len, split_tokens, n_splits;
  float scale_log2;
};

template <int CK, int CV>
struct DecodeCfg {
  static constexpr int UK = unit_bytes(CK);
  static constexpr int UV = unit_bytes(CV);
  static constexpr int STAGE = UK + UV;
  static constexpr int NS_RAW = kWarpSmemBudget / STAGE;
  static constexpr int NS = NS_RAW < 2 ? 2 : (NS_RAW > 8 ? 8 : NS_RAW);
  static constexpr int WARP_SMEM = NS * STAGE;
  static constexpr int SMEM = kDecodeWarps * WARP_SMEM;
  static_assert(SMEM >= kDecodeWarps * (8 * 128 + 16) * 4, "reduction area must fit");
};

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
}

// Head-dim index of accumulator row (m-row) of m-tile mt for the V codec.
template <int CV>
__device__ __forceinline__ int v_dim(int mt, int mrow) {
  if (CV == KVQ_Q4_0) {
    const int b = mt >> 1, hh = mt & 1;
    return 32 * b + 8 * hh + (mrow & 7) + (mrow >> 3) * 16;
  }
  return 16 * mt + 2 * (mrow & 7) + (mrow >> 3);
}

// S (16 tokens x 8 heads) of one unit, already multiplied by scale*log2(e).
template <int CK>
__device__ __forceinline__ void unit_scores(const uint8_t *ku, int lane, const uint32_t (&qb)[8][2],
                                            float scale_log2, float (&s)[4]) {
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
        const uint32_t a0[4] = {u4_pair_minus8(W0), u4_pair_minus8(W1), u4_pair_minus8(W0 >> 8),
                                u4_pair_minus8(W1 >> 8)};
        const uint32_t a1[4] = {u4_pair_minus8(W0 >> 4), u4_pair_minus8(W1 >> 4),
                                u4_pair_minus8(W0 >> 12), u4_pair_minus8(W1 >> 12)};
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
template <int CV>
__device__ __forceinline__ void unit_pv(const uint8_t *vu, int lane, uint32_t B0, uint32_t B1,
                                        int nvalid, float (&o)[8][4]) {
  const int tig = lane & 3;
  // token validity masks for the halves this thread holds: (t0,t1)=(2tig,2tig+1), (t2,t3)=+8
  uint32_t m01 = 0xffffffffu, m23 = 0xffffffffu;
  if (nvalid < 16) {
    m01 = (2 * tig < nvalid ? 0x0000ffffu : 0u) | (2 * tig + 1 < nvalid ? 0xffff0000u : 0u);
    m23 = (2 * tig + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * tig + 9 < nvalid ? 0xffff0000u : 0u);
  }
  if (CV == KVQ_F16) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const uint4 r = lds128(vu + mt * 512 + lane * 16);
      const uint32_t a[4] = {r.x & m01, r.y & m01, r.z & m23, r.w & m23};
      mma16816(o[mt], a, B0, B1);
    }
  } else {
    const uint4 s01 = lds128(vu + unit_scale_offset(CV) + tig * 32);
    const uint4 s23 = lds128(vu + unit_scale_offset(CV) + tig * 32 + 16);
    const uint32_t dp01[4] = {s01.x & m01, s01.z & m01, s23.x & m01, s23.z & m01};
    const uint32_t dp23[4] = {s01.y & m23, s01.w & m23, s23.y & m23, s23.w & m23};
    if (CV == KVQ_Q8_0) {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t bp0 = hmul2_bits(B0, dp01[b]), bp1 = hmul2_bits(B1, dp23[b]);
        const uint4 w = lds128(vu + b * 512 + lane * 16);
        const uint32_t a0[4] = {s8_pair_02(w.x), s8_pair_13(w.x), s8_pair_02(w.y), s8_pair_13(w.y)};
        const uint32_t a1[4] = {s8_pair_02(w.z), s8_pair_13(w.z), s8_pair_02(w.w), s8_pair_13(w.w)};
        mma16816(o[2 * b], a0, bp0, bp1);
        mma16816(o[2 * b + 1], a1, bp0, bp1);
      }
    } else {
#pragma unroll
      for (int jv = 0; jv < 2; ++jv) {
        const uint4 w = lds128(vu + jv * 512 + lane * 16);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const int mt = 4 * jv + qq, b = mt >> 1;
          const uint32_t bp0 = hmul2_bits(B0, dp01[b]), bp1 = hmul2_bits(B1, dp23[b]);
          const uint32_t W = ws[qq];
          const uint32_t a[4] = {u4_pair_minus8(W), u4_pair_minus8(W >> 4), u4_pair_minus8(W >> 8),
                                 u4_pair_minus8(W >> 12)};
          mma16816(o[mt], a, bp0, bp1);
        }
      }
    }
  }
}

template <int CK, int CV>
__global__ void __launch_bounds__(kDecodeWarps * 32, 2) decode_split_kernel(const DecodeParams p) {
  using C = DecodeCfg<CK, CV>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t bars[kDecodeWarps][C::NS];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y / p.n_hgroups, hg = blockIdx.y % p.n_hgroups;
  const int seq = blockIdx.z;

  int len = p.seq_lens[seq];
  if (len > p.max_len) {
    if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) set_err(p.err, KVQ_DEVERR_MAXLEN);
    len = p.max_len;
  }
  const int t0 = split * p.split_tokens;
  if (t0 >= len) return;  // whole CTA: empty split
  const int t1 = min(len, t0 + p.split_tokens);
  const int n_units = (t1 - t0 + kUnitTokens - 1) / kUnitTokens;
  const int my_n = n_units > warp ? (n_units - warp + kDecodeWarps - 1) / kDecodeWarps : 0;

  const int64_t units_per_stream = p.capacity / kUnitTokens;
  const int64_t stream = static_cast<int64_t>(seq) * p.n_kv + kvh;
  const int64_t u0 = stream * units_per_stream + t0 / kUnitTokens;
  const uint8_t *kbase = p.k_cache + u0 * C::UK;
  const uint8_t *vbase = p.v_cache + u0 * C::UV;
  uint8_t *ring = smem + warp * C::WARP_SMEM;
  uint64_t *wb = bars[warp];

  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < C::NS; ++s) mbar_init(&wb[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  auto issue = [&](int k) {  // lane 0 only: load unit (warp + k*WARPS) into stage k % NS
    const int j = warp + k * kDecodeWarps;
    const int s = k % C::NS;
    uint8_t *dst = ring + s * C::STAGE;
    mbar_arrive_expect_tx(&wb[s], C::STAGE);
    bulk_copy_g2s(dst, kbase + static_cast<int64_t>(j) * C::UK, C::UK, &wb[s]);
    bulk_copy_g2s(dst + C::UK, vbase + static_cast<int64_t>(j) * C::UV, C::UV, &wb[s]);
  };
  const int pre = my_n < C::NS ? my_n : C::NS;
  if (lane == 0)
    for (int k = 0; k < pre; ++k) issue(k);

  // B fragments of Q (n = query head g of this group), with the per-codec
  // ordering of the k (head-dim) index that matches the K unit layout.
  const int hq = hg * 8 + g;
  const bool hvalid = hq < p.G;
  uint32_t qb[8][2];
  {
    const __half *qrow = p.q + (static_cast<int64_t>(seq) * p.n_q + kvh * p.G + (hvalid ? hq : 0)) * kD;
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

  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.0f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
  bool ok = true;
  int k_fail = my_n;

  for (int k = 0; k < my_n; ++k) {
    const int s = k % C::NS;
    const uint32_t phase = static_cast<uint32_t>(k / C::NS) & 1u;
    const bool got = mbar_wait_bounded(&wb[s], phase);
    if (!__all_sync(0xffffffffu, got)) {  // warp-uniform decision
      ok = false;
      k_fail = k;
      if (lane == 0) set_err(p.err, KVQ_DEVERR_TIMEOUT);
      break;
    }
    const uint8_t *ku = ring + s * C::STAGE;
    const uint8_t *vu = ku + C::UK;
    const int j = warp + k * kDecodeWarps;
    const int nvalid = min(kUnitTokens, t1 - (t0 + j * kUnitTokens));

    float sc[4];
    unit_scores<CK>(ku, lane, qb, p.scale_log2, sc);
    if (nvalid < kUnitTokens) {
      if (g >= nvalid) sc[0] = sc[1] = -INFINITY;
      if (g + 8 >= nvalid) sc[2] = sc[3] = -INFINITY;
    }
    float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
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
      m0 = mn0;
      m1 = mn1;
    }
    const float p0 = fast_exp2(sc[0] - m0), p1 = fast_exp2(sc[1] - m1);
    const float p2 = fast_exp2(sc[2] - m0), p3 = fast_exp2(sc[3] - m1);
    l0 += p0 + p2;
    l1 += p1 + p3;
    const uint32_t B0 = movmatrix_trans(pack_half2(p0, p1));
    const uint32_t B1 = movmatrix_trans(pack_half2(p2, p3));
    unit_pv<CV>(vu, lane, B0, B1, nvalid, o);

    __syncwarp();
    if (lane == 0 && k + C::NS < my_n) {
      fence_proxy_async_smem();
      issue(k + C::NS);
    }
  }
  if (!ok) {
    // Drain copies still in flight into this warp's ring before the CTA moves on.
    const int issued = min(my_n, k_fail + C::NS);
    for (int k = k_fail; k < issued; ++k)
      mbar_wait_bounded(&wb[k % C::NS], static_cast<uint32_t>(k / C::NS) & 1u);
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.0f;
  }

#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  __syncthreads();  // every warp is done with its ring: reuse it for the CTA merge
  float *red_o = reinterpret_cast<float *>(smem);                  // [warp][8 heads][128]
  float *red_ml = red_o + kDecodeWarps * 8 * kD;                   // [warp][8][2]
  {
    float *wo = red_o + warp * 8 * kD;
    const int h0 = 2 * tig, h1 = 2 * tig + 1;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int dlo = v_dim<CV>(mt, g), dhi = v_dim<CV>(mt, g + 8);
      wo[h0 * kD + dlo] = ok ? o[mt][0] : 0.0f;
      wo[h1 * kD + dlo] = ok ? o[mt][1] : 0.0f;
      wo[h0 * kD + dhi] = ok ? o[mt][2] : 0.0f;
      wo[h1 * kD + dhi] = ok ? o[mt][3] : 0.0f;
    }
    if (g == 0) {
      red_ml[(warp * 8 + h0) * 2 + 0] = m0;
      red_ml[(warp * 8 + h0) * 2 + 1] = l0;
      red_ml[(warp * 8 + h1) * 2 + 0] = m1;
      red_ml[(warp * 8 + h1) * 2 + 1] = l1;
    }
  }
  __syncthreads();
  const int heads_here = min(8, p.G - hg * 8);
  for (int idx = threadIdx.x; idx < heads_here * kD; idx += kDecodeWarps * 32) {
    const int hh = idx / kD, d = idx % kD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, red_ml[(w * 8 + hh) * 2]);
    float acc = 0.0f, L = 0.0f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) {
      const float mw = red_ml[(w * 8 + hh) * 2];
      const float sw = mw == -INFINITY ? 0.0f : fast_exp2(mw - M);
      acc = fmaf(sw, red_o[(w * 8 + hh) * kD + d], acc);
      L = fmaf(sw, red_ml[(w * 8 + hh) * 2 + 1], L);
    }
    const int head = kvh * p.G + hg * 8 + hh;
    const int64_t slot = (static_cast<int64_t>(seq) * p.n_q + head) * p.n_splits + split;
    p.part_o[slot * kD + d] = acc;
    if (d == 0) p.part_ml[slot] = make_float2(M, L);
  }
}

struct MergeParams {
  const float *part_o;
  const float2 *part_ml;
  const int32_t *seq_lens;
  __half *out;
  float *lse;
  int n_seqs, n_q, max_len, split_tokens, n_splits;
};

// One warp per (sequence, query head): log-sum-exp merge of the split partials.
__global__ void __launch_bounds__(128) decode_merge_kernel(const MergeParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + warp;
  if (row >= p.n_seqs * p.n_q) return;
  const int seq = row / p.n_q;
  int len = p.seq_lens[seq];
  len = len < p.max_len ? len : p.max_len;
  int nv = len > 0 ? (len + p.split_tokens - 1) / p.split_tokens : 0;
  nv = nv < p.n_splits ? nv : p.n_splits;
  const float2 *ml = p.part_ml + static_cast<int64_t>(row) * p.n_splits;
  const float *po = p.part_o + static_cast<int64_t>(row) * p.n_splits * kD;
  float M = -INFINITY;
  for (int i = lane; i < nv; i += 32) M = fmaxf(M, ml[i].x);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float L = 0.0f;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (M != -INFINITY) {
    for (int i = 0; i < nv; ++i) {
      const float2 v = ml[i];
      const float w = v.x == -INFINITY ? 0.0f : fast_exp2(v.x - M);
      const float4 x = reinterpret_cast<const float4 *>(po + static_cast<int64_t>(i) * kD)[lane];
      L = fmaf(w, v.y, L);
      acc.x = fmaf(w, x.x, acc.x);
      acc.y = fmaf(w, x.y, acc.y);
      acc.z = fmaf(w, x.z, acc.z);
      acc.w = fmaf(w, x.w, acc.w);
    }
  }
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  __half2 *dst = reinterpret_cast<__half2 *>(p.out + static_cast<int64_t>(row) * kD) + lane * 2;
  dst[0] = __floats2half2_rn(acc.x * inv, acc.y * inv);
  dst[1] = __floats2half2_rn(acc.z * inv, acc.w * inv);
  if (p.lse && lane == 0) p.lse[row] = L > 0.0f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
}

template <int CK, int CV>
cudaError_t launch_split(const DecodeParams &p, dim3 grid, cudaStream_t stream) {
  using C = DecodeCfg<CK, CV>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<CK, CV>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  decode_split_kernel<CK, CV><<<grid, kDecodeWarps * 32, C::SMEM, stream>>>(p);
  return cudaGetLastError();
}

template <int CK>
cudaError_t launch_split_v(int cv, const DecodeParams &p, dim3 grid, cudaStream_t stream) {
  switch (cv) {
    case KVQ_F16: return launch_split<CK, KVQ_F16>(p, grid, stream);
    case KVQ_Q8_0: return launch_split<CK, KVQ_Q8_0>(p, grid, stream);
    default: return launch_split<CK, KVQ_Q4_0>(p, grid, stream);
  }
}

}  // namespace

DecodePlan plan_decode(const kvq_layer &L, int max_len, int num_sms) {
  DecodePlan pl;
  const int G = L.n_q_heads / L.n_kv_heads;
  pl.n_hgroups = (G + 7) / 8;
  const int64_t streams = static_cast<int64_t>(L.n_seqs) * L.n_kv_heads * pl.n_hgroups;
  const int64_t max_units = (max_len + kUnitTokens - 1) / kUnitTokens;
  // Aim at ~4 waves of two resident CTAs per SM; at least two units per warp.
  const int64_t target = static_cast<int64_t>(num_sms > 0 ? num_sms : 148) * 2 * 4;
  int64_t split_units = (streams * max_units + target - 1) / target;
  const int64_t min_units = 2 * kDecodeWarps;
  if (split_units < min_units) split_units = min_units;
  if (split_units > max_units) split_units = max_units > 0 ? max_units : 1;
  pl.split_tokens = static_cast<int>(split_units * kUnitTokens);
  pl.n_splits = static_cast<int>((max_len + pl.split_tokens - 1) / pl.split_tokens);
  if (pl.n_splits < 1) pl.n_splits = 1;
  const int64_t slots = static_cast<int64_t>(L.n_seqs) * L.n_q_heads * pl.n_splits;
  pl.ws_o_bytes = slots * kD * sizeof(float);
  pl.ws_bytes = pl.ws_o_bytes + slots * sizeof(float2);
  return pl;
}

cudaError_t launch_decode(const kvq_layer &L, const DecodePlan &pl, const void *q, float scale,
                          void *out, float *lse, int max_len, void *workspace,
                          cudaStream_t stream) {
  DecodeParams p;
  p.k_cache = static_cast<const uint8_t *>(L.k_cache);
  p.v_cache = static_cast<const uint8_t *>(L.v_cache);
  p.seq_lens = L.seq_lens;
  p.q = static_cast<const __half *>(q);
  p.part_o = static_cast<float *>(workspace);
  p.part_ml = reinterpret_cast<float2 *>(static_cast<uint8_t *>(workspace) + pl.ws_o_bytes);
  p.err = L.err;
  p.n_seqs = L.n_seqs;
  p.n_kv = L.n_kv_heads;
  p.n_q = L.n_q_heads;
  p.G = L.n_q_heads / L.n_kv_heads;
  p.n_hgroups = pl.n_hgroups;
  p.capacity = L.capacity;
  p.max_len = max_len;
  p.split_tokens = pl.split_tokens;
  p.n_splits = pl.n_splits;
  p.scale_log2 = scale * 1.4426950408889634f;
  const dim3 grid(pl.n_splits, L.n_kv_heads * pl.n_hgroups, L.n_seqs);
  cudaError_t e;
  switch (L.codec_k) {
    case KVQ_F16: e = launch_split_v<KVQ_F16>(L.codec_v, p, grid, stream); break;
    case KVQ_Q8_0: e = launch_split_v<KVQ_Q8_0>(L.codec_v, p, grid, stream); break;
    default: e = launch_split_v<KVQ_Q4_0>(L.codec_v, p, grid, stream); break;
  }
  if (e != cudaSuccess) return e;
  MergeParams mp;
  mp.part_o = p.part_o;
  mp.part_ml = p.part_ml;
  mp.seq_lens = L.seq_lens;
  mp.out = static_cast<__half *>(out);
  mp.lse = lse;
  mp.n_seqs = L.n_seqs;
  mp.n_q = L.n_q_heads;
  mp.max_len = max_len;
  mp.split_tokens = pl.split_tokens;
  mp.n_splits = pl.n_splits;
  const int rows = L.n_seqs * L.n_q_heads;
  decode_merge_kernel<<<(rows + 3) / 4, 128, 0, stream>>>(mp);
  return cudaGetLastError();
}

}  // namespace kvq
