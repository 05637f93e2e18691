// kvq_encode.cuh -- the row encoders of the cache codecs (device code shared
// by the append, re-encode and fused decode-step kernels).
//
// Block codecs of the "Codecs" table of the buun-llama-cpp listing (q8_0 8.5
// and q4_0 4.5 bits per value, 32-value blocks with an fp16 scale) and the
// rotated turbo4 rows, with the fp32 encoder formulas of include/kvq.h,
// evaluated with explicit IEEE round-to-nearest operations so that the bytes
// are reproducible bit for bit.  One warp encodes one 128-value row: lane l
// holds dims 4l..4l+3.
#pragma once

#include <cuda_runtime.h>

#include "kvq_device.cuh"

namespace kvq {
namespace {

// The integers the encoders take from the quotients x/d, without a division
// or a float-to-int conversion per value.  t = RN(x * RN(1/d)) lies within
// |x/d| * 3 * 2^-24 of RN(x/d) (two roundings of relative size 2^-24).
// Where t is far enough from the boundary at which the encoder's integer
// changes, t gives the same integer as RN(x/d) (tests below); elsewhere the
// encoder divides exactly.  Integers come from the 1.5 * 2^23 addition: for
// |y| < 2^22, RN(y + 1.5 * 2^23) holds RN-to-nearest-integer(y) in its low
// mantissa bits.  The bytes are those of the exact division.
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23
constexpr int kRoundMagicBits = 0x4B400000;

// q8_0: q = round-half-away(RN(x/d)) with |x/d| <= 127 (1 + 2^-23), so
// |t - RN(x/d)| < 2^-15.4.  t more than 2^-14 away from every half-integer
// rounds the same way, and there round-half-away equals round-to-nearest.
__device__ __forceinline__ int q8_from_quotient(float x, float d, float rcp) {
  const float t = __fmul_rn(x, rcp);
  const float tm = __fadd_rn(t, kRoundMagic);
  const float dist = fabsf(__fsub_rn(t, __fsub_rn(tm, kRoundMagic)));  // to the nearest integer
  if (fabsf(__fsub_rn(dist, 0.5f)) > 0x1p-14f) return __float_as_int(tm) - kRoundMagicBits;
  return static_cast<int>(roundf(__fdiv_rn(x, d)));
}

// q4_0 and turbo4: q = min(15, trunc(RN(RN(x/d) + 8.5))) with |x/d| <= 8 (1 +
// 2^-23): u = RN(t + 8.5) lies within 2^-18.5 of the exact path's value, so
// u more than 2^-17 away from every integer truncates the same way
// (floor(u) = the integer nearest to u - 0.5, which is exact there).
__device__ __forceinline__ int q4_from_quotient(float x, float d, float rcp) {
  const float u = __fadd_rn(__fmul_rn(x, rcp), 8.5f);
  const float fm = __fadd_rn(__fsub_rn(u, 0.5f), kRoundMagic);
  const float fr = __fsub_rn(u, __fsub_rn(fm, kRoundMagic));  // u - floor(u)
  const int v = (fr > 0x1p-17f && fr < 1.0f - 0x1p-17f)
                    ? __float_as_int(fm) - kRoundMagicBits
                    : static_cast<int>(__fadd_rn(__fdiv_rn(x, d), 8.5f));  // truncation; u >= 0.5
  return v > 15 ? 15 : v;
}

// q8_0: amax over the 8 lanes of the block, d = amax/127, q = round(x/d).
__device__ __forceinline__ void encode_q8(const float (&x)[4], int (&q)[4], __half &d16) {
  float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const float d = __fdiv_rn(a, 127.0f);
  d16 = __float2half_rn(d);
  const float rcp = d != 0.0f ? __frcp_rn(d) : 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = d != 0.0f ? q8_from_quotient(x[i], d, rcp) : 0;
}

// q4_0: signed value of largest magnitude (lowest dim wins ties), d = m/-8,
// q = min(15, trunc(x/d + 8.5)).
__device__ __forceinline__ void encode_q4(const float (&x)[4], int lane, int (&q)[4], __half &d16) {
  float best = fabsf(x[0]);
  float m = x[0];
  int idx = 4 * lane;
#pragma unroll
  for (int i = 1; i < 4; ++i) {
    const float a = fabsf(x[i]);
    if (a > best) { best = a; m = x[i]; idx = 4 * lane + i; }
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const float om = __shfl_xor_sync(0xffffffffu, m, o);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
    if (ob > best || (ob == best && oi < idx)) { best = ob; m = om; idx = oi; }
  }
  const float d = __fdiv_rn(m, -8.0f);
  d16 = __float2half_rn(d);
  const float rcp = d != 0.0f ? __frcp_rn(d) : 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = d != 0.0f ? q4_from_quotient(x[i], d, rcp) : 8;
}

// turbo4: signs, FWHT and the factor 1/8 (the rotation of the row, exact
// order of the definition), then the q4_0 rule over all 128 rotated values
// (32 lanes, lowest dim wins ties).
__device__ __forceinline__ void encode_turbo4(const float (&x)[4], int lane, int (&q)[4],
                                              __half &d16) {
  float y[4] = {x[0], x[1], x[2], x[3]};
  turbo_flip_lane(y, lane);
  fwht128_warp(y, lane);
#pragma unroll
  for (int i = 0; i < 4; ++i) y[i] *= 0.125f;
  float best = fabsf(y[0]);
  float m = y[0];
  int idx = 4 * lane;
#pragma unroll
  for (int i = 1; i < 4; ++i) {
    const float a = fabsf(y[i]);
    if (a > best) { best = a; m = y[i]; idx = 4 * lane + i; }
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const float om = __shfl_xor_sync(0xffffffffu, m, o);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
    if (ob > best || (ob == best && oi < idx)) { best = ob; m = om; idx = oi; }
  }
  const float d = __fdiv_rn(m, -8.0f);
  d16 = __float2half_rn(d);
  const float rcp = d != 0.0f ? __frcp_rn(d) : 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = d != 0.0f ? q4_from_quotient(y[i], d, rcp) : 8;
}

__device__ __forceinline__ void st_u16(uint8_t *p, uint32_t v) {
  *reinterpret_cast<uint16_t *>(p) = static_cast<uint16_t>(v);
}

// Write one row (token row r of `unit`) from lane-held data.
template <int SIDE>
__device__ __forceinline__ void store_row(int codec, uint8_t *unit, int r, int lane,
                                          const uint2 raw, const int (&q)[4], __half d16) {
  const int g = r & 7, rh = r >> 3, tig = (r & 7) >> 1, par = r & 1;
  const int b = lane >> 3, lb = lane & 7;  // block and lane-in-block
  if (codec == KVQ_F16) {
    if (SIDE == 0) {
      const int h = (lane >> 2) & 1, w = lane & 3;
      *reinterpret_cast<uint2 *>(unit + (2 * b + rh) * 512 + (4 * g + w) * 16 + h * 8) = raw;
    } else {
      const uint16_t v[4] = {static_cast<uint16_t>(raw.x), static_cast<uint16_t>(raw.x >> 16),
                             static_cast<uint16_t>(raw.y), static_cast<uint16_t>(raw.y >> 16)};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int d = 4 * lane + i, mt = d >> 4, gq = (d & 15) >> 1, s = d & 1;
        *reinterpret_cast<uint16_t *>(unit + mt * 512 + (4 * gq + tig) * 16 +
                                      (rh * 4 + s * 2 + par) * 2) = v[i];
      }
    }
    return;
  }
  const uint16_t dbits = __half_as_ushort(d16);
  if (codec == KVQ_Q8_0) {
    if (SIDE == 0) {
      const uint32_t word = (q[0] & 0xff) | ((q[1] & 0xff) << 8) | ((q[2] & 0xff) << 16) |
                            (static_cast<uint32_t>(q[3] & 0xff) << 24);
      const int h = lb >> 2, w = lane & 3;
      *reinterpret_cast<uint32_t *>(unit + b * 512 + (4 * g + w) * 16 + (2 * rh + h) * 4) = word;
      if (lb == 0) st_u16(unit + 2048 + g * 16 + rh * 8 + b * 2, dbits);
    } else {
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int d = 4 * lane + 2 * p, mt = d >> 4, gq = (d & 15) >> 1;
        st_u16(unit + (mt >> 1) * 512 + (4 * gq + tig) * 16 + ((mt & 1) * 2 + rh) * 4 + par * 2,
               (q[2 * p] & 0xff) | ((q[2 * p + 1] & 0xff) << 8));
      }
      if (lb == 0) st_u16(unit + 2048 + tig * 32 + b * 8 + rh * 4 + par * 2, dbits);
    }
    return;
  }
  // q4_0 and turbo4: canonical byte jc of block (group) b = q[jc] | q[jc+16]
  // << 4; lanes lb<4 hold jc = 4lb..4lb+3 and fetch the high nibbles from
  // lane lb+4 of the same block.
  int hi[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) hi[i] = __shfl_down_sync(0xffffffffu, q[i], 4);
  if (lb < 4) {
    uint32_t bytes[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) bytes[i] = (q[i] & 0xf) | ((hi[i] & 0xf) << 4);
    if (SIDE == 0) {
      const uint32_t word = bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (bytes[3] << 24);
      *reinterpret_cast<uint32_t *>(unit + (b >> 1) * 512 + (4 * g + lb) * 16 +
                                    ((b & 1) * 2 + rh) * 4) = word;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int jc = 4 * lb + i, mt = 2 * b + (jc >> 3), gq = jc & 7;
        unit[(mt >> 2) * 512 + (4 * gq + tig) * 16 + (mt & 3) * 4 + par * 2 + rh] =
            static_cast<uint8_t>(bytes[i]);
      }
    }
  }
  if (codec == KVQ_TURBO4) {  // one scale per row
    if (lane == 0)
      st_u16(unit + (SIDE == 0 ? 1024 + g * 4 + rh * 2 : 1024 + tig * 8 + rh * 4 + par * 2),
             dbits);
    return;
  }
  if (lb == 0) {
    const int off = SIDE == 0 ? 1024 + g * 16 + rh * 8 + b * 2
                              : 1024 + tig * 32 + b * 8 + rh * 4 + par * 2;
    st_u16(unit + off, dbits);
  }
}

// Encode one fp16 row (lane l holds its dims 4l..4l+3 in `raw`) with
// `codec` into token row r of `unit` (all 32 lanes of the warp).
template <int SIDE>
__device__ __forceinline__ void encode_row_into(int codec, const uint2 raw, uint8_t *unit, int r,
                                                int lane) {
  float x[4];
  {
    const __half2 h01 = *reinterpret_cast<const __half2 *>(&raw.x);
    const __half2 h23 = *reinterpret_cast<const __half2 *>(&raw.y);
    x[0] = __low2float(h01); x[1] = __high2float(h01);
    x[2] = __low2float(h23); x[3] = __high2float(h23);
  }
  int q[4] = {0, 0, 0, 0};
  __half d16 = __float2half_rn(0.0f);
  if (codec == KVQ_Q8_0) encode_q8(x, q, d16);
  else if (codec == KVQ_Q4_0) encode_q4(x, lane, q, d16);
  else if (codec == KVQ_TURBO4) encode_turbo4(x, lane, q, d16);
  store_row<SIDE>(codec, unit, r, lane, raw, q, d16);
}

}  // namespace
}  // namespace kvq
