// kvq_device.cuh -- device helpers shared by the libkvq kernels (sm_103a).
//
// Warp-level tensor-core MMA (m16n8k16, fp16 in, fp32 accumulate), fragment
// transposes, exact small-integer -> fp16 conversions, mbarrier-tracked bulk
// async copies with bounded waits, and the unit geometry of the cache layout
// documented in include/kvq.h.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kD = 128;          // head_dim
constexpr int kUnitTokens = 16;  // tokens per layout unit

__host__ __device__ constexpr int row_bytes(int codec) {
  return codec == KVQ_F16 ? 256 : codec == KVQ_Q8_0 ? 136 : codec == KVQ_Q4_0 ? 72 : 66;
}
__host__ __device__ constexpr int unit_bytes(int codec) { return kUnitTokens * row_bytes(codec); }
// Byte offset of the scale area inside a unit (q8_0 / q4_0 / turbo4 only).
__host__ __device__ constexpr int unit_scale_offset(int codec) {
  return codec == KVQ_Q8_0 ? 2048 : 1024;
}
// Codecs whose quants are nibbles in the q4_0 places of the unit.
__host__ __device__ constexpr bool nibble_codec(int codec) {
  return codec == KVQ_Q4_0 || codec == KVQ_TURBO4;
}

// ---------------------------------------------------------------- turbo4 rotation

// SplitMix64 (Steele, Lea and Flood, OOPSLA 2014): output n (0-based) of the
// generator seeded with `seed`; the state advances by 0x9E3779B97F4A7C15 per
// output and is mixed by two xor-shift-multiply steps and an xor-shift.
__host__ __device__ constexpr uint64_t splitmix64_at(uint64_t seed, int n) {
  const uint64_t z0 = seed + 0x9E3779B97F4A7C15ull * static_cast<uint64_t>(n + 1);
  const uint64_t z1 = (z0 ^ (z0 >> 30)) * 0xBF58476D1CE4E5B9ull;
  const uint64_t z2 = (z1 ^ (z1 >> 27)) * 0x94D049BB133111EBull;
  return z2 ^ (z2 >> 31);
}
// turbo4 sign flips as a 128-bit mask: bit j set <=> s_j = -1 (bit 63 of
// output j from seed 0x4B5651).  Word w holds dims 32w .. 32w + 31.
__host__ __device__ constexpr uint32_t turbo_sign_word(int w) {
  uint32_t m = 0;
  for (int j = 0; j < 32; ++j)
    m |= static_cast<uint32_t>(splitmix64_at(0x4B5651ull, 32 * w + j) >> 63) << j;
  return m;
}
__device__ __forceinline__ uint32_t turbo_signs(int w) {
  constexpr uint32_t w0 = turbo_sign_word(0), w1 = turbo_sign_word(1), w2 = turbo_sign_word(2),
                     w3 = turbo_sign_word(3);
  return w == 0 ? w0 : w == 1 ? w1 : w == 2 ? w2 : w3;
}

// Unnormalised Sylvester-order FWHT of a 128-vector held four per lane (lane
// l: elements 4l .. 4l + 3): stages h = 1, 2 inside the lane, then h = 4 ..
// 64 against lane l ^ (h / 4); every output is the single fp32 addition or
// subtraction (lower - upper) of the pair, as in the definition.
__device__ __forceinline__ void fwht128_warp(float (&v)[4], int lane) {
  const float a0 = __fadd_rn(v[0], v[1]), a1 = __fsub_rn(v[0], v[1]);
  const float a2 = __fadd_rn(v[2], v[3]), a3 = __fsub_rn(v[2], v[3]);
  v[0] = __fadd_rn(a0, a2);
  v[2] = __fsub_rn(a0, a2);
  v[1] = __fadd_rn(a1, a3);
  v[3] = __fsub_rn(a1, a3);
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
      v[i] = upper ? __fsub_rn(o, v[i]) : __fadd_rn(v[i], o);
    }
  }
}

// Sign flips of the four elements 4l .. 4l + 3 held by lane l.
__device__ __forceinline__ void turbo_flip_lane(float (&v)[4], int lane) {
  const uint32_t bits = turbo_signs(lane >> 3) >> (4 * (lane & 7));
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if ((bits >> i) & 1u) v[i] = -v[i];
}

// x^ = s * H y^ / 16 for a row held four per lane (exact in fp32 for
// decoded turbo4 values).
__device__ __forceinline__ void turbo_unrotate_lane(float (&v)[4], int lane) {
  fwht128_warp(v, lane);
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] *= 0.0625f;
  turbo_flip_lane(v, lane);
}

// y^ = d16 * (n - 8) of token row r of a turbo4 unit (exact in fp32), lane l
// holding rotated elements 4l .. 4l + 3: lanes 8b + lb with lb < 4 read the
// low nibbles of canonical bytes 4 lb .. 4 lb + 3 of group b, lanes lb >= 4
// the high nibbles of bytes 4 (lb - 4) .. (elements + 16).
template <int SIDE>
__device__ __forceinline__ void turbo4_row_rotated(const uint8_t *unit, int r, int lane,
                                                   float (&y)[4]) {
  const int g = r & 7, rh = r >> 3, tig = (r & 7) >> 1, par = r & 1;
  const int b = lane >> 3, lb = lane & 7, l4 = lb & 3, hi = lb >> 2;
  uint32_t bytes[4];
  if (SIDE == 0) {
    const uint32_t word = *reinterpret_cast<const uint32_t *>(
        unit + (b >> 1) * 512 + (4 * g + l4) * 16 + ((b & 1) * 2 + rh) * 4);
#pragma unroll
    for (int i = 0; i < 4; ++i) bytes[i] = (word >> (8 * i)) & 0xffu;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int jc = 4 * l4 + i, mt = 2 * b + (jc >> 3), gq = jc & 7;
      bytes[i] = unit[(mt >> 2) * 512 + (4 * gq + tig) * 16 + (mt & 3) * 4 + par * 2 + rh];
    }
  }
  const float d = __half2float(*reinterpret_cast<const __half *>(
      unit + 1024 + (SIDE == 0 ? g * 4 + rh * 2 : tig * 8 + rh * 4 + par * 2)));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int n = hi ? static_cast<int>(bytes[i] >> 4) : static_cast<int>(bytes[i] & 0xfu);
    y[i] = d * static_cast<float>(n - 8);
  }
}

// The rotated query H (s * q) / 16 of the head held by one quad of lanes in
// the tensor-core fragment order: lane tig holds dims 16c + 4 tig + i as
// v[c][i] (c < 8, i < 4).  Stages on bits 0-1 (i) and 4-6 (c) stay in the
// lane, bits 2-3 (tig) go across the quad; the order of the stages does not
// matter here (the query side is rounded to fp16 afterwards anyway).
__device__ __forceinline__ void turbo_rotate_q_quad(float (&v)[8][4], int tig) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t bits = turbo_signs(c >> 1) >> (16 * (c & 1) + 4 * tig);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if ((bits >> i) & 1u) v[c][i] = -v[c][i];
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float a0 = v[c][0] + v[c][1], a1 = v[c][0] - v[c][1];
    const float a2 = v[c][2] + v[c][3], a3 = v[c][2] - v[c][3];
    v[c][0] = a0 + a2; v[c][2] = a0 - a2; v[c][1] = a1 + a3; v[c][3] = a1 - a3;
  }
#pragma unroll
  for (int m = 1; m < 4; m <<= 1) {
    const bool upper = (tig & m) != 0;
#pragma unroll
    for (int c = 0; c < 8; ++c)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float o = __shfl_xor_sync(0xffffffffu, v[c][i], m);
        v[c][i] = upper ? o - v[c][i] : v[c][i] + o;
      }
  }
#pragma unroll
  for (int h = 1; h < 8; h <<= 1)
#pragma unroll
    for (int c = 0; c < 8; ++c)
      if ((c & h) == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float a = v[c][i], b = v[c + h][i];
          v[c][i] = a + b;
          v[c + h][i] = a - b;
        }
      }
#pragma unroll
  for (int c = 0; c < 8; ++c)
#pragma unroll
    for (int i = 0; i < 4; ++i) v[c][i] *= 0.0625f;
}

// ---------------------------------------------------------------- tensor-core MMA

// D = A(16x16, row) * B(16x8, col) + C, fp16 inputs, fp32 accumulators.
// a[0]=(row g, k 2t..2t+1) a[1]=(row g+8, k 2t..) a[2]=(row g, k 2t+8..) a[3]=(row g+8, k 2t+8..)
// b[0]=(k 2t..2t+1, col g) b[1]=(k 2t+8.., col g); c/d: [0..1]=(row g, col 2t..) [2..3]=(row g+8)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose an 8x8 fp16 matrix held as one m8n8 fragment per warp.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t lop3_and_xor(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;  // (a & b) ^ c
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;  // (a & b) | c
  asm("lop3.b32 %0, %1, %2, %3, 0xea;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t lop3_xor_and(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;  // (a ^ b) & c
  asm("lop3.b32 %0, %1, %2, %3, 0x28;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Element-wise a * b + c and a + b on fp32 pairs, one instruction each.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// D = A * B + C with C in other registers than D (same operands as mma16816).
__device__ __forceinline__ void mma16816c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1, const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}

// Signed bytes 0 and 2 of w as an exact fp16 pair (byte 0 in the low half).
// Each byte is biased to x+128 and placed in the mantissa of 1024, giving
// 1152 + x exactly; subtracting 1152 leaves x.
__device__ __forceinline__ uint32_t s8_pair_02(uint32_t w) {
  return hsub2_bits(lop3_and_xor(w, 0x00ff00ffu, 0x64806480u), 0x64806480u);
}
// Signed bytes 1 and 3.
__device__ __forceinline__ uint32_t s8_pair_13(uint32_t w) {
  return hsub2_bits(lop3_and_xor(w >> 8, 0x00ff00ffu, 0x64806480u), 0x64806480u);
}
// Nibbles at bits 0..3 and 16..19 of w as the exact fp16 pair (n - 8):
// the nibble lands in the mantissa of 1024; subtracting 1032 leaves n - 8.
__device__ __forceinline__ uint32_t u4_pair_minus8(uint32_t w) {
  return hsub2_bits(lop3_and_or(w, 0x000f000fu, 0x64006400u), 0x64086408u);
}
// Nibbles at bits 4..7 and 20..23 of w as the exact fp16 pair (n - 8),
// without a shift: masked in place they give 1024 + 16 n, and one fused
// multiply-add by 1/16 and -72 leaves n - 8 (every step exact in fp16).
__device__ __forceinline__ uint32_t u4_pair_minus8_hi(uint32_t w) {
  const uint32_t x = lop3_and_or(w, 0x00f000f0u, 0x64006400u);
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;\n" : "=r"(r) : "r"(x), "r"(0x2c002c00u), "r"(0xd480d480u));
  return r;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------- mbarrier + bulk copy

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// 1-D bulk async copy global -> shared, completion counted on an mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(phase)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;\n" : "=l"(t));
  return t;
}

// Wait for the given phase of an mbarrier, giving up after ~limit_ns or as
// soon as *abort (a shared flag, optional) becomes non-zero.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t phase,
                                                  const int *abort = nullptr,
                                                  uint64_t limit_ns = 1000000000ull) {
  if (mbar_try_wait(bar, phase)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, phase)) return true;
    if ((it & 63u) == 63u) {
      if (abort && *reinterpret_cast<const volatile int *>(abort)) return false;
      if (globaltimer_ns() - t0 > limit_ns) return false;
    }
  }
}

// Plain shared-memory vector load: ordered after the memory-clobbering waits.
__device__ __forceinline__ uint4 lds128(const void *p) {
  return *reinterpret_cast<const uint4 *>(p);
}
__device__ __forceinline__ uint2 lds64(const void *p) {
  return *reinterpret_cast<const uint2 *>(p);
}

// Paged layers: a page is kPageUnits units (256 tokens) of every kv head of
// one sequence; unit j of (sequence s, kv head h) is pool unit
// (page * n_kv + h) * kPageUnits + j % kPageUnits with page =
// table[s * pages_per_seq + j / kPageUnits].  page_of returns that entry, or
// -1 when it is outside [0, n_pages).
constexpr int kPageUnits = 16;
__device__ __forceinline__ int page_of(const int32_t *table, int pages_per_seq, int n_pages,
                                       int s, int64_t page_idx) {
  const int pg = table[static_cast<int64_t>(s) * pages_per_seq + page_idx];
  return (pg >= 0 && pg < n_pages) ? pg : -1;
}

__device__ __forceinline__ void set_err(int32_t *err, int32_t bit) {
  if (err) atomicOr(err, bit);
}

// turbo4 keys: the B fragments of the rotated query H (s * q) / 16 in the
// nibble codecs' k order, as an fp16 pair per value: qb = fp16(q_r) and
// qlo = fp16(q_r - qb), so that qb + qlo carries q_r to within 2^-22 of its
// size (two MMAs take the place of one); `ld` reads the 4 halves at a row
// offset (global or shared memory).
template <typename Ld>
__device__ __forceinline__ void rotated_q_frags(const __half *qrow, bool hvalid, int tig,
                                                uint32_t (&qb)[8][2], uint32_t (&qlo)[8][2],
                                                Ld ld) {
  float v[8][4];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint2 r = make_uint2(0u, 0u);
    if (hvalid) r = ld(qrow + 16 * c + 4 * tig);
    const __half2 h01 = *reinterpret_cast<const __half2 *>(&r.x);
    const __half2 h23 = *reinterpret_cast<const __half2 *>(&r.y);
    v[c][0] = __low2float(h01); v[c][1] = __high2float(h01);
    v[c][2] = __low2float(h23); v[c][3] = __high2float(h23);
  }
  turbo_rotate_q_quad(v, tig);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    qb[c][0] = pack_half2(v[c][0], v[c][2]);
    qb[c][1] = pack_half2(v[c][1], v[c][3]);
    const float2 h0 = __half22float2(*reinterpret_cast<const __half2 *>(&qb[c][0]));
    const float2 h1 = __half22float2(*reinterpret_cast<const __half2 *>(&qb[c][1]));
    qlo[c][0] = pack_half2(v[c][0] - h0.x, v[c][2] - h0.y);
    qlo[c][1] = pack_half2(v[c][1] - h1.x, v[c][3] - h1.y);
  }
}

// Programmatic dependent launch: wait for the previous grid on the stream to
// complete (and its writes to be visible), and let the next grid launch early.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Opt `kernel` in to `bytes` of dynamic shared memory on the current device.
// The setting belongs to the device, so it is made once per device ordinal
// (`done` holds one bit per ordinal; ordinals >= 64 set it on every call).
template <typename Kernel>
inline cudaError_t smem_optin(Kernel kernel, int bytes, std::atomic<uint64_t> &done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel on the stream drains; it must call
// grid_dependency_wait() before touching that kernel's results.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace kvq
