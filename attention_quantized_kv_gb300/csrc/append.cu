// append.cu -- quantize-on-append: encode new K/V rows into the cache.
//
// Block codecs of the "Codecs" table of the buun-llama-cpp listing (q8_0 8.5
// and q4_0 4.5 bits per value, 32-value blocks with an fp16 scale), with the
// fp32 encoder formulas of include/kvq.h, evaluated with explicit IEEE
// round-to-nearest operations so that the bytes are reproducible bit for bit.
//
// One warp encodes one 128-value row: lane l holds dims 4l..4l+3, so each
// 32-value block is 8 lanes and its amax / signed max is a 3-step xor-shuffle
// reduction.  Each lane then writes its part of the row straight into the
// row's places in the 16-token unit (see the layout in include/kvq.h).
#include <cuda_runtime.h>

#include <algorithm>

#include "kvq_device.cuh"
#include "kvq_encode.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

// Read one row (token row r of `unit`) into the lane-held form of store_row:
// lane l gets dims 4l..4l+3 as fp32, the decoded values x^ = d16 * q (q8_0),
// d16 * (n - 8) (q4_0), s * H (d16 * (n - 8)) / 16 (turbo4) or the fp16
// values, all exact in fp32.
template <int SIDE>
__device__ __forceinline__ void load_row(int codec, const uint8_t *unit, int r, int lane,
                                         float (&x)[4]) {
  const int g = r & 7, rh = r >> 3, tig = (r & 7) >> 1, par = r & 1;
  const int b = lane >> 3, lb = lane & 7;
  if (codec == KVQ_F16) {
    if (SIDE == 0) {
      const int h = (lane >> 2) & 1, w = lane & 3;
      const uint2 raw =
          *reinterpret_cast<const uint2 *>(unit + (2 * b + rh) * 512 + (4 * g + w) * 16 + h * 8);
      const __half2 h01 = *reinterpret_cast<const __half2 *>(&raw.x);
      const __half2 h23 = *reinterpret_cast<const __half2 *>(&raw.y);
      x[0] = __low2float(h01); x[1] = __high2float(h01);
      x[2] = __low2float(h23); x[3] = __high2float(h23);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int d = 4 * lane + i, mt = d >> 4, gq = (d & 15) >> 1, sb = d & 1;
        x[i] = __half2float(*reinterpret_cast<const __half *>(
            unit + mt * 512 + (4 * gq + tig) * 16 + (rh * 4 + sb * 2 + par) * 2));
      }
    }
    return;
  }
  if (codec == KVQ_Q8_0) {
    int q[4];
    int soff;
    if (SIDE == 0) {
      const int h = lb >> 2, w = lane & 3;
      const uint32_t word =
          *reinterpret_cast<const uint32_t *>(unit + b * 512 + (4 * g + w) * 16 + (2 * rh + h) * 4);
#pragma unroll
      for (int i = 0; i < 4; ++i) q[i] = static_cast<int8_t>((word >> (8 * i)) & 0xffu);
      soff = 2048 + g * 16 + rh * 8 + b * 2;
    } else {
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        const int d = 4 * lane + 2 * pp, mt = d >> 4, gq = (d & 15) >> 1;
        const uint32_t v = *reinterpret_cast<const uint16_t *>(
            unit + (mt >> 1) * 512 + (4 * gq + tig) * 16 + ((mt & 1) * 2 + rh) * 4 + par * 2);
        q[2 * pp] = static_cast<int8_t>(v & 0xffu);
        q[2 * pp + 1] = static_cast<int8_t>(v >> 8);
      }
      soff = 2048 + tig * 32 + b * 8 + rh * 4 + par * 2;
    }
    const float d = __half2float(*reinterpret_cast<const __half *>(unit + soff));
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = d * static_cast<float>(q[i]);
    return;
  }
  if (codec == KVQ_TURBO4) {
    turbo4_row_rotated<SIDE>(unit, r, lane, x);
    turbo_unrotate_lane(x, lane);
    return;
  }
  // q4_0: lanes lb < 4 hold canonical bytes jc = 4lb..4lb+3 (low nibbles),
  // lanes lb + 4 the same bytes' high nibbles.
  const int l4 = lb & 3, hi = lb >> 2;
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
  const int soff = SIDE == 0 ? 1024 + g * 16 + rh * 8 + b * 2
                             : 1024 + tig * 32 + b * 8 + rh * 4 + par * 2;
  const float d = __half2float(*reinterpret_cast<const __half *>(unit + soff));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int n = hi ? static_cast<int>(bytes[i] >> 4) : static_cast<int>(bytes[i] & 0xfu);
    x[i] = d * static_cast<float>(n - 8);
  }
}

struct AppendParams {
  const __half *x[2];  // k_new, v_new: [n_seqs][max_new][n_kv][128]
  uint8_t *cache[2];
  int codec[2];
  int32_t *seq_lens;  // read by every row; advanced only by append_small_kernel
  const int32_t *n_new;
  int32_t *err;
  const int32_t *table;  // paged layers: block table; nullptr: contiguous
  int n_seqs, n_kv, max_new, capacity, pages_per_seq, n_pages;
};

constexpr int kAppendWarps = 8;

__device__ __forceinline__ void append_row(const AppendParams &p, int64_t row, int lane) {
  const int64_t rows_per_side = static_cast<int64_t>(p.n_seqs) * p.max_new * p.n_kv;
  const int side = row >= rows_per_side ? 1 : 0;
  const int64_t rr = row - side * rows_per_side;
  const int kvh = static_cast<int>(rr % p.n_kv);
  const int i = static_cast<int>((rr / p.n_kv) % p.max_new);
  const int s = static_cast<int>(rr / (static_cast<int64_t>(p.n_kv) * p.max_new));
  if (i >= p.n_new[s]) return;
  const int64_t pos = static_cast<int64_t>(p.seq_lens[s]) + i;
  if (pos < 0 || pos >= p.capacity) {
    if (lane == 0) set_err(p.err, KVQ_DEVERR_CAPACITY);
    return;
  }
  const uint2 raw = reinterpret_cast<const uint2 *>(p.x[side] + rr * kD)[lane];
  const int codec = p.codec[side];
  int64_t unit_idx;
  if (p.table) {
    const int pg =
        page_of(p.table, p.pages_per_seq, p.n_pages, s, pos / (kUnitTokens * kPageUnits));
    if (pg < 0) {
      if (lane == 0) set_err(p.err, KVQ_DEVERR_PAGE);
      return;
    }
    unit_idx = (static_cast<int64_t>(pg) * p.n_kv + kvh) * kPageUnits +
               (pos / kUnitTokens) % kPageUnits;
  } else {
    unit_idx = (static_cast<int64_t>(s) * p.n_kv + kvh) * (p.capacity / kUnitTokens) +
               pos / kUnitTokens;
  }
  uint8_t *unit = p.cache[side] + unit_idx * unit_bytes(codec);
  const int r = static_cast<int>(pos % kUnitTokens);
  if (side == 0) encode_row_into<0>(codec, raw, unit, r, lane);
  else encode_row_into<1>(codec, raw, unit, r, lane);
}

// One warp per row (grid covers all rows).
// Every kernel here lets the next kernel of the stream launch at once (it
// waits for this grid's completion before it reads anything this grid
// writes), so that its prologue overlaps this one.
__global__ void __launch_bounds__(kAppendWarps * 32) append_kernel(AppendParams p) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kAppendWarps + (threadIdx.x >> 5);
  const int64_t rows = 2ll * p.n_seqs * p.max_new * p.n_kv;
  if (row < rows) append_row(p, row, lane);
}

// Small appends (a decode step): one CTA whose warps take all rows, then,
// once every row has read its position, advances the lengths itself.
__global__ void __launch_bounds__(kAppendWarps * 32) append_small_kernel(AppendParams p,
                                                                        int update_lens) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t rows = 2ll * p.n_seqs * p.max_new * p.n_kv;
  for (int64_t row = threadIdx.x >> 5; row < rows; row += kAppendWarps) append_row(p, row, lane);
  if (update_lens) {
    __syncthreads();
    for (int s = threadIdx.x; s < p.n_seqs; s += kAppendWarps * 32) {
      const int v = p.seq_lens[s] + p.n_new[s];
      p.seq_lens[s] = v > p.capacity ? p.capacity : v;
    }
  }
}

__global__ void update_lens_kernel(int32_t *seq_lens, const int32_t *n_new, int n_seqs,
                                   int capacity) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s < n_seqs) {
    const int v = seq_lens[s] + n_new[s];
    seq_lens[s] = v > capacity ? capacity : v;
  }
}

constexpr int64_t kSmallAppendRows = 64;  // at most 8 rows per warp

struct RequantParams {
  const uint8_t *src;
  uint8_t *dst;
  const int32_t *seq_lens;
  int32_t *err;
  const int32_t *table;  // paged layers: block table; nullptr: contiguous
  int src_codec, dst_codec, n_kv, capacity, pages_per_seq, n_pages;
  int units_per_stream;  // block re-encode: units per (seq, kv head) stream
  int64_t n_units;       //                  in all
};

constexpr int kRqUnits = 8;  // units per CTA of the re-encode kernel
static_assert(kPageUnits % kRqUnits == 0, "a run of units must lie inside one page");

// turbo4 on either side: one CTA per run of kRqUnits 16-token units of one
// (sequence, kv head) stream.  The source units are copied into shared memory with coalesced
// 16-byte loads (all of them requested before any is used); warp w then
// re-encodes rows w, w + 16, ... below the sequence's length there (decode
// exactly to fp32, then the append encoder of the new codec; an f16 target
// rounds to fp16) into a shared copy of the destination units, which go out
// with coalesced 16-byte stores.  The unit holding the sequence's last tokens
// first reads its destination bytes, so that its rows past the length keep
// them.  SC / DC: source and destination codecs (compile-time, so that the
// row decode and encode carry no codec dispatch).
template <int SIDE, int SC, int DC>
__global__ void __launch_bounds__(kUnitTokens * 32) requant_kernel(RequantParams p) {
  extern __shared__ uint4 rq_smem[];
  grid_dependency_wait();
  const int kvh = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int len = min(p.seq_lens[s], p.capacity);
  const int u0 = blockIdx.x * kRqUnits;
  const int n_units = min(kRqUnits, (len + kUnitTokens - 1) / kUnitTokens - u0);
  if (n_units > 0) {
    // first unit of the run (a run lies inside one page: kPageUnits % kRqUnits == 0)
    int64_t uidx;
    if (p.table) {
      const int pg = page_of(p.table, p.pages_per_seq, p.n_pages, s, u0 / kPageUnits);
      if (pg < 0) {
        if (threadIdx.x == 0) set_err(p.err, KVQ_DEVERR_PAGE);
        return;  // whole CTA
      }
      uidx = (static_cast<int64_t>(pg) * p.n_kv + kvh) * kPageUnits + u0 % kPageUnits;
    } else {
      uidx = (static_cast<int64_t>(s) * p.n_kv + kvh) * (p.capacity / kUnitTokens) + u0;
    }
    constexpr int sb = unit_bytes(SC), db = unit_bytes(DC);
    uint4 *sbuf = rq_smem;
    uint4 *dbuf = rq_smem + kRqUnits * sb / 16;
    const uint4 *su = reinterpret_cast<const uint4 *>(p.src + uidx * sb);
    uint4 *du = reinterpret_cast<uint4 *>(p.dst + uidx * db);
    for (int i = threadIdx.x; i < n_units * sb / 16; i += blockDim.x) sbuf[i] = su[i];
    if ((u0 + n_units) * kUnitTokens > len) {  // the last unit is partial
      const int base = (n_units - 1) * db / 16;
      for (int i = threadIdx.x; i < db / 16; i += blockDim.x) dbuf[base + i] = du[base + i];
    }
    __syncthreads();
    const int rows = min(n_units * kUnitTokens, len - u0 * kUnitTokens);
    for (int row = warp; row < rows; row += kUnitTokens) {
      const int ul = row / kUnitTokens, r = row % kUnitTokens;
      float x[4];
      load_row<SIDE>(SC, reinterpret_cast<const uint8_t *>(sbuf) + ul * sb, r, lane, x);
      int q[4] = {0, 0, 0, 0};
      __half d16 = __float2half_rn(0.0f);
      uint2 raw = make_uint2(0u, 0u);
      if (DC == KVQ_Q8_0) {
        encode_q8(x, q, d16);
      } else if (DC == KVQ_Q4_0) {
        encode_q4(x, lane, q, d16);
      } else if (DC == KVQ_TURBO4) {
        encode_turbo4(x, lane, q, d16);
      } else {
        const __half2 h01 = __floats2half2_rn(x[0], x[1]), h23 = __floats2half2_rn(x[2], x[3]);
        raw.x = *reinterpret_cast<const uint32_t *>(&h01);
        raw.y = *reinterpret_cast<const uint32_t *>(&h23);
      }
      store_row<SIDE>(DC, reinterpret_cast<uint8_t *>(dbuf) + ul * db, r, lane, raw, q, d16);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n_units * db / 16; i += blockDim.x) du[i] = dbuf[i];
  }
  grid_launch_dependents();
}

// ---------------------------------------------------------------------------
// Re-encode between the block codecs (f16, q8_0, q4_0): one thread per
// (unit, token row, 32-value block), so the block's amax or signed maximum is
// a serial scan in registers and its divisions are taken once per block.
// Every warp of the persistent grid works alone, with no CTA-wide barrier:
// it walks 16-token units of the flattened [seq][kv head][unit] space (unit
// j goes to warp j % (all warps)) through kRbStages shared-memory stages of
// its own.  Lane 0 bulk-copies the source unit j + kRbStages * (all warps)
// into a stage as soon as the warp is done with it, so kRbStages - 1 units
// per warp are in flight while one is encoded; each lane encodes two of the
// unit's 64 (row, block) items and stores the encoded pieces straight to the
// destination (rows past a sequence's length are not written).
constexpr int kRbWarps = 8;
constexpr int kRbThreads = kRbWarps * 32;
constexpr int kRbStages = 2;  // source stages per warp: a warp's unit i uses stage i % kRbStages

// K side: for every codec the 32 values of block b of row r lie in four
// pieces w = 0..3, piece w holding dims 32b + {4w..4w+3, 16+4w..16+4w+3} in
// this order (f16: 16 bytes at (2b+rh)*512 + 64g + 16w; q8_0: 8 quants at
// b*512 + 64g + 16w + 8rh; q4_0: canonical bytes 4w..4w+3 at
// (b>>1)*512 + 64g + 16w + ((b&1)*2+rh)*4, low nibbles the first four
// values, high nibbles the last four).  A thread visits its pieces in the
// order w = (k + (g >> 1)) & 3, k = 0..3, which puts the eight threads of a
// shared-memory phase (rows g = 0..7) on distinct banks.
__host__ __device__ constexpr int rq_piece_dim(int w, int v) {
  return v < 4 ? 4 * w + v : 16 + 4 * w + (v - 4);
}

// A chunk: the 8 values of one piece (K side) or of the same dims on the V
// side, value v being dim rq_piece_dim(w, v) of the block.  V side (tig =
// g >> 1, par = g & 1): f16 dim e at (2b + (e>>4))*512 + (4gq+tig)*16 +
// (rh*4 + s*2 + par)*2 with gq = (e&15)>>1, s = e&1; q8_0 quant pair (e, e+1),
// e even, at b*512 + (4gq+tig)*16 + ((e>>4)*2 + rh)*4 + par*2; q4_0 canonical
// byte jc (dims jc and jc + 16) at (b>>1)*512 + (4(jc&7)+tig)*16 +
// (2(b&1) + (jc>>3))*4 + par*2 + rh.
struct RowGeo {
  int g, rh, tig, par, b;
};

__device__ __forceinline__ int rq_v_f16_off(const RowGeo &q, int e) {
  return (2 * q.b + (e >> 4)) * 512 + (4 * ((e & 15) >> 1) + q.tig) * 16 +
         (q.rh * 4 + (e & 1) * 2 + q.par) * 2;
}
__device__ __forceinline__ int rq_v_q8_off(const RowGeo &q, int e) {  // e even
  return q.b * 512 + (4 * ((e & 15) >> 1) + q.tig) * 16 + ((e >> 4) * 2 + q.rh) * 4 + q.par * 2;
}
__device__ __forceinline__ int rq_v_q4_off(const RowGeo &q, int jc) {
  return (q.b >> 1) * 512 + (4 * (jc & 7) + q.tig) * 16 + (2 * (q.b & 1) + (jc >> 3)) * 4 +
         q.par * 2 + q.rh;
}
__device__ __forceinline__ int rq_k_off(int codec, const RowGeo &q, int w) {
  return codec == KVQ_F16    ? (2 * q.b + q.rh) * 512 + 64 * q.g + 16 * w
         : codec == KVQ_Q8_0 ? q.b * 512 + 64 * q.g + 16 * w + 8 * q.rh
                             : (q.b >> 1) * 512 + 64 * q.g + 16 * w + ((q.b & 1) * 2 + q.rh) * 4;
}

// The chunk's values, decoded exactly to fp32 (d: the source block's scale).
template <int SIDE, int SC>
__device__ __forceinline__ void rq_load_chunk(const uint8_t *u, const RowGeo &q, int w, float d,
                                              float (&x)[8]) {
  if (SC == KVQ_F16) {
    uint32_t h[4];
    if (SIDE == 0) {
      const uint4 raw = *reinterpret_cast<const uint4 *>(u + rq_k_off(SC, q, w));
      h[0] = raw.x; h[1] = raw.y; h[2] = raw.z; h[3] = raw.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e0 = rq_piece_dim(w, 2 * i);
        h[i] = static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(u + rq_v_f16_off(q, e0))) |
               (static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(
                    u + rq_v_f16_off(q, e0 + 1)))
                << 16);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h[i]));
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  } else if (SC == KVQ_Q8_0) {
    uint32_t lo, hi;  // quants of values 0..3 and 4..7, one per byte
    if (SIDE == 0) {
      const uint2 raw = *reinterpret_cast<const uint2 *>(u + rq_k_off(SC, q, w));
      lo = raw.x;
      hi = raw.y;
    } else {
      const uint32_t p0 = *reinterpret_cast<const uint16_t *>(u + rq_v_q8_off(q, 4 * w));
      const uint32_t p1 = *reinterpret_cast<const uint16_t *>(u + rq_v_q8_off(q, 4 * w + 2));
      const uint32_t p2 = *reinterpret_cast<const uint16_t *>(u + rq_v_q8_off(q, 16 + 4 * w));
      const uint32_t p3 = *reinterpret_cast<const uint16_t *>(u + rq_v_q8_off(q, 18 + 4 * w));
      lo = p0 | (p1 << 16);
      hi = p2 | (p3 << 16);
    }
#pragma unroll
    for (int v = 0; v < 8; ++v)
      x[v] = d * static_cast<float>(
                     static_cast<int8_t>(((v < 4 ? lo : hi) >> (8 * (v & 3))) & 0xffu));
  } else {
    uint32_t raw;  // canonical bytes 4w..4w+3
    if (SIDE == 0) {
      raw = *reinterpret_cast<const uint32_t *>(u + rq_k_off(SC, q, w));
    } else {
      raw = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        raw |= static_cast<uint32_t>(u[rq_v_q4_off(q, 4 * w + i)]) << (8 * i);
    }
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const int n = static_cast<int>((raw >> (8 * (v & 3) + (v < 4 ? 0 : 4))) & 0xfu);
      x[v] = d * static_cast<float>(n - 8);
    }
  }
}

// Bytes 0 of a, b, c, d as one word (a in the lowest byte).
__device__ __forceinline__ uint32_t low_bytes4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}
// Four byte lanes holding 0..16, each clamped to 15 (16 - (16 >> 4)).
__device__ __forceinline__ uint32_t clamp15x4(uint32_t w) { return w - ((w >> 4) & 0x01010101u); }

// Store a chunk: f16 from x; else the codes k, words whose lowest byte is
// the code (q8_0: q & 0xff; q4_0: the level 0..16 before the clamp to 15).
template <int SIDE, int DC>
__device__ __forceinline__ void rq_store_chunk(uint8_t *u, const RowGeo &q, int w,
                                               const float (&x)[8], const uint32_t (&k)[8]) {
  if (DC == KVQ_F16) {
    uint32_t h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 t = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
      h[i] = *reinterpret_cast<const uint32_t *>(&t);
    }
    if (SIDE == 0) {
      *reinterpret_cast<uint4 *>(u + rq_k_off(DC, q, w)) = make_uint4(h[0], h[1], h[2], h[3]);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e0 = rq_piece_dim(w, 2 * i);
        *reinterpret_cast<uint16_t *>(u + rq_v_f16_off(q, e0)) = static_cast<uint16_t>(h[i]);
        *reinterpret_cast<uint16_t *>(u + rq_v_f16_off(q, e0 + 1)) =
            static_cast<uint16_t>(h[i] >> 16);
      }
    }
  } else if (DC == KVQ_Q8_0) {
    const uint32_t lo = low_bytes4(k[0], k[1], k[2], k[3]), hi = low_bytes4(k[4], k[5], k[6], k[7]);
    if (SIDE == 0) {
      *reinterpret_cast<uint2 *>(u + rq_k_off(DC, q, w)) = make_uint2(lo, hi);
    } else {
      uint16_t *const pr[4] = {reinterpret_cast<uint16_t *>(u + rq_v_q8_off(q, 4 * w)),
                               reinterpret_cast<uint16_t *>(u + rq_v_q8_off(q, 4 * w + 2)),
                               reinterpret_cast<uint16_t *>(u + rq_v_q8_off(q, 16 + 4 * w)),
                               reinterpret_cast<uint16_t *>(u + rq_v_q8_off(q, 18 + 4 * w))};
      *pr[0] = static_cast<uint16_t>(lo);
      *pr[1] = static_cast<uint16_t>(lo >> 16);
      *pr[2] = static_cast<uint16_t>(hi);
      *pr[3] = static_cast<uint16_t>(hi >> 16);
    }
  } else {
    const uint32_t lo = clamp15x4(low_bytes4(k[0], k[1], k[2], k[3]));
    const uint32_t hi = clamp15x4(low_bytes4(k[4], k[5], k[6], k[7]));
    const uint32_t word = lo | (hi << 4);  // canonical bytes 4w..4w+3
    if (SIDE == 0) {
      *reinterpret_cast<uint32_t *>(u + rq_k_off(DC, q, w)) = word;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        u[rq_v_q4_off(q, 4 * w + i)] = static_cast<uint8_t>(word >> (8 * i));
    }
  }
}

// The quotient path of q8_from_quotient / q4_from_quotient on one chunk, two
// values per instruction: k[v] gets the fast path's code (its lowest byte;
// q4_0: the level before the clamp), and lo / hi collect the chunk's
// distances from the rounding boundaries (q8_0: hi = the largest distance
// to the nearest integer; q4_0: lo, hi = the range of u - floor(u)), which
// say whether the fast path is the exact one for every value.
template <int DC>
__device__ __forceinline__ void rq_codes_fast(const float (&x)[8], float rcp, uint32_t (&k)[8],
                                              float &lo, float &hi) {
  const float2 r2 = make_float2(rcp, rcp), m2 = make_float2(kRoundMagic, kRoundMagic);
  const float2 nm2 = make_float2(-kRoundMagic, -kRoundMagic), n1 = make_float2(-1.0f, -1.0f);
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    if (DC == KVQ_Q8_0) {
      const float2 t = __fmul2_rn(make_float2(x[j], x[j + 1]), r2);
      const float2 tm = __fadd2_rn(t, m2);
      const float2 fr = __ffma2_rn(__fadd2_rn(tm, nm2), n1, t);  // t - round(t)
      hi = fmaxf(hi, fmaxf(fabsf(fr.x), fabsf(fr.y)));
      k[j] = __float_as_uint(tm.x);
      k[j + 1] = __float_as_uint(tm.y);
    } else {
      const float2 u =
          __fadd2_rn(__fmul2_rn(make_float2(x[j], x[j + 1]), r2), make_float2(8.5f, 8.5f));
      const float2 fm = __fadd2_rn(__fadd2_rn(u, make_float2(-0.5f, -0.5f)), m2);
      const float2 fr = __ffma2_rn(__fadd2_rn(fm, nm2), n1, u);  // u - floor(u)
      lo = fminf(lo, fminf(fr.x, fr.y));
      hi = fmaxf(hi, fmaxf(fr.x, fr.y));
      k[j] = __float_as_uint(fm.x);
      k[j + 1] = __float_as_uint(fm.y);
    }
  }
}

// One (unit, row, block) item: decode the block exactly and encode it with
// the append encoder of DC (q8_0: d = amax / 127; q4_0: d = m / -8 with m the
// signed value of largest magnitude, lowest dim on ties; the quotient rule
// of q8_from_quotient / q4_from_quotient), in two passes over the chunks
// (the block's statistics, then the codes) so that few values are live.
// The codes take the two-at-a-time fast path; if any value of the block
// lies too near its rounding boundary, the block is encoded again value by
// value with the exact path.
template <int SIDE, int SC, int DC>
__device__ __forceinline__ void rq_encode_item(const uint8_t *su, uint8_t *du, int r, int b) {
  RowGeo q;
  q.g = r & 7;
  q.rh = r >> 3;
  q.tig = q.g >> 1;
  q.par = q.g & 1;
  q.b = b;
  const int rot = SIDE == 0 ? q.g >> 1 : 0;  // K side: the piece order (c + rot) & 3
  const int soff =
      SIDE == 0 ? q.g * 16 + q.rh * 8 + b * 2 : q.tig * 32 + b * 8 + q.rh * 4 + q.par * 2;
  const float ds = SC == KVQ_F16 ? 0.0f
                                 : __half2float(*reinterpret_cast<const __half *>(
                                       su + unit_scale_offset(SC) + soff));
  const uint32_t zero[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (DC == KVQ_F16) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int w = (c + rot) & 3;
      float x[8];
      rq_load_chunk<SIDE, SC>(su, q, w, ds, x);
      rq_store_chunk<SIDE, DC>(du, q, w, x, zero);
    }
    return;
  }
  // pass 1: amax (q8_0) or the largest and smallest value (q4_0)
  float pmax, nmin;
  if (SIDE == 0 && SC == KVQ_F16) {  // on the fp16 values themselves (exact)
    __half2 hp = __float2half2_rn(-65504.0f), hn = __float2half2_rn(65504.0f);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 raw = *reinterpret_cast<const uint4 *>(su + rq_k_off(SC, q, (c + rot) & 3));
      const uint32_t h[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 v = *reinterpret_cast<const __half2 *>(&h[i]);
        if (DC == KVQ_Q8_0) {
          hp = __hmax2(hp, __habs2(v));
        } else {
          hp = __hmax2(hp, v);
          hn = __hmin2(hn, v);
        }
      }
    }
    pmax = fmaxf(__low2float(hp), __high2float(hp));
    nmin = fminf(__low2float(hn), __high2float(hn));
  } else {
    pmax = DC == KVQ_Q8_0 ? 0.0f : -INFINITY;
    nmin = INFINITY;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float x[8];
      rq_load_chunk<SIDE, SC>(su, q, (c + rot) & 3, ds, x);
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        if (DC == KVQ_Q8_0) {
          pmax = fmaxf(pmax, fabsf(x[v]));
        } else {
          pmax = fmaxf(pmax, x[v]);
          nmin = fminf(nmin, x[v]);
        }
      }
    }
  }
  float d;
  if (DC == KVQ_Q8_0) {
    d = __fdiv_rn(pmax, 127.0f);
  } else {
    float m = pmax > -nmin ? pmax : nmin;
    if (pmax == -nmin) {  // both signs reach the largest magnitude (or all zero)
      float best = -1.0f;
      int idx = 32;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int w = (c + rot) & 3;
        float x[8];
        rq_load_chunk<SIDE, SC>(su, q, w, ds, x);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const float a = fabsf(x[v]);
          const int dim = rq_piece_dim(w, v);
          if (a > best || (a == best && dim < idx)) { best = a; m = x[v]; idx = dim; }
        }
      }
    }
    d = __fdiv_rn(m, -8.0f);
  }
  *reinterpret_cast<__half *>(du + unit_scale_offset(DC) + soff) = __float2half_rn(d);
  const float rcp = d != 0.0f ? __frcp_rn(d) : 0.0f;
  // pass 2: the codes
  float lo = 1.0f, hi = 0.0f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int w = (c + rot) & 3;
    float x[8];
    uint32_t k[8];
    rq_load_chunk<SIDE, SC>(su, q, w, ds, x);
    if (d != 0.0f) {
      rq_codes_fast<DC>(x, rcp, k, lo, hi);
    } else {
#pragma unroll
      for (int v = 0; v < 8; ++v) k[v] = DC == KVQ_Q8_0 ? 0u : 8u;
    }
    rq_store_chunk<SIDE, DC>(du, q, w, x, k);
  }
  const bool exact =
      DC == KVQ_Q8_0 ? hi < 0.5f - 0x1p-14f : (lo > 0x1p-17f && hi < 1.0f - 0x1p-17f);
  if (d != 0.0f && !exact) {  // rare: some quotient near a boundary
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int w = (c + rot) & 3;
      float x[8];
      uint32_t k[8];
      rq_load_chunk<SIDE, SC>(su, q, w, ds, x);
#pragma unroll
      for (int v = 0; v < 8; ++v)
        k[v] = static_cast<uint32_t>(DC == KVQ_Q8_0 ? q8_from_quotient(x[v], d, rcp)
                                                    : q4_from_quotient(x[v], d, rcp));
      rq_store_chunk<SIDE, DC>(du, q, w, x, k);
    }
  }
}

template <int SIDE, int SC, int DC>
__global__ void __launch_bounds__(kRbThreads, DC == KVQ_Q4_0 ? 2 : 3)
    rq_block_kernel(RequantParams p) {
  constexpr int sb = unit_bytes(SC), db = unit_bytes(DC);
  extern __shared__ __align__(128) uint8_t rb_smem[];
  __shared__ __align__(8) uint64_t full[kRbWarps][kRbStages];
  // lane 0 describes each unit when it issues its copy: the rows below the
  // length (0: nothing to do) and the unit's index in the cache or pool
  struct UnitInfo {
    int rows, pad;
    int64_t uidx;
  };
  __shared__ UnitInfo info[kRbWarps][kRbStages];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t *const stage0 = rb_smem + warp * kRbStages * sb;
  if (lane == 0) {
    for (int q = 0; q < kRbStages; ++q) mbar_init(&full[warp][q], 1);
    fence_mbar_init();
  }
  __syncwarp();
  grid_dependency_wait();

  // The unit's global reads (its sequence's length, its block-table entry)
  // go out one unit ahead (prepare), so that their latency hides behind the
  // encoding of the current unit.
  struct UnitPre {
    int s, kvh, u, len, pg;
  };
  const uint32_t ups = static_cast<uint32_t>(p.units_per_stream);
  auto prepare = [&](int64_t j) {
    const uint32_t jj = static_cast<uint32_t>(j);  // n_units < 2^31 (checked by the host)
    const uint32_t t = jj / ups;
    UnitPre pr;
    pr.kvh = static_cast<int>(t % static_cast<uint32_t>(p.n_kv));
    pr.s = static_cast<int>(t / static_cast<uint32_t>(p.n_kv));
    pr.u = static_cast<int>(jj - t * ups);
    pr.len = p.seq_lens[pr.s];
    pr.pg = p.table ? page_of(p.table, p.pages_per_seq, p.n_pages, pr.s, pr.u / kPageUnits) : 0;
    return pr;
  };
  auto issue = [&](const UnitPre &pr, int st) {  // lane 0
    UnitInfo ui;
    ui.rows = max(0, min(kUnitTokens, min(pr.len, p.capacity) - pr.u * kUnitTokens));
    ui.pad = 0;
    ui.uidx = 0;
    if (ui.rows > 0) {
      if (p.table) {
        if (pr.pg < 0) {
          set_err(p.err, KVQ_DEVERR_PAGE);
          ui.rows = 0;
        } else {
          ui.uidx = (static_cast<int64_t>(pr.pg) * p.n_kv + pr.kvh) * kPageUnits +
                    pr.u % kPageUnits;
        }
      } else {
        ui.uidx = static_cast<int64_t>(pr.s * p.n_kv + pr.kvh) * ups + pr.u;
      }
    }
    info[warp][st] = ui;
    // an empty unit only completes the stage's barrier phase
    const uint32_t bytes = ui.rows > 0 ? static_cast<uint32_t>(sb) : 0u;
    mbar_arrive_expect_tx(&full[warp][st], bytes);
    if (bytes) bulk_copy_g2s(stage0 + st * sb, p.src + ui.uidx * sb, bytes, &full[warp][st]);
  };

  const int64_t W = static_cast<int64_t>(gridDim.x) * kRbWarps;
  const int64_t j0 = static_cast<int64_t>(blockIdx.x) * kRbWarps + warp;
  int64_t issued = 0;  // lane 0: units issued (the i-th into stage i % kRbStages)
  if (lane == 0) {
    for (int64_t j = j0; j < p.n_units && issued < kRbStages; j += W, ++issued)
      issue(prepare(j), static_cast<int>(issued));
  }
  __syncwarp();
  int i = 0;
  for (int64_t j = j0; j < p.n_units; j += W, ++i) {
    const int st = i % kRbStages;
    const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(
                                                  &full[warp][st],
                                                  static_cast<uint32_t>(i / kRbStages) & 1u));
    if (!got) {
      if (lane == 0) set_err(p.err, KVQ_DEVERR_TIMEOUT);
      break;
    }
    const UnitInfo ui = info[warp][st];
    const int64_t jn = j + kRbStages * W;  // the unit that takes this stage next
    UnitPre pre{};
    if (lane == 0 && jn < p.n_units) pre = prepare(jn);
#pragma unroll 1
    for (int t = 0; t < 2; ++t) {  // items lane and lane + 32: row item & 15, block item >> 4
      const int item = lane + 32 * t, r = item & 15, b = item >> 4;
      if (r < ui.rows)
        rq_encode_item<SIDE, SC, DC>(stage0 + st * sb, p.dst + ui.uidx * db, r, b);
    }
    __syncwarp();  // every lane is done with the stage
    if (lane == 0 && jn < p.n_units) {
      fence_proxy_async_smem();
      issue(pre, st);
      ++issued;
    }
    __syncwarp();
  }
  if (lane == 0) {
    // after a timeout: the copies still in flight into this warp's stages
    // (units i .. issued - 1)
    for (int64_t q = i; q < issued; ++q)
      mbar_wait_bounded(&full[warp][q % kRbStages], static_cast<uint32_t>(q / kRbStages) & 1u);
  }
  grid_launch_dependents();
}

template <int SIDE, int SC, int DC>
cudaError_t launch_requant_t(const RequantParams &p, dim3 grid, int smem, int num_sms,
                             cudaStream_t stream) {
  static std::atomic<uint64_t> optin{0};
  if constexpr (SC != KVQ_TURBO4 && DC != KVQ_TURBO4) {  // block codecs: a thread per block
    constexpr int rb_smem = kRbWarps * kRbStages * unit_bytes(SC);
    const cudaError_t e = smem_optin(rq_block_kernel<SIDE, SC, DC>, rb_smem, optin);
    if (e != cudaSuccess) return e;
    static std::atomic<int> per_sm{0};  // resident CTAs per SM
    if (per_sm.load() == 0) {
      int n = 0;
      const cudaError_t eo = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &n, rq_block_kernel<SIDE, SC, DC>, kRbThreads, rb_smem);
      if (eo != cudaSuccess) return eo;
      per_sm.store(n > 0 ? n : 1);
    }
    const int64_t g =
        std::min<int64_t>((p.n_units + kRbWarps - 1) / kRbWarps,
                          static_cast<int64_t>(per_sm.load()) * (num_sms > 0 ? num_sms : 148));
    if (g <= 0) return cudaSuccess;
    return launch_pdl(rq_block_kernel<SIDE, SC, DC>, dim3(static_cast<unsigned>(g)),
                      dim3(kRbThreads), rb_smem, stream, p);
  } else {  // turbo4 rotates whole rows: a warp per row
    const cudaError_t e = smem_optin(requant_kernel<SIDE, SC, DC>, kRqUnits * 2 * 4096, optin);
    if (e != cudaSuccess) return e;
    return launch_pdl(requant_kernel<SIDE, SC, DC>, grid, dim3(kUnitTokens * 32), smem, stream,
                      p);
  }
}

template <int SIDE, int SC>
cudaError_t launch_requant_d(int dc, const RequantParams &p, dim3 grid, int smem, int num_sms,
                             cudaStream_t stream) {
  switch (dc) {
    case KVQ_F16: return launch_requant_t<SIDE, SC, KVQ_F16>(p, grid, smem, num_sms, stream);
    case KVQ_Q8_0: return launch_requant_t<SIDE, SC, KVQ_Q8_0>(p, grid, smem, num_sms, stream);
    case KVQ_Q4_0: return launch_requant_t<SIDE, SC, KVQ_Q4_0>(p, grid, smem, num_sms, stream);
    default: return launch_requant_t<SIDE, SC, KVQ_TURBO4>(p, grid, smem, num_sms, stream);
  }
}

template <int SIDE>
cudaError_t launch_requant_c(int sc, int dc, const RequantParams &p, dim3 grid, int smem,
                             int num_sms, cudaStream_t stream) {
  switch (sc) {
    case KVQ_F16: return launch_requant_d<SIDE, KVQ_F16>(dc, p, grid, smem, num_sms, stream);
    case KVQ_Q8_0: return launch_requant_d<SIDE, KVQ_Q8_0>(dc, p, grid, smem, num_sms, stream);
    case KVQ_Q4_0: return launch_requant_d<SIDE, KVQ_Q4_0>(dc, p, grid, smem, num_sms, stream);
    default: return launch_requant_d<SIDE, KVQ_TURBO4>(dc, p, grid, smem, num_sms, stream);
  }
}

cudaError_t launch_requant_s(int side, int sc, int dc, const RequantParams &p, dim3 grid,
                             int smem, int num_sms, cudaStream_t stream) {
  return side == 0 ? launch_requant_c<0>(sc, dc, p, grid, smem, num_sms, stream)
                   : launch_requant_c<1>(sc, dc, p, grid, smem, num_sms, stream);
}

}  // namespace

cudaError_t launch_requant(const kvq_layer &L, int side, int dst_codec, void *dst_cache,
                           cudaStream_t stream, int num_sms) {
  RequantParams p;
  p.src = static_cast<const uint8_t *>(side == 0 ? L.k_cache : L.v_cache);
  p.dst = static_cast<uint8_t *>(dst_cache);
  p.seq_lens = L.seq_lens;
  p.err = L.err;
  p.table = L.pages_per_seq > 0 ? L.block_table : nullptr;
  p.pages_per_seq = L.pages_per_seq;
  p.n_pages = L.n_pages;
  p.src_codec = side == 0 ? L.codec_k : L.codec_v;
  p.dst_codec = dst_codec;
  p.n_kv = L.n_kv_heads;
  p.capacity = L.capacity;
  const int units = L.capacity / kUnitTokens;
  p.units_per_stream = units;
  p.n_units = static_cast<int64_t>(units) * L.n_kv_heads * L.n_seqs;
  if (p.n_units >= (int64_t{1} << 31)) return cudaErrorInvalidValue;  // 32-bit unit indices
  const dim3 grid((units + kRqUnits - 1) / kRqUnits, L.n_kv_heads, L.n_seqs);  // turbo4 kernel
  const int smem = kRqUnits * (unit_bytes(p.src_codec) + unit_bytes(dst_codec));
  return launch_requant_s(side, p.src_codec, dst_codec, p, grid, smem, num_sms, stream);
}

cudaError_t launch_append(const kvq_layer &L, const void *k_new, const void *v_new,
                          const int32_t *n_new, int max_new, int update_lens,
                          cudaStream_t stream) {
  AppendParams p;
  p.x[0] = static_cast<const __half *>(k_new);
  p.x[1] = static_cast<const __half *>(v_new);
  p.cache[0] = static_cast<uint8_t *>(L.k_cache);
  p.cache[1] = static_cast<uint8_t *>(L.v_cache);
  p.codec[0] = L.codec_k;
  p.codec[1] = L.codec_v;
  p.seq_lens = L.seq_lens;
  p.n_new = n_new;
  p.err = L.err;
  p.table = L.pages_per_seq > 0 ? L.block_table : nullptr;
  p.n_seqs = L.n_seqs;
  p.n_kv = L.n_kv_heads;
  p.max_new = max_new;
  p.capacity = L.capacity;
  p.pages_per_seq = L.pages_per_seq;
  p.n_pages = L.n_pages;
  const int64_t rows = 2ll * L.n_seqs * max_new * L.n_kv_heads;
  if (rows <= kSmallAppendRows) {
    return launch_pdl(append_small_kernel, dim3(1), dim3(kAppendWarps * 32), 0, stream, p,
                      update_lens);
  }
  const int64_t blocks = (rows + kAppendWarps - 1) / kAppendWarps;
  cudaError_t e = launch_pdl(append_kernel, dim3(static_cast<unsigned>(blocks)),
                             dim3(kAppendWarps * 32), 0, stream, p);
  if (e != cudaSuccess || !update_lens) return e;
  return launch_pdl(update_lens_kernel, dim3((L.n_seqs + 127) / 128), dim3(128), 0, stream,
                    L.seq_lens, n_new, L.n_seqs, L.capacity);
}

}  // namespace kvq
