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
};

constexpr int kRqUnits = 8;  // units per CTA of the re-encode kernel
static_assert(kPageUnits % kRqUnits == 0, "a run of units must lie inside one page");

// One CTA per run of kRqUnits 16-token units of one (sequence, kv head)
// stream.  The source units are copied into shared memory with coalesced
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

template <int SIDE, int SC, int DC>
cudaError_t launch_requant_t(const RequantParams &p, dim3 grid, int smem, cudaStream_t stream) {
  static std::atomic<uint64_t> optin{0};
  const cudaError_t e = smem_optin(requant_kernel<SIDE, SC, DC>, kRqUnits * 2 * 4096, optin);
  if (e != cudaSuccess) return e;
  return launch_pdl(requant_kernel<SIDE, SC, DC>, grid, dim3(kUnitTokens * 32), smem, stream, p);
}

template <int SIDE, int SC>
cudaError_t launch_requant_d(int dc, const RequantParams &p, dim3 grid, int smem,
                             cudaStream_t stream) {
  switch (dc) {
    case KVQ_F16: return launch_requant_t<SIDE, SC, KVQ_F16>(p, grid, smem, stream);
    case KVQ_Q8_0: return launch_requant_t<SIDE, SC, KVQ_Q8_0>(p, grid, smem, stream);
    case KVQ_Q4_0: return launch_requant_t<SIDE, SC, KVQ_Q4_0>(p, grid, smem, stream);
    default: return launch_requant_t<SIDE, SC, KVQ_TURBO4>(p, grid, smem, stream);
  }
}

template <int SIDE>
cudaError_t launch_requant_c(int sc, int dc, const RequantParams &p, dim3 grid, int smem,
                             cudaStream_t stream) {
  switch (sc) {
    case KVQ_F16: return launch_requant_d<SIDE, KVQ_F16>(dc, p, grid, smem, stream);
    case KVQ_Q8_0: return launch_requant_d<SIDE, KVQ_Q8_0>(dc, p, grid, smem, stream);
    case KVQ_Q4_0: return launch_requant_d<SIDE, KVQ_Q4_0>(dc, p, grid, smem, stream);
    default: return launch_requant_d<SIDE, KVQ_TURBO4>(dc, p, grid, smem, stream);
  }
}

cudaError_t launch_requant_s(int side, int sc, int dc, const RequantParams &p, dim3 grid,
                             int smem, cudaStream_t stream) {
  return side == 0 ? launch_requant_c<0>(sc, dc, p, grid, smem, stream)
                   : launch_requant_c<1>(sc, dc, p, grid, smem, stream);
}

}  // namespace

cudaError_t launch_requant(const kvq_layer &L, int side, int dst_codec, void *dst_cache,
                           cudaStream_t stream) {
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
  const dim3 grid((units + kRqUnits - 1) / kRqUnits, L.n_kv_heads, L.n_seqs);
  const int smem = kRqUnits * (unit_bytes(p.src_codec) + unit_bytes(dst_codec));
  return launch_requant_s(side, p.src_codec, dst_codec, p, grid, smem, stream);
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
