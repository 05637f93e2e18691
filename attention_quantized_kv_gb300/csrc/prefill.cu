// prefill.cu -- causal attention of one prefill chunk (ubatch) on the
// 5th-generation tensor cores.
//
// The chunk's queries attend every earlier key of the sequence plus the
// chunk's own keys up to their position (the ubatch prefill described in the
// serverAppConfigs commit log: the prompt is processed in ubatches whose
// buffers are sized by the ubatch alone; the chunk's K/V are quantize-appended
// first, then attended in their quantized form).
//
// Three kernels:
//  1. dequant_tiles: the attended keys of both sides, dequantized (x^ = d * q,
//     rounded once to fp16; f16 is copied), written to the workspace as
//     128-key tiles already in the tensor core's shared-memory operand layout
//     (two 64-dim halves of 128 rows x 128 bytes, 128-byte swizzle), so that
//     the attention kernel moves each tile with one 32 KB bulk async copy.
//     Each key is dequantized once per chunk, not once per query block.
//  2. prefill_attn: persistent CTAs, one per SM.  A work item is (kv head,
//     pair of its query heads, 128-query tile); both heads read the same K/V
//     tiles.  An item is a run of key-tile steps (one per 128-key tile its
//     queries attend), and each CTA takes an equal contiguous slice of all
//     steps in (kv head, pair, query tile) order: whole items plus pieces of
//     at most two more.  A piece writes its rows as partials (unnormalised O,
//     max, sum) and the CTA moves on.  Roles (12 warps): warps 0-3
//     and 4-7 are the softmax warpgroups of the pair's two heads (one query
//     row per thread, TMEM lane quadrant = warp % 4); warp 8 is the
//     producer, streaming K and V tiles into a two-stage ring by bulk async
//     copies on mbarriers; one thread of warp 9 issues tcgen05.mma: S_e =
//     Q_e K^T (M = 128 queries, N = 128 keys, K = 128 dims, fp16 in, fp32
//     accumulate) into head e's TMEM columns, then O_e += P_e V with P_e
//     (fp16) read from TMEM and O_e accumulated in TMEM; warps 10-11 are
//     idle (registers go to a CTA in groups of four warps).  MMAs are issued
//     S0 S1 PV0 S0' PV1 S1' ..., so each head's softmax overlaps the tensor
//     core's work for the other head.  The softmax runs in the log2 domain in
//     two passes over the S row in TMEM (row max with the causal mask, then
//     exp2, row sum and tcgen05.st of P over the S columns).  The running max
//     used for P is only raised (and O, l rescaled) when a row's max grows by
//     more than 2^8, which keeps O rescales rare and the result exact (the
//     same max scales O and l).
//  3. piece_merge: the items split over several CTAs, merged by log-sum-exp
//     once the attention kernel has completed (a CTA per item and head, a
//     thread per query row), so that no CTA waits at its end for the merge.
#include <cuda_runtime.h>

#include <algorithm>

#include <math.h>

#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kBM = 128;                       // query rows per CTA
constexpr int kBN = 128;                       // keys per tile
constexpr int kTileBytes = kBN * kD * 2;       // 32 KB: one side of one tile
constexpr int kHalfBytes = kTileBytes / 2;     // one 64-dim half
constexpr int kStages = 2;
// warps 0-3, 4-7: softmax of heads 0, 1; 8: producer; 9: MMA; 10-11 idle.
// (Registers are allocated to a CTA in groups of four warps, so ten warps
// would cost as much as twelve.)
constexpr int kThreads = 384;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kRescaleThreshold = 8.0f;      // log2 units

// ------------------------------------------------------------------ tcgen05 helpers

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
// Shared-memory matrix descriptor: 128-byte swizzle, given leading/stride
// byte offsets.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor, kind::f16: fp16 A and B, fp32 D, M = 128, N = 128.
__host__ __device__ constexpr uint32_t idesc_f16(int b_mn_major) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (0u << 15) |
         (static_cast<uint32_t>(b_mn_major) << 16) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
}
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

// 32 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
// 16 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st32f(uint32_t taddr, const float (&v)[32]) {
  uint32_t a[16], b[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) { a[i] = __float_as_uint(v[i]); b[i] = __float_as_uint(v[16 + i]); }
  tmem_st16(taddr, a);
  tmem_st16(taddr + 16, b);
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Byte offset of element (row, dim) inside a 128-row tile in the operand
// layout: two 64-dim halves of 128 rows x 128 bytes; inside a half the 16-byte
// chunk index is XOR-ed with (row % 8) (128-byte swizzle).
__host__ __device__ __forceinline__ int tile_offset(int row, int dim) {
  return (dim >> 6) * kHalfBytes + row * 128 + ((((dim & 63) >> 3) ^ (row & 7)) << 4) +
         (dim & 7) * 2;
}

// ------------------------------------------------------------------ dequant pre-pass

// One 32-value block b of token row r of a unit (a shared-memory copy of the
// cache unit), dequantized: x^ = d * q exactly in fp32, per the cache layout.
template <int CODEC, int SIDE>
__device__ __forceinline__ void load_block(const uint8_t *unit, int r, int b, float (&x)[32]) {
  // Loads are as wide as the layout keeps the block's values together: the
  // K side holds 4 consecutive dims of a row in one 32-bit word (q8_0) or 8
  // bytes (f16), the V side 2 consecutive dims in 16 (q8_0) or 32 (f16) bits.
  const int g = r & 7, rh = r >> 3, tig = (r & 7) >> 1, par = r & 1;
  if (CODEC == KVQ_F16) {
    if (SIDE == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {  // dims 4i .. 4i + 3 of the block
        const uint2 w = *reinterpret_cast<const uint2 *>(
            unit + (2 * b + rh) * 512 + (4 * g + (i & 3)) * 16 + (i >> 2) * 8);
        const __half2 h01 = *reinterpret_cast<const __half2 *>(&w.x);
        const __half2 h23 = *reinterpret_cast<const __half2 *>(&w.y);
        x[4 * i] = __low2float(h01); x[4 * i + 1] = __high2float(h01);
        x[4 * i + 2] = __low2float(h23); x[4 * i + 3] = __high2float(h23);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int d = 32 * b + e, mt = d >> 4, gq = (d & 15) >> 1;
        x[e] = __half2float(*reinterpret_cast<const __half *>(
            unit + mt * 512 + (4 * gq + tig) * 16 + (rh * 4 + (d & 1) * 2 + par) * 2));
      }
    }
    return;
  }
  const int soff = CODEC == KVQ_Q8_0
                       ? (SIDE == 0 ? 2048 + g * 16 + rh * 8 + b * 2
                                    : 2048 + tig * 32 + b * 8 + rh * 4 + par * 2)
                       : (SIDE == 0 ? 1024 + g * 16 + rh * 8 + b * 2
                                    : 1024 + tig * 32 + b * 8 + rh * 4 + par * 2);
  const float dsc = __half2float(*reinterpret_cast<const __half *>(unit + soff));
  if (CODEC == KVQ_Q8_0) {
    if (SIDE == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {  // dims 4i .. 4i + 3: one word
        const uint32_t w = *reinterpret_cast<const uint32_t *>(
            unit + b * 512 + (4 * g + (i & 3)) * 16 + (2 * rh + (i >> 2)) * 4);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          x[4 * i + k] = dsc * static_cast<float>(static_cast<int8_t>((w >> (8 * k)) & 0xffu));
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {  // dims 2i, 2i + 1: one 16-bit pair
        const int d = 32 * b + 2 * i, mt = d >> 4, gq = (d & 15) >> 1;
        const uint32_t v = *reinterpret_cast<const uint16_t *>(
            unit + (mt >> 1) * 512 + (4 * gq + tig) * 16 + ((mt & 1) * 2 + rh) * 4 + par * 2);
        x[2 * i] = dsc * static_cast<float>(static_cast<int8_t>(v & 0xffu));
        x[2 * i + 1] = dsc * static_cast<float>(static_cast<int8_t>(v >> 8));
      }
    }
  } else {
    if (SIDE == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // canonical bytes 4i .. 4i + 3: one word
        const uint32_t w = *reinterpret_cast<const uint32_t *>(
            unit + (b >> 1) * 512 + (4 * g + i) * 16 + ((b & 1) * 2 + rh) * 4);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int v = (w >> (8 * k)) & 0xff, jc = 4 * i + k;
          x[jc] = dsc * static_cast<float>((v & 0xf) - 8);
          x[jc + 16] = dsc * static_cast<float>((v >> 4) - 8);
        }
      }
    } else {
#pragma unroll
      for (int jc = 0; jc < 16; ++jc) {  // canonical byte jc: dims jc (low) and jc+16 (high)
        const int mt = 2 * b + (jc >> 3), gq = jc & 7;
        const int v = unit[(mt >> 2) * 512 + (4 * gq + tig) * 16 + (mt & 3) * 4 + par * 2 + rh];
        x[jc] = dsc * static_cast<float>((v & 0xf) - 8);
        x[jc + 16] = dsc * static_cast<float>((v >> 4) - 8);
      }
    }
  }
}

struct DequantParams {
  const uint8_t *cache[2];
  int codec[2];
  uint8_t *tiles[2];   // [n_kv][n_tiles][32 KB]
  const int32_t *seq_lens;
  int32_t *err;
  const int32_t *table;  // paged layers: block table; nullptr: contiguous
  int seq, n_kv, capacity, kv_len, n_tiles, pages_per_seq, n_pages;
  int buf_bytes;         // one shared buffer: a tile's units of the wider side's codec
};

// Persistent CTAs of 256 threads over the work items (side, kv head, tile),
// item w = (side * n_kv + kv head) * n_tiles + tile; CTA c takes w = c,
// c + grid, ...  An item's units (at most eight, inside one page) arrive by
// one bulk copy into one of two shared buffers, the next item's while the
// current one is dequantized: each thread takes (key row, 32-value block)
// items, dequantizes the block there and writes four 16-byte chunks of the
// swizzled fp16 tile.
constexpr int kDqThreads = 256;
constexpr int kDqUnits = kBN / kUnitTokens;  // units per tile

template <int CODEC, int SIDE>
__device__ __forceinline__ void dequant_tile(const DequantParams &p, const uint8_t *units_sh,
                                             int tile, int kvh) {
  constexpr int UB = unit_bytes(CODEC);
  uint8_t *dst = p.tiles[SIDE] + (static_cast<int64_t>(kvh) * p.n_tiles + tile) * kTileBytes;
  if (CODEC == KVQ_TURBO4) {
    // a warp per key row: y^ from the nibbles, then x^ = s * H y^ / 16 across
    // the warp (exact), rounded to fp16 once like every other codec
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll 1
    for (int row = warp; row < kBN; row += kDqThreads / 32) {
      float x[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (tile * kBN + row < p.kv_len) {  // warp-uniform
        turbo4_row_rotated<SIDE>(units_sh + (row / kUnitTokens) * UB, row % kUnitTokens, lane, x);
        turbo_unrotate_lane(x, lane);
      }
      *reinterpret_cast<uint2 *>(dst + tile_offset(row, 4 * lane)) =
          make_uint2(pack_half2(x[0], x[1]), pack_half2(x[2], x[3]));
    }
  } else {
#pragma unroll 1
    for (int item = threadIdx.x; item < kBN * 4; item += kDqThreads) {
      const int row = item >> 2, b = item & 3;
      const int key = tile * kBN + row;
      float x[32];
      if (key < p.kv_len) {
        load_block<CODEC, SIDE>(units_sh + (row / kUnitTokens) * UB, row % kUnitTokens, b, x);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = 0.0f;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 w;
        w.x = pack_half2(x[8 * c + 0], x[8 * c + 1]);
        w.y = pack_half2(x[8 * c + 2], x[8 * c + 3]);
        w.z = pack_half2(x[8 * c + 4], x[8 * c + 5]);
        w.w = pack_half2(x[8 * c + 6], x[8 * c + 7]);
        *reinterpret_cast<uint4 *>(dst + tile_offset(row, 32 * b + 8 * c)) = w;
      }
    }
  }
}

template <int SIDE>
__device__ __forceinline__ void dequant_tile_c(const DequantParams &p, const uint8_t *units_sh,
                                               int tile, int kvh) {
  const int codec = p.codec[SIDE];
  if (codec == KVQ_F16) dequant_tile<KVQ_F16, SIDE>(p, units_sh, tile, kvh);
  else if (codec == KVQ_Q8_0) dequant_tile<KVQ_Q8_0, SIDE>(p, units_sh, tile, kvh);
  else if (codec == KVQ_Q4_0) dequant_tile<KVQ_Q4_0, SIDE>(p, units_sh, tile, kvh);
  else dequant_tile<KVQ_TURBO4, SIDE>(p, units_sh, tile, kvh);
}

__global__ void __launch_bounds__(kDqThreads, 4) dequant_tiles_kernel(const DequantParams p) {
  extern __shared__ __align__(128) uint8_t dq_sh[];  // two buffers of p.buf_bytes
  __shared__ uint64_t full[2];
  if (threadIdx.x == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependency_wait();
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.seq_lens[p.seq] < p.kv_len)
    set_err(p.err, KVQ_DEVERR_SEQLEN);
  const int n_work = 2 * p.n_kv * p.n_tiles;
  const int64_t units = p.capacity / kUnitTokens;
  const int units_kv = (p.kv_len + kUnitTokens - 1) / kUnitTokens;
  // thread 0: bulk-copy item w's units into buffer `buf`
  auto issue = [&](int w, int buf) {
    const int side = w / (p.n_kv * p.n_tiles);
    const int kvh = (w / p.n_tiles) % p.n_kv, tile = w % p.n_tiles;
    const int ub = unit_bytes(side ? p.codec[1] : p.codec[0]);
    const int u_first = tile * kDqUnits;
    const int n_u = min(kDqUnits, units_kv - u_first);
    int64_t uidx;
    if (p.table) {  // a tile lies inside one page (kPageUnits % kDqUnits == 0)
      int pg = page_of(p.table, p.pages_per_seq, p.n_pages, p.seq, u_first / kPageUnits);
      if (pg < 0) {
        set_err(p.err, KVQ_DEVERR_PAGE);
        pg = 0;  // read pool page 0 in its place
      }
      uidx = (static_cast<int64_t>(pg) * p.n_kv + kvh) * kPageUnits + u_first % kPageUnits;
    } else {
      uidx = (static_cast<int64_t>(p.seq) * p.n_kv + kvh) * units + u_first;
    }
    const uint32_t bytes = n_u > 0 ? static_cast<uint32_t>(n_u * ub) : 0u;
    mbar_arrive_expect_tx(&full[buf], bytes);
    const uint8_t *src = (side ? p.cache[1] : p.cache[0]) + uidx * ub;
    if (bytes) bulk_copy_g2s(dq_sh + buf * p.buf_bytes, src, bytes, &full[buf]);
  };
  int issued = 0;  // thread 0: items issued (the k-th into buffer k & 1)
  if (threadIdx.x == 0 && static_cast<int>(blockIdx.x) < n_work) {
    issue(blockIdx.x, 0);
    issued = 1;
  }
  int i = 0;
  bool ok = true;
  for (int w = blockIdx.x; w < n_work; w += gridDim.x, ++i) {
    const int buf = i & 1;
    // the other buffer was last read in item i - 1 (the barrier below ended it)
    if (threadIdx.x == 0 && w + static_cast<int>(gridDim.x) < n_work) {
      fence_proxy_async_smem();
      issue(w + gridDim.x, buf ^ 1);
      ++issued;
    }
    const bool got = __syncthreads_and(
        mbar_wait_bounded(&full[buf], static_cast<uint32_t>(i >> 1) & 1u) ? 1 : 0);
    if (!got) {
      if (threadIdx.x == 0) set_err(p.err, KVQ_DEVERR_TIMEOUT);
      ok = false;
      break;
    }
    const int side = w / (p.n_kv * p.n_tiles);
    const int kvh = (w / p.n_tiles) % p.n_kv, tile = w % p.n_tiles;
    const uint8_t *units_sh = dq_sh + buf * p.buf_bytes;
    if (side == 0) dequant_tile_c<0>(p, units_sh, tile, kvh);
    else dequant_tile_c<1>(p, units_sh, tile, kvh);
    __syncthreads();  // every thread is done with this buffer
  }
  if (!ok && threadIdx.x == 0) {  // after a timeout: the copies still in flight
    for (int k = i; k < issued; ++k)
      mbar_wait_bounded(&full[k & 1], static_cast<uint32_t>(k >> 1) & 1u, nullptr, 100000000ull);
  }
  grid_launch_dependents();
}

// ------------------------------------------------------------------ attention

struct AttnParams {
  const uint8_t *ktiles;  // [n_kv][n_tiles][32 KB]
  const uint8_t *vtiles;
  const __half *q;        // [n_tok][n_q][128]
  __half *out;
  float *lse;
  int32_t *err;
  float *part;            // partial slots [slot][2][128][kPartStride]: O (unnormalised), m, l
  int n_q, G, n_tok, q_start, kv_len, n_tiles;
  int npairs, n_qt, n_items;
  int64_t Tq;             // key-tile steps of one (kv head, head pair) group: sum over q tiles
  int64_t W;              // all key-tile steps: groups * Tq
  float scale_log2;
};

constexpr int kPartStride = 132;  // floats per partial row: 128 O, m, l, 2 pad (16-byte rows)

struct __align__(8) AttnBars {
  uint64_t kfull[kStages], vfull[kStages], kempty[kStages], vempty[kStages];
  uint64_t sfull[2], pfull[2], odone[2], segdone[2], qready[2], ofree[2], drain;
};

// Key tiles attended by query tile qt (128 rows; the last may be short).
__device__ __forceinline__ int qt_tiles_of(int q_start, int n_tok, int qt) {
  const int rows_end = min(kBM * (qt + 1), n_tok);
  return (q_start + rows_end + kBN - 1) / kBN;
}
__device__ __forceinline__ int qt_tiles(const AttnParams &p, int qt) {
  return qt_tiles_of(p.q_start, p.n_tok, qt);
}

// The work is the list of items (group g = kv head * npairs + head pair,
// query tile qt), item index g * n_qt + qt, each item a run of qt_tiles(qt)
// key-tile steps.  CTA c takes the steps [W c / P, W (c + 1) / P): whole
// items, plus pieces of the first and last ones.  A segment is one item's
// piece [j_lo, j_hi) of steps.
//
// Step j of an item reads key tile (j + rot) % nt rather than tile j.  The
// item's rotation puts its tiles in step with every CTA's own clock: the
// owner of the item's last step starts the item (or its piece of it) at the
// point of its slice where it reads tile 0 + (its slice position) mod nt, so
// that at any moment the CTAs working on one kv head read about the same
// tile.  The ~19 CTAs of a kv head then share each tile through L2 instead of
// each reading the whole kv head from HBM at its own pace.  (Softmax over
// the tiles in any order gives the same result up to rounding; the causal
// mask follows the tile, not the step.)
struct Segment {
  int g, qt, j_lo, j_hi, nt;  // nt: the item's key tiles
  int rot;                    // step j reads key tile (j + rot) % nt
  int64_t start;              // the item's first step
};
struct SegIter {
  int64_t s, s1;
  int g, qt;
  int64_t item_start;  // first step of item (g, qt)
  __device__ __forceinline__ void init(const AttnParams &p, int64_t s0, int64_t s_end) {
    s = s0;
    s1 = s_end;
    g = static_cast<int>(s0 / p.Tq);
    int64_t base = static_cast<int64_t>(g) * p.Tq;
    qt = 0;
    while (qt + 1 < p.n_qt && base + qt_tiles(p, qt) <= s0) {
      base += qt_tiles(p, qt);
      ++qt;
    }
    item_start = base;
  }
  __device__ __forceinline__ bool next(const AttnParams &p, Segment &seg) {
    if (s >= s1) return false;
    const int nt = qt_tiles(p, qt);
    seg.g = g;
    seg.qt = qt;
    seg.nt = nt;
    seg.start = item_start;
    {
      // the owner of the item's last step and the first step of its slice
      const int64_t P = gridDim.x;
      const int64_t last = item_start + nt - 1;
      const int64_t c_last = ((last + 1) * P - 1) / p.W;
      const int64_t slice0 = p.W * c_last / P;
      const int64_t r = (item_start - slice0) % nt;
      seg.rot = static_cast<int>(r < 0 ? r + nt : r);
    }
    seg.j_lo = static_cast<int>(s - item_start);
    const int64_t end = min(s1, item_start + nt);
    seg.j_hi = static_cast<int>(end - item_start);
    s = end;
    if (end == item_start + nt) {  // on to the next item
      item_start += nt;
      if (++qt == p.n_qt) {
        qt = 0;
        ++g;
      }
    }
    return true;
  }
};

// Persistent CTAs (one per SM) over a balanced split of the key-tile steps of
// all (128-query block, pair of query heads of one kv head) items: both
// heads read the same K and V tiles.  Head e of the pair has its own Q tile,
// S buffer (TMEM columns 128e..), O accumulator (256 + 128e..) and softmax
// warpgroup (head 0: warps 0-3, head 1: warps 4-7; a warp's TMEM lane
// quadrant is warp % 4).  The MMA thread issues, per key tile j,
//   S0(j)  S1(j)  PV0(j)  S0(j+1)  PV1(j)  S1(j+1)  PV0(j+1) ...
// so that each warpgroup's softmax of tile j overlaps the tensor core's work
// for the other head.  An S buffer is rewritten only after the PV that read
// its P, in issue order (tcgen05.mma from one thread executes in order).
// A segment that covers a whole item writes its rows; the pieces of a split
// item are written as partials (unnormalised O, m, l) for piece_merge_kernel.
__global__ void __launch_bounds__(kThreads, 1) prefill_attn_kernel(const AttnParams p) {
  const int64_t P = gridDim.x;
  const int64_t s0 = p.W * blockIdx.x / P, s1 = p.W * (blockIdx.x + 1) / P;
  if (s0 >= s1) return;  // whole CTA: no work (the grid is at most W, so never)

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned operand area: Q0, Q1 (32 KB each), K stages, V stages.
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sq = smem;
  uint8_t *sk = smem + 2 * kTileBytes;
  uint8_t *sv = sk + kStages * kTileBytes;
  __shared__ AttnBars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t idesc_qk = idesc_f16(0), idesc_pv = idesc_f16(1);
  // softmax warpgroup of this warp (-1: producer, MMA or idle warp)
  const int e = warp < 8 ? (warp >> 2) : -1;
  auto seg_two = [&](const Segment &sg) { return 2 * (sg.g % p.npairs) + 1 < p.G; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.kfull[s], 1);
      mbar_init(&bars.vfull[s], 1);
      mbar_init(&bars.kempty[s], 1);
      mbar_init(&bars.vempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.sfull[b], 1);
      mbar_init(&bars.pfull[b], 4);  // one arrival per softmax warp
      mbar_init(&bars.odone[b], 1);
      mbar_init(&bars.segdone[b], 1);
      mbar_init(&bars.qready[b], 4);  // the segment's Q written, one arrival per warp
      mbar_init(&bars.ofree[b], 4);   // the segment's O read, one arrival per warp
    }
    mbar_init(&bars.drain, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&tmem_base_sh, 512);

  grid_dependency_wait();  // the dequantized tiles come from the previous kernel

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t tm_s[2] = {tmem, tmem + 128};
  const uint32_t tm_o[2] = {tmem + 256, tmem + 384};

  if (warp == kProducerWarp) {
    // ---------------- producer: K and V tiles into the two-stage ring
    if (lane == 0) {
      SegIter it;
      it.init(p, s0, s1);
      Segment sg;
      int t = 0;  // tiles issued by this CTA
      bool ok = true;
      while (ok && it.next(p, sg)) {
        const int kvh = sg.g / p.npairs;
        const uint8_t *kt = p.ktiles + static_cast<int64_t>(kvh) * p.n_tiles * kTileBytes;
        const uint8_t *vt = p.vtiles + static_cast<int64_t>(kvh) * p.n_tiles * kTileBytes;
        for (int j = sg.j_lo; j < sg.j_hi; ++j, ++t) {
          const int s = t % kStages;
          const int64_t tile = (j + sg.rot) % sg.nt;
          const uint32_t ph = static_cast<uint32_t>(t / kStages - 1) & 1u;
          if (t >= kStages && !mbar_wait_bounded(&bars.kempty[s], ph, &abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&bars.kfull[s], kTileBytes);
          bulk_copy_g2s(sk + s * kTileBytes, kt + tile * kTileBytes, kTileBytes, &bars.kfull[s]);
          if (t >= kStages && !mbar_wait_bounded(&bars.vempty[s], ph, &abort_flag)) {
            // the V copy of this tile was not started: drain below counts t + 1 K copies
            mbar_wait_bounded(&bars.kfull[s], static_cast<uint32_t>(t / kStages) & 1u, nullptr,
                              100000000ull);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars.vfull[s], kTileBytes);
          bulk_copy_g2s(sv + s * kTileBytes, vt + tile * kTileBytes, kTileBytes, &bars.vfull[s]);
        }
      }
      // After an abort, wait (bounded) for the copies still landing in the ring.
      if (!ok || *reinterpret_cast<volatile int *>(&abort_flag)) {
        for (int u = max(0, t - kStages); u < t; ++u) {
          mbar_wait_bounded(&bars.kfull[u % kStages], static_cast<uint32_t>(u / kStages) & 1u,
                            nullptr, 100000000ull);
          mbar_wait_bounded(&bars.vfull[u % kStages], static_cast<uint32_t>(u / kStages) & 1u,
                            nullptr, 100000000ull);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer (one thread)
    if (lane == 0) {
      const uint32_t q_addr[2] = {smem_u32(sq), smem_u32(sq + kTileBytes)};
      // S_e = Q_e K^T of ring tile t into TMEM buffer e
      auto qk = [&](int eh, int t) {
        const uint32_t k_addr = smem_u32(sk + (t % kStages) * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          mma_ss(tm_s[eh], smem_desc(q_addr[eh] + off, 16, 1024), smem_desc(k_addr + off, 16, 1024),
                 idesc_qk, kk > 0);
        }
        mma_commit(&bars.sfull[eh]);
      };
      // O_e (+)= P_e V of ring tile t: keys 16kk..16kk+15 are P columns 8kk..
      // (fp16 pairs) and V rows 16kk.. (two 8-row groups)
      auto pv = [&](int eh, int t, bool first) {
        const uint32_t v_addr = smem_u32(sv + (t % kStages) * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tm_o[eh], tm_s[eh] + kk * 8, smem_desc(v_addr + kk * 2048, kHalfBytes, 1024),
                 idesc_pv, (!first || kk > 0) ? 1u : 0u);
        mma_commit(&bars.odone[eh]);
      };
      SegIter it;
      it.init(p, s0, s1);
      Segment sg;
      int t = 0;            // ring tile index
      int u[2] = {0, 0};    // tiles per head (sfull / pfull / odone phases)
      int k[2] = {0, 0};    // segments per head (ready / segdone phases)
      bool ok = true;
      while (ok && it.next(p, sg)) {
        const bool two = seg_two(sg);
        const int n = sg.j_hi - sg.j_lo;
        // Q of this segment written (its S can start while the previous
        // segment's O is still being read; the first PV waits for that)
        ok = mbar_wait_bounded(&bars.qready[0], static_cast<uint32_t>(k[0]) & 1u, &abort_flag) &&
             (!two || mbar_wait_bounded(&bars.qready[1], static_cast<uint32_t>(k[1]) & 1u, &abort_flag)) &&
             mbar_wait_bounded(&bars.kfull[t % kStages], static_cast<uint32_t>(t / kStages) & 1u,
                               &abort_flag);
        if (!ok) break;
        tc_fence_after();
        qk(0, t);
        if (two) qk(1, t);
        mma_commit(&bars.kempty[t % kStages]);
        for (int jj = 0; jj < n && ok; ++jj, ++t) {
          const int s = t % kStages;
          const bool more = jj + 1 < n;
          ok = mbar_wait_bounded(&bars.pfull[0], static_cast<uint32_t>(u[0]) & 1u, &abort_flag) &&
               mbar_wait_bounded(&bars.vfull[s], static_cast<uint32_t>(t / kStages) & 1u, &abort_flag) &&
               (jj > 0 || k[0] == 0 ||
                mbar_wait_bounded(&bars.ofree[0], static_cast<uint32_t>(k[0] - 1) & 1u, &abort_flag));
          if (!ok) break;
          tc_fence_after();
          pv(0, t, jj == 0);
          ++u[0];
          if (!two) mma_commit(&bars.vempty[s]);
          if (more) {
            ok = mbar_wait_bounded(&bars.kfull[(t + 1) % kStages],
                                   static_cast<uint32_t>((t + 1) / kStages) & 1u, &abort_flag);
            if (!ok) break;
            tc_fence_after();
            qk(0, t + 1);
            if (!two) mma_commit(&bars.kempty[(t + 1) % kStages]);
          }
          if (two) {
            ok = mbar_wait_bounded(&bars.pfull[1], static_cast<uint32_t>(u[1]) & 1u, &abort_flag) &&
                 (jj > 0 || k[1] == 0 ||
                  mbar_wait_bounded(&bars.ofree[1], static_cast<uint32_t>(k[1] - 1) & 1u, &abort_flag));
            if (!ok) break;
            tc_fence_after();
            pv(1, t, jj == 0);
            ++u[1];
            mma_commit(&bars.vempty[s]);
            if (more) {
              qk(1, t + 1);
              mma_commit(&bars.kempty[(t + 1) % kStages]);
            }
          }
        }
        if (!ok) break;
        // the segment's O is complete once every MMA issued so far is
        mma_commit(&bars.segdone[0]);
        ++k[0];
        if (two) {
          mma_commit(&bars.segdone[1]);
          ++k[1];
        }
      }
      if (!ok) {
        set_err(p.err, KVQ_DEVERR_TIMEOUT);
        atomicExch(&abort_flag, 1);
      }
      // drain: completes when every MMA this thread issued has finished
      // (TMEM is freed after it).
      mma_commit(&bars.drain);
      mbar_wait_bounded(&bars.drain, 0, nullptr, 100000000ull);
    }
  } else if (e >= 0) {
    // ---------------- softmax warpgroup of head e: thread = query row
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tms = tm_s[e], tmo = tm_o[e];
    uint8_t *dstq = sq + e * kTileBytes;
    SegIter it;
    it.init(p, s0, s1);
    Segment sg;
    int u = 0, kseg = 0;  // tiles and segments of this head
    bool ok = true;
    // Q rows of this head of segment `q` into its operand tile, then tell the
    // MMA thread.
    auto load_q = [&](const Segment &q) {
      const int hq = (q.g / p.npairs) * p.G + 2 * (q.g % p.npairs) + e;
      const int qq0 = q.qt * kBM;
      const bool have = r < min(kBM, p.n_tok - qq0);
      const uint4 *src = reinterpret_cast<const uint4 *>(
          p.q + (static_cast<int64_t>(qq0 + (have ? r : 0)) * p.n_q + hq) * kD);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint4 v = have ? src[c] : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4 *>(dstq + tile_offset(r, c * 8)) = v;
      }
      fence_proxy_async_smem();  // generic-proxy writes, read by the tensor core
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.qready[e]);
    };
    // the next segment this head takes part in (e == 1 skips single heads)
    auto next_mine = [&](SegIter &i2, Segment &q) {
      while (i2.next(p, q))
        if (e == 0 || seg_two(q)) return true;
      return false;
    };
    bool have_seg = next_mine(it, sg);
    if (have_seg) load_q(sg);
    while (have_seg) {
      const int kvh = sg.g / p.npairs, hp = sg.g % p.npairs;
      const int head = kvh * p.G + 2 * hp + e;
      const int q0 = sg.qt * kBM;
      const int rows = min(kBM, p.n_tok - q0);
      const int pos = p.q_start + q0 + r;  // absolute position of this query
      float m = -INFINITY, l = 0.0f;
      // After an abort (ok false) the segment loop still runs to the end with
      // no waits, so that both warpgroups pass the same named barriers.
      for (int j = sg.j_lo; j < sg.j_hi && ok; ++j, ++u) {
        ok = mbar_wait_bounded(&bars.sfull[e], static_cast<uint32_t>(u) & 1u, &abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0) atomicExch(&abort_flag, 1);
          break;
        }
        tc_fence_after();
        const int kbase = ((j + sg.rot) % sg.nt) * kBN;
        // Tiles crossing some row's position (warp-uniform test): the scores of
        // keys past the row's position are overwritten with -inf in TMEM, so
        // that pass 2 needs no mask.
        const bool diag = __any_sync(0xffffffffu, kbase + kBN - 1 > pos);
        // Pass 1: row max of the raw scores (scale > 0 keeps the order), read
        // from TMEM 64 columns at a time, 8 independent partial maxima of
        // three-input max instructions.  The row is read again for P (pass 2),
        // which keeps it out of registers.
        float mp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mp[i] = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; c += 2) {
          float v0[32], v1[32];
          tmem_ld32(tms + lane_off + c * 32, v0);
          tmem_ld32(tms + lane_off + (c + 1) * 32, v1);
          tmem_wait_ld();
          if (diag) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if (kbase + c * 32 + i > pos) v0[i] = -INFINITY;
              if (kbase + (c + 1) * 32 + i > pos) v1[i] = -INFINITY;
            }
            tmem_st32f(tms + lane_off + c * 32, v0);
            tmem_st32f(tms + lane_off + (c + 1) * 32, v1);
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) mp[i & 7] = fmax3(mp[i & 7], v0[i], v1[i]);
        }
        if (diag) tmem_wait_st();
        const float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                               fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7]))) * p.scale_log2;
        // Raise a row's running max only when it grew by more than the
        // threshold.  tcgen05.ld/st are warp-collective, so the O rescale runs
        // for the whole warp when any of its rows needs it (factor 1 elsewhere).
        const bool raise = mx > m + kRescaleThreshold || m == -INFINITY;
        const float mnew = raise ? fmaxf(mx, m) : m;
        const float a = (raise && m != -INFINITY) ? fast_exp2(m - mnew) : 1.0f;
        if (__any_sync(0xffffffffu, raise && m != -INFINITY)) {
          // O holds the sum of P V over this segment's earlier tiles: wait for
          // the last PV (tile u - 1 of this head), rescale in TMEM
          bool got = mbar_wait_bounded(&bars.odone[e], static_cast<uint32_t>(u - 1) & 1u, &abort_flag);
          got = __all_sync(0xffffffffu, got);
          if (!got) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float v[32];
            tmem_ld32(tmo + lane_off + c * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= a;
            tmem_st32f(tmo + lane_off + c * 32, v);
          }
          tmem_wait_st();
        }
        l *= a;
        m = mnew;
        // Pass 2: P = exp2(s * scale_log2 - m) as fp16 pairs over the first 64
        // columns of the S buffer (P chunk c lands on columns already read);
        // scale-and-offset and the row sum (4 partial pairs) in f32x2 ops.
        float2 sp2[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                         make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
        // A piece of an item past some rows' positions leaves those rows with
        // every key masked (m = -inf): their P is 0, not exp2(-inf + inf).
        const float nm = m == -INFINITY ? 0.0f : -m;
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nm2 = make_float2(nm, nm);
#pragma unroll
        for (int c = 0; c < 4; c += 2) {
          float v0[32], v1[32];
          tmem_ld32(tms + lane_off + c * 32, v0);
          tmem_ld32(tms + lane_off + (c + 1) * 32, v1);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float *v = h ? v1 : v0;
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 tt = fma2(make_float2(v[2 * i], v[2 * i + 1]), sc2, nm2);
              const float2 x = make_float2(fast_exp2(tt.x), fast_exp2(tt.y));
              sp2[i & 3] = add2(sp2[i & 3], x);
              pk[i] = pack_half2(x.x, x.y);
            }
            tmem_st16(tms + lane_off + (c + h) * 16, pk);
          }
        }
        const float2 s01 = add2(sp2[0], sp2[1]), s23 = add2(sp2[2], sp2[3]);
        const float2 s4 = add2(s01, s23);
        l += s4.x + s4.y;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.pfull[e]);
      }
      // The next segment's Q can go in now: this segment's last S has been
      // read, so its QK MMAs are done with the Q tile.
      Segment nsg;
      const bool have_next = next_mine(it, nsg);
      if (have_next) load_q(nsg);
      // the segment's O: wait for its last MMA
      if (ok) ok = mbar_wait_bounded(&bars.segdone[e], static_cast<uint32_t>(kseg) & 1u, &abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      ++kseg;
      tc_fence_after();
      const bool whole = sg.j_lo == 0 && sg.j_hi == sg.nt;
      const int64_t item = static_cast<int64_t>(sg.g) * p.n_qt + sg.qt;
      const int64_t row = static_cast<int64_t>(q0 + r) * p.n_q + head;
      float *prow = p.part +
                    ((static_cast<int64_t>(blockIdx.x) + item) * 2 * kBM + e * kBM + r) * kPartStride;
      if (whole) {
        const float inv = l > 0.0f ? 1.0f / l : 0.0f;
        __half *dst = p.out + row * kD;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float v[32];
          tmem_ld32(tmo + lane_off + c * 32, v);
          tmem_wait_ld();
          if (r < rows) {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = pack_half2(v[2 * i] * inv, v[2 * i + 1] * inv);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              reinterpret_cast<uint4 *>(dst + c * 32)[i] =
                  make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
        }
        tc_fence_before();  // O read: the next segment's first PV may overwrite it
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.ofree[e]);
        if (p.lse && r < rows)
          p.lse[row] = l > 0.0f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
        sg = nsg;
        have_seg = have_next;
        continue;
      }
      // A piece of a split item: write the partial row (O as accumulated, in
      // the scale of m; m in log2 units; l) into slot blockIdx.x + item; the
      // merge kernel behind this one combines the item's pieces.
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(tmo + lane_off + c * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i)
          reinterpret_cast<float4 *>(prow + c * 32)[i] =
              make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
      tc_fence_before();  // O read: the next segment's first PV may overwrite it
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.ofree[e]);
      reinterpret_cast<float2 *>(prow + kD)[0] = make_float2(m, l);
      sg = nsg;
      have_seg = have_next;
    }
    if (!ok) {
      if (lane == 0) {
        set_err(p.err, KVQ_DEVERR_TIMEOUT);
        atomicExch(&abort_flag, 1);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ piece merge

struct PieceMergeParams {
  const float *part;  // the attention kernel's partial slots
  __half *out;
  float *lse;
  int n_q, G, n_tok, q_start, npairs, n_qt;
  int64_t Tq, W;
  int grid;           // the attention kernel's CTAs
};

// The items that the attention kernel split over several CTAs, merged by
// log-sum-exp after it has completed: o = sum_c 2^(m_c - M) o_c / L with
// M = max_c m_c and L = sum_c 2^(m_c - M) l_c over the item's pieces
// c = c_first..c_last (the CTAs owning its first and last step), summed in
// that order.  Grid (item, head of its pair, quarter of the 128 rows); a
// thread per (query row, 8 dims), so that many small threads keep the reads
// of the partial rows in flight: each requests the (m, l) of up to four
// pieces at once, then its 8 dims of two pieces at a time.  Items that one
// CTA took whole were written by the attention kernel; their CTAs return.
constexpr int kMergeRowsPerCta = 32;
constexpr int kMergeThreads = kMergeRowsPerCta * (kD / 8);

__global__ void __launch_bounds__(kMergeThreads) piece_merge_kernel(const PieceMergeParams p) {
  __shared__ int64_t owners[2];
  grid_dependency_wait();  // the partials are complete
  const int item = blockIdx.x, e = blockIdx.y;
  const int g = item / p.n_qt, qt = item % p.n_qt;
  if (e == 1 && 2 * (g % p.npairs) + 1 >= p.G) return;  // a pair with one head
  if (threadIdx.x == 0) {  // the owners of the item's first and last step, once per CTA
    int64_t start = static_cast<int64_t>(g) * p.Tq;
    for (int q = 0; q < qt; ++q) start += qt_tiles_of(p.q_start, p.n_tok, q);
    const int nt = qt_tiles_of(p.q_start, p.n_tok, qt);
    const int64_t P = p.grid;
    owners[0] = ((start + 1) * P - 1) / p.W;  // owner of step s: ((s + 1) P - 1) / W
    owners[1] = ((start + nt) * P - 1) / p.W;
  }
  __syncthreads();
  const int64_t c_first = owners[0], c_last = owners[1];
  if (c_first == c_last) return;
  const int r = blockIdx.z * kMergeRowsPerCta + (threadIdx.x >> 4), cc = threadIdx.x & 15;
  const int q0 = qt * kBM;
  if (r >= min(kBM, p.n_tok - q0)) return;
  const int head = (g / p.npairs) * p.G + 2 * (g % p.npairs) + e;
  const int64_t row = static_cast<int64_t>(q0 + r) * p.n_q + head;
  auto part_row = [&](int64_t c) {
    return p.part + ((c + item) * 2 * kBM + e * kBM + r) * kPartStride;
  };
  auto ml_of = [&](int64_t c) {
    return c <= c_last ? __ldcg(reinterpret_cast<const float2 *>(part_row(c) + kD))
                       : make_float2(-INFINITY, 0.0f);
  };
  // (m, l) of the first four pieces in one round trip (an item rarely has
  // more), the rest four at a time
  float2 ml[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) ml[i] = ml_of(c_first + i);
  float M = fmaxf(fmaxf(ml[0].x, ml[1].x), fmaxf(ml[2].x, ml[3].x));
  for (int64_t c0 = c_first + 4; c0 <= c_last; c0 += 4) {
#pragma unroll
    for (int i = 0; i < 4; ++i) M = fmaxf(M, ml_of(c0 + i).x);
  }
  float L = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (ml[i].x != -INFINITY) L = fmaf(fast_exp2(ml[i].x - M), ml[i].y, L);
  for (int64_t c0 = c_first + 4; c0 <= c_last; c0 += 4) {
    float2 mr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) mr[i] = ml_of(c0 + i);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (mr[i].x != -INFINITY) L = fmaf(fast_exp2(mr[i].x - M), mr[i].y, L);
  }
  float4 acc[2] = {make_float4(0.0f, 0.0f, 0.0f, 0.0f), make_float4(0.0f, 0.0f, 0.0f, 0.0f)};
  for (int64_t c0 = c_first; c0 <= c_last; c0 += 2) {
    float4 x[2][2];
    float w[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const bool have = c0 + k <= c_last;
      const float *pr = part_row(have ? c0 + k : c0);
      const int64_t j = c0 + k - c_first;  // ml[] holds pieces 0..3 (selected, not indexed)
      const float mk = !have ? -INFINITY
                       : j == 0 ? ml[0].x : j == 1 ? ml[1].x : j == 2 ? ml[2].x
                       : j == 3 ? ml[3].x : __ldcg(pr + kD);
      w[k] = mk == -INFINITY ? 0.0f : fast_exp2(mk - M);
      x[k][0] = have ? __ldcg(reinterpret_cast<const float4 *>(pr + cc * 8)) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      x[k][1] = have ? __ldcg(reinterpret_cast<const float4 *>(pr + cc * 8) + 1) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (c0 + k > c_last) break;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        acc[i].x = fmaf(w[k], x[k][i].x, acc[i].x);
        acc[i].y = fmaf(w[k], x[k][i].y, acc[i].y);
        acc[i].z = fmaf(w[k], x[k][i].z, acc[i].z);
        acc[i].w = fmaf(w[k], x[k][i].w, acc[i].w);
      }
    }
  }
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  *reinterpret_cast<uint4 *>(p.out + row * kD + cc * 8) =
      make_uint4(pack_half2(acc[0].x * inv, acc[0].y * inv), pack_half2(acc[0].z * inv, acc[0].w * inv),
                 pack_half2(acc[1].x * inv, acc[1].y * inv), pack_half2(acc[1].z * inv, acc[1].w * inv));
  if (p.lse && cc == 0) p.lse[row] = L > 0.0f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
  grid_launch_dependents();
}

}  // namespace

// Key tiles attended by query tile qt of a chunk (host copy of qt_tiles).
static int64_t host_qt_tiles(int q_start, int n_q_tok, int qt) {
  const int64_t rows_end = std::min<int64_t>(static_cast<int64_t>(kBM) * (qt + 1), n_q_tok);
  return (q_start + rows_end + kBN - 1) / kBN;
}

PrefillPlan plan_prefill(const kvq_layer &L, int q_start, int n_q_tok, int num_sms) {
  PrefillPlan pl;
  pl.kv_tokens = static_cast<int64_t>(q_start) + n_q_tok;
  const int64_t n_tiles = (pl.kv_tokens + kBN - 1) / kBN;
  pl.kv_tokens_pad = n_tiles * kBN;
  pl.ws_k_bytes = static_cast<int64_t>(L.n_kv_heads) * n_tiles * kTileBytes;
  const int G = L.n_q_heads / L.n_kv_heads;
  pl.npairs = (G + 1) / 2;
  pl.n_qt = (n_q_tok + kBM - 1) / kBM;
  pl.n_items = static_cast<int64_t>(L.n_kv_heads) * pl.npairs * pl.n_qt;
  pl.Tq = 0;
  for (int qt = 0; qt < pl.n_qt; ++qt) pl.Tq += host_qt_tiles(q_start, n_q_tok, qt);
  pl.W = static_cast<int64_t>(L.n_kv_heads) * pl.npairs * pl.Tq;
  pl.sms = num_sms > 0 ? num_sms : 148;
  pl.grid = std::max<int64_t>(1, std::min<int64_t>(pl.sms, pl.W));
  // the partial slots after the K and V tiles
  pl.part_off = 2 * pl.ws_k_bytes;
  pl.part_bytes = (pl.grid + pl.n_items) * 2 * kBM * kPartStride * 4;
  pl.ws_bytes = pl.part_off + pl.part_bytes;
  return pl;
}

cudaError_t launch_prefill(const kvq_layer &L, const PrefillPlan &pl, int seq, int q_start,
                           int n_q_tok, const void *q, float scale, void *out, float *lse,
                           void *workspace, cudaStream_t stream) {
  const int n_tiles = static_cast<int>(pl.kv_tokens_pad / kBN);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  DequantParams dp;
  dp.cache[0] = static_cast<const uint8_t *>(L.k_cache);
  dp.cache[1] = static_cast<const uint8_t *>(L.v_cache);
  dp.codec[0] = L.codec_k;
  dp.codec[1] = L.codec_v;
  dp.tiles[0] = ws;
  dp.tiles[1] = ws + pl.ws_k_bytes;
  dp.seq_lens = L.seq_lens;
  dp.err = L.err;
  dp.table = L.pages_per_seq > 0 ? L.block_table : nullptr;
  dp.pages_per_seq = L.pages_per_seq;
  dp.n_pages = L.n_pages;
  dp.seq = seq;
  dp.n_kv = L.n_kv_heads;
  dp.capacity = L.capacity;
  dp.kv_len = static_cast<int>(pl.kv_tokens);
  dp.n_tiles = n_tiles;
  dp.buf_bytes = kBN / kUnitTokens * std::max(unit_bytes(L.codec_k), unit_bytes(L.codec_v));
  const int dq_smem = 2 * dp.buf_bytes;
  // opted in once per device for the widest codec (f16 units), whatever this
  // layer's codecs are
  static std::atomic<uint64_t> dq_optin{0};
  cudaError_t e = smem_optin(dequant_tiles_kernel, 2 * kDqUnits * unit_bytes(KVQ_F16), dq_optin);
  if (e != cudaSuccess) return e;
  int dq_per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&dq_per_sm, dequant_tiles_kernel, kDqThreads,
                                                    dq_smem);
  if (e != cudaSuccess) return e;
  const int64_t dq_work = 2 * static_cast<int64_t>(L.n_kv_heads) * n_tiles;
  const int64_t dq_grid =
      std::max<int64_t>(1, std::min<int64_t>(dq_work, static_cast<int64_t>(std::max(dq_per_sm, 1)) * pl.sms));
  e = launch_pdl(dequant_tiles_kernel, dim3(static_cast<unsigned>(dq_grid)), dim3(kDqThreads),
                 dq_smem, stream, dp);
  if (e != cudaSuccess) return e;

  AttnParams ap;
  ap.ktiles = ws;
  ap.vtiles = ws + pl.ws_k_bytes;
  ap.q = static_cast<const __half *>(q);
  ap.out = static_cast<__half *>(out);
  ap.lse = lse;
  ap.err = L.err;
  ap.part = reinterpret_cast<float *>(ws + pl.part_off);
  ap.n_q = L.n_q_heads;
  ap.G = L.n_q_heads / L.n_kv_heads;
  ap.n_tok = n_q_tok;
  ap.q_start = q_start;
  ap.kv_len = static_cast<int>(pl.kv_tokens);
  ap.n_tiles = n_tiles;
  ap.npairs = pl.npairs;
  ap.n_qt = pl.n_qt;
  ap.n_items = static_cast<int>(pl.n_items);
  ap.Tq = pl.Tq;
  ap.W = pl.W;
  ap.scale_log2 = scale * 1.4426950408889634f;
  const int smem = (2 + 2 * kStages) * kTileBytes + 1024;
  static std::atomic<uint64_t> optin{0};
  e = smem_optin(prefill_attn_kernel, smem, optin);
  if (e != cudaSuccess) return e;
  e = launch_pdl(prefill_attn_kernel, dim3(static_cast<unsigned>(pl.grid)), dim3(kThreads), smem,
                 stream, ap);
  if (e != cudaSuccess) return e;
  PieceMergeParams mp;
  mp.part = ap.part;
  mp.out = ap.out;
  mp.lse = lse;
  mp.n_q = ap.n_q;
  mp.G = ap.G;
  mp.n_tok = n_q_tok;
  mp.q_start = q_start;
  mp.npairs = pl.npairs;
  mp.n_qt = pl.n_qt;
  mp.Tq = pl.Tq;
  mp.W = pl.W;
  mp.grid = static_cast<int>(pl.grid);
  return launch_pdl(piece_merge_kernel,
                    dim3(static_cast<unsigned>(pl.n_items), 2, kBM / kMergeRowsPerCta),
                    dim3(kMergeThreads), 0, stream, mp);
}

}  // namespace kvq
