/*
 * kvq.h -- C ABI of libkvq: attention over a block-quantized KV cache on one
 * GB300 (sm_103a).
 *
 * Operations (all asynchronous on the caller's CUDA stream):
 *   kv_append_quantize   quantize new K/V rows into the cache (f16 / q8_0 / q4_0)
 *   attn_decode          split-K decode attention over every cached key
 *   attn_prefill_chunk   causal attention of one prefill chunk (ubatch)
 *   kv_requantize        degrade one (layer, side) tensor to another codec
 *   kvq_aggregate_bpv    aggregate bits per value of a set of tensors
 *   kvq_ladder_next      the next step of the banded classic degrade ladder
 *
 * Sources.  The codecs and their sizes follow the "Codecs" table of the
 * buun-llama-cpp listing (f16 16.0, q8_0 8.5, q4_0 4.5 bits per value); the
 * per-(layer, side) codec choice follows its "VBR -- Variable Bit-Rate KV
 * Cache" section (the classic F16 -> Q8_0 -> Q4_0 ladder, K and V typed
 * independently, flash attention mandatory); the asymmetric K=f16 / V=q8_0
 * contract, the ubatch-sized prefill chunks and the 256-aligned per-slot
 * pools follow the serverAppConfigs commit log (frank_small_unit.bats
 * commit).  Softmax attention is the plain definition: o = softmax(scale *
 * q K^T) V over the attended keys, K and V dequantized.
 *
 * Ownership.  The caller allocates every buffer (cache, lengths, inputs,
 * outputs, workspace) in device memory and keeps it alive until the work on
 * the stream has finished.  The library never allocates, frees or
 * synchronizes; it keeps no state between calls besides cached device
 * attributes.
 *
 * Errors.  Every entry point validates its arguments on the host before any
 * launch and returns a kvq_status; it never aborts.  Conditions that only the
 * device can see (a length that passes capacity, a wait that timed out) set
 * bits in the optional device word kvq_layer.err (KVQ_DEVERR_*) and the
 * affected rows are skipped.
 *
 * ------------------------------------------------------------------------
 * Block codecs (head_dim 128 = four 32-value blocks per row):
 *   f16  : 128 fp16 values.                              256 bytes / row
 *   q8_0 : per block fp16 d16 + 32 int8 q.               136 bytes / row
 *          amax = max|x| (fp32); d = amax / 127 (fp32, IEEE RN division);
 *          q = round-half-away-from-zero(x / d) (IEEE RN division), or 0 when
 *          d == 0; d16 = fp16_RN(d).  x^ = d16 * q.
 *   q4_0 : per block fp16 d16 + 16 bytes of nibbles.      72 bytes / row
 *          m = the signed x with the largest |x| (lowest index wins ties);
 *          d = m / -8 (fp32 RN); t = x / d (fp32 RN; 0 when d == 0);
 *          u = t + 8.5 (fp32 RN); q = min(15, trunc(u));
 *          canonical byte j = q[j] | q[j+16] << 4; d16 = fp16_RN(d).
 *          x^ = d16 * (q - 8).
 *   turbo4: a Walsh-Hadamard-rotated 4-bit row (the turbo4 row of the
 *          "Codecs" table of the buun-llama-cpp listing, 4.125 bits per value;
 *          the FWHT with random sign flips of its TCQ "How it works" list;
 *          the scale and levels are this library's reading).   66 bytes / row
 *          signs s_j = -1 where bit 63 of output j (j = 0..127) of SplitMix64
 *          (Steele, Lea, Flood 2014) seeded with 0x4B5651 is set, else +1;
 *          t = s * x; unnormalised FWHT of t in Sylvester order, stages
 *          h = 1, 2, ..., 64 turning each pair (j, j + h), j & h == 0, into
 *          (a + b, a - b) with fp32 RN additions; y = t / 8; then the q4_0
 *          rule over all 128 values of y (one d16 per row); canonical byte
 *          16 g + j (group g < 4, j < 16) = q[32g + j] | q[32g + j + 16] << 4.
 *          Decoded: y^ = d16 * (q - 8) and x^ = s * H y^ / 16, exact in fp32.
 *          Attention never forms x^: q . x^ = (H (s * q) / 16) . y^, so the
 *          kernels rotate the query once, accumulate V in the rotated space
 *          and rotate the output back once.
 *   The canonical row is the row's four blocks end to end (d16 little-endian
 *   before each block's quants); for turbo4 the row's d16 then its 64 bytes.
 *
 * Cache layout (one layer, one side):
 *   [n_seqs][n_kv_heads][capacity / 16 units][unit_bytes]
 *   A unit holds 16 consecutive tokens (unit_bytes = 16 * row bytes: 4096,
 *   2176, 1152, 1056).  Inside a unit, canonical byte cb of token row r (0..15) is
 *   placed as follows (all integer arithmetic; g = r & 7, rh = r >> 3,
 *   tig = (r & 7) >> 1, par = r & 1):
 *   K side
 *     f16  value d, byte k:  b=d>>5, h=(d>>4)&1, w=(d>>2)&3, i=d&3
 *          -> (2b+rh)*512 + (4g+w)*16 + h*8 + i*2 + k
 *     q8_0 quant of dim 32b+e: h=e>>4, w=(e>>2)&3, i=e&3
 *          -> b*512 + (4g+w)*16 + (2rh+h)*4 + i
 *          scale byte k of block b -> 2048 + g*16 + rh*8 + b*2 + k
 *     q4_0 canonical byte jc (0..15) of block b: w=jc>>2, i=jc&3
 *          -> (b>>1)*512 + (4g+w)*16 + ((b&1)*2+rh)*4 + i
 *          scale byte k of block b -> 1024 + g*16 + rh*8 + b*2 + k
 *     turbo4 canonical byte jc of group b: as q4_0's byte jc of block b;
 *          scale byte k -> 1024 + g*4 + rh*2 + k
 *   V side
 *     f16  value d, byte k:  mt=d>>4, gq=(d&15)>>1, s=d&1
 *          -> mt*512 + (4gq+tig)*16 + (rh*4+s*2+par)*2 + k
 *     q8_0 quant of dim d: mt=d>>4, gq=(d&15)>>1, s=d&1
 *          -> (mt>>1)*512 + (4gq+tig)*16 + ((mt&1)*2+rh)*4 + par*2 + s
 *          scale byte k of block b -> 2048 + tig*32 + b*8 + rh*4 + par*2 + k
 *     q4_0 canonical byte jc of block b: mt=2b+(jc>>3), gq=jc&7
 *          -> (mt>>2)*512 + (4gq+tig)*16 + (mt&3)*4 + par*2 + rh
 *          scale byte k of block b -> 1024 + tig*32 + b*8 + rh*4 + par*2 + k
 *     turbo4 canonical byte jc of group b: as q4_0's byte jc of block b;
 *          scale byte k -> 1024 + tig*8 + rh*4 + par*2 + k
 *   The layout stores exactly the canonical bytes (8.5 / 4.5 / 16 / 4.125
 *   bits per value); it only orders them so that each thread of the decode kernel
 *   reads its tensor-core operand fragments with aligned 16-byte loads.
 *
 * Paged layout (kvq_layer.pages_per_seq > 0; block-level KV management as in
 * the vLLM PagedAttention entry of the buun-llama-cpp references, with the
 * pool shared by the sequences and 256-aligned as in the serverAppConfigs
 * commit log):
 *   a page is 256 tokens (16 units) of every kv head of one sequence; each
 *   side's pool is [n_pages][n_kv_heads][16 units][unit_bytes]
 *   (kvq_pool_bytes()); block_table[s][p] is the pool page that holds
 *   tokens 256p .. 256p + 255 of sequence s (-1: not mapped).  Unit j of
 *   (sequence s, kv head h) is pool unit
 *   (block_table[s][j / 16] * n_kv_heads + h) * 16 + j % 16.  capacity is
 *   then pages_per_seq * 256.  Every page a call touches (tokens below the
 *   length, or being appended) must be mapped to a page in [0, n_pages);
 *   otherwise the device sets KVQ_DEVERR_PAGE and skips the row (append,
 *   re-encode) or reads pool page 0 in its place (attention).
 * ------------------------------------------------------------------------
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Codec of one (layer, side) cache tensor. */
typedef enum { KVQ_F16 = 0, KVQ_Q8_0 = 1, KVQ_Q4_0 = 2, KVQ_TURBO4 = 3 } kvq_codec;

/* Host-side status returned by every entry point. */
typedef enum {
    KVQ_OK = 0,
    KVQ_EINVAL = 1,       /* null pointer, non-positive size, bad index, n_q % n_kv != 0 */
    KVQ_EUNSUPPORTED = 2, /* head_dim != 128 or unknown codec */
    KVQ_ECAPACITY = 3,    /* a host-known position passes capacity */
    KVQ_EALIGN = 4,       /* capacity not a multiple of 256, or a misaligned pointer */
    KVQ_EWORKSPACE = 5,   /* workspace null or smaller than the *_workspace query says */
    KVQ_ECUDA = 6         /* a CUDA runtime call or a launch failed */
} kvq_status;

/* Bits OR-ed into *kvq_layer.err by the device (the word is never cleared). */
#define KVQ_DEVERR_CAPACITY 1 /* append: seq_lens[s] + n_new[s] > capacity; rows skipped */
#define KVQ_DEVERR_MAXLEN 2   /* decode: seq_lens[s] > max_len; keys past max_len ignored */
#define KVQ_DEVERR_TIMEOUT 4  /* a bounded wait on an async copy gave up */
#define KVQ_DEVERR_SEQLEN 8   /* prefill: seq_lens[seq] < q_start + n_q_tok */
#define KVQ_DEVERR_PAGE 16    /* paged: a block-table entry outside [0, n_pages) */
#define KVQ_DEVERR_EVICT 32   /* kv_compact: an eviction list not increasing below the length */

/* One layer's cache.  All pointers are device pointers owned by the caller.
 * k_cache / v_cache: kvq_cache_bytes() bytes each (kvq_pool_bytes() when
 * paged), 16-byte aligned, in the layouts above.  seq_lens: int32[n_seqs],
 * the number of valid tokens of each sequence.  err: optional int32 error
 * word (NULL to skip). */
typedef struct kvq_layer {
    int32_t n_seqs;
    int32_t n_kv_heads;
    int32_t n_q_heads;  /* multiple of n_kv_heads; head h reads kv head h / (n_q/n_kv) */
    int32_t head_dim;   /* must be 128 */
    int32_t capacity;   /* tokens per (seq, kv head) stream; multiple of 256 */
    int32_t codec_k;    /* kvq_codec of the K side */
    int32_t codec_v;    /* kvq_codec of the V side */
    int32_t pages_per_seq; /* 0: contiguous caches; > 0: paged (capacity = 256 * this) */
    void *k_cache;
    void *v_cache;
    int32_t *seq_lens;
    int32_t *err;
    const int32_t *block_table; /* paged: int32 [n_seqs][pages_per_seq], device; else NULL */
    int32_t n_pages;            /* paged: pages in each side's pool; else 0 */
    int32_t reserved;           /* must be 0 */
} kvq_layer;

/* Human-readable name of a status code (static string). */
KVQ_API const char *kvq_status_str(int status);

/* Bytes of one canonical row (256 / 136 / 72 for head_dim 128), or -1. */
KVQ_API int64_t kvq_row_bytes(int codec, int32_t head_dim);

/* Bytes of one side's page pool: n_pages * n_kv_heads * 256 * row bytes, or
 * -1 on bad arguments. */
KVQ_API int64_t kvq_pool_bytes(int codec, int32_t n_pages, int32_t n_kv_heads, int32_t head_dim);

/* Bytes of one side's cache for the given geometry, or -1 on bad arguments. */
KVQ_API int64_t kvq_cache_bytes(int codec, int32_t n_seqs, int32_t n_kv_heads, int32_t capacity,
                        int32_t head_dim);

/* Quantize-on-append (block codecs above).
 * k_new, v_new: fp16 [n_seqs][max_new][n_kv_heads][128], 8-byte aligned.
 * n_new: device int32[n_seqs], rows to append per sequence (0..max_new).
 * Row i < n_new[s] of sequence s is encoded with the side's codec and written
 * at token position seq_lens[s] + i.  When update_lens != 0, seq_lens[s] +=
 * n_new[s] afterwards (stream-ordered).  Positions past capacity set
 * KVQ_DEVERR_CAPACITY and are skipped. */
KVQ_API int kv_append_quantize(const kvq_layer *layer, const void *k_new, const void *v_new,
                       const int32_t *n_new, int32_t max_new, int32_t update_lens,
                       void *stream);

/* Workspace bytes that attn_decode needs for this layer and max_len. */
KVQ_API int attn_decode_workspace(const kvq_layer *layer, int32_t max_len, size_t *bytes);

/* Decode attention: every query head of every sequence attends all
 * seq_lens[s] cached keys (split-K over the token axis; two launches: the
 * split kernel writes partials, the merge kernel combines them by
 * log-sum-exp).  The first 64 KiB of the workspace are a counter region that
 * must be zero before the first call (zero-fill the workspace once after
 * allocating it); every call that completes without KVQ_DEVERR_TIMEOUT
 * leaves it zero again, so one workspace serves any number of calls and
 * layers without clearing.  Calls that may run concurrently need separate
 * workspaces.  Limits: 1024 sequences and 16383 streams (sequence x kv head
 * x group of 8 query heads) per call, else KVQ_EINVAL.
 * q: fp16 [n_seqs][n_q_heads][128] (8-byte aligned); out: fp16
 * [n_seqs][n_q_heads][128]; lse: optional fp32 [n_seqs][n_q_heads] natural-log
 * sum-exp of the scaled scores (NULL to skip).  max_len bounds every
 * seq_lens[s] (1..capacity).  workspace: device, 16-byte aligned, at least
 * attn_decode_workspace() bytes.  A sequence of length 0 gives out = 0 and
 * lse = -inf. */
KVQ_API int attn_decode(const kvq_layer *layer, const void *q, float scale, void *out, float *lse,
                int32_t max_len, void *workspace, size_t ws_bytes, void *stream);

/* One decode step of a layer with no launch for the append: quantize-on-append
 * of one new token per sequence (the kv_append_quantize row encoding, at position
 * seq_lens[s]), then attn_decode over seq_lens[s] + 1 keys, then
 * seq_lens[s] += 1.  The result (cache bytes, lengths, out, lse) is that of
 * kv_append_quantize(n_new = 1 for every sequence, update_lens = 1)
 * followed by attn_decode on the same stream (a new token's keys enter the
 * typed cache before it is attended, as in the serverAppConfigs commit log,
 * frank_small_unit.bats commit), fused so that the append costs no launch
 * of its own.
 * k_new, v_new: fp16 [n_seqs][n_kv_heads][128], 8-byte aligned.  A sequence
 * whose length is already capacity (or negative) gets no new token (sets
 * KVQ_DEVERR_CAPACITY) and attends its existing keys.  max_len must bound
 * every new length.  The workspace is attn_decode_workspace(layer, max_len)
 * bytes, with the same zero-between-calls contract as attn_decode; its
 * 64 KiB counter region also counts the CTAs that have read the lengths.
 * Other arguments and limits are those of attn_decode. */
KVQ_API int attn_decode_append(const kvq_layer *layer, const void *k_new, const void *v_new,
                               const void *q, float scale, void *out, float *lse,
                               int32_t max_len, void *workspace, size_t ws_bytes, void *stream);

/* attn_decode without a workspace argument, for callers that cannot allocate
 * device memory where they run attention (an interface that hands them only
 * the input and output buffers, a loop where a device allocation is not
 * allowed, a fully committed memory budget).  There is no counterpart in the
 * source material; it is a convenience of this library.  The scratch that
 * attn_decode keeps in the caller's workspace lives instead in one 8 MiB
 * device array inside the library (reserved on every GPU that loads it, until
 * the process exits); nothing is allocated.  The first call on a device looks
 * the array up (cudaGetSymbolAddress) and must come before any stream capture.
 * The array is shared by all calls and keeps the previous call's contents:
 * its counter region is cleared on `stream` before each launch, and calls
 * that can overlap on the GPU race on it, so issue them in order on one
 * stream.  A layer whose attn_decode_workspace() exceeds 8 MiB is refused
 * with KVQ_EWORKSPACE.  Arguments and results are those of attn_decode. */
KVQ_API int attn_decode_noalloc(const kvq_layer *layer, const void *q, float scale, void *out,
                                float *lse, int32_t max_len, void *stream);

/* Workspace bytes that attn_prefill_chunk needs for a chunk ending at
 * q_start + n_q_tok. */
KVQ_API int attn_prefill_workspace(const kvq_layer *layer, int32_t q_start, int32_t n_q_tok,
                           size_t *bytes);

/* Causal attention of one prefill chunk of sequence `seq`: query i (absolute
 * position q_start + i) of head h attends keys 0 .. q_start + i of kv head
 * h / (n_q/n_kv).  The chunk's own keys must already be appended.
 * q: fp16 [n_q_tok][n_q_heads][128] (16-byte aligned); out: fp16
 * [n_q_tok][n_q_heads][128] (16-byte aligned); lse: optional fp32
 * [n_q_tok][n_q_heads]; scale > 0.  The keys and values are dequantized once
 * into the workspace as fp16 (each value rounded once to fp16, the tensor-core
 * operand type).  workspace: device, 16-byte aligned, at least
 * attn_prefill_workspace() bytes. */
KVQ_API int attn_prefill_chunk(const kvq_layer *layer, int32_t seq, int32_t q_start, int32_t n_q_tok,
                       const void *q, float scale, void *out, float *lse, void *workspace,
                       size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Degrade ladder ("VBR -- Variable Bit-Rate KV Cache" section of the
 * buun-llama-cpp listing: the cache degrades one (layer, side) tensor at a
 * time down the classic f16 -> q8_0 -> q4_0 ladder; the classic order is
 * strictly banded, every movable tensor reaching q8_0 before any reaches
 * q4_0; degrades stop at the last step whose aggregate bits per value stays
 * at or above the floor).
 * ------------------------------------------------------------------------ */

/* Re-encode side `side` (0 = K, 1 = V) of the layer with codec dst_codec into
 * dst_cache: for every sequence s and kv head, tokens [0, seq_lens[s]) are
 * decoded (exactly, as fp32: d16 * q, d16 * (n - 8), or the fp16 value) and
 * encoded again with the append encoder of dst_codec (an f16 target rounds to
 * fp16); tokens past the length are not written.  From f16 the result equals
 * appending the original rows with dst_codec.
 * dst_cache: device, kvq_cache_bytes(dst_codec, ...) bytes, 16-byte aligned,
 * not overlapping the source (the degrade is done out of place; the caller
 * then points the layer's side at dst_cache and sets its codec).  Any pair of
 * codecs is accepted. */
KVQ_API int kv_requantize(const kvq_layer *layer, int32_t side, int32_t dst_codec, void *dst_cache,
                          void *stream);

/* Aggregate bits per value of n tensors holding equally many values: the mean
 * of the codecs' bits per value (16, 8.5, 4.5).  -1 on bad arguments.  Host
 * only. */
KVQ_API double kvq_aggregate_bpv(const int32_t *codecs, int32_t n);

/* The next degrade step of the banded classic ladder for n tensors with the
 * given codecs.  order: the n_order movable tensor indices in price order
 * (tensors missing from it are pinned and never move); NULL with n_order = 0
 * means every tensor in index order.  The first tensor in order still above
 * q8_0 goes to q8_0; once none is, the first one still above q4_0 goes to
 * q4_0; the step is taken only if the aggregate bits per value afterwards is
 * >= floor_bpv.  On KVQ_OK, *tensor and *codec hold the step, or *tensor = -1
 * when no step remains.  Host only. */
KVQ_API int kvq_ladder_next(const int32_t *codecs, int32_t n, const int32_t *order,
                            int32_t n_order, double floor_bpv, int32_t *tensor, int32_t *codec);

/* ------------------------------------------------------------------------
 * Probe-scored eviction (the "Sparse KV eviction" item of the "How It Works"
 * section of the GitHot listing of VITRIOL: an attention probe, a q.K softmax
 * with exponential decay, scores the cells; the lowest-scored middle cells
 * are evicted first; the sink cells at the start and the recent cells at the
 * end are protected).
 * Scores are fp32 [n_seqs][capacity] by logical position, for contiguous and
 * paged layers alike.
 * ------------------------------------------------------------------------ */

/* Fold one probe into the scores: for every sequence s and token
 * t < seq_lens[s],
 *   mass_t = sum over the query heads h of exp(scale * q_h . k^_t - lse[s][h])
 * (the softmax weight head h puts on t; k^ the decoded key of h's kv head) and
 *   scores[s][t] = decay * scores[s][t] + mass_t.
 * Entries at t >= seq_lens[s] are not touched.  q: fp16 [n_seqs][n_q][128]
 * (8-byte aligned), the query of the decode step; lse: fp32 [n_seqs][n_q],
 * the natural-log log-sum-exp that attn_decode wrote for the same q, scale
 * and cache (the probe reads K once more and never recomputes it); scores:
 * device, 4-byte aligned.  Results are deterministic (a fixed summation
 * order). */
KVQ_API int kv_probe_scores(const kvq_layer *layer, const void *q, float scale, const float *lse,
                            float decay, float *scores, void *stream);

/* For every sequence s, the min(n_evict, len - n_recent - n_sink) positions t
 * in [n_sink, len - n_recent) with the smallest (scores[s][t], t) pairs
 * (equal scores: the lower position first; -0 equals +0; NaN scores are
 * outside the contract and order after every number), written in increasing
 * order to evict[s][0 ..); n_evicted[s] = their count (0 when the middle
 * range is empty).  evict: device int32 [n_seqs][n_evict]; n_evicted: device
 * int32 [n_seqs]; n_sink, n_recent >= 0, n_evict >= 0. */
KVQ_API int kv_evict_select(const kvq_layer *layer, const float *scores, int32_t n_sink,
                            int32_t n_recent, int32_t n_evict, int32_t *evict,
                            int32_t *n_evicted, void *stream);

/* Remove the listed tokens from both sides of every sequence: the kept tokens
 * t < seq_lens[s] move down in order into k_dst / v_dst, bytes unchanged
 * (same codecs and layout as the layer's caches, same block table for a paged
 * layer).  evict: device int32 [n_seqs][max_evict], the n_evicted[s] first
 * entries of row s increasing and below seq_lens[s] (as kv_evict_select
 * writes them; otherwise the device sets KVQ_DEVERR_EVICT and the result is
 * unspecified but in bounds).  Inside the last unit written, rows past the new
 * length are zero; units past it are not written.  Optional (null to skip):
 * scores_dst[s][w] = scores[s][source of w] for w below the new length, and
 * lens_dst[s] = seq_lens[s] - n_evicted[s].  Every destination is out of
 * place (it must not overlap the layer's caches or the scores); the caller
 * then points the layer at k_dst, v_dst and lens_dst.  k_dst, v_dst: 16-byte
 * aligned, kvq_cache_bytes (kvq_pool_bytes for a paged layer) of the codecs. */
KVQ_API int kv_compact(const kvq_layer *layer, const int32_t *evict, const int32_t *n_evicted,
                       int32_t max_evict, void *k_dst, void *v_dst, const float *scores,
                       float *scores_dst, int32_t *lens_dst, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
