// kvq_launch.h -- internal launch entry points shared between the C ABI
// translation unit and the kernel translation units of libkvq.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

cudaError_t launch_append(const kvq_layer &L, const void *k_new, const void *v_new,
                          const int32_t *n_new, int max_new, int update_lens,
                          cudaStream_t stream);

// Re-encode one side of the layer into dst_cache (dst_codec): tokens below
// each sequence's length (append.cu).
cudaError_t launch_requant(const kvq_layer &L, int side, int dst_codec, void *dst_cache,
                           cudaStream_t stream, int num_sms);

constexpr int kDecodeMaxSeqs = 1024;         // sequences per attn_decode call
// counter region at the workspace start (zero between calls); its last word
// counts the CTAs of a fused decode step that have read the lengths
constexpr int kDecodeTicketBytes = 64 * 1024;
constexpr int kDecodeMaxStreams = kDecodeTicketBytes / 4 - 1;  // streams per call

struct DecodePlan {
  int n_hgroups = 1;      // groups of up to 8 query heads per kv head
  int grid = 1;           // CTAs, each an equal slice of the (stream, unit) space
  int64_t slots = 0;      // partial slots: grid + streams
  int64_t ticket_bytes = 0;  // workspace: the counter region (zero between calls)
  int64_t ml_bytes = 0;   //            (max, sum) per slot and head
  int64_t o_bytes = 0;    //            unnormalised output per slot and head
  int64_t ws_bytes = 0;
};

DecodePlan plan_decode(const kvq_layer &L, int max_len, int num_sms);
// k_new / v_new (fused decode step, fp16 [n_seqs][n_kv][128]): append one
// token per sequence before attending, and advance the lengths.
cudaError_t launch_decode(const kvq_layer &L, const DecodePlan &pl, const void *q, float scale,
                          void *out, float *lse, int max_len, void *workspace,
                          cudaStream_t stream, const void *k_new = nullptr,
                          const void *v_new = nullptr);

struct PrefillPlan {
  int64_t kv_tokens = 0;     // keys attended by the chunk: q_start + n_q_tok
  int64_t kv_tokens_pad = 0; // rounded up to the attention tile
  int64_t ws_k_bytes = 0;    // fp16 K staging [n_kv][kv_tokens_pad][128] (V the same)
  int npairs = 0, n_qt = 0;  // query-head pairs per kv head, 128-query tiles
  int64_t n_items = 0;       // (kv head, head pair, query tile) work items
  int64_t Tq = 0, W = 0;     // key-tile steps per (kv head, pair); in all
  int64_t sms = 0;           // the device's SMs
  int64_t grid = 0;          // persistent CTAs (at most one per SM)
  int64_t part_off = 0, part_bytes = 0;
  int64_t ws_bytes = 0;
};

PrefillPlan plan_prefill(const kvq_layer &L, int q_start, int n_q_tok, int num_sms);
cudaError_t launch_prefill(const kvq_layer &L, const PrefillPlan &pl, int seq, int q_start,
                           int n_q_tok, const void *q, float scale, void *out, float *lse,
                           void *workspace, cudaStream_t stream);

// Probe-scored eviction (evict.cu).
cudaError_t launch_probe(const kvq_layer &L, const void *q, float scale, const float *lse,
                         float decay, float *scores, cudaStream_t stream);
cudaError_t launch_evict_select(const kvq_layer &L, const float *scores, int n_sink,
                                int n_recent, int n_evict, int32_t *evict, int32_t *n_evicted,
                                cudaStream_t stream);
cudaError_t launch_compact(const kvq_layer &L, const int32_t *evict, const int32_t *n_evicted,
                           int max_evict, void *k_dst, void *v_dst, const float *scores,
                           float *scores_dst, int32_t *lens_dst, cudaStream_t stream);

}  // namespace kvq
