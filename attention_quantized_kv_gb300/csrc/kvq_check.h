// kvq_check.h -- host-side argument validation shared by every entry point of
// libkvq, so that all of them apply the same rules (include/kvq.h: "Errors").
#pragma once

#include <stdint.h>

#include "../../include/kvq.h"
#include "kvq_launch.h"

namespace kvq {

constexpr int kHeadDim = 128;

inline bool valid_codec(int c) {
  return c == KVQ_F16 || c == KVQ_Q8_0 || c == KVQ_Q4_0 || c == KVQ_TURBO4;
}

inline bool aligned(const void *p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// The layer descriptor: geometry, codecs, cache pointers and their
// alignment, and (paged layers) the block table.
inline int check_layer(const kvq_layer *L) {
  if (!L) return KVQ_EINVAL;
  if (L->head_dim != kHeadDim) return KVQ_EUNSUPPORTED;
  if (!valid_codec(L->codec_k) || !valid_codec(L->codec_v)) return KVQ_EUNSUPPORTED;
  if (L->n_seqs <= 0 || L->n_kv_heads <= 0 || L->n_q_heads <= 0 || L->capacity <= 0 ||
      L->reserved != 0)
    return KVQ_EINVAL;
  if (L->n_q_heads % L->n_kv_heads != 0) return KVQ_EINVAL;
  if (!L->k_cache || !L->v_cache || !L->seq_lens) return KVQ_EINVAL;
  if (L->capacity % 256 != 0) return KVQ_EALIGN;
  if (L->pages_per_seq < 0) return KVQ_EINVAL;
  if (L->pages_per_seq > 0) {  // paged: a block table over pools of n_pages pages
    if (!L->block_table || L->n_pages <= 0) return KVQ_EINVAL;
    if (static_cast<int64_t>(L->pages_per_seq) * 256 != L->capacity) return KVQ_EINVAL;
    if (!aligned(L->block_table, 4)) return KVQ_EALIGN;
  }
  if (!aligned(L->k_cache, 16) || !aligned(L->v_cache, 16) || !aligned(L->seq_lens, 4) ||
      (L->err && !aligned(L->err, 4)))
    return KVQ_EALIGN;
  return KVQ_OK;
}

// Decode streams: (sequence, kv head, group of up to 8 query heads).
inline bool decode_shape_ok(const kvq_layer *L) {
  const int64_t G = L->n_q_heads / L->n_kv_heads;
  const int64_t streams = static_cast<int64_t>(L->n_seqs) * L->n_kv_heads * ((G + 7) / 8);
  return L->n_seqs <= kDecodeMaxSeqs && streams <= kDecodeMaxStreams;
}

// Everything a decode call checks before its scratch memory: the layer, the
// query and output pointers and max_len.
inline int check_decode_call(const kvq_layer *L, const void *q, const void *out,
                             const float *lse, int32_t max_len) {
  const int st = check_layer(L);
  if (st != KVQ_OK) return st;
  if (!q || !out || max_len <= 0) return KVQ_EINVAL;
  if (!decode_shape_ok(L)) return KVQ_EINVAL;
  if (max_len > L->capacity) return KVQ_ECAPACITY;
  if (!aligned(q, 8) || !aligned(out, 8) || (lse && !aligned(lse, 4))) return KVQ_EALIGN;
  return KVQ_OK;
}

}  // namespace kvq
