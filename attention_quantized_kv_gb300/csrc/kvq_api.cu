// kvq_api.cu -- the C ABI of libkvq (include/kvq.h): argument validation on
// the host, launch planning, and dispatch to the kernels.  Nothing here
// allocates, frees or synchronizes device memory.
#include <cuda_runtime.h>

#include <stdint.h>

#include "../../include/kvq.h"
#include "kvq_check.h"
#include "kvq_launch.h"

namespace {

using kvq::aligned;
using kvq::check_layer;
using kvq::decode_shape_ok;
using kvq::kHeadDim;
using kvq::valid_codec;

int device_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace

extern "C" {

const char *kvq_status_str(int status) {
  switch (status) {
    case KVQ_OK: return "KVQ_OK";
    case KVQ_EINVAL: return "KVQ_EINVAL: invalid argument";
    case KVQ_EUNSUPPORTED: return "KVQ_EUNSUPPORTED: head_dim or codec not supported";
    case KVQ_ECAPACITY: return "KVQ_ECAPACITY: position past the cache capacity";
    case KVQ_EALIGN: return "KVQ_EALIGN: misaligned pointer or capacity not a multiple of 256";
    case KVQ_EWORKSPACE: return "KVQ_EWORKSPACE: workspace missing or too small";
    case KVQ_ECUDA: return "KVQ_ECUDA: CUDA runtime error";
    default: return "KVQ: unknown status";
  }
}

int64_t kvq_row_bytes(int codec, int32_t head_dim) {
  if (head_dim != kHeadDim || !valid_codec(codec)) return -1;
  return codec == KVQ_F16 ? 256 : codec == KVQ_Q8_0 ? 136 : codec == KVQ_Q4_0 ? 72 : 66;
}

int64_t kvq_pool_bytes(int codec, int32_t n_pages, int32_t n_kv_heads, int32_t head_dim) {
  const int64_t rb = kvq_row_bytes(codec, head_dim);
  if (rb < 0 || n_pages <= 0 || n_kv_heads <= 0) return -1;
  return rb * 256 * n_kv_heads * static_cast<int64_t>(n_pages);
}

int64_t kvq_cache_bytes(int codec, int32_t n_seqs, int32_t n_kv_heads, int32_t capacity,
                        int32_t head_dim) {
  const int64_t rb = kvq_row_bytes(codec, head_dim);
  if (rb < 0 || n_seqs <= 0 || n_kv_heads <= 0 || capacity <= 0 || capacity % 256 != 0)
    return -1;
  return rb * n_seqs * n_kv_heads * static_cast<int64_t>(capacity);
}

int kv_append_quantize(const kvq_layer *layer, const void *k_new, const void *v_new,
                       const int32_t *n_new, int32_t max_new, int32_t update_lens,
                       void *stream) {
  int st = check_layer(layer);
  if (st != KVQ_OK) return st;
  if (max_new < 0 || !n_new) return KVQ_EINVAL;
  if (max_new > layer->capacity) return KVQ_ECAPACITY;
  if (max_new > 0 && (!k_new || !v_new)) return KVQ_EINVAL;
  if (!aligned(k_new, 8) || !aligned(v_new, 8) || !aligned(n_new, 4)) return KVQ_EALIGN;
  const cudaError_t e = kvq::launch_append(*layer, k_new, v_new, n_new, max_new, update_lens,
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

int attn_decode_workspace(const kvq_layer *layer, int32_t max_len, size_t *bytes) {
  int st = check_layer(layer);
  if (st != KVQ_OK) return st;
  if (!decode_shape_ok(layer)) return KVQ_EINVAL;
  if (!bytes || max_len <= 0) return KVQ_EINVAL;
  if (max_len > layer->capacity) return KVQ_ECAPACITY;
  const int sms = device_sms();
  if (sms <= 0) return KVQ_ECUDA;
  *bytes = static_cast<size_t>(kvq::plan_decode(*layer, max_len, sms).ws_bytes);
  return KVQ_OK;
}

int attn_decode(const kvq_layer *layer, const void *q, float scale, void *out, float *lse,
                int32_t max_len, void *workspace, size_t ws_bytes, void *stream) {
  const int st = kvq::check_decode_call(layer, q, out, lse, max_len);
  if (st != KVQ_OK) return st;
  if (!workspace) return KVQ_EWORKSPACE;
  if (!aligned(workspace, 16)) return KVQ_EALIGN;
  const int sms = device_sms();
  if (sms <= 0) return KVQ_ECUDA;
  const kvq::DecodePlan pl = kvq::plan_decode(*layer, max_len, sms);
  if (ws_bytes < static_cast<size_t>(pl.ws_bytes)) return KVQ_EWORKSPACE;
  const cudaError_t e = kvq::launch_decode(*layer, pl, q, scale, out, lse, max_len, workspace,
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

int attn_decode_append(const kvq_layer *layer, const void *k_new, const void *v_new,
                       const void *q, float scale, void *out, float *lse, int32_t max_len,
                       void *workspace, size_t ws_bytes, void *stream) {
  int st = check_layer(layer);
  if (st != KVQ_OK) return st;
  if (!k_new || !v_new || !q || !out || max_len <= 0) return KVQ_EINVAL;
  if (!decode_shape_ok(layer)) return KVQ_EINVAL;
  if (max_len > layer->capacity) return KVQ_ECAPACITY;
  if (!aligned(k_new, 8) || !aligned(v_new, 8) || !aligned(q, 8) || !aligned(out, 8) ||
      (lse && !aligned(lse, 4)))
    return KVQ_EALIGN;
  if (!workspace) return KVQ_EWORKSPACE;
  if (!aligned(workspace, 16)) return KVQ_EALIGN;
  const int sms = device_sms();
  if (sms <= 0) return KVQ_ECUDA;
  const kvq::DecodePlan pl = kvq::plan_decode(*layer, max_len, sms);
  if (ws_bytes < static_cast<size_t>(pl.ws_bytes)) return KVQ_EWORKSPACE;
  const cudaError_t e = kvq::launch_decode(*layer, pl, q, scale, out, lse, max_len, workspace,
                                           static_cast<cudaStream_t>(stream), k_new, v_new);
  return e == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

int attn_prefill_workspace(const kvq_layer *layer, int32_t q_start, int32_t n_q_tok,
                           size_t *bytes) {
  int st = check_layer(layer);
  if (st != KVQ_OK) return st;
  if (!bytes || q_start < 0 || n_q_tok <= 0) return KVQ_EINVAL;
  if (static_cast<int64_t>(q_start) + n_q_tok > layer->capacity) return KVQ_ECAPACITY;
  const kvq::PrefillPlan pl =
      kvq::plan_prefill(*layer, q_start, n_q_tok, device_sms());
  *bytes = static_cast<size_t>(pl.ws_bytes);
  return KVQ_OK;
}

int attn_prefill_chunk(const kvq_layer *layer, int32_t seq, int32_t q_start, int32_t n_q_tok,
                       const void *q, float scale, void *out, float *lse, void *workspace,
                       size_t ws_bytes, void *stream) {
  int st = check_layer(layer);
  if (st != KVQ_OK) return st;
  if (!q || !out || q_start < 0 || n_q_tok <= 0 || seq < 0 || seq >= layer->n_seqs ||
      !(scale > 0.0f))
    return KVQ_EINVAL;
  if (static_cast<int64_t>(q_start) + n_q_tok > layer->capacity) return KVQ_ECAPACITY;
  if (!aligned(q, 16) || !aligned(out, 16) || (lse && !aligned(lse, 4))) return KVQ_EALIGN;
  if (!workspace) return KVQ_EWORKSPACE;
  if (!aligned(workspace, 16)) return KVQ_EALIGN;
  const kvq::PrefillPlan pl =
      kvq::plan_prefill(*layer, q_start, n_q_tok, device_sms());
  if (ws_bytes < static_cast<size_t>(pl.ws_bytes)) return KVQ_EWORKSPACE;
  const cudaError_t e = kvq::launch_prefill(*layer, pl, seq, q_start, n_q_tok, q, scale, out, lse,
                                            workspace, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

int kv_requantize(const kvq_layer *layer, int32_t side, int32_t dst_codec, void *dst_cache,
                  void *stream) {
  int st = check_layer(layer);
  if (st != KVQ_OK) return st;
  if (side != 0 && side != 1) return KVQ_EINVAL;
  if (!valid_codec(dst_codec)) return KVQ_EUNSUPPORTED;
  if (!dst_cache) return KVQ_EINVAL;
  if (!aligned(dst_cache, 16)) return KVQ_EALIGN;
  // out of place: the destination must not overlap the source
  const void *src = side == 0 ? layer->k_cache : layer->v_cache;
  const int src_codec = side == 0 ? layer->codec_k : layer->codec_v;
  const uint8_t *s0 = static_cast<const uint8_t *>(src);
  const uint8_t *d0 = static_cast<const uint8_t *>(dst_cache);
  const bool paged = layer->pages_per_seq > 0;
  const int64_t sb = paged ? kvq_pool_bytes(src_codec, layer->n_pages, layer->n_kv_heads, kHeadDim)
                           : kvq_cache_bytes(src_codec, layer->n_seqs, layer->n_kv_heads,
                                             layer->capacity, kHeadDim);
  const int64_t db = paged ? kvq_pool_bytes(dst_codec, layer->n_pages, layer->n_kv_heads, kHeadDim)
                           : kvq_cache_bytes(dst_codec, layer->n_seqs, layer->n_kv_heads,
                                             layer->capacity, kHeadDim);
  if (d0 < s0 + sb && s0 < d0 + db) return KVQ_EINVAL;
  const cudaError_t e =
      kvq::launch_requant(*layer, side, dst_codec, dst_cache, static_cast<cudaStream_t>(stream),
                          device_sms());
  return e == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

static bool overlaps(const void *a, int64_t na, const void *b, int64_t nb) {
  const uint8_t *x = static_cast<const uint8_t *>(a), *y = static_cast<const uint8_t *>(b);
  return x < y + nb && y < x + na;
}

// Bytes of one side's cache (or pool, for a paged layer).
static int64_t side_bytes(const kvq_layer *L, int codec) {
  return L->pages_per_seq > 0
             ? kvq_pool_bytes(codec, L->n_pages, L->n_kv_heads, kHeadDim)
             : kvq_cache_bytes(codec, L->n_seqs, L->n_kv_heads, L->capacity, kHeadDim);
}

int kv_probe_scores(const kvq_layer *layer, const void *q, float scale, const float *lse,
                    float decay, float *scores, void *stream) {
  int st = check_layer(layer);
  if (st != KVQ_OK) return st;
  if (!q || !lse || !scores) return KVQ_EINVAL;
  if (!aligned(q, 8) || !aligned(lse, 4) || !aligned(scores, 4)) return KVQ_EALIGN;
  const cudaError_t e = kvq::launch_probe(*layer, q, scale, lse, decay, scores,
                                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

int kv_evict_select(const kvq_layer *layer, const float *scores, int32_t n_sink,
                    int32_t n_recent, int32_t n_evict, int32_t *evict, int32_t *n_evicted,
                    void *stream) {
  int st = check_layer(layer);
  if (st != KVQ_OK) return st;
  if (!scores || !evict || !n_evicted || n_sink < 0 || n_recent < 0 || n_evict < 0)
    return KVQ_EINVAL;
  if (!aligned(scores, 4) || !aligned(evict, 4) || !aligned(n_evicted, 4)) return KVQ_EALIGN;
  const cudaError_t e =
      kvq::launch_evict_select(*layer, scores, n_sink, n_recent, n_evict, evict, n_evicted,
                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

int kv_compact(const kvq_layer *layer, const int32_t *evict, const int32_t *n_evicted,
               int32_t max_evict, void *k_dst, void *v_dst, const float *scores,
               float *scores_dst, int32_t *lens_dst, void *stream) {
  int st = check_layer(layer);
  if (st != KVQ_OK) return st;
  if (!evict || !n_evicted || max_evict < 0 || !k_dst || !v_dst) return KVQ_EINVAL;
  if ((scores == nullptr) != (scores_dst == nullptr)) return KVQ_EINVAL;
  if (!aligned(evict, 4) || !aligned(n_evicted, 4) || !aligned(k_dst, 16) ||
      !aligned(v_dst, 16) || (scores && !aligned(scores, 4)) ||
      (scores_dst && !aligned(scores_dst, 4)) || (lens_dst && !aligned(lens_dst, 4)))
    return KVQ_EALIGN;
  const int64_t kb = side_bytes(layer, layer->codec_k), vb = side_bytes(layer, layer->codec_v);
  if (overlaps(k_dst, kb, layer->k_cache, kb) || overlaps(k_dst, kb, layer->v_cache, vb) ||
      overlaps(v_dst, vb, layer->k_cache, kb) || overlaps(v_dst, vb, layer->v_cache, vb) ||
      overlaps(k_dst, kb, v_dst, vb))
    return KVQ_EINVAL;
  const int64_t sb = static_cast<int64_t>(layer->n_seqs) * layer->capacity * 4;
  if (scores && overlaps(scores, sb, scores_dst, sb)) return KVQ_EINVAL;
  if (lens_dst && overlaps(lens_dst, 4 * layer->n_seqs, layer->seq_lens, 4 * layer->n_seqs))
    return KVQ_EINVAL;
  const cudaError_t e =
      kvq::launch_compact(*layer, evict, n_evicted, max_evict, k_dst, v_dst, scores, scores_dst,
                          lens_dst, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

double kvq_aggregate_bpv(const int32_t *codecs, int32_t n) {
  if (!codecs || n <= 0) return -1.0;
  double sum = 0.0;
  for (int32_t i = 0; i < n; ++i) {
    const int64_t rb = kvq_row_bytes(codecs[i], kHeadDim);
    if (rb < 0) return -1.0;
    sum += static_cast<double>(rb) * 8.0 / kHeadDim;
  }
  return sum / n;
}

int kvq_ladder_next(const int32_t *codecs, int32_t n, const int32_t *order, int32_t n_order,
                    double floor_bpv, int32_t *tensor, int32_t *codec) {
  if (!codecs || n <= 0 || !tensor || !codec || n_order < 0 || (n_order > 0 && !order))
    return KVQ_EINVAL;
  for (int32_t i = 0; i < n; ++i)
    if (!valid_codec(codecs[i])) return KVQ_EUNSUPPORTED;
  for (int32_t i = 0; i < n_order; ++i)
    if (order[i] < 0 || order[i] >= n) return KVQ_EINVAL;
  const bool all = order == nullptr;
  const int32_t m = all ? n : n_order;
  *tensor = -1;
  *codec = -1;
  double total = 0.0;
  for (int32_t i = 0; i < n; ++i) total += kvq_row_bytes(codecs[i], kHeadDim) * 8.0 / kHeadDim;
  const int rungs[2] = {KVQ_Q8_0, KVQ_Q4_0};
  for (int k = 0; k < 2; ++k) {
    for (int32_t i = 0; i < m; ++i) {
      const int32_t t = all ? i : order[i];
      if (codecs[t] < rungs[k]) {  // codec ids grow as bits shrink
        const double after = total - kvq_row_bytes(codecs[t], kHeadDim) * 8.0 / kHeadDim +
                             kvq_row_bytes(rungs[k], kHeadDim) * 8.0 / kHeadDim;
        if (after / n < floor_bpv) return KVQ_OK;
        *tensor = t;
        *codec = rungs[k];
        return KVQ_OK;
      }
    }
  }
  return KVQ_OK;
}

}  // extern "C"
