// prefill.cu -- causal attention of one prefill chunk (placeholder until the
// tensor-core kernel lands: the entry point reports "unsupported").
#include <cuda_runtime.h>

#include "kvq_launch.h"

namespace kvq {

PrefillPlan plan_prefill(const kvq_layer &L, int q_start, int n_q_tok) {
  PrefillPlan pl;
  pl.kv_tokens = static_cast<int64_t>(q_start) + n_q_tok;
  pl.kv_tokens_pad = (pl.kv_tokens + 127) / 128 * 128;
  pl.ws_k_bytes = static_cast<int64_t>(L.n_kv_heads) * pl.kv_tokens_pad * 128 * 2;
  pl.ws_bytes = 2 * pl.ws_k_bytes;
  return pl;
}

cudaError_t launch_prefill(const kvq_layer &, const PrefillPlan &, int, int, int, const void *,
                           float, void *, float *, void *, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace kvq
