// decode_noalloc.cu -- attn_decode_noalloc: decode attention whose scratch
// lives in a fixed array inside the library instead of a caller workspace.
//
// Who needs it: callers that cannot allocate device memory where they run
// attention -- a plug-in or callback interface that receives only the input
// and output buffers and has no handle to an allocator; a latency-critical
// loop where a device allocation (which may synchronize the device) is not
// allowed; a process whose device memory budget is fully committed up front.
// For them the split-K partials and the per-stream arrival counters of the
// decode kernel sit in one file-scope device array of kNoAllocScratchBytes
// (8 MiB), which every GPU that loads this library reserves until the
// process exits.
//
// Rules of use:
//  * The first call on a device looks the array's device address up with
//    cudaGetSymbolAddress (with that device current) and caches it; make that
//    first call before any stream capture begins.
//  * Every call shares the one array and it keeps what the previous call left
//    there; the arrival counters are cleared (cudaMemsetAsync on the call's
//    stream) before each launch.  Calls that may overlap on the GPU -- on
//    different streams or from different host threads without ordering --
//    race on the array and must not be issued.
//  * A layer whose decode scratch (attn_decode_workspace) exceeds the array is
//    refused with KVQ_EWORKSPACE before anything is launched.
//  * Nothing here allocates: no cudaMalloc, cudaFree or allocating library call.
#include <cuda_runtime.h>

#include <mutex>
#include <stdint.h>

#include "../../include/kvq.h"
#include "kvq_launch.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 8u << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_decode_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {nullptr};
int g_num_sms[kMaxDevices] = {0};

// Device address of the scratch array (and the SM count) for the current
// device, looked up once per device.
int scratch_for_current_device(void **addr, int *sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVQ_ECUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return KVQ_ECUDA;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return KVQ_ECUDA;
    g_scratch_addr[dev] = p;
    g_num_sms[dev] = n;
  }
  *addr = g_scratch_addr[dev];
  *sms = g_num_sms[dev];
  return KVQ_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" {

int attn_decode_noalloc(const kvq_layer *L, const void *q, float scale, void *out, float *lse,
                        int32_t max_len, void *stream) {
  // Argument checks (the same rules as attn_decode).
  if (!L) return KVQ_EINVAL;
  if (L->head_dim != 128) return KVQ_EUNSUPPORTED;
  const bool codecs_ok = L->codec_k >= KVQ_F16 && L->codec_k <= KVQ_TURBO4 &&
                         L->codec_v >= KVQ_F16 && L->codec_v <= KVQ_TURBO4;
  if (!codecs_ok) return KVQ_EUNSUPPORTED;
  if (L->n_seqs <= 0 || L->n_kv_heads <= 0 || L->n_q_heads <= 0 || L->capacity <= 0 ||
      L->reserved != 0 || L->n_q_heads % L->n_kv_heads != 0)
    return KVQ_EINVAL;
  if (!L->k_cache || !L->v_cache || !L->seq_lens || !q || !out || max_len <= 0)
    return KVQ_EINVAL;
  if (L->capacity % 256 != 0) return KVQ_EALIGN;
  if (L->pages_per_seq < 0) return KVQ_EINVAL;
  if (L->pages_per_seq > 0 &&
      (!L->block_table || L->n_pages <= 0 ||
       static_cast<int64_t>(L->pages_per_seq) * 256 != L->capacity))
    return KVQ_EINVAL;
  if (!aligned(L->k_cache, 16) || !aligned(L->v_cache, 16) || !aligned(L->seq_lens, 4) ||
      (L->err && !aligned(L->err, 4)) || !aligned(q, 8) || !aligned(out, 8) ||
      (lse && !aligned(lse, 4)))
    return KVQ_EALIGN;
  if (max_len > L->capacity) return KVQ_ECAPACITY;
  const int64_t G = L->n_q_heads / L->n_kv_heads;
  const int64_t streams = static_cast<int64_t>(L->n_seqs) * L->n_kv_heads * ((G + 7) / 8);
  if (L->n_seqs > kvq::kDecodeMaxSeqs || streams > kvq::kDecodeMaxStreams) return KVQ_EINVAL;

  void *scratch = nullptr;
  int sms = 0;
  const int st = scratch_for_current_device(&scratch, &sms);
  if (st != KVQ_OK) return st;
  const kvq::DecodePlan pl = kvq::plan_decode(*L, max_len, sms);
  if (pl.ws_bytes > static_cast<int64_t>(kNoAllocScratchBytes)) return KVQ_EWORKSPACE;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The per-stream arrival counters must start at zero.
  if (cudaMemsetAsync(scratch, 0, static_cast<size_t>(streams) * 4, s) != cudaSuccess)
    return KVQ_ECUDA;
  const cudaError_t e = kvq::launch_decode(*L, pl, q, scale, out, lse, max_len, scratch, s);
  return e == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

}  // extern "C"
