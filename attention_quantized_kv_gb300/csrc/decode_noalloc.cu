// decode_noalloc.cu -- attn_decode_noalloc: decode attention whose scratch
// lives in a fixed array inside the library instead of a caller workspace.
//
// Who needs it: callers that cannot allocate device memory where they run
// attention -- a plug-in or callback interface that receives only the input
// and output buffers and has no handle to an allocator; a latency-critical
// loop where a device allocation (which may synchronize the device) is not
// allowed; a process whose device memory budget is fully committed up front.
// For them the split-K partials and the counter region of the decode
// kernels sit in one file-scope device array of kNoAllocScratchBytes
// (8 MiB), which every GPU that loads this library reserves until the
// process exits.
//
// Rules of use:
//  * The first call on a device looks the array's device address up with
//    cudaGetSymbolAddress (with that device current) and caches it; make that
//    first call before any stream capture begins.
//  * Every call shares the one array and it keeps what the previous call left
//    there; its counter region (the first 64 KiB) is cleared (cudaMemsetAsync
//    on the call's stream) before each launch.  Calls that may overlap on the
//    GPU -- on different streams or from different host threads without
//    ordering -- race on the array and must not be issued.
//  * A layer whose decode scratch (attn_decode_workspace) exceeds the array is
//    refused with KVQ_EWORKSPACE before anything is launched.
//  * Nothing here allocates: no cudaMalloc, cudaFree or allocating library call.
#include <cuda_runtime.h>

#include <mutex>
#include <stdint.h>

#include "../../include/kvq.h"
#include "kvq_check.h"
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

}  // namespace

extern "C" {

int attn_decode_noalloc(const kvq_layer *L, const void *q, float scale, void *out, float *lse,
                        int32_t max_len, void *stream) {
  // Argument checks: the same function attn_decode uses.
  const int chk = kvq::check_decode_call(L, q, out, lse, max_len);
  if (chk != KVQ_OK) return chk;

  void *scratch = nullptr;
  int sms = 0;
  const int st = scratch_for_current_device(&scratch, &sms);
  if (st != KVQ_OK) return st;
  const kvq::DecodePlan pl = kvq::plan_decode(*L, max_len, sms);
  if (pl.ws_bytes > static_cast<int64_t>(kNoAllocScratchBytes)) return KVQ_EWORKSPACE;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The counter region at the start of the scratch must start at zero; the
  // previous call may have left anything there.
  if (cudaMemsetAsync(scratch, 0, static_cast<size_t>(kvq::kDecodeTicketBytes), s) !=
      cudaSuccess)
    return KVQ_ECUDA;
  const cudaError_t e = kvq::launch_decode(*L, pl, q, scale, out, lse, max_len, scratch, s);
  return e == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

}  // extern "C"
