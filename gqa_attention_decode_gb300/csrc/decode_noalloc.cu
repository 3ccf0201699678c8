// decode_noalloc.cu -- gqa_attn_decode_noalloc: decode for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where they
// run attention: code running inside a custom allocator or memory pool that must
// not re-enter it, runtimes that forbid allocation after start-up, and hosts that
// simply have no allocator to hand.  gqa_attn_decode needs a caller-provided
// workspace for its per-split partials; this entry point instead uses a fixed
// scratch array that lives in the library's own static device memory.
//
// The array is reserved on every GPU that loads the library and stays reserved
// until the process exits.  Every call shares it, so calls whose GPU work
// overlaps (different streams, or different host threads on the same device)
// race on it and must be serialised by the caller.  The decode writes every
// partial it later reads within the same call, so nothing has to be cleared
// between calls.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/gqa_attn.h"

namespace {

// File-scope scratch: GQA_NOALLOC_SCRATCH_BYTES bytes, 256-byte aligned.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GQA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct NoallocDevice {
  bool ready = false;
  int num_sms = 0;
  void *scratch = nullptr;  // device address of g_noalloc_scratch on this device
};

std::mutex g_noalloc_mutex;
NoallocDevice g_noalloc_devices[kMaxDevices];

// Once per device, with that device current: look up the device address of the
// scratch array (the host-side name is only a stand-in) and the SM count.
int noalloc_setup(NoallocDevice **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoallocDevice &st = g_noalloc_devices[dev];
  if (!st.ready) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return GQA_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
      return GQA_ERR_CUDA;
    st.scratch = ptr;
    st.num_sms = sms;
    st.ready = true;
  }
  *out = &st;
  return GQA_OK;
}

}  // namespace

extern "C" GQA_API int gqa_attn_decode_noalloc(const gqa_bf16_t *q, const gqa_bf16_t *k_cache,
                                               const gqa_bf16_t *v_cache,
                                               const int32_t *seqlens, int B, int H_q, int H_kv,
                                               int S_max, int d, float scale, int num_splits,
                                               gqa_bf16_t *o, float *lse, gqa_stream_t stream) {
  if (B == 0) {
    return gqa_attn_decode(q, k_cache, v_cache, seqlens, B, H_q, H_kv, S_max, d, scale,
                           num_splits, o, lse, nullptr, 0, stream);
  }
  NoallocDevice *st = nullptr;
  int rc = noalloc_setup(&st);
  if (rc != GQA_OK) return rc;
  const size_t need =
      gqa_attn_decode_workspace_size(B, H_q, H_kv, S_max, d, st->num_sms, num_splits);
  if (need == 0) return GQA_ERR_INVALID_ARG;
  if (need > (size_t)GQA_NOALLOC_SCRATCH_BYTES) return GQA_ERR_WORKSPACE;
  return gqa_attn_decode(q, k_cache, v_cache, seqlens, B, H_q, H_kv, S_max, d, scale, num_splits,
                         o, lse, st->scratch, (size_t)GQA_NOALLOC_SCRATCH_BYTES, stream);
}
