// kvq_noalloc.cu -- decode attention for callers that cannot allocate.
//
// Some callers cannot allocate device memory when they run decode: an
// application that must not call cudaMalloc/cudaFree after start-up (those
// calls may synchronize the device and can fail once memory is committed), or
// a plugin whose host framework owns all device memory and gives it no
// allocator.  kvq_decode_attention_noalloc serves them: its split-K scratch
// is a file-scope static device array, so the call needs no workspace.
//
// The array holds kNoAllocScratchBytes and stays resident on every GPU that
// loads this library until the process exits.  Every call shares it, and it
// keeps the last call's contents; the decode kernels write every partial they
// later read, so nothing needs clearing between calls.  Calls that overlap on
// the GPU (other streams, other host threads) race on the array.
#include <mutex>

#include "kvq_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)KVQ_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Host code must not use this name as a device address: it is a host-side
// stand-in.  Device addresses come from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, resolved once per
// device (on the first call made with that device current).
cudaError_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" kvq_status kvq_decode_attention_noalloc(kvq_cache* cache, int layer, const void* q_bf16,
                                                   int num_q_heads, const int32_t* page_table,
                                                   int max_pages_per_seq, const int32_t* seq_lens,
                                                   int batch, float sm_scale, void* out_bf16,
                                                   kvq_stream stream) {
  // A NULL cache, invalid sizes (INVALID_ARG) or an unsupported shape
  // (UNSUPPORTED) leave no workspace size; the workspace entry point, called
  // without one, validates the same arguments in the same order and returns
  // that status and message before any device work.
  const size_t need =
      cache ? kvq_decode_workspace_size(cache, batch, num_q_heads, max_pages_per_seq) : 0;
  if (need == 0)
    return kvq_decode_attention(cache, layer, q_bf16, num_q_heads, page_table, max_pages_per_seq,
                                seq_lens, batch, sm_scale, out_bf16, nullptr, 0, stream);
  if (need > kNoAllocScratchBytes) {
    kvq::set_error_message("kvq_decode_attention_noalloc: these sizes need %zu bytes of scratch, "
                          "more than its static %zu-byte array; use kvq_decode_attention with a "
                          "caller-provided workspace",
                          need, kNoAllocScratchBytes);
    return KVQ_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_on_current_device(&scratch);
  if (e != cudaSuccess) {
    kvq::set_error_message("kvq_decode_attention_noalloc: cudaGetSymbolAddress: %s",
                          cudaGetErrorString(e));
    return KVQ_ERR_CUDA;
  }
  return kvq_decode_attention(cache, layer, q_bf16, num_q_heads, page_table, max_pages_per_seq,
                              seq_lens, batch, sm_scale, out_bf16, scratch, kNoAllocScratchBytes,
                              stream);
}
