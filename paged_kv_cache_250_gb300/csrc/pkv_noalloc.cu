// pkv_noalloc.cu -- decode attention for callers that cannot allocate device
// memory.
//
// pkv_paged_decode_attention needs a caller-provided workspace for its split
// partials and arrival counters.  Some callers have no way to provide one:
// code running where device allocation is forbidden or unavailable (inside a
// framework's custom-op hook with no allocator handle, plugins loaded into an
// engine that owns all device memory, or code paths that must not call
// cudaMalloc because it can synchronise the device).  This entry point runs
// the same kernel on a fixed scratch array that lives in the library's own
// device image, so it allocates nothing at call time.
#include <cuda_runtime.h>

#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

// The scratch every call of pkv_paged_decode_attention_noalloc uses.  Each
// GPU that loads the library holds these bytes until the process exits.
static __device__ __align__(256) unsigned char g_decode_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.  Host code only
// sees a stand-in for the symbol; its device address must be asked for once
// per device, with that device current.
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" pkv_status pkv_paged_decode_attention_noalloc(
    const pkv_cache_desc* desc, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, int32_t batch,
    int32_t max_blocks_per_seq, int32_t max_context_len_hint, float scale, void* out,
    pkv_dtype q_dtype, pkv_dtype out_dtype, pkv_stream_t stream) {
  if (batch == 0 || pkv_decode_workspace_bytes(desc, batch, max_blocks_per_seq,
                                               max_context_len_hint) == 0) {
    // nothing to do, or invalid arguments: the regular entry point returns
    // the precise status without launching anything
    return pkv_paged_decode_attention(desc, q, k_cache, v_cache, block_tables, context_lens,
                                      batch, max_blocks_per_seq, max_context_len_hint, scale,
                                      out, q_dtype, out_dtype, nullptr, 0, stream);
  }
  const size_t need =
      pkv_decode_workspace_bytes(desc, batch, max_blocks_per_seq, max_context_len_hint);
  if (need > (size_t)PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return PKV_ERR_CUDA;
  // every argument is checked before anything is put on the stream
  const pkv_status st = pkv::decode_validate(
      desc, q, k_cache, v_cache, block_tables, context_lens, batch, max_blocks_per_seq,
      max_context_len_hint, scale, out, q_dtype, out_dtype, scratch,
      (size_t)PKV_NOALLOC_SCRATCH_BYTES);
  if (st != PKV_OK) return st;
  // the arrival counters must start at zero whatever an earlier call left
  if (pkv::decode_workspace_clear(scratch, (size_t)PKV_NOALLOC_SCRATCH_BYTES, desc, batch,
                                  max_blocks_per_seq, max_context_len_hint,
                                  reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PKV_ERR_CUDA;
  return pkv_paged_decode_attention(desc, q, k_cache, v_cache, block_tables, context_lens,
                                    batch, max_blocks_per_seq, max_context_len_hint, scale, out,
                                    q_dtype, out_dtype, scratch,
                                    (size_t)PKV_NOALLOC_SCRATCH_BYTES, stream);
}
