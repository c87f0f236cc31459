// Split-K decode kernels, several query tokens per sequence, f16 cache.
#include "pkv_decode_impl.cuh"

namespace pkv {
cudaError_t launch_decode_multi_f16(const DecodeLaunch& l) {
  if (l.q_bf16 != false) return cudaErrorNotSupported;
  return dispatch_split_multi<kCacheF16, false>(l);
}
}  // namespace pkv
