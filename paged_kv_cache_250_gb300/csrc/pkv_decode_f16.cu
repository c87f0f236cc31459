// Split-K decode kernels for a f16 cache (q in f16).
#include "pkv_decode_impl.cuh"

namespace pkv {
cudaError_t launch_decode_f16(const DecodeLaunch& l) {
  if (l.q_bf16 != false) return cudaErrorNotSupported;
  return dispatch_split<kCacheF16, false>(l);
}
}  // namespace pkv
