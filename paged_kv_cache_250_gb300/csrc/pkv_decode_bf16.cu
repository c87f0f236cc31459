// Split-K decode kernels for a bf16 cache (q in bf16).
#include "pkv_decode_impl.cuh"

namespace pkv {
cudaError_t launch_decode_bf16(const DecodeLaunch& l) {
  if (l.q_bf16 != true) return cudaErrorNotSupported;
  return dispatch_split<kCacheBF16, true>(l);
}
}  // namespace pkv
