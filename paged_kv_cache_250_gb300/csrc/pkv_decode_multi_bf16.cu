// Split-K decode kernels, several query tokens per sequence, bf16 cache.
#include "pkv_decode_impl.cuh"

namespace pkv {
cudaError_t launch_decode_multi_bf16(const DecodeLaunch& l) {
  if (l.q_bf16 != true) return cudaErrorNotSupported;
  return dispatch_split_multi<kCacheBF16, true>(l);
}
}  // namespace pkv
