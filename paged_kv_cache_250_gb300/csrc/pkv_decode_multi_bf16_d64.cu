// Multi-query decode kernels (several query tokens per sequence), bf16 cache,
// head_dim 64.
#include "pkv_decode_mq.cuh"

namespace pkv {
cudaError_t launch_decode_multi_bf16_d64(const DecodeLaunch& l) {
  return mq::dispatch_split_multi_d<kCacheBF16, true, 64>(l);
}
}  // namespace pkv
