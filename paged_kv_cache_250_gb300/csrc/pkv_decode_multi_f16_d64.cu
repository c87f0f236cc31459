// Multi-query decode kernels (several query tokens per sequence), fp16 cache,
// head_dim 64.
#include "pkv_decode_mq.cuh"

namespace pkv {
cudaError_t launch_decode_multi_f16_d64(const DecodeLaunch& l) {
  return mq::dispatch_split_multi_d<kCacheF16, false, 64>(l);
}
}  // namespace pkv
