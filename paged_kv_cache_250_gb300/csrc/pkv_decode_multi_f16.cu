// Multi-query decode kernels (several query tokens per sequence), fp16 cache,
// head_dim 128; head_dim 64 is in pkv_decode_multi_f16_d64.cu.
#include "pkv_decode_mq.cuh"

namespace pkv {
cudaError_t launch_decode_multi_f16(const DecodeLaunch& l) {
  if (l.q_bf16 != false) return cudaErrorNotSupported;
  if (l.p.d == 64) return launch_decode_multi_f16_d64(l);
  if (l.p.d != 128) return cudaErrorNotSupported;
  return mq::dispatch_split_multi_d<kCacheF16, false, 128>(l);
}
}  // namespace pkv
