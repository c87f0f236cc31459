// Multi-query decode kernels (several query tokens per sequence), E4M3 (fp8)
// cache with per-head scales, fp16 q.
#include "pkv_decode_mq.cuh"

namespace pkv {
cudaError_t launch_decode_multi_e4m3_f16q(const DecodeLaunch& l) {
  if (l.p.d != 128) return cudaErrorNotSupported;
  return mq::dispatch_split_multi_d<kCacheE4M3, false, 128>(l);
}
}  // namespace pkv
