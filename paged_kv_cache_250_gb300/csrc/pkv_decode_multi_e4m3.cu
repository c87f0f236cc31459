// Multi-query decode kernels (several query tokens per sequence), E4M3 (fp8)
// cache with per-head scales, bf16 q (used as fp16 in the contractions);
// fp16 q is in pkv_decode_multi_e4m3_f16q.cu.
#include "pkv_decode_mq.cuh"

namespace pkv {
cudaError_t launch_decode_multi_e4m3(const DecodeLaunch& l) {
  if (!l.q_bf16) return launch_decode_multi_e4m3_f16q(l);
  if (l.p.d != 128) return cudaErrorNotSupported;
  return mq::dispatch_split_multi_d<kCacheE4M3, true, 128>(l);
}
}  // namespace pkv
