// Multi-query decode kernels (q_len > 1 per sequence) for an E4M3 cache with
// one fp32 scale per (token, KV head) for K and for V, bf16 q; fp16 q is in
// pkv_decode_multi_e4m3_tok_f16q.cu.
#include "pkv_decode_mq.cuh"

namespace pkv {
cudaError_t launch_decode_multi_e4m3_tok(const DecodeLaunch& l) {
  if (!l.q_bf16) return launch_decode_multi_e4m3_tok_f16q(l);
  if (l.p.d != 128) return cudaErrorNotSupported;
  return mq::dispatch_split_multi_d<kCacheE4M3Tok, true, 128>(l);
}
}  // namespace pkv
