// Multi-query decode kernels (q_len > 1 per sequence) for an E4M3 cache with
// one fp32 scale per (token, KV head) for K and for V; q in fp16 or bf16.
#include "pkv_decode_impl.cuh"

namespace pkv {
cudaError_t launch_decode_multi_e4m3_tok(const DecodeLaunch& l) {
  return l.q_bf16 ? dispatch_split_multi<kCacheE4M3Tok, true>(l)
                  : dispatch_split_multi<kCacheE4M3Tok, false>(l);
}
}  // namespace pkv
