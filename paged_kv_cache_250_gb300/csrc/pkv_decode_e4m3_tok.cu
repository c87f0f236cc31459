// Split-K decode kernels for an E4M3 (fp8) cache with one fp32 scale per
// (token, KV head) for K and for V; q in fp16 or bf16 and used as fp16 in the
// tensor-core contractions.
#include "pkv_decode_impl.cuh"

namespace pkv {
cudaError_t launch_decode_e4m3_tok(const DecodeLaunch& l) {
  return l.q_bf16 ? dispatch_split<kCacheE4M3Tok, true>(l)
                  : dispatch_split<kCacheE4M3Tok, false>(l);
}
}  // namespace pkv
