// Split-K decode kernels, several query tokens per sequence, E4M3 (fp8)
// cache; q in fp16 or bf16 and used as fp16 in the contractions.
#include "pkv_decode_impl.cuh"

namespace pkv {
cudaError_t launch_decode_multi_e4m3(const DecodeLaunch& l) {
  return l.q_bf16 ? dispatch_split_multi<kCacheE4M3, true>(l)
                  : dispatch_split_multi<kCacheE4M3, false>(l);
}
}  // namespace pkv
