// Block copy for copy-on-write of shared prefixes.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

// One CTA copies one block of one cache (blockIdx.y: 0 = K, 1 = V; 2 = the
// block's per-token scales, when the cache has them) in 16-byte pieces; the
// copy streams (evict-first loads and stores), since nothing reads it back
// soon.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const CopyParams c) {
  const int i = blockIdx.x;
  const int32_t src = c.src[i], dst = c.dst[i];
  if (src < 0 || src >= c.NB || dst < 0 || dst >= c.NB) {
    if (threadIdx.x == 0 && blockIdx.y == 0) report_error(c.err_word, PKV_ERR_BOUNDS);
    return;
  }
  if (blockIdx.y == 2) {
    const int64_t n = c.scales_per_block;
    for (int64_t j = threadIdx.x; j < n; j += blockDim.x)
      c.scales[(int64_t)dst * n + j] = c.scales[(int64_t)src * n + j];
    return;
  }
  char* base = static_cast<char*>(blockIdx.y == 0 ? c.k_cache : c.v_cache);
  const uint4* from = reinterpret_cast<const uint4*>(base + (int64_t)src * c.block_bytes);
  uint4* to = reinterpret_cast<uint4*>(base + (int64_t)dst * c.block_bytes);
  const int64_t n16 = c.block_bytes / 16;
  for (int64_t j = threadIdx.x; j < n16; j += blockDim.x) __stcs(to + j, __ldcs(from + j));
}

cudaError_t launch_copy_blocks(const CopyParams& c, int32_t n, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  copy_blocks_kernel<<<dim3((unsigned)n, c.scales != nullptr ? 3 : 2), 256, 0, stream>>>(c);
  return cudaGetLastError();
}

}  // namespace pkv
