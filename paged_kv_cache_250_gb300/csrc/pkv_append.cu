// Append/scatter kernel.
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

// ---------------------------------------------------------------------------
// Append / scatter.  One thread moves 8 elements (16 bytes) of one (token,
// KV head) row of K and the same of V into slot_mapping[token]: block =
// slot / P, offset = slot % P ("KV Cache & Flash Attention."
// (kvcache-7e2.pages.dev), PagedAttention section).  Negative slots are
// skipped; slots past the pool are reported, never written.  For an E4M3
// cache each value is divided by its head's scale (IEEE fp32) and encoded
// round-to-nearest-even with saturation to +-448.
// Largest magnitude of eight 16-bit values.
template <bool IN_BF16>
__device__ __forceinline__ float amax8(uint4 in) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = unpack2<IN_BF16>(w[i]);
    m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
  }
  return m;
}

template <int CACHE, bool IN_BF16>
__global__ void append_kernel(const AppendParams a) {
  // let a dependent decode kernel start its prologue while this one runs
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int per_row = a.d >> 3;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t row = tid / per_row;
  if (row >= (int64_t)a.T * a.Hkv) return;
  const int part = (int)(tid - row * per_row);
  const int t = (int)(row / a.Hkv);
  const int h = (int)(row - (int64_t)t * a.Hkv);
  int64_t slot;
  if (a.slot_mapping != nullptr) {
    slot = a.slot_mapping[t];
  } else {  // the newest position of sequence t (none when it is empty)
    const int c = a.context_lens[t];
    if (c <= 0 || c > a.MBS * kPageSize) return;  // lengths are checked by the attention
    const int blk = a.block_tables[(int64_t)t * a.MBS + (c - 1) / kPageSize];
    if (blk < 0 || blk >= a.NB) return;  // reported by the attention's own lookup
    slot = (int64_t)blk * kPageSize + (c - 1) % kPageSize;
  }
  if (slot < 0) return;
  if (slot >= (int64_t)a.NB * kPageSize) {
    if (part == 0) report_error(a.err_word, PKV_ERR_BOUNDS);
    return;
  }
  const int64_t blk = slot / kPageSize;
  const int64_t off = slot - blk * kPageSize;
  const int64_t dst = ((blk * a.Hkv + h) * kPageSize + off) * per_row + part;
  const uint4 kin = reinterpret_cast<const uint4*>(a.k)[row * per_row + part];
  const uint4 vin = reinterpret_cast<const uint4*>(a.v)[row * per_row + part];
  if constexpr (CACHE == kCacheE4M3) {
    reinterpret_cast<uint2*>(a.k_cache)[dst] = quantize8<IN_BF16>(kin, a.k_scale[h]);
    reinterpret_cast<uint2*>(a.v_cache)[dst] = quantize8<IN_BF16>(vin, a.v_scale[h]);
  } else if constexpr (CACHE == kCacheE4M3Tok) {
    // The row's own scale: its largest magnitude over 448 in IEEE fp32 (1 for
    // an all-zero row).  A row is the 16 lanes of one half-warp (d = 128).
    float ak = amax8<IN_BF16>(kin), av = amax8<IN_BF16>(vin);
    const unsigned half = 0xffffu << (threadIdx.x & 16);
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) {
      ak = fmaxf(ak, __shfl_xor_sync(half, ak, off));
      av = fmaxf(av, __shfl_xor_sync(half, av, off));
    }
    const float ks = ak > 0.f ? __fdiv_rn(ak, 448.f) : 1.f;
    const float vs = av > 0.f ? __fdiv_rn(av, 448.f) : 1.f;
    reinterpret_cast<uint2*>(a.k_cache)[dst] = quantize8<IN_BF16>(kin, ks);
    reinterpret_cast<uint2*>(a.v_cache)[dst] = quantize8<IN_BF16>(vin, vs);
    if (part == 0) {  // pool [NB][Hkv][2][P]: the page's K scales, then its V scales
      float* sp = a.scale_out + (blk * a.Hkv + h) * 2 * kPageSize + off;
      sp[0] = ks;
      sp[kPageSize] = vs;
    }
  } else {
    reinterpret_cast<uint4*>(a.k_cache)[dst] = kin;
    reinterpret_cast<uint4*>(a.v_cache)[dst] = vin;
  }
}

cudaError_t launch_append(const AppendParams& a, CacheKind cache, bool in_bf16,
                          cudaStream_t stream) {
  const int64_t threads_total = (int64_t)a.T * a.Hkv * (a.d / 8);
  if (threads_total == 0) return cudaSuccess;
  const int block = 256;
  const int64_t grid = (threads_total + block - 1) / block;
  if (grid > 0x7fffffff) return cudaErrorInvalidValue;
  if (cache == kCacheE4M3) {
    if (in_bf16)
      append_kernel<kCacheE4M3, true><<<(unsigned)grid, block, 0, stream>>>(a);
    else
      append_kernel<kCacheE4M3, false><<<(unsigned)grid, block, 0, stream>>>(a);
  } else if (cache == kCacheE4M3Tok) {
    if (a.d != 128) return cudaErrorNotSupported;  // a row is one half-warp
    if (in_bf16)
      append_kernel<kCacheE4M3Tok, true><<<(unsigned)grid, block, 0, stream>>>(a);
    else
      append_kernel<kCacheE4M3Tok, false><<<(unsigned)grid, block, 0, stream>>>(a);
  } else {
    append_kernel<kCacheBF16, false><<<(unsigned)grid, block, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace pkv
