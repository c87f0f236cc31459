// Split-combine and append/scatter kernels.
#include <math.h>

#include "pkv_decode_impl.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

// ---------------------------------------------------------------------------
// Split combine.  One CTA per (sequence, KV head); one thread per 4 output
// elements of one query head.  Merges the chunks' (m, l, o) by bringing each
// to the common maximum M with exp2(m - M) and dividing once by the merged
// sum ("KV Cache & FlashAttention" (deepforge.srivtx.xyz), running-summary
// paragraph; "KV Cache & Flash Attention." (kvcache-7e2.pages.dev), Flash
// Attention section, one division per output row).  Chunks with l == 0
// contribute nothing; a sequence with no tokens gets a zero row.
template <typename OutT>
__device__ __forceinline__ void store4(OutT* dst, float4 v);

template <>
__device__ __forceinline__ void store4<float>(float* dst, float4 v) {
  *reinterpret_cast<float4*>(dst) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* dst, float4 v) {
  uint2 u;
  u.x = pack2<true>(v.x, v.y);
  u.y = pack2<true>(v.z, v.w);
  *reinterpret_cast<uint2*>(dst) = u;
}
template <>
__device__ __forceinline__ void store4<__half>(__half* dst, float4 v) {
  uint2 u;
  u.x = pack2<false>(v.x, v.y);
  u.y = pack2<false>(v.z, v.w);
  *reinterpret_cast<uint2*>(dst) = u;
}

template <typename OutT>
__global__ void combine_kernel(const DecodeParams p, int G) {
  const int s = blockIdx.x;
  const int b = s / p.Hkv;
  const int h = s - b * p.Hkv;
  const int per_head = p.d >> 2;
  const int head = threadIdx.x / per_head;
  const int d0 = (threadIdx.x - head * per_head) * 4;
  if (head >= G) return;
  const int ctx = p.context_lens[b];
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (ctx > 0 && ctx <= p.MBS * kPageSize) {
    const int first = p.seg_info[2 * s];
    const int cnt = p.seg_info[2 * s + 1];
    float M = -INFINITY;
    for (int k = 0; k < cnt; ++k) {
      const float2 ml =
          *reinterpret_cast<const float2*>(p.part_ml + ((int64_t)(first + k) * G + head) * 2);
      if (ml.y > 0.f) M = fmaxf(M, ml.x);
    }
    if (M > -INFINITY) {
      float L = 0.f;
      for (int k = 0; k < cnt; ++k) {
        const int64_t c = (int64_t)(first + k) * G + head;
        const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + c * 2);
        if (!(ml.y > 0.f)) continue;
        const float w = exp2f(ml.x - M);
        L += w * ml.y;
        const float4 v = *reinterpret_cast<const float4*>(p.part_o + c * p.d + d0);
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
      }
      const float inv = 1.0f / L;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
    }
  }
  OutT* dst = reinterpret_cast<OutT*>(p.out) + ((int64_t)b * p.Hq + h * G + head) * p.d + d0;
  store4<OutT>(dst, acc);
}

cudaError_t launch_combine(const DecodeLaunch& l) {
  const int threads = l.group * (l.p.d / 4);
  const int blocks = l.p.B * l.p.Hkv;
  if (blocks == 0) return cudaSuccess;
  switch (l.out_dtype) {
    case PKV_F32:
      combine_kernel<float><<<blocks, threads, 0, l.stream>>>(l.p, l.group);
      break;
    case PKV_BF16:
      combine_kernel<__nv_bfloat16><<<blocks, threads, 0, l.stream>>>(l.p, l.group);
      break;
    case PKV_F16:
      combine_kernel<__half><<<blocks, threads, 0, l.stream>>>(l.p, l.group);
      break;
    default:
      return cudaErrorNotSupported;
  }
  return cudaGetLastError();
}

size_t decode_smem_bytes(int32_t d, CacheKind cache, int32_t B) {
  const int elem = cache == kCacheE4M3 ? 1 : 2;
  const int stage = 2 * kPageSize * d * elem;
  int stages = (96 * 1024) / (kDecodeWarps * stage);
  stages = stages < 2 ? 2 : (stages > 8 ? 8 : stages);
  size_t bytes = 1024;                                  // alignment slack
  bytes += decode_ring_bytes(stage, stages);            // K/V page ring
  bytes += (size_t)kDecodeWarps * stages * 8;           // mbarriers
  bytes += (size_t)kDecodeWarps * 64 * 16;              // descriptor windows
  bytes += (size_t)(2 * B + 1) * 4;                     // prefix sums + lengths
  return bytes;
}

// ---------------------------------------------------------------------------
// Append / scatter.  One thread moves 8 elements (16 bytes) of one (token,
// KV head) row of K and the same of V into slot_mapping[token]: block =
// slot / P, offset = slot % P ("KV Cache & Flash Attention."
// (kvcache-7e2.pages.dev), PagedAttention section).  Negative slots are
// skipped; slots past the pool are reported, never written.  For an E4M3
// cache each value is divided by its head's scale (IEEE fp32) and encoded
// round-to-nearest-even with saturation to +-448.
template <bool IN_BF16>
__device__ __forceinline__ uint2 quantize8(uint4 in, float scale) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
  uint32_t outw[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float2 a = unpack2<IN_BF16>(w[2 * i]);
    const float2 b = unpack2<IN_BF16>(w[2 * i + 1]);
    const uint16_t lo = f32x2_to_e4m3x2(__fdiv_rn(a.x, scale), __fdiv_rn(a.y, scale));
    const uint16_t hi = f32x2_to_e4m3x2(__fdiv_rn(b.x, scale), __fdiv_rn(b.y, scale));
    outw[i] = (uint32_t)lo | ((uint32_t)hi << 16);
  }
  return make_uint2(outw[0], outw[1]);
}

template <int CACHE, bool IN_BF16>
__global__ void append_kernel(const AppendParams a) {
  const int per_row = a.d >> 3;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t row = tid / per_row;
  if (row >= (int64_t)a.T * a.Hkv) return;
  const int part = (int)(tid - row * per_row);
  const int t = (int)(row / a.Hkv);
  const int h = (int)(row - (int64_t)t * a.Hkv);
  const int64_t slot = a.slot_mapping[t];
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
  if constexpr (CACHE != kCacheE4M3) {
    reinterpret_cast<uint4*>(a.k_cache)[dst] = kin;
    reinterpret_cast<uint4*>(a.v_cache)[dst] = vin;
  } else {
    reinterpret_cast<uint2*>(a.k_cache)[dst] = quantize8<IN_BF16>(kin, a.k_scale[h]);
    reinterpret_cast<uint2*>(a.v_cache)[dst] = quantize8<IN_BF16>(vin, a.v_scale[h]);
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
  } else {
    append_kernel<kCacheBF16, false><<<(unsigned)grid, block, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace pkv
