// pkv_internal.h -- host-side contract between the C-ABI layer (pkv_api.cu)
// and the kernel launchers.  Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

constexpr int kPageSize = 16;  // tokens per block: the only page size built
constexpr int kDecodeWarps = 4;
constexpr int kDecodeCtasPerSm = 2;

enum CacheKind { kCacheF16 = 0, kCacheBF16 = 1, kCacheE4M3 = 2 };

// Arguments of the split kernel (one warp = one contiguous share of all
// (sequence, KV head, page) units) and of the split-combine kernel.
struct DecodeParams {
  const void* q;               // [B][Hq][d]
  const int32_t* block_tables; // [B][MBS]
  const int32_t* context_lens; // [B]
  void* out;                   // [B][Hq][d]
  float* part_o;               // [chunks][G][d]   unnormalised partial outputs
  float* part_ml;              // [chunks][G][2]   (running max in log2 units, sum)
  int32_t* seg_info;           // [B*Hkv][2]       (first chunk id, chunk count)
  const float* k_scale;        // FP8 only
  const float* v_scale;        // FP8 only
  int32_t* err_word;
  int32_t B, Hq, Hkv, d, NB, MBS;
  int32_t num_warps_total;     // warps in the split launch
  float scale_log2;            // softmax scale * log2(e)
};

struct DecodeLaunch {
  DecodeParams p;
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  int32_t group;               // Hq / Hkv
  CacheKind cache;
  bool q_bf16;
  pkv_dtype out_dtype;
  int32_t ctas;
  cudaStream_t stream;
};

struct AppendParams {
  void* k_cache;
  void* v_cache;
  const int64_t* slot_mapping;
  const void* k;
  const void* v;
  const float* k_scale;
  const float* v_scale;
  int32_t* err_word;
  int32_t T, Hkv, d, NB;
};

// Dynamic shared memory the split kernel needs for a batch of B sequences.
size_t decode_smem_bytes(int32_t d, CacheKind cache, int32_t B);

// Returns a CUDA error (cudaSuccess when both kernels were enqueued) or
// cudaErrorNotSupported when no kernel is built for the combination.
cudaError_t launch_decode_f16(const DecodeLaunch& l);
cudaError_t launch_decode_bf16(const DecodeLaunch& l);
cudaError_t launch_decode_e4m3(const DecodeLaunch& l);
cudaError_t launch_combine(const DecodeLaunch& l);
cudaError_t launch_append(const AppendParams& a, CacheKind cache, bool in_bf16,
                          cudaStream_t stream);

}  // namespace pkv
