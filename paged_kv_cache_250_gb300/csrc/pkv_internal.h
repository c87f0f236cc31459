// pkv_internal.h -- host-side contract between the C-ABI layer (pkv_api.cu)
// and the kernel launchers.  Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

constexpr int kPageSize = 16;  // tokens per block: the only page size built
constexpr int kDecodeWarps = 4;     // warps per CTA of the 16-bit and multi-query kernels
constexpr int kDecodeWarpsFp8 = 6;  // of the single-token E4M3 kernel (more warps hide
                                    // the latency of the byte-to-fp16 conversions)
constexpr int kDecodeCtasPerSm = 2;

// E4M3: one fp32 scale per KV head; E4M3 per token: one K and one V scale per
// (block, KV head, slot), in one pool [NB][Hkv][2][P] (a page's 16 K scales,
// then its 16 V scales: one 128-byte line).
enum CacheKind { kCacheF16 = 0, kCacheBF16 = 1, kCacheE4M3 = 2, kCacheE4M3Tok = 3 };
__host__ __device__ constexpr bool cache_is_fp8(CacheKind c) { return c == kCacheE4M3 || c == kCacheE4M3Tok; }

// A CTA's share holds at least about kRangeMin cost units (fewer CTAs run
// when the batch is small: a short context is not worth splitting) and is
// walked in pieces of at most kRangeMax pages.
constexpr int kRangeMin = 32;
constexpr int kRangeMax = 64;
// Cost of starting a (sequence, KV head) segment, in pages, when shares are
// cut (a state merge, an output write and a pipeline refill).
constexpr int kSegCost = 12;

// Shared-memory plan of the single-token decode kernel (pkv_decode_impl.cuh;
// host and device agree on it).
__host__ __device__ constexpr int decode_warps(CacheKind c) {
  return cache_is_fp8(c) ? kDecodeWarpsFp8 : kDecodeWarps;
}
// page descriptors per warp: two pieces of at most ceil(kRangeMax / warps)
// pages each, rounded up to a power of two
__host__ __device__ constexpr int decode_desc_ring(int nw) { return nw <= 4 ? 64 : 32; }
__host__ __device__ constexpr int decode_lane_state(int d) { return 4 + 4 * (d / 16); }
// merge buffer (floats): two whole warp states for the barrier tree, or the
// compact states (two column pairs each) of all warps but one for the
// asynchronous hand-off
__host__ __device__ constexpr int decode_mbuf_floats(int d, int nw) {
  return 2 * decode_lane_state(d) * 32 > (nw - 1) * decode_lane_state(d) * 16
             ? 2 * decode_lane_state(d) * 32
             : (nw - 1) * decode_lane_state(d) * 16;
}
__host__ __device__ constexpr int decode_stage_bytes(int d, CacheKind c) {
  return 2 * kPageSize * d * (cache_is_fp8(c) ? 1 : 2);
}
// per-token scales of one staged page (K then V), kept beside the page ring
__host__ __device__ constexpr int decode_scale_bytes(CacheKind c) {
  return c == kCacheE4M3Tok ? 2 * kPageSize * 4 : 0;
}
// alignment slack + descriptor rings + merge buffers + merge flags +
// mbarriers (8 stages max per warp, 4 slots for the flush hand-off)
__host__ __device__ constexpr int decode_fixed_smem(int d, CacheKind c) {
  return 1024 + decode_warps(c) * decode_desc_ring(decode_warps(c)) * 8 +
         decode_mbuf_floats(d, decode_warps(c)) * 4 + 2 * decode_warps(c) * 4 +
         decode_warps(c) * 8 * 8 + 32;
}
// Ring depth: as many K+V page slots per warp as fit two CTAs per SM (228 KB
// per SM, 1 KB reserved per CTA) with room for the per-sequence arrays of a
// 128-sequence batch; between 2 and 8.
constexpr int kDecodeSmemTarget = 113 * 1024;
__host__ __device__ constexpr int decode_clamp_stages(int s) { return s < 2 ? 2 : (s > 8 ? 8 : s); }
__host__ __device__ constexpr int decode_stages(int d, CacheKind c) {
  return decode_clamp_stages((kDecodeSmemTarget - decode_fixed_smem(d, c) - 2600) /
                             (decode_warps(c) * (decode_stage_bytes(d, c) + decode_scale_bytes(c))));
}

// Columns of the multi-query kernel (pkv_decode_mq.cuh) built for nc (query
// token, head) pairs per KV head (nc = group x query tokens, a power of two
// from 2 to 64): MMA column groups of 8, cw of them per warp, and sl warps
// ("slices") that compute disjoint column ranges of every page; the other
// kDecodeWarps / sl warps of a slice share its pages.
__host__ __device__ constexpr int mq_cw(int nc) { return nc <= 8 ? 1 : 2; }
__host__ __device__ constexpr int mq_sl(int nc) { return nc <= 16 ? 1 : nc / 16; }
// columns a partial slot holds (at least 8, whatever the call)
__host__ __device__ constexpr int decode_part_cols(int nc) { return nc < 8 ? 8 : nc; }
// floats of one warp's online-softmax state per lane: (m, l) for two
// columns and O^T fragments, per column group
__host__ __device__ constexpr int mq_lane_state(int d, int nc) {
  return mq_cw(nc) * (4 + 4 * (d / 16));
}
// merge buffers: two warp states (none when every warp owns its columns)
__host__ __device__ constexpr int mq_mbuf_bytes(int d, int nc) {
  return mq_sl(nc) == kDecodeWarps ? 0 : 2 * mq_lane_state(d, nc) * 32 * 4;
}
constexpr int kDescN = 128;      // page descriptors (int4) in the CTA's ring
constexpr int kDescBlock = 32;   // descriptors written by one fill (one per lane)
constexpr int kSmemInts = 96;    // flags, counters, merge flags, ordinal issued per slot
constexpr int kFlushBars = 16;   // mbarriers of the segment-end hand-off
// bytes per ring slot: the K and V page, their per-token scales, the slot's
// mbarrier and its pending-consumer count
__host__ __device__ constexpr int mq_slot_bytes(int d, CacheKind c) {
  return decode_stage_bytes(d, c) + decode_scale_bytes(c) + 8 + 4;
}
__host__ __device__ constexpr int mq_fixed_smem(int d, int nc) {
  return 1024 + kFlushBars * 8 + 16 + kDescN * 16 + mq_mbuf_bytes(d, nc) + kSmemInts * 4;
}
// Ring slots of a CTA: as many K+V pages as fit two CTAs per SM with room for
// the per-sequence arrays of a 128-sequence batch; between 4 and 28.
__host__ __device__ constexpr int mq_clamp_ring(int r) { return r < 4 ? 4 : (r > 28 ? 28 : r); }
__host__ __device__ constexpr int mq_ring(int d, CacheKind c, int nc) {
  return mq_clamp_ring((kDecodeSmemTarget - mq_fixed_smem(d, nc) - 2600) / mq_slot_bytes(d, c));
}

// Arguments of the decode kernel (one CTA = one contiguous share of all
// (sequence, KV head, page) units; split partials merged in-kernel).
struct DecodeParams {
  const void* q;               // [B][Hq][d]
  const int32_t* block_tables; // [B][MBS]
  const int32_t* context_lens; // [B]
  void* out;                   // [B][Hq][d]
  float* part_o;               // [max ctas+B*Hkv][cols][d] unnormalised partial outputs
  float* part_ml;              // [max ctas+B*Hkv][cols][2] (reference max in log2 units, sum)
  int32_t* tickets;            // [B*Hkv]  pages stored per segment (x slices); zero between calls
  const float* k_scale;        // FP8 only
  const float* v_scale;        // FP8 only
  int32_t* err_word;
  int32_t B, Hq, Hkv, d, NB, MBS;
  pkv_dtype out_dtype;
  int32_t qlen;                // query tokens per sequence (q, out are [B][qlen][Hq][d])
  const void* k_new;           // fused append: new K rows [B][Hkv][d] (NULL: none)
  const void* v_new;           // fused append: new V rows
  void* k_cache;               // the caches (pages prefetched into L2; fused append writes)
  void* v_cache;
  int32_t kv_bf16;             // fused append: k_new / v_new are bf16 (else fp16)
  int32_t window;              // > 0: query at position t sees t - window + 1 .. t (and sinks)
  int32_t sinks;               // with a window: positions 0 .. sinks - 1 stay visible
  int32_t early_prologue;      // 1: read lengths/tables before waiting on the previous kernel
  int32_t trigger_next;        // 1: let the next kernel on the stream launch at once
  float scale_log2;            // softmax scale * log2(e)
};

struct DecodeLaunch {
  DecodeParams p;
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  int32_t group;               // Hq / Hkv
  int32_t qcap;                // query tokens the kernel is built for (>= p.qlen; 1, 2, 4, 8)
  CacheKind cache;
  bool q_bf16;
  int32_t ctas;
  cudaStream_t stream;
};

struct AppendParams {
  void* k_cache;
  void* v_cache;
  const int64_t* slot_mapping;   // NULL: token t goes to position context_lens[t] - 1
  const int32_t* block_tables;   // of sequence t, through its block table
  const int32_t* context_lens;
  int32_t MBS;
  float* scale_out;              // E4M3 per token: the scale pool [NB][Hkv][2][P] the
                                 // rows' scales go to (NULL otherwise)
  const void* k;
  const void* v;
  const float* k_scale;
  const float* v_scale;
  int32_t* err_word;
  int32_t T, Hkv, d, NB;
};

// Dynamic shared memory the single-token kernel needs for a batch of B
// sequences.
// The "deep" form of the per-token E4M3 kernel: its segment ends go through
// the barrier tree (two whole warp states in the merge buffer instead of the
// others' compact states), which leaves room for one more page slot per warp
// (four instead of three) when the batch's per-sequence arrays are small
// (up to about 100 sequences at d 128).
__host__ __device__ constexpr int decode_fixed_smem_deep(int d, CacheKind c) {
  return 1024 + decode_warps(c) * decode_desc_ring(decode_warps(c)) * 8 +
         2 * decode_lane_state(d) * 32 * 4 + 2 * decode_warps(c) * 4 + decode_warps(c) * 8 * 8 +
         32;
}
__host__ __device__ constexpr int decode_stages_deep(int d, CacheKind c) {
  return decode_clamp_stages((kDecodeSmemTarget - decode_fixed_smem_deep(d, c)) /
                             (decode_warps(c) * (decode_stage_bytes(d, c) + decode_scale_bytes(c))));
}
inline size_t decode_smem_bytes_form(int32_t d, CacheKind cache, int32_t B, bool deep) {
  return (size_t)(deep ? decode_fixed_smem_deep(d, cache) : decode_fixed_smem(d, cache)) +
         (size_t)decode_warps(cache) * (deep ? decode_stages_deep(d, cache) : decode_stages(d, cache)) *
             (decode_stage_bytes(d, cache) + decode_scale_bytes(cache)) +
         (size_t)(5 * B + 2) * 4;
}
// whether a single-token launch of B sequences takes the deep form
inline bool decode_use_deep(int32_t d, CacheKind cache, int32_t B) {
  return cache == kCacheE4M3Tok && decode_stages_deep(d, cache) > decode_stages(d, cache) &&
         decode_smem_bytes_form(d, cache, B, true) <= (size_t)kDecodeSmemTarget;
}
inline size_t decode_smem_bytes(int32_t d, CacheKind cache, int32_t B) {
  return decode_smem_bytes_form(d, cache, B, decode_use_deep(d, cache, B));
}
// The same for the multi-query kernel built for nc columns.
inline size_t mq_smem_bytes(int32_t d, CacheKind cache, int32_t B, int32_t nc) {
  return (size_t)mq_fixed_smem(d, nc) + (size_t)mq_ring(d, cache, nc) * mq_slot_bytes(d, cache) +
         (size_t)(5 * B + 2) * 4;
}

// Returns a CUDA error (cudaSuccess when the kernel was enqueued) or
// cudaErrorNotSupported when no kernel is built for the combination.
cudaError_t launch_decode_f16(const DecodeLaunch& l);
cudaError_t launch_decode_bf16(const DecodeLaunch& l);
cudaError_t launch_decode_e4m3(const DecodeLaunch& l);
cudaError_t launch_decode_e4m3_tok(const DecodeLaunch& l);
cudaError_t launch_decode_multi_f16(const DecodeLaunch& l);
cudaError_t launch_decode_multi_bf16(const DecodeLaunch& l);
cudaError_t launch_decode_multi_e4m3(const DecodeLaunch& l);
cudaError_t launch_decode_multi_e4m3_tok(const DecodeLaunch& l);
cudaError_t launch_decode_multi_f16_d64(const DecodeLaunch& l);
cudaError_t launch_decode_multi_bf16_d64(const DecodeLaunch& l);
cudaError_t launch_decode_multi_e4m3_f16q(const DecodeLaunch& l);
cudaError_t launch_decode_multi_e4m3_tok_f16q(const DecodeLaunch& l);
// The argument checks of pkv_paged_decode_attention, with nothing launched.
pkv_status decode_validate(const pkv_cache_desc* desc, const void* q, const void* k_cache,
                           const void* v_cache, const int32_t* block_tables,
                           const int32_t* context_lens, int32_t batch, int32_t max_blocks_per_seq,
                           int32_t max_context_len_hint, float scale, const void* out,
                           pkv_dtype q_dtype, pkv_dtype out_dtype, const void* workspace,
                           size_t workspace_bytes);
// Clears, on the stream, the parts of a decode workspace that must be zero
// when a call begins (whatever an earlier, failed call left there).
cudaError_t decode_workspace_clear(void* workspace, size_t workspace_bytes,
                                   const pkv_cache_desc* d, int32_t batch, int32_t mbs,
                                   int32_t hint, cudaStream_t stream);

cudaError_t launch_append(const AppendParams& a, CacheKind cache, bool in_bf16,
                          cudaStream_t stream);

struct CopyParams {
  void* k_cache;
  void* v_cache;
  const int32_t* src;
  const int32_t* dst;
  int32_t* err_word;
  int64_t block_bytes;  // one block of one cache: Hkv * P * d * element bytes
  int32_t NB;
  float* scales;        // E4M3 per token: the scale pool, copied with its block
  int32_t scales_per_block;  // Hkv * 2 * P
};

cudaError_t launch_copy_blocks(const CopyParams& c, int32_t n, cudaStream_t stream);

// Paged prefill (pkv_prefill.cu): one CTA per 256 query rows, 256 / g new
// tokens of one sequence times the g query heads of one KV head.
struct PrefillParams {
  const int32_t* q_start;       // [B+1] first query row of each sequence
  const int32_t* context_lens;  // [B]
  const int32_t* block_tables;  // [B][MBS]
  void* out;                    // [total_q][Hq][d]
  int32_t* err_word;
  int32_t B, Hq, Hkv, NB, MBS, total_q, tiles_per_seq;
  pkv_dtype out_dtype;
  float scale_log2;
};
struct PrefillLaunch {
  PrefillParams p;
  CUtensorMap tmap_q;  // [total_q][Hq][d], boxes of 128 / g tokens x g heads x 64
  CUtensorMap tmap_k;  // the cache maps of the decode kernel
  CUtensorMap tmap_v;
  bool bf16;
  int32_t d;           // head dim: 64 or 128
  cudaStream_t stream;
};
size_t prefill_smem_bytes(int d);
cudaError_t launch_prefill(const PrefillLaunch& l);

}  // namespace pkv
