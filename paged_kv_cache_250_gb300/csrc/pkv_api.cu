// pkv_api.cu -- the C ABI (include/pkv.h): argument validation, launch
// sizing, tensor-map encoding and kernel dispatch.  No allocation, no
// synchronisation, no state beyond a per-device SM-count cache.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

using pkv::kPageSize;

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

int sm_count_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  if (dev < kMaxDevices) {
    int cached = g_sm_count[dev].load(std::memory_order_relaxed);
    if (cached > 0) return cached;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return -1;
  if (dev < kMaxDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
  return n;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shape checks shared by both calls.
pkv_status check_desc(const pkv_cache_desc* d) {
  if (d == nullptr || d->struct_size != sizeof(pkv_cache_desc)) return PKV_ERR_INVALID_ARG;
  if (d->num_blocks <= 0 || d->page_size <= 0 || d->num_kv_heads <= 0 ||
      d->num_q_heads <= 0 || d->head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  if (d->num_q_heads % d->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if (d->page_size != kPageSize) return PKV_ERR_UNSUPPORTED;
  const int g = d->num_q_heads / d->num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return PKV_ERR_UNSUPPORTED;
  switch (d->cache_dtype) {
    case PKV_F16:
    case PKV_BF16:
      if (d->head_dim != 64 && d->head_dim != 128) return PKV_ERR_UNSUPPORTED;
      break;
    case PKV_FP8_E4M3:
    case PKV_FP8_E4M3_TOKEN:
      if (d->head_dim != 128) return PKV_ERR_UNSUPPORTED;
      if (d->k_scale == nullptr) return PKV_ERR_INVALID_ARG;
      if (d->cache_dtype == PKV_FP8_E4M3 && d->v_scale == nullptr) return PKV_ERR_INVALID_ARG;
      // per token: one pool, a page's scales copied as one 128-byte line
      if (d->cache_dtype == PKV_FP8_E4M3_TOKEN && !aligned(d->k_scale, 128))
        return PKV_ERR_INVALID_ARG;
      break;
    default:
      return PKV_ERR_UNSUPPORTED;
  }
  const int64_t rows = (int64_t)d->num_blocks * d->num_kv_heads * d->page_size;
  if (rows >= (int64_t)1 << 31) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

pkv::CacheKind kind_of(pkv_dtype t) {
  switch (t) {
    case PKV_FP8_E4M3: return pkv::kCacheE4M3;
    case PKV_FP8_E4M3_TOKEN: return pkv::kCacheE4M3Tok;
    case PKV_BF16: return pkv::kCacheBF16;
    default: return pkv::kCacheF16;
  }
}
bool is_fp8(pkv_dtype t) { return t == PKV_FP8_E4M3 || t == PKV_FP8_E4M3_TOKEN; }

struct WsLayout {
  size_t ml_off, o_off, ticket_bytes, total;
  int ctas;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace: from the front, the split partials (one slot per CTA of the
// largest grid plus one per segment, slot cta + seg, each with room for the
// (query token, head) columns of a group: 8, or group x query tokens when
// that is more); at the very end of the caller's buffer, one page ticket per
// segment.  Only the tickets must be zero when a call starts, and a completed
// call leaves them at zero.  The partials' size grows with the batch and the
// columns and the tickets sit at the end, so a workspace sized for batch B
// and q_len Q serves every call with the same descriptor, a batch of at most
// B and at most Q query tokens: a smaller call's tickets are the tail of a
// larger call's, and no call's partials reach the tickets of any such call.
int nc_of(const pkv_cache_desc* d, int32_t qlen) {
  const int g = d->num_q_heads / d->num_kv_heads;
  const int qc = qlen <= 1 ? 1 : (qlen <= 2 ? 2 : (qlen <= 4 ? 4 : 8));
  return g * qc;
}
WsLayout ws_layout(const pkv_cache_desc* d, int32_t batch, int32_t mbs, int32_t hint,
                   int num_sms, int nc) {
  const int64_t g = pkv::decode_part_cols(nc);
  const int64_t cap = (int64_t)mbs * kPageSize;
  const int64_t len = (hint > 0 && hint < cap) ? hint : cap;
  const int64_t np_max = (len + kPageSize - 1) / kPageSize;
  const int64_t segs = (int64_t)batch * d->num_kv_heads;
  const int64_t pages_bound = segs * np_max;
  // at least eight pages per CTA (two per warp of a four-warp CTA); at most
  // kDecodeCtasPerSm CTAs per SM
  int64_t ctas = (pages_bound + 2 * pkv::kDecodeWarps - 1) / (2 * pkv::kDecodeWarps);
  const int64_t max_ctas = (int64_t)num_sms * pkv::kDecodeCtasPerSm;
  if (ctas > max_ctas) ctas = max_ctas;
  if (ctas < 1) ctas = 1;
  const int64_t slots = max_ctas + segs;
  WsLayout w;
  w.ctas = (int)ctas;
  w.ml_off = 0;
  w.o_off = align256(w.ml_off + (size_t)slots * g * 2 * sizeof(float));
  w.ticket_bytes = (size_t)segs * sizeof(int32_t);
  w.total = align256(w.o_off + (size_t)slots * g * d->head_dim * sizeof(float) + w.ticket_bytes);
  return w;
}

// The tickets of a call: the last ticket_bytes of the caller's buffer.
size_t ticket_offset(size_t workspace_bytes, const WsLayout& w) {
  return (workspace_bytes & ~(size_t)3) - w.ticket_bytes;
}

}  // namespace

namespace pkv {
cudaError_t decode_workspace_clear(void* workspace, size_t workspace_bytes,
                                   const pkv_cache_desc* d, int32_t batch, int32_t mbs,
                                   int32_t hint, cudaStream_t stream) {
  int sms = 0, dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const WsLayout w = ws_layout(d, batch, mbs, hint, sms, nc_of(d, 1));
  char* ws = static_cast<char*>(workspace);
  return cudaMemsetAsync(ws + ticket_offset(workspace_bytes, w), 0, w.ticket_bytes, stream);
}
}  // namespace pkv

namespace {

pkv_status encode_cache_map(CUtensorMap* map, const void* cache, const pkv_cache_desc* d) {
  auto fn = encode_fn();
  if (fn == nullptr) return PKV_ERR_CUDA;
  const bool fp8 = is_fp8(d->cache_dtype);
  const cuuint64_t elem = fp8 ? 1 : 2;
  const cuuint64_t dims[2] = {(cuuint64_t)d->head_dim,
                              (cuuint64_t)d->num_blocks * d->num_kv_heads * d->page_size};
  const cuuint64_t strides[1] = {(cuuint64_t)d->head_dim * elem};
  const cuuint32_t box[2] = {(cuuint32_t)(128 / elem), (cuuint32_t)d->page_size};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                  const_cast<void*>(cache), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status append_checks(const pkv_cache_desc* desc, const void* k_cache, const void* v_cache,
                         const int64_t* slot_mapping, const void* k, const void* v,
                         int32_t num_tokens, pkv_dtype kv_dtype) {
  if (!k_cache || !v_cache || !slot_mapping || !k || !v) return PKV_ERR_INVALID_ARG;
  if (kv_dtype != PKV_F16 && kv_dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
  if (!is_fp8(desc->cache_dtype) && kv_dtype != desc->cache_dtype)
    return PKV_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k, 16) || !aligned(v, 16) ||
      !aligned(slot_mapping, 8))
    return PKV_ERR_INVALID_ARG;
  (void)num_tokens;
  return PKV_OK;
}

pkv_status decode_checks(const pkv_cache_desc* desc, const void* q, const void* k_cache,
                         const void* v_cache, const int32_t* block_tables,
                         const int32_t* context_lens, int32_t batch, int32_t max_blocks_per_seq,
                         int32_t max_context_len_hint, float scale, const void* out,
                         pkv_dtype q_dtype, pkv_dtype out_dtype, const void* workspace,
                         size_t workspace_bytes, int32_t qlen = 1) {
  pkv_status st = check_desc(desc);
  if (st != PKV_OK) return st;
  if (batch < 0 || max_blocks_per_seq <= 0 || max_context_len_hint < 0)
    return PKV_ERR_INVALID_ARG;
  if (batch == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return PKV_ERR_INVALID_ARG;
  if ((int64_t)batch * max_blocks_per_seq >= ((int64_t)1 << 31)) return PKV_ERR_UNSUPPORTED;
  if ((int64_t)max_blocks_per_seq * kPageSize >= ((int64_t)1 << 31)) return PKV_ERR_UNSUPPORTED;
  if (q_dtype != PKV_F16 && q_dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
  if (!is_fp8(desc->cache_dtype) && q_dtype != desc->cache_dtype)
    return PKV_ERR_INVALID_ARG;
  if (out_dtype != PKV_F16 && out_dtype != PKV_BF16 && out_dtype != PKV_F32)
    return PKV_ERR_UNSUPPORTED;
  if (!(scale == scale)) return PKV_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4))
    return PKV_ERR_INVALID_ARG;
  if (qlen < 1 || qlen > 8) return PKV_ERR_UNSUPPORTED;
  const pkv::CacheKind cache = kind_of(desc->cache_dtype);
  const int nc = nc_of(desc, qlen);
  const size_t smem = qlen == 1 ? pkv::decode_smem_bytes(desc->head_dim, cache, batch)
                                 : pkv::mq_smem_bytes(desc->head_dim, cache, batch, nc);
  if (smem > 227 * 1024) return PKV_ERR_UNSUPPORTED;
  const int sms = sm_count_current_device();
  if (sms <= 0) return PKV_ERR_CUDA;
  const WsLayout w = ws_layout(desc, batch, max_blocks_per_seq, max_context_len_hint, sms, nc);
  if (workspace == nullptr || workspace_bytes < w.total || !aligned(workspace, 256))
    return PKV_ERR_WORKSPACE;
  return PKV_OK;
}

}  // namespace

namespace pkv {
pkv_status decode_validate(const pkv_cache_desc* desc, const void* q, const void* k_cache,
                           const void* v_cache, const int32_t* block_tables,
                           const int32_t* context_lens, int32_t batch, int32_t max_blocks_per_seq,
                           int32_t max_context_len_hint, float scale, const void* out,
                           pkv_dtype q_dtype, pkv_dtype out_dtype, const void* workspace,
                           size_t workspace_bytes) {
  return decode_checks(desc, q, k_cache, v_cache, block_tables, context_lens, batch,
                       max_blocks_per_seq, max_context_len_hint, scale, out, q_dtype, out_dtype,
                       workspace, workspace_bytes);
}
}  // namespace pkv

namespace {

pkv_status decode_impl(const pkv_cache_desc* desc, const void* q, const void* k_cache,
                       const void* v_cache, const int32_t* block_tables,
                       const int32_t* context_lens, int32_t batch, int32_t max_blocks_per_seq,
                       int32_t max_context_len_hint, float scale, void* out, pkv_dtype q_dtype,
                       pkv_dtype out_dtype, void* workspace, size_t workspace_bytes,
                       pkv_stream_t stream, int early_prologue, int32_t qlen = 1,
                       int32_t window = 0, int32_t sinks = 0, const void* k_new = nullptr,
                       const void* v_new = nullptr, pkv_dtype kv_dtype = PKV_BF16,
                       int trigger_next = 0) {
  pkv_status st = decode_checks(desc, q, k_cache, v_cache, block_tables, context_lens, batch,
                                max_blocks_per_seq, max_context_len_hint, scale, out, q_dtype,
                                out_dtype, workspace, workspace_bytes, qlen);
  if (st != PKV_OK || batch == 0) return st;
  const int sms = sm_count_current_device();
  const WsLayout w =
      ws_layout(desc, batch, max_blocks_per_seq, max_context_len_hint, sms, nc_of(desc, qlen));
  pkv::DecodeLaunch l;
  st = encode_cache_map(&l.tmap_k, k_cache, desc);
  if (st != PKV_OK) return st;
  st = encode_cache_map(&l.tmap_v, v_cache, desc);
  if (st != PKV_OK) return st;
  char* ws = static_cast<char*>(workspace);
  l.p.q = q;
  l.p.block_tables = block_tables;
  l.p.context_lens = context_lens;
  l.p.out = out;
  l.p.tickets = reinterpret_cast<int32_t*>(ws + ticket_offset(workspace_bytes, w));
  l.p.part_ml = reinterpret_cast<float*>(ws + w.ml_off);
  l.p.part_o = reinterpret_cast<float*>(ws + w.o_off);
  l.p.k_scale = desc->k_scale;
  l.p.v_scale = desc->v_scale;
  l.p.err_word = desc->err_word;
  l.p.B = batch;
  l.p.Hq = desc->num_q_heads;
  l.p.Hkv = desc->num_kv_heads;
  l.p.d = desc->head_dim;
  l.p.NB = desc->num_blocks;
  l.p.MBS = max_blocks_per_seq;
  l.p.out_dtype = out_dtype;
  l.p.early_prologue = early_prologue;
  l.p.trigger_next = trigger_next;
  l.p.qlen = qlen;
  l.p.window = window;
  l.p.k_new = k_new;
  l.p.v_new = v_new;
  l.p.k_cache = const_cast<void*>(k_cache);
  l.p.v_cache = const_cast<void*>(v_cache);
  l.p.kv_bf16 = kv_dtype == PKV_BF16 ? 1 : 0;
  l.p.sinks = window > 0 ? sinks : 0;
  l.p.scale_log2 = scale * 1.4426950408889634f;
  l.group = desc->num_q_heads / desc->num_kv_heads;
  // query-token capacity of the kernel: 1, or the smallest of 2, 4, 8 that
  // holds qlen
  l.qcap = nc_of(desc, qlen) / l.group;
  l.cache = kind_of(desc->cache_dtype);
  l.q_bf16 = (q_dtype == PKV_BF16);
  l.ctas = w.ctas;
  l.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (l.qcap == 1) {
    switch (l.cache) {
      case pkv::kCacheF16: e = pkv::launch_decode_f16(l); break;
      case pkv::kCacheBF16: e = pkv::launch_decode_bf16(l); break;
      case pkv::kCacheE4M3: e = pkv::launch_decode_e4m3(l); break;
      default: e = pkv::launch_decode_e4m3_tok(l); break;
    }
  } else {
    switch (l.cache) {
      case pkv::kCacheF16: e = pkv::launch_decode_multi_f16(l); break;
      case pkv::kCacheBF16: e = pkv::launch_decode_multi_bf16(l); break;
      case pkv::kCacheE4M3: e = pkv::launch_decode_multi_e4m3(l); break;
      default: e = pkv::launch_decode_multi_e4m3_tok(l); break;
    }
  }
  if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

extern "C" {

pkv_status pkv_kv_append(const pkv_cache_desc* desc, void* k_cache, void* v_cache,
                         const int64_t* slot_mapping, const void* k, const void* v,
                         int32_t num_tokens, pkv_dtype kv_dtype, pkv_stream_t stream) {
  pkv_status st = check_desc(desc);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  st = append_checks(desc, k_cache, v_cache, slot_mapping, k, v, num_tokens, kv_dtype);
  if (st != PKV_OK) return st;
  pkv::AppendParams a;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.slot_mapping = slot_mapping;
  a.block_tables = nullptr;
  a.context_lens = nullptr;
  a.MBS = 0;
  a.scale_out = nullptr;
  if (desc->cache_dtype == PKV_FP8_E4M3_TOKEN)  // the scale pool takes the rows' scales
    a.scale_out = const_cast<float*>(desc->k_scale);
  a.k = k;
  a.v = v;
  a.k_scale = desc->k_scale;
  a.v_scale = desc->v_scale;
  a.err_word = desc->err_word;
  a.T = num_tokens;
  a.Hkv = desc->num_kv_heads;
  a.d = desc->head_dim;
  a.NB = desc->num_blocks;
  cudaError_t e = pkv::launch_append(a, kind_of(desc->cache_dtype), kv_dtype == PKV_BF16,
                                     reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_copy_blocks(const pkv_cache_desc* desc, void* k_cache, void* v_cache,
                           const int32_t* src_blocks, const int32_t* dst_blocks, int32_t n,
                           pkv_stream_t stream) {
  pkv_status st = check_desc(desc);
  if (st != PKV_OK) return st;
  if (n < 0) return PKV_ERR_INVALID_ARG;
  if (n == 0) return PKV_OK;
  if (!k_cache || !v_cache || !src_blocks || !dst_blocks) return PKV_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(src_blocks, 4) ||
      !aligned(dst_blocks, 4))
    return PKV_ERR_INVALID_ARG;
  pkv::CopyParams c;
  c.k_cache = k_cache;
  c.v_cache = v_cache;
  c.src = src_blocks;
  c.dst = dst_blocks;
  c.err_word = desc->err_word;
  c.block_bytes = (int64_t)desc->num_kv_heads * desc->page_size * desc->head_dim *
                  (is_fp8(desc->cache_dtype) ? 1 : 2);
  c.scales = nullptr;  // per-token scales travel with their block
  if (desc->cache_dtype == PKV_FP8_E4M3_TOKEN) c.scales = const_cast<float*>(desc->k_scale);
  c.scales_per_block = desc->num_kv_heads * 2 * desc->page_size;
  c.NB = desc->num_blocks;
  const cudaError_t e = pkv::launch_copy_blocks(c, n, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

size_t pkv_decode_workspace_bytes(const pkv_cache_desc* desc, int32_t batch,
                                  int32_t max_blocks_per_seq, int32_t max_context_len_hint) {
  return pkv_decode_workspace_bytes_multi(desc, batch, 1, max_blocks_per_seq,
                                          max_context_len_hint);
}

size_t pkv_decode_workspace_bytes_multi(const pkv_cache_desc* desc, int32_t batch,
                                        int32_t q_len, int32_t max_blocks_per_seq,
                                        int32_t max_context_len_hint) {
  if (check_desc(desc) != PKV_OK || batch < 0 || max_blocks_per_seq <= 0) return 0;
  if (q_len < 1 || q_len > 8) return 0;
  if (batch == 0) return 0;
  const int sms = sm_count_current_device();
  if (sms <= 0) return 0;
  return ws_layout(desc, batch, max_blocks_per_seq, max_context_len_hint, sms,
                   nc_of(desc, q_len)).total;
}

pkv_status pkv_paged_decode_attention(const pkv_cache_desc* desc, const void* q,
                                      const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, const int32_t* context_lens,
                                      int32_t batch, int32_t max_blocks_per_seq,
                                      int32_t max_context_len_hint, float scale, void* out,
                                      pkv_dtype q_dtype, pkv_dtype out_dtype, void* workspace,
                                      size_t workspace_bytes, pkv_stream_t stream) {
  return decode_impl(desc, q, k_cache, v_cache, block_tables, context_lens, batch,
                     max_blocks_per_seq, max_context_len_hint, scale, out, q_dtype, out_dtype,
                     workspace, workspace_bytes, stream, /*early_prologue=*/0);
}

pkv_status pkv_paged_decode_attention_multi(
    const pkv_cache_desc* desc, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, int32_t batch, int32_t q_len,
    int32_t max_blocks_per_seq, int32_t max_context_len_hint, float scale, void* out,
    pkv_dtype q_dtype, pkv_dtype out_dtype, void* workspace, size_t workspace_bytes,
    pkv_stream_t stream) {
  pkv_status st = check_desc(desc);
  if (st != PKV_OK) return st;
  if (q_len < 1) return PKV_ERR_INVALID_ARG;
  if (q_len > 8) return PKV_ERR_UNSUPPORTED;
  return decode_impl(desc, q, k_cache, v_cache, block_tables, context_lens, batch,
                     max_blocks_per_seq, max_context_len_hint, scale, out, q_dtype, out_dtype,
                     workspace, workspace_bytes, stream, /*early_prologue=*/0, q_len);
}

pkv_status pkv_paged_decode_attention_window(
    const pkv_cache_desc* desc, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, int32_t batch, int32_t q_len,
    int32_t window, int32_t sinks, int32_t max_blocks_per_seq, int32_t max_context_len_hint,
    float scale, void* out, pkv_dtype q_dtype, pkv_dtype out_dtype, void* workspace,
    size_t workspace_bytes, pkv_stream_t stream) {
  pkv_status st = check_desc(desc);
  if (st != PKV_OK) return st;
  if (q_len < 1 || window < 0 || sinks < 0) return PKV_ERR_INVALID_ARG;
  if (q_len > 8) return PKV_ERR_UNSUPPORTED;
  return decode_impl(desc, q, k_cache, v_cache, block_tables, context_lens, batch,
                     max_blocks_per_seq, max_context_len_hint, scale, out, q_dtype, out_dtype,
                     workspace, workspace_bytes, stream, /*early_prologue=*/0, q_len, window,
                     sinks);
}

pkv_status pkv_decode_step(const pkv_cache_desc* desc, const void* q, void* k_cache,
                           void* v_cache, const int64_t* slot_mapping, const void* k,
                           const void* v, pkv_dtype kv_dtype, const int32_t* block_tables,
                           const int32_t* context_lens, int32_t batch,
                           int32_t max_blocks_per_seq, int32_t max_context_len_hint,
                           float scale, void* out, pkv_dtype q_dtype, pkv_dtype out_dtype,
                           void* workspace, size_t workspace_bytes, pkv_stream_t stream) {
  // Validate everything before the first launch, so an error launches nothing.
  pkv_status st = decode_checks(desc, q, k_cache, v_cache, block_tables, context_lens, batch,
                                max_blocks_per_seq, max_context_len_hint, scale, out, q_dtype,
                                out_dtype, workspace, workspace_bytes);
  if (st != PKV_OK) return st;
  if (batch > 0) {
    st = append_checks(desc, k_cache, v_cache, slot_mapping, k, v, batch, kv_dtype);
    if (st != PKV_OK) return st;
  }
  st = pkv_kv_append(desc, k_cache, v_cache, slot_mapping, k, v, batch, kv_dtype, stream);
  if (st != PKV_OK) return st;
  return decode_impl(desc, q, k_cache, v_cache, block_tables, context_lens, batch,
                     max_blocks_per_seq, max_context_len_hint, scale, out, q_dtype, out_dtype,
                     workspace, workspace_bytes, stream, /*early_prologue=*/1);
}

pkv_status pkv_paged_prefill_attention(const pkv_cache_desc* desc, const void* q,
                                       const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables,
                                       const int32_t* context_lens, const int32_t* q_start,
                                       int32_t batch, int32_t total_q, int32_t max_q_len,
                                       int32_t max_blocks_per_seq, float scale, void* out,
                                       pkv_dtype q_dtype, pkv_dtype out_dtype,
                                       pkv_stream_t stream) {
  pkv_status st = check_desc(desc);
  if (st != PKV_OK) return st;
  if (batch < 0 || total_q < 0 || max_q_len < 0 || max_blocks_per_seq <= 0)
    return PKV_ERR_INVALID_ARG;
  if (batch == 0 || total_q == 0 || max_q_len == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !q_start || !out)
    return PKV_ERR_INVALID_ARG;
  if (desc->cache_dtype != PKV_F16 && desc->cache_dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
  if (desc->head_dim != 64 && desc->head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (q_dtype != desc->cache_dtype) return PKV_ERR_INVALID_ARG;
  if (out_dtype != PKV_F16 && out_dtype != PKV_BF16 && out_dtype != PKV_F32)
    return PKV_ERR_UNSUPPORTED;
  if (!(scale > 0.f)) return PKV_ERR_INVALID_ARG;  // the kernel takes row maxima unscaled
  if ((int64_t)batch * max_blocks_per_seq >= ((int64_t)1 << 31)) return PKV_ERR_UNSUPPORTED;
  if ((int64_t)max_blocks_per_seq * kPageSize >= ((int64_t)1 << 31)) return PKV_ERR_UNSUPPORTED;
  if ((int64_t)total_q * desc->num_q_heads >= ((int64_t)1 << 31)) return PKV_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(q_start, 4))
    return PKV_ERR_INVALID_ARG;
  pkv::PrefillLaunch l;
  st = encode_cache_map(&l.tmap_k, k_cache, desc);
  if (st != PKV_OK) return st;
  st = encode_cache_map(&l.tmap_v, v_cache, desc);
  if (st != PKV_OK) return st;
  auto fn = encode_fn();
  if (fn == nullptr) return PKV_ERR_CUDA;
  const cuuint64_t hd = (cuuint64_t)desc->head_dim;
  const cuuint64_t dims[3] = {hd, (cuuint64_t)desc->num_q_heads, (cuuint64_t)total_q};
  const cuuint64_t strides[2] = {hd * 2, (cuuint64_t)desc->num_q_heads * hd * 2};
  const int G = desc->num_q_heads / desc->num_kv_heads;  // a box: 128 / G tokens x G heads
  const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(128 / G)};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (fn(&l.tmap_q, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(q), dims, strides, box,
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return PKV_ERR_CUDA;
  l.p.q_start = q_start;
  l.p.context_lens = context_lens;
  l.p.block_tables = block_tables;
  l.p.out = out;
  l.p.err_word = desc->err_word;
  l.p.B = batch;
  l.p.Hq = desc->num_q_heads;
  l.p.Hkv = desc->num_kv_heads;
  l.p.NB = desc->num_blocks;
  l.p.MBS = max_blocks_per_seq;
  l.p.total_q = total_q;
  l.p.tiles_per_seq = (max_q_len + 256 / G - 1) / (256 / G);  // a CTA: 256 / G tokens
  l.p.out_dtype = out_dtype;
  l.p.scale_log2 = scale * 1.4426950408889634f;
  l.bf16 = desc->cache_dtype == PKV_BF16;
  l.d = desc->head_dim;
  l.stream = reinterpret_cast<cudaStream_t>(stream);
  if ((int64_t)batch * l.p.tiles_per_seq >= ((int64_t)1 << 31)) return PKV_ERR_UNSUPPORTED;
  return pkv::launch_prefill(l) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_decode_step_fused(const pkv_cache_desc* desc, const void* q, void* k_cache,
                                 void* v_cache, const void* k, const void* v,
                                 pkv_dtype kv_dtype, const int32_t* block_tables,
                                 const int32_t* context_lens, int32_t batch,
                                 int32_t max_blocks_per_seq, int32_t max_context_len_hint,
                                 float scale, void* out, pkv_dtype q_dtype, pkv_dtype out_dtype,
                                 void* workspace, size_t workspace_bytes, int32_t flags,
                                 pkv_stream_t stream) {
  pkv_status st = decode_checks(desc, q, k_cache, v_cache, block_tables, context_lens, batch,
                                max_blocks_per_seq, max_context_len_hint, scale, out, q_dtype,
                                out_dtype, workspace, workspace_bytes);
  if (st != PKV_OK || batch == 0) return st;
  if (!k || !v) return PKV_ERR_INVALID_ARG;
  if (kv_dtype != PKV_F16 && kv_dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
  if (!is_fp8(desc->cache_dtype) && kv_dtype != desc->cache_dtype)
    return PKV_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(v, 16)) return PKV_ERR_INVALID_ARG;
  if ((flags & ~PKV_STEP_OVERLAP) != 0) return PKV_ERR_INVALID_ARG;
  const int overlap = (flags & PKV_STEP_OVERLAP) ? 1 : 0;
  if (is_fp8(desc->cache_dtype)) {
    // E4M3: the append kernel (each sequence's newest position, from its
    // table), then the attention overlapping its tail
    pkv::AppendParams a;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.slot_mapping = nullptr;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.MBS = max_blocks_per_seq;
    a.scale_out = nullptr;
    if (desc->cache_dtype == PKV_FP8_E4M3_TOKEN) a.scale_out = const_cast<float*>(desc->k_scale);
    a.k = k;
    a.v = v;
    a.k_scale = desc->k_scale;
    a.v_scale = desc->v_scale;
    a.err_word = desc->err_word;
    a.T = batch;
    a.Hkv = desc->num_kv_heads;
    a.d = desc->head_dim;
    a.NB = desc->num_blocks;
    if (pkv::launch_append(a, kind_of(desc->cache_dtype), kv_dtype == PKV_BF16,
                           reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
      return PKV_ERR_CUDA;
    return decode_impl(desc, q, k_cache, v_cache, block_tables, context_lens, batch,
                       max_blocks_per_seq, max_context_len_hint, scale, out, q_dtype, out_dtype,
                       workspace, workspace_bytes, stream, /*early_prologue=*/1, 1, 0, 0,
                       nullptr, nullptr, kv_dtype, /*trigger_next=*/overlap);
  }
  return decode_impl(desc, q, k_cache, v_cache, block_tables, context_lens, batch,
                     max_blocks_per_seq, max_context_len_hint, scale, out, q_dtype, out_dtype,
                     workspace, workspace_bytes, stream, /*early_prologue=*/overlap, 1, 0, 0, k,
                     v, kv_dtype, /*trigger_next=*/overlap);
}

uint64_t pkv_kv_bytes_per_token(int32_t layers, int32_t kv_heads, int32_t head_dim,
                                int32_t elem_bytes) {
  if (layers < 0 || kv_heads < 0 || head_dim < 0 || elem_bytes < 0) return 0;
  return 2ull * (uint64_t)layers * (uint64_t)kv_heads * (uint64_t)head_dim *
         (uint64_t)elem_bytes;
}

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG: invalid argument";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED: shape or dtype not built";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA: CUDA call failed";
    case PKV_ERR_BOUNDS: return "PKV_ERR_BOUNDS: slot, block id or context length out of range";
    case PKV_ERR_TIMEOUT: return "PKV_ERR_TIMEOUT: a bounded device wait gave up";
  }
  return "unknown pkv_status";
}

int32_t pkv_version(void) { return 100; }

}  // extern "C"
