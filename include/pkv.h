/*
 * pkv.h -- C ABI of the paged-KV decode-attention library (libpkv.so).
 *
 * One decode step for one attention layer is two calls on the caller's CUDA
 * stream:
 *
 *   1. pkv_kv_append: write the new token's K and V rows into the cache
 *      pages named by a slot mapping.
 *   2. pkv_paged_decode_attention: for every sequence and query head, one
 *      (1,N) attention row over the cached keys and values, read through the
 *      sequence's block table.
 *
 * pkv_decode_step validates and enqueues both; pkv_decode_step_fused does
 * both in one kernel, each new row going to its sequence's newest position.
 *
 * Sources (web pages):
 *   [KVFA] "KV Cache & Flash Attention." (kvcache-7e2.pages.dev)
 *   [DF]   "KV Cache & FlashAttention" (deepforge.srivtx.xyz)
 *   [AP]   "KV cache, paged, flash and sparse attention" (abhishekpatel.co)
 *
 * Conventions shared by every entry point
 *   - All buffers are owned by the caller.  The library allocates and frees
 *     nothing and keeps no state beyond a per-device cache of the SM count.
 *   - Pointers are DEVICE pointers unless the comment says host.  The
 *     descriptor itself is a host struct.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  They return once the kernels are enqueued and never
 *     synchronise.
 *   - Argument errors are reported before any launch.  Launch failures
 *     return PKV_ERR_CUDA.  Data-dependent errors found on the device (a slot
 *     or block-table entry outside the pool, a context longer than the table)
 *     skip the offending work and are recorded in the optional device word
 *     `err_word` (first error wins; the library never clears it).  No kernel
 *     traps.
 *   - Cache layout ("HND"): k_cache and v_cache are [num_blocks][num_kv_heads]
 *     [page_size][head_dim] elements of `cache_dtype`, so one (block, KV head)
 *     page is a contiguous run of page_size * head_dim elements.  The base
 *     address must be 16-byte aligned.
 *   - Query head hq reads KV head hq / (num_q_heads / num_kv_heads).
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so this header needs no CUDA. */
typedef struct CUstream_st* pkv_stream_t;

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1, /* null pointer, bad size, Hq % Hkv != 0, ...    */
  PKV_ERR_UNSUPPORTED = 2, /* valid but not built: head_dim, group, dtype  */
  PKV_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required    */
  PKV_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed          */
  PKV_ERR_BOUNDS = 5,      /* device: slot / block id / context out of range */
  PKV_ERR_TIMEOUT = 6      /* device: a bounded wait gave up                */
} pkv_status;

typedef enum {
  PKV_F16 = 0,
  PKV_BF16 = 1,
  PKV_FP8_E4M3 = 2, /* OCP E4M3 (bias 7, max 448, no infinities)         */
  PKV_F32 = 3,
  PKV_FP8_E4M3_TOKEN = 4 /* E4M3 cache, one fp32 scale per token and head  */
} pkv_dtype;

/* Shape of the paged cache, shared by both calls.
 * Supported: page_size 16; head_dim 64 or 128 (128 for FP8_E4M3);
 * num_q_heads / num_kv_heads in {1, 2, 4, 8}; cache_dtype F16, BF16 or
 * FP8_E4M3; num_blocks * num_kv_heads * page_size < 2^31. */
typedef struct {
  uint32_t struct_size;  /* sizeof(pkv_cache_desc); checked               */
  int32_t num_blocks;    /* physical blocks in the pool (NB)               */
  int32_t page_size;     /* tokens per block (P)                           */
  int32_t num_kv_heads;  /* Hkv                                            */
  int32_t num_q_heads;   /* Hq, a multiple of Hkv                          */
  int32_t head_dim;      /* d                                              */
  pkv_dtype cache_dtype; /* F16 | BF16 | FP8_E4M3                          */
  const float* k_scale;  /* FP8_E4M3: device fp32 [Hkv], stored K = k/scale.
                            FP8_E4M3_TOKEN: the scale pool, device fp32
                            [NB][Hkv][2][P], 128-byte aligned: for each
                            (block, KV head) the P slots' K scales, then
                            their V scales; written by the append.
                            NULL for 16-bit caches.                        */
  const float* v_scale;  /* FP8_E4M3: device fp32 [Hkv] for V; unused
                            otherwise                                       */
  int32_t* err_word;     /* optional device int32; NULL = do not report    */
} pkv_cache_desc;

/* Flags of pkv_decode_step_fused. */
#define PKV_STEP_OVERLAP 1

/* Append (scatter) new K/V rows into their cache slots.
 * [KVFA] KV-cache section (append one K and one V per token) and
 * PagedAttention section (position -> (block, offset)); [AP] "Following one
 * new token through the cache".
 *   slot_mapping int64 [num_tokens]: slot = block * page_size + offset; a
 *                negative slot skips the token; a slot >= num_blocks *
 *                page_size is a device-detected PKV_ERR_BOUNDS.
 *   k, v         [num_tokens][num_kv_heads][head_dim] of kv_dtype (F16 or
 *                BF16; for 16-bit caches it must equal cache_dtype).
 *   For FP8_E4M3 caches each element is divided by its head's scale in IEEE
 *   fp32 and encoded round-to-nearest-even with saturation to +-448.
 *   For FP8_E4M3_TOKEN caches each (token, KV head) row of K, and of V, gets
 *   its own scale, the row's largest magnitude divided by 448 in IEEE fp32
 *   (1 for an all-zero row), written to the slot's K (or V) entry of the
 *   scale pool;
 *   the row is then encoded under it as above ([KVFA] memory-cost section:
 *   the cache is quantized to fp8; Flash Attention section: FP8 with finer-
 *   grained scales).  head_dim 128.
 *   Slots written by two tokens of one call race; the caller avoids it. */
PKV_API pkv_status pkv_kv_append(const pkv_cache_desc* desc, void* k_cache,
                         void* v_cache, const int64_t* slot_mapping,
                         const void* k, const void* v, int32_t num_tokens,
                         pkv_dtype kv_dtype, pkv_stream_t stream);

/* Bytes of device workspace pkv_paged_decode_attention / pkv_decode_step
 * need for these sizes on the current device (it depends on the SM count).
 * Returns 0 on invalid arguments or without a device.  The workspace holds
 * the split partials and one arrival counter per (sequence, KV head).  It
 * must be zero-filled once before its first use (e.g. cudaMemsetAsync);
 * every call that completes leaves the counters at zero again, so it can be
 * reused without clearing.  A workspace sized for a batch B serves every call
 * with the same descriptor and a batch of at most B (any max_blocks_per_seq
 * and hint); pass its full size.  After a call that reported
 * PKV_ERR_TIMEOUT, zero it again.  Calls that share a workspace must not
 * overlap.  It serves the multi-query and windowed calls for
 * (num_q_heads / num_kv_heads) * q_len <= 8. */
PKV_API size_t pkv_decode_workspace_bytes(const pkv_cache_desc* desc, int32_t batch,
                                  int32_t max_blocks_per_seq,
                                  int32_t max_context_len_hint);

/* The same for the multi-query and windowed calls with up to q_len (1 .. 8)
 * query tokens per sequence: their split partials hold group * q_len
 * columns (rounded up to a power of two).  A workspace sized for (B, Q)
 * serves every call with the same descriptor, a batch of at most B and at
 * most Q query tokens.  Returns 0 on invalid arguments or without a device. */
PKV_API size_t pkv_decode_workspace_bytes_multi(const pkv_cache_desc* desc, int32_t batch,
                                        int32_t q_len, int32_t max_blocks_per_seq,
                                        int32_t max_context_len_hint);

/* Decode attention for one layer.
 * [KVFA] KV-cache section ((1,N) row per step), Flash Attention and
 * online-softmax sections (running max and sum, rescale by exp(m_old -
 * m_new)), PagedAttention section (the kernel takes the page table and
 * gathers K and V); [DF] running-summary paragraph.
 *   q             [batch][num_q_heads][head_dim] of q_dtype (F16 | BF16;
 *                 for 16-bit caches equal to cache_dtype).  With an FP8
 *                 cache the kernel meets q on the fp16 MMA: a bf16 q is
 *                 first scaled, per query head, by a power of two that
 *                 brings its largest element into [2^14, 2^15), and the
 *                 score scale undoes it, so any finite bf16 q is taken
 *                 whole (elements more than 2^28 below their head's largest
 *                 keep fewer bits).
 *   block_tables  int32 [batch][max_blocks_per_seq]; entry p of row b is the
 *                 block holding tokens p*P .. p*P+P-1 of sequence b.  Rows
 *                 may share blocks (prefix sharing); entries past a
 *                 sequence's last page are never read.
 *   context_lens  int32 [batch]; tokens attended, including one appended by
 *                 a preceding pkv_kv_append on the same stream.  0 gives a
 *                 zero output row; > max_blocks_per_seq * P is a device-
 *                 detected PKV_ERR_BOUNDS (that sequence's output is zero).
 *   max_context_len_hint  0, or an upper bound on context_lens used only to
 *                 size the launch; the kernel reads the true lengths.
 *   scale         softmax scale applied to q.k (usually 1/sqrt(head_dim)).
 *   out           [batch][num_q_heads][head_dim] of out_dtype (F16 | BF16 |
 *                 F32), rounded to nearest even.  Must not alias inputs.
 *   workspace     device buffer of at least pkv_decode_workspace_bytes(),
 *                 256-byte aligned, zero-filled before its first use (see
 *                 pkv_decode_workspace_bytes); not shared with concurrent
 *                 calls.
 * Results are bitwise repeatable for the same inputs, sizes and device: the
 * work split depends only on the context lengths and the SM count, and
 * partial sums are always added in the same order.
 * The kernel keeps five int32 per sequence in shared memory beside its page
 * ring: batches past about 6000 sequences at head_dim 128 (6076 for 16-bit,
 * 5979 for per-head and 7093 for per-token E4M3 caches) do not fit and
 * return PKV_ERR_UNSUPPORTED.
 * The kernel is launched as a programmatic dependent of the preceding
 * kernel on the stream but waits for it to complete before reading any
 * input, so ordinary stream order holds. */
PKV_API pkv_status pkv_paged_decode_attention(
    const pkv_cache_desc* desc, const void* q, const void* k_cache,
    const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int32_t batch, int32_t max_blocks_per_seq,
    int32_t max_context_len_hint, float scale, void* out, pkv_dtype q_dtype,
    pkv_dtype out_dtype, void* workspace, size_t workspace_bytes,
    pkv_stream_t stream);

/* Decode attention for q_len new tokens per sequence at once, causal among
 * themselves (verifying drafted tokens: [KVFA] speculative-decoding section,
 * where the target model scores the prefix and the drafted tokens in one
 * forward pass).  Token j (0 <= j < q_len) of sequence b sits at position
 * context_lens[b] - q_len + j and attends to positions 0 .. that position;
 * the new tokens' K and V must already be in the cache (pkv_kv_append with
 * batch * q_len rows), and context_lens counts them.  A token that sees no
 * position (context_lens[b] < q_len) gets a zero row.
 *   q, out        [batch][q_len][num_q_heads][head_dim].
 *   q_len         1 .. 8 at any group size; larger returns
 *                 PKV_ERR_UNSUPPORTED.  q_len 1 is pkv_paged_decode_attention.
 *                 Up to 8 (query token, head) pairs of a KV head share one
 *                 tensor-core column block; 16 take two per warp, and 32 or
 *                 64 split every page's columns over 2 or 4 warps, so each
 *                 page is still read from memory once.
 *   workspace     of at least pkv_decode_workspace_bytes_multi(q_len) bytes
 *                 (pkv_decode_workspace_bytes suffices while
 *                 (num_q_heads / num_kv_heads) * q_len <= 8).
 * For q_len > 1 each CTA's pages go to whichever of its warps is free first,
 * so repeated calls can differ by the order in which fp32 partial sums are
 * added (a few units in the last place of an fp32 output); q_len 1 is
 * bitwise repeatable.
 * Other arguments and guarantees as for pkv_paged_decode_attention. */
PKV_API pkv_status pkv_paged_decode_attention_multi(
    const pkv_cache_desc* desc, const void* q, const void* k_cache,
    const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int32_t batch, int32_t q_len,
    int32_t max_blocks_per_seq, int32_t max_context_len_hint, float scale,
    void* out, pkv_dtype q_dtype, pkv_dtype out_dtype, void* workspace,
    size_t workspace_bytes, pkv_stream_t stream);

/* pkv_paged_decode_attention_multi under a sliding window with attention
 * sinks ([AP] "Sparse attention: stop looking at everything": a token sees
 * only the previous w tokens plus a few global tokens at the start; [KVFA]
 * eviction paragraph: the window drops the oldest tokens, the first few are
 * always kept).  Token j, at position t = context_lens[b] - q_len + j, attends
 * to the positions u <= t with u >= t - window + 1 (itself included) or
 * u < sinks.
 *   window        0: no window (the call is pkv_paged_decode_attention_multi
 *                 and sinks is ignored); > 0: the window length in tokens.
 *   sinks         >= 0 leading positions every token keeps seeing.
 * Pages that no token of the sequence sees (wholly between the sink pages
 * and the first page of token 0's window) are neither loaded nor looked up:
 * their block-table entries are never read and may be anything, so a caller
 * may hand those blocks back to its pool.  Negative window or sinks, or
 * q_len < 1, return PKV_ERR_INVALID_ARG.  Other arguments and guarantees as
 * for pkv_paged_decode_attention_multi. */
PKV_API pkv_status pkv_paged_decode_attention_window(
    const pkv_cache_desc* desc, const void* q, const void* k_cache,
    const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int32_t batch, int32_t q_len, int32_t window,
    int32_t sinks, int32_t max_blocks_per_seq, int32_t max_context_len_hint,
    float scale, void* out, pkv_dtype q_dtype, pkv_dtype out_dtype,
    void* workspace, size_t workspace_bytes, pkv_stream_t stream);

/* One whole decode step: pkv_kv_append of one new token per sequence
 * (slot_mapping, k, v have `batch` rows) followed by
 * pkv_paged_decode_attention, validated together before anything is
 * launched.  The attention kernel is launched as a programmatic dependent
 * of the append kernel: it reads context_lens and block_tables and plans
 * its work while the append runs, and waits for the append to complete
 * before reading any cache page.  context_lens must already count the
 * appended token.  Arguments as for the two calls above. */
PKV_API pkv_status pkv_decode_step(
    const pkv_cache_desc* desc, const void* q, void* k_cache, void* v_cache,
    const int64_t* slot_mapping, const void* k, const void* v, pkv_dtype kv_dtype,
    const int32_t* block_tables, const int32_t* context_lens, int32_t batch,
    int32_t max_blocks_per_seq, int32_t max_context_len_hint, float scale,
    void* out, pkv_dtype q_dtype, pkv_dtype out_dtype, void* workspace,
    size_t workspace_bytes, pkv_stream_t stream);

/* Paged prefill attention: a chunk of new tokens per sequence, whose K and V
 * are already in the cache, attends causally over the sequence's whole
 * context through its block table ([KVFA] opening section: the prefill phase
 * processes the prompt in one parallel pass; continuous-batching section:
 * chunked prefill reads each sequence's pages through its table).  Row j of
 * sequence b's chunk sits at position context_lens[b] - n_b + j (n_b its
 * row count) and attends to positions 0 .. that position.  Runs on the
 * tensor cores (tcgen05, accumulators in tensor memory); 16-bit caches with
 * head_dim 64 or 128 (others return PKV_ERR_UNSUPPORTED).
 *   q             [total_q][num_q_heads][head_dim] of q_dtype (= cache_dtype);
 *                 sequence b's rows are q_start[b] .. q_start[b + 1] - 1.
 *   q_start       int32 [batch + 1], device, non-decreasing, q_start[batch]
 *                 <= total_q.
 *   max_q_len     host: an upper bound on q_start[b + 1] - q_start[b]; it
 *                 sizes the launch.
 *   context_lens  tokens of each sequence, the chunk included (>= n_b).
 *   scale         > 0 (the softmax scale); otherwise PKV_ERR_INVALID_ARG.
 *   out           [total_q][num_q_heads][head_dim] of out_dtype (F16 | BF16 |
 *                 F32).
 * A sequence whose row count or length breaks these rules is a device-
 * detected PKV_ERR_BOUNDS and its output rows are not written.  A table
 * entry outside [0, num_blocks) in a page the chunk sees is PKV_ERR_BOUNDS
 * too: that page is read as zeros, never from outside the pool, and the
 * sequence's rows are written but meaningless.  No workspace.  Inputs are read after the preceding kernel on the stream
 * completes (the kernel is launched as a programmatic dependent).  Results
 * are deterministic: each output row is one CTA's fixed sequence of MMAs. */
PKV_API pkv_status pkv_paged_prefill_attention(
    const pkv_cache_desc* desc, const void* q, const void* k_cache,
    const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, const int32_t* q_start, int32_t batch,
    int32_t total_q, int32_t max_q_len, int32_t max_blocks_per_seq,
    float scale, void* out, pkv_dtype q_dtype, pkv_dtype out_dtype,
    pkv_stream_t stream);

/* One decode step in ONE kernel: pkv_decode_step with each sequence's new
 * token placed at its position context_lens[b] - 1, i.e. in block
 * block_tables[b][(context_lens[b] - 1) / P] at offset (context_lens[b] - 1)
 * % P ([KVFA] KV-cache section: append, then attend over all tokens;
 * PagedAttention section: position -> (block, offset)).  With a 16-bit
 * cache the warp that stages that page writes the new K and V row into its
 * staged copy, which this pass attends to, and into the cache, for later
 * steps: one launch, no slot mapping.  With an E4M3 cache the call enqueues
 * two kernels: the append (each row to its sequence's newest position,
 * encoded as pkv_kv_append encodes it), then the attention overlapping its
 * tail.  Either way the cache bytes are those pkv_kv_append writes.
 *   k, v          [batch][num_kv_heads][head_dim] of kv_dtype (F16 or BF16;
 *                 for 16-bit caches it must equal cache_dtype).  A sequence
 *                 with context_lens[b] == 0 appends nothing.
 *   flags         0, or PKV_STEP_OVERLAP: context_lens and block_tables are
 *                 not written by the kernel launched just before this call
 *                 on the stream (host copies and earlier kernels may write
 *                 them).  The kernel then reads them, and lays out its work,
 *                 while that kernel finishes (programmatic dependent
 *                 launch), and lets the next kernel on the stream launch
 *                 before it ends (a programmatic dependent must wait for it
 *                 before reading its outputs, as that launch mode requires).
 *                 Every other input is read after the preceding kernel
 *                 completes.  Without the flag every input is.  Other bits
 *                 return PKV_ERR_INVALID_ARG.
 * The block receiving a new row must not be read at that row by another
 * sequence of the same call (copy it first: pkv_copy_blocks).  Other
 * arguments and guarantees as for pkv_paged_decode_attention. */
PKV_API pkv_status pkv_decode_step_fused(
    const pkv_cache_desc* desc, const void* q, void* k_cache, void* v_cache,
    const void* k, const void* v, pkv_dtype kv_dtype,
    const int32_t* block_tables, const int32_t* context_lens, int32_t batch,
    int32_t max_blocks_per_seq, int32_t max_context_len_hint, float scale,
    void* out, pkv_dtype q_dtype, pkv_dtype out_dtype, void* workspace,
    size_t workspace_bytes, int32_t flags, pkv_stream_t stream);

/* Size of the fixed device scratch behind pkv_paged_decode_attention_noalloc
 * (32 MiB, held by every GPU that loads the library until the process ends). */
#define PKV_NOALLOC_SCRATCH_BYTES (32u << 20)

/* pkv_paged_decode_attention without a caller workspace.  The pages have no
 * counterpart to this call; it exists for callers that cannot allocate device
 * memory when they attend (a custom-op hook with no allocator handle, a plugin
 * inside an engine that owns all device memory, a path that must not call
 * cudaMalloc because it may synchronise the device).  It runs the same kernel
 * on a fixed scratch array in the library's own device image and allocates
 * nothing.
 *   - Shapes whose workspace (pkv_decode_workspace_bytes) exceeds
 *     PKV_NOALLOC_SCRATCH_BYTES return PKV_ERR_WORKSPACE; other argument
 *     errors are those of pkv_paged_decode_attention.  Every argument is
 *     checked before anything is put on the stream.
 *   - The first call on each device looks up the scratch array's device
 *     address (cudaGetSymbolAddress) and keeps it for the life of the
 *     process.  The kept address belongs to the device's primary context (the
 *     one the CUDA runtime uses): calls from another context on the device,
 *     or after a cudaDeviceReset, are not supported.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; each call first clears, on `stream`, the part that must start
 *     at zero.  Calls whose executions overlap on the GPU (other streams,
 *     other threads) race on the scratch and give wrong results: order them.
 * Arguments otherwise as for pkv_paged_decode_attention. */
PKV_API pkv_status pkv_paged_decode_attention_noalloc(
    const pkv_cache_desc* desc, const void* q, const void* k_cache,
    const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int32_t batch, int32_t max_blocks_per_seq,
    int32_t max_context_len_hint, float scale, void* out, pkv_dtype q_dtype,
    pkv_dtype out_dtype, pkv_stream_t stream);

/* Copy whole cache blocks, all KV heads of K and of V: block dst_blocks[i]
 * receives block src_blocks[i], for i < n (copy-on-write for shared
 * prefixes).  [AP] "Paged attention: stop reserving empty tables": sequences
 * point at the same physical blocks for a shared beginning, copying only if
 * one of them would change a block; [KVFA] PagedAttention section: sharing a
 * prefix hands the second sequence ceil(prefix / P) of the same blocks, so
 * the last may be partly filled and must be copied before either sequence
 * appends into it.  The pages have no function of this name; it is the copy
 * step of that scheme.
 *   src_blocks, dst_blocks  device int32 [n].  A pair with an id outside
 *                 [0, num_blocks) is skipped and reported as PKV_ERR_BOUNDS
 *                 in err_word.  A block may be a destination at most once
 *                 per call and must not also be a source in that call
 *                 (the copies run concurrently).
 * Asynchronous on `stream`; n == 0 launches nothing. */
PKV_API pkv_status pkv_copy_blocks(const pkv_cache_desc* desc, void* k_cache,
                                   void* v_cache, const int32_t* src_blocks,
                                   const int32_t* dst_blocks, int32_t n,
                                   pkv_stream_t stream);

/* Cache bytes per token across all layers: 2 * layers * kv_heads * head_dim
 * * elem_bytes ([AP] "Opening the hood: how big is the notebook?"; [DF]
 * cache-size paragraph).  Host-only. */
PKV_API uint64_t pkv_kv_bytes_per_token(int32_t layers, int32_t kv_heads,
                                int32_t head_dim, int32_t elem_bytes);

/* Static, human-readable name of a status code.  Host-only. */
PKV_API const char* pkv_status_string(pkv_status status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH.  Host-only. */
PKV_API int32_t pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
