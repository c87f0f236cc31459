// pkv_decode_mq.cuh -- split-K flash-decoding kernel over a paged KV cache for
// several query tokens per sequence (multi-query and windowed decode), with
// the split combine fused in.  Single-token decode is pkv_decode_impl.cuh.
//
// What it computes: for every sequence b and query head hq, one (1,N)
// attention row softmax(scale * q K^T) V over the sequence's cached tokens,
// read through its block table.  Sources: "KV Cache & Flash Attention."
// (kvcache-7e2.pages.dev), Flash Attention and online-softmax sections
// (running max m and sum l, rescale by exp(m_old - m_new), one division at
// the end) and PagedAttention section (block = table[pos / P], offset =
// pos % P, gathered at lookup time); "KV Cache & FlashAttention"
// (deepforge.srivtx.xyz), running-summary paragraph (partial sums and
// partial outputs are brought to a common maximum by the same factor).
//
// Schedule.  The (sequence b, KV head h, page) units are laid out b-major,
// then h, then page, on a cost line where a page costs 1 and the start of a
// (b, h) "segment" kSegCost more; the line is cut into contiguous shares of
// equal cost (at least kRangeMin each), one per CTA of a persistent grid (two
// CTAs per SM), so ragged lengths never leave an SM idle.
//
// Within a CTA the share's pages are numbered 0 .. N-1 (ordinals) and flow
// through one ring of R shared-memory slots (ordinal o in slot o % R): every
// slot holds one K page and one V page of one (block, KV head), loaded by
// 2-D TMA tile copies that complete on the slot's mbarrier.  Warps claim the
// next two ordinals from a shared counter whenever they are free, so the
// CTA's pages go to whichever warp is ready; a page's slot is refilled with
// ordinal o + R as soon as it has been read.  Page descriptors (TMA row, the
// tokens that count, sequence, KV head) are looked up from the block table
// by the lanes of one warp, 32 at a time, two blocks ahead of the claims.
//
// Columns.  A kernel is built for NC = G x QC (query token, head) columns of
// one KV head.  Up to 8 columns fit one MMA's N; 16 are two column groups in
// one warp; for 32 and 64 the warps split into SL slices that compute
// disjoint column ranges of every page (each page is read by one warp of each
// slice, and its slot is refilled after the last of them).
//
// Segment ends.  Each warp accumulates its own online-softmax state per
// segment; when it claims a page of a later segment it hands the state over
// (the merge is order-independent).  For up to 4 columns three warps drop
// their state into shared memory behind an mbarrier and keep streaming while
// a rotating fourth merges and writes; otherwise the warps of a slice merge
// by a barrier tree.  A segment wholly inside one share is normalised and
// written at once; a segment cut by share boundaries gets one partial
// (m, l, o) per CTA, in slot cta + segment, and a page-count ticket; the CTA
// whose pages complete the segment merges the partials (the split combine),
// in slot order.  Nothing waits on another CTA.
//
// Math per page (16 tokens), on warp-level tensor-core MMAs:
//   S^T[16 tok][8] = K[16][d] . Q^T[d][8]   K via ldmatrix from the swizzled
//                                           page, Q^T resident in registers;
//                                           the 8 columns are (query token,
//                                           head) pairs (zero-padded)
//   online softmax in registers (log2 domain); the running max only moves
//   when a tile's max exceeds it by more than 2^8, which keeps every weight
//   p <= 256 and is exact because l and o use the same reference;
//   O^T[d][8] += V^T[d][16] . P^T[16][8]    V^T via ldmatrix.trans, P^T via
//                                           movmatrix; P is split into hi + lo
//                                           16-bit parts (two MMAs) so the
//                                           weights keep ~16 mantissa bits.
// E4M3 pages are converted to fp16 in registers (exact) after the ldmatrix;
// the per-head K scale is folded into the score scale and the V scale into
// the output.
#pragma once

#include <cuda.h>
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace mq {

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per bounded wait
constexpr float kRescaleThreshold = 8.0f;         // log2 units
constexpr int kMergeBarrier = 1;                  // named barrier id (0 = __syncthreads)
constexpr int kSliceBarrier0 = 2;                 // named barriers 2 .. 5: one per slice
// A descriptor holds the tokens from the page's start to the context's end,
// capped here (enough for the causal limits of up to 8 query tokens).
constexpr int kRemCap = 2 * kPageSize;
constexpr int kRemMask = 63;       // descriptor y, bits 0-5: tokens to the context's end
constexpr int kWinFlag = 1 << 17;  // descriptor: a sliding window masks rows of this page
constexpr int kDescBlocks = kDescN / kDescBlock;
constexpr int kFillAhead = 2;      // descriptor blocks filled ahead of the claims

template <int N>
struct Int {  // a compile-time count passed to a generic lambda
  static constexpr int value = N;
};

template <int D, int CACHE, int NC>
struct DecodeCfg {
  static constexpr int kElem = cache_is_fp8((CacheKind)CACHE) ? 1 : 2;
  static constexpr int kRowBytes = D * kElem;              // bytes per token row
  static constexpr int kBoxes = kRowBytes / 128;           // 128-byte TMA boxes per row
  static constexpr int kBoxBytes = kPageSize * 128;        // one box of a page
  static constexpr int kTileBytes = kPageSize * kRowBytes; // one K (or V) page
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kScaleBytes = decode_scale_bytes((CacheKind)CACHE);  // per slot
  static constexpr int kKSteps = D / 16;  // k-steps of the QK contraction
  static constexpr int kMTiles = D / 16;  // 16-row tiles of O^T
  static constexpr int kRing = mq_ring(D, (CacheKind)CACHE, NC);
  static constexpr int kCW = mq_cw(NC);       // column groups per warp
  static constexpr int kSL = mq_sl(NC);       // slices
  static constexpr int kPS = kDecodeWarps / kSL;  // warps per slice
  static constexpr int kPartCols = decode_part_cols(NC);
  static constexpr int kLaneState = mq_lane_state(D, NC);  // per CW groups
  static constexpr int kGroupState = 4 + 4 * kMTiles;          // one column group
  static_assert(kRowBytes % 128 == 0, "rows must be whole 128-byte boxes");
  static_assert(kRing <= 28, "descriptor ring reuse needs R <= 28");
};

// Byte offset of 16-byte chunk `chunk` of token row `tok` inside a page
// loaded as 128-byte-swizzled boxes of 16 rows.
__device__ __forceinline__ uint32_t swz(int tok, int chunk) {
  return (uint32_t)((chunk >> 3) * (kPageSize * 128) + tok * 128 +
                    (((chunk & 7) ^ (tok & 7)) << 4));
}

__device__ __forceinline__ void merge_barrier() {
  asm volatile("bar.sync %0, %1;" ::"n"(kMergeBarrier), "n"(kDecodeWarps * 32) : "memory");
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ int ld_volatile_s32(const int* p) {
  return *reinterpret_cast<const volatile int*>(p);
}
__device__ __forceinline__ void st_volatile_s32(int* p, int v) {
  *reinterpret_cast<volatile int*>(p) = v;
}

template <typename OutT>
__device__ __forceinline__ void store_out(void* base, int64_t idx, float v);
template <>
__device__ __forceinline__ void store_out<float>(void* base, int64_t idx, float v) {
  reinterpret_cast<float*>(base)[idx] = v;
}
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(void* base, int64_t idx, float v) {
  reinterpret_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
}
template <>
__device__ __forceinline__ void store_out<__half>(void* base, int64_t idx, float v) {
  reinterpret_cast<__half*>(base)[idx] = __float2half_rn(v);
}

__device__ __forceinline__ void store_out_rt(pkv_dtype t, void* base, int64_t idx, float v) {
  if (t == PKV_F32) store_out<float>(base, idx, v);
  else if (t == PKV_BF16) store_out<__nv_bfloat16>(base, idx, v);
  else store_out<__half>(base, idx, v);
}

// G query heads share a KV head; QC is the number of query tokens per
// sequence the kernel is built for (p.qlen <= QC of them are real).  The
// NC = QC * G (query token, head) pairs of a group are the MMA columns.
template <int D, int G, int QC, int CACHE, bool QBF16>
__global__ void __launch_bounds__(kDecodeWarps * 32, kDecodeCtasPerSm)
    decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv) {
  constexpr int NC = G * QC;
  using C = DecodeCfg<D, CACHE, NC>;
  constexpr bool kBF = (CACHE == kCacheBF16);  // mma operand type (else fp16)
  constexpr int R = C::kRing;
  constexpr int NW = kDecodeWarps;
  constexpr int kMT = C::kMTiles;
  constexpr int CW = C::kCW, SL = C::kSL, PS = C::kPS, PC = C::kPartCols;
  constexpr int kGS = C::kGroupState;
  constexpr bool kFp8 = cache_is_fp8((CacheKind)CACHE);
  constexpr bool kTok = CACHE == kCacheE4M3Tok;  // one scale per token and KV head
  // the one-kernel step writes new rows in the main loop for 16-bit caches
  // only (E4M3 steps enqueue the append kernel first)
  constexpr bool kFusedAppend = QC == 1 && !kFp8;
  static_assert(8 * CW * SL >= NC && NC <= 64, "column layout");
  static_assert(!kFusedAppend || SL == 1, "a fused append stages a page for one warp");

  // the next kernel on the stream may launch (a programmatic dependent waits
  // for this one to complete before it reads what this one writes)
  if (p.trigger_next) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!p.early_prologue) griddep_wait();

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const int slice = warp % SL;  // the column range this warp computes
  const int sw = warp / SL;     // its rank among the warps of its slice

  // ---- shared memory (decode_smem_bytes mirrors this plan)
  const uint32_t ring = base;                                  // [R] K+V pages
  const uint32_t scl = base + (uint32_t)(R * C::kStageBytes);  // [R] per-token scales
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(base_ptr + (size_t)R * (C::kStageBytes + C::kScaleBytes));
  uint64_t* fbar = bars + R;  // [kFlushBars] segment-end hand-off
  const size_t desc_off =
      ((size_t)R * (C::kStageBytes + C::kScaleBytes) + (size_t)(R + kFlushBars) * 8 + 15) &
      ~(size_t)15;
  int4* desc = reinterpret_cast<int4*>(base_ptr + desc_off);  // [kDescN]
  float* mbuf = reinterpret_cast<float*>(desc + kDescN);       // two warp states
  int* sint = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(mbuf) + mq_mbuf_bytes(D, NC));
  int* desc_ready = sint;      // [kDescBlocks] descriptor block held by each ring block
  int* claim = sint + 8;       // [SL] next ordinal of each slice
  int* sflag = sint + 12;      // [0] a bounded wait gave up
  int* mflag = sint + 16;      // [2 NW] segments a warp's tickets completed
  int* slot_pend = sint + 32;  // [R] slices still to read each slot
  int* slot_ord = sint + 64;   // [R] ordinal last issued into each slot (-1: none)
  int32_t* pfx = sint + kSmemInts;     // [B+1] pages
  int32_t* nzp = pfx + (p.B + 1);      // [B+1] non-empty seqs
  int32_t* ctxs = nzp + (p.B + 1);     // [B]
  int32_t* gns = ctxs + p.B;  // [B] pages before a sliding window's gap (all pages if none)
  int32_t* gsk = gns + p.B;   // [B] pages the gap skips
  const int64_t Gn = gridDim.x;

  // ---- prologue: pages per sequence, prefix sums of pages and of non-empty
  // sequences
  if (tid == 0) {
    pfx[0] = 0;
    nzp[0] = 0;
  }
  if (tid < kSmemInts) sint[tid] = (tid < 8 || tid >= 64) ? -1 : (tid >= 32 ? SL : 0);
  for (int b = tid; b < p.B; b += blockDim.x) {
    int c = p.context_lens[b];
    int np = 0;
    if (c < 0 || c > p.MBS * kPageSize) {
      if (blockIdx.x == 0) report_error(p.err_word, PKV_ERR_BOUNDS);
      c = 0;
    } else {
      np = (c + kPageSize - 1) / kPageSize;
    }
    // with a sliding window the pages between the sink pages and the first
    // page any query's window reaches are never read: a sequence's units are
    // its visible pages only
    int ns = np, sk = 0;
    if (p.window > 0 && np > 0) {
      const int lo = max(0, c - p.qlen - p.window + 1);  // first position of query 0's window
      const int fw = lo / kPageSize;
      const int nsp = (min(c, p.sinks) + kPageSize - 1) / kPageSize;
      if (fw > nsp) {
        ns = nsp;
        sk = fw - nsp;
      }
    }
    ctxs[b] = c;
    gns[b] = ns;
    gsk[b] = sk;
    pfx[b + 1] = np - sk;
    nzp[b + 1] = np > 0 ? 1 : 0;
  }
  if (warp == 0) {
    if (lane < R) mbar_init(smem_u32(&bars[lane]), 1);
    if constexpr (PS > 1) {
      if (lane < SL) {  // per slice: full (even, odd flushes), empty
        mbar_init(smem_u32(fbar + 4 * lane + 0), (PS - 1) * 32);
        mbar_init(smem_u32(fbar + 4 * lane + 1), (PS - 1) * 32);
        mbar_init(smem_u32(fbar + 4 * lane + 2), 32);
      }
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp < 2) {  // inclusive scans: warp 0 pages, warp 1 non-empty sequences
    int32_t* arr = warp == 0 ? pfx : nzp;
    int carry = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int idx = b0 + lane + 1;
      int v = (idx <= p.B) ? arr[idx] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += u;
      }
      if (idx <= p.B) arr[idx] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();

  const int64_t W = (int64_t)p.Hkv * pfx[p.B];  // all (b, h, page) units
  // Shares are equal in cost, not in pages: a page costs 1 and the start of a
  // segment kSegCost more (the state merge, output write and pipeline refill
  // a segment change takes), so CTAs whose share holds many short segments
  // get fewer pages.  Unit x of segment (b, h) costs from
  //   X(x) = Hkv (pfx[b] + kSegCost nzp[b]) + h (np_b + kSegCost) + kSegCost + (x - start)
  // and CTA c owns the units with c T / Gs <= X(x) < (c+1) T / Gs, T the total
  // cost, Gs the CTAs given work (each about kRangeMin pages or more).
  const int64_t Tc = W + (int64_t)p.Hkv * kSegCost * nzp[p.B];
  const int64_t Gs_raw = (Tc + kRangeMin - 1) / kRangeMin;
  const int64_t Gs = Gs_raw < Gn ? (Gs_raw > 0 ? Gs_raw : 1) : Gn;
  auto seq_cost0 = [&](int b) -> int64_t {
    return (int64_t)p.Hkv * (pfx[b] + (int64_t)kSegCost * nzp[b]);
  };
  // first unit whose cost position is >= P (W when none)
  auto unit_at_cost = [&](int64_t P) -> int64_t {
    if (P >= Tc) return W;
    int a = 0, z = p.B;
    while (z - a > 1) {
      const int mid = (a + z) >> 1;
      if (seq_cost0(mid) <= P) a = mid; else z = mid;
    }
    const int64_t np = pfx[a + 1] - pfx[a];
    const int64_t r = P - seq_cost0(a);
    const int64_t hh = r / (np + kSegCost);
    const int64_t off = r - hh * (np + kSegCost) - kSegCost;
    return (int64_t)p.Hkv * pfx[a] + hh * np + (off > 0 ? off : 0);
  };
  const int64_t sh_lo = blockIdx.x < Gs ? unit_at_cost((Tc * blockIdx.x + Gs - 1) / Gs) : W;
  const int64_t sh_hi = blockIdx.x < Gs ? unit_at_cost((Tc * (blockIdx.x + 1) + Gs - 1) / Gs) : W;
  const int N = (int)(sh_hi - sh_lo);  // this CTA's pages
  // the CTA whose share holds unit x of sequence b, KV head h
  auto cta_of = [&](int64_t x, int b, int64_t h) -> int64_t {
    const int64_t np = pfx[b + 1] - pfx[b];
    const int64_t start = (int64_t)p.Hkv * pfx[b] + h * np;
    const int64_t X = seq_cost0(b) + h * (np + kSegCost) + kSegCost + (x - start);
    return X * Gs / Tc;
  };
  auto seq_of = [&](int64_t x) -> int {
    int a = 0, z = p.B;
    while (z - a > 1) {
      const int mid = (a + z) >> 1;
      if ((int64_t)p.Hkv * pfx[mid] <= x) a = mid; else z = mid;
    }
    return a;
  };
  // Segments with pages are numbered in order: gsid(b, h) = nzp[b] Hkv + h.
  // The share's segments are gsid g0 .. g0 + nseg - 1, flushed in that order
  // by every warp.
  auto gsid_of_unit = [&](int64_t x) -> int {
    const int b = seq_of(x);
    const int64_t np = pfx[b + 1] - pfx[b];
    return nzp[b] * p.Hkv + (int)((x - (int64_t)p.Hkv * pfx[b]) / np);
  };
  const int g0 = N > 0 ? gsid_of_unit(sh_lo) : 0;
  const int nseg = N > 0 ? gsid_of_unit(sh_hi - 1) - g0 + 1 : 0;
  auto seq_of_gsid = [&](int g) -> int {  // the (non-empty) sequence of segment g
    const int k = g / p.Hkv;
    int a = 0, z = p.B;
    while (z - a > 1) {
      const int mid = (a + z) >> 1;
      if (nzp[mid] <= k) a = mid; else z = mid;
    }
    return a;
  };
  // A descriptor's y: tokens from the page's start to the context's end
  // (capped at kRemCap), then, for a page a sliding window cuts, the rows
  // before query 0's window start and the sink rows, and a flag.
  auto page_info = [&](int b, int pg) -> int {
    const int pos = pg * kPageSize;
    int y = min(kRemCap, ctxs[b] - pos);
    if (p.window > 0) {
      const int wr = ctxs[b] - p.qlen - p.window + 1 - pos;  // query 0: rows >= wr visible
      const int sr = p.sinks - pos;                          // rows < sr always visible
      if (wr + p.qlen - 1 > 0 && sr < kPageSize) {
        const int wrc = wr < -8 ? -8 : (wr > 24 ? 24 : wr);
        const int src = sr < 0 ? 0 : sr;
        y |= (src << 6) | ((wrc + 8) << 11) | kWinFlag;
      }
    }
    return y;
  };

  // ---- descriptors: one per ordinal, {TMA row or -1, page_info, b, h}, in
  // a ring of kDescN written 32 at a time by the lanes of one warp.  The
  // table loads are issued first (fill_issue) and the ring written a page
  // later (fill_commit), so they never stall the warp.
  int fi_f = -1, fi_blk = -1, fi_info = 0, fi_b = 0, fi_h = 0;
  bool fi_has = false;  // this lane's ordinal is in the share
  auto fill_issue = [&](int f) {
    fi_f = f;
    const int o = f * kDescBlock + lane;
    fi_has = o < N;
    if (fi_has) {
      const int64_t x = sh_lo + o;
      const int b = seq_of(x);
      const int np = pfx[b + 1] - pfx[b];
      const int64_t rr = x - (int64_t)p.Hkv * pfx[b];
      const int h = (int)(rr / np);
      const int pgu = (int)(rr - (int64_t)h * np);  // unit within the segment
      const int pg = pgu < gns[b] ? pgu : pgu + gsk[b];
      fi_blk = p.block_tables[(int64_t)b * p.MBS + pg];
      fi_info = page_info(b, pg);
      fi_b = b;
      fi_h = h;
      if (o == 0 || pgu == 0) {  // a segment starts here: warm its q rows in L2
        for (int i = 0; i < p.qlen; ++i) {
          const char* qp = reinterpret_cast<const char*>(p.q) +
                           (((int64_t)b * p.qlen + i) * p.Hq + h * G) * D * 2;
          for (int off = 0; off < G * D * 2; off += 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(qp + off));
        }
      }
    }
  };
  auto fill_commit = [&]() {
    if (fi_f < 0) return;
    if (fi_has) {
      int row = -1;
      if (fi_blk >= 0 && fi_blk < p.NB) row = (fi_blk * p.Hkv + fi_h) * kPageSize;
      else report_error(p.err_word, PKV_ERR_BOUNDS);
      desc[(fi_f * kDescBlock + lane) % kDescN] = make_int4(row, fi_info, fi_b, fi_h);
    }
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      st_volatile_s32(&desc_ready[fi_f % kDescBlocks], fi_f);
    }
    fi_f = -1;
  };
  // bounded wait until the descriptor of ordinal o is written (one lane)
  auto desc_wait = [&](int o) -> bool {
    const int f = o / kDescBlock;
    if (ld_volatile_s32(&desc_ready[f % kDescBlocks]) != f) {
      uint64_t t0, t1;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
      while (ld_volatile_s32(&desc_ready[f % kDescBlocks]) != f) {
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
        if (t1 - t0 > kWaitLimitNs) return false;
        __nanosleep(64);
      }
    }
    __threadfence_block();
    return true;
  };

  if (lane == 0) {
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  const uint64_t pol = l2_policy_evict_first();

  // the first two descriptor blocks need nothing the previous kernel writes
  // (lengths and tables only)
  if (warp < kFillAhead && warp * kDescBlock < N) {
    fill_issue(warp);
    fill_commit();
  }
  __syncthreads();

  // From here on the kernel touches data the previous kernel on the stream may
  // write (cache pages, q, outputs, workspace): wait for it.
  if (p.early_prologue) griddep_wait();

  // one thread: load ordinal o into slot o % R
  auto issue = [&](int o) {
    const int4 dsc = desc[o % kDescN];
    const int slot = o % R;
    const uint32_t bar = smem_u32(&bars[slot]);
    const uint32_t kt = ring + (uint32_t)(slot * C::kStageBytes);
    const uint32_t vt = kt + C::kTileBytes;
    // a reader of ordinal o waits on the slot's barrier only once this is
    // o: the barrier is then in o's phase (its previous phase, ordinal o - R,
    // completed and was read), so its parity test cannot be satisfied by a
    // phase one behind
    st_volatile_s32(&slot_ord[slot], o);
    if (dsc.x >= 0) {
      mbar_arrive_expect_tx(bar, C::kStageBytes + C::kScaleBytes);
#pragma unroll
      for (int bx = 0; bx < C::kBoxes; ++bx) {
        tma_load_2d(kt + bx * C::kBoxBytes, &tmk, bar, bx * (128 / C::kElem), dsc.x, pol);
        tma_load_2d(vt + bx * C::kBoxBytes, &tmv, bar, bx * (128 / C::kElem), dsc.x, pol);
      }
      if constexpr (kTok) {  // the page's 16 K scales, then its 16 V scales: one line
        bulk_load(scl + (uint32_t)(slot * C::kScaleBytes), p.k_scale + 2 * dsc.x,
                  C::kScaleBytes, bar, pol);
      }
    } else {
      mbar_arrive(bar);  // nothing to load; complete the phase
    }
  };
  if (lane == 0) {
    const int n0 = N < R ? N : R;
    for (int o = warp; o < n0; o += NW) issue(o);
  }

  // sequences with no tokens get a zero output row (spread over CTAs)
  for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
    if (pfx[b + 1] != pfx[b]) continue;
    const int64_t row0 = (int64_t)b * p.qlen * p.Hq * D;
    for (int i = tid; i < p.qlen * p.Hq * D; i += blockDim.x)
      store_out_rt(p.out_dtype, p.out, row0 + i, 0.f);
  }

  // ---- per-lane fragment coordinates
  const int c4 = lane & 3;   // C-fragment column pair: columns 2*c4, 2*c4+1 of a group
  const int r8 = lane >> 2;  // C-fragment row: token r8 / r8+8, or O^T row r8 / r8+8
  const int qk_tok = (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix row, K page
  const int qk_chunk_hi = lane >> 4;
  const int pv_tok = (lane & 7) + (lane >> 4) * 8;        // ldmatrix row, V page (trans)
  const int pv_chunk_hi = (lane >> 3) & 1;

  // d of O^T rows r8 and r8 + 8 in m-tile mt
  auto d_of = [&](int mt, int half) -> int {
    if constexpr (!kFp8) return 16 * mt + r8 + 8 * half;
    else return 32 * (mt >> 1) + 2 * r8 + (mt & 1) + 16 * half;
  };
  // first column of column group cg of this warp
  auto col_base = [&](int cg) -> int { return (slice * CW + cg) * 8; };

  uint32_t qf[C::kKSteps][CW][2];
  float o[kMT][CW][4];
  float m2[CW][2], l2[CW][2];
  // score scale in log2 units (E4M3: times the K scale) for the lane's two
  // C-fragment columns 2 c4 and 2 c4 + 1 of each group
  float c2a[CW], c2b[CW];

  auto reset_state = [&]() {
#pragma unroll
    for (int cg = 0; cg < CW; ++cg) {
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][cg][e] = 0.f;
      m2[cg][0] = m2[cg][1] = -INFINITY;
      l2[cg][0] = l2[cg][1] = 0.f;
    }
  };

  // row of q / out for column c of segment (b, h): query token c / G,
  // query head h * G + c % G; the column is real when c < G * p.qlen
  auto col_row = [&](int b, int h, int c) -> int64_t {
    return ((int64_t)b * p.qlen + c / G) * p.Hq + h * G + c % G;
  };
  auto col_real = [&](int c) -> bool { return c < NC && c < G * p.qlen; };

  auto load_q = [&](int b, int h) {
#pragma unroll
    for (int cg = 0; cg < CW; ++cg) {
      const int col = col_base(cg) + r8;  // B-fragment column n = lane / 4
      const bool real = col_real(col);
      const uint16_t* qrow =
          reinterpret_cast<const uint16_t*>(p.q) + (real ? col_row(b, h, col) : 0) * D;
      if constexpr (!kFp8) {
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
          uint32_t b0 = 0, b1 = 0;
          if (real) {
            b0 = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c4);
            b1 = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c4 + 8);
          }
          qf[ks][cg][0] = b0;
          qf[ks][cg][1] = b1;
        }
        c2a[cg] = c2b[cg] = p.scale_log2;
      } else {
        // FP8 pages meet q on the fp16 MMA.  A bf16 q can lie outside fp16's
        // range, so each column is brought to [2^14, 2^15) by a power of two
        // (exact), which the column's score scale undoes (also exact).
        uint2 raw4[C::kKSteps];
        float amax = 0.f;
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
          raw4[ks] = make_uint2(0u, 0u);
          if (real) raw4[ks] = *reinterpret_cast<const uint2*>(qrow + 16 * ks + 4 * c4);
          if constexpr (QBF16) {
            const float2 f01 = unpack2<true>(raw4[ks].x), f23 = unpack2<true>(raw4[ks].y);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(f01.x), fabsf(f01.y)),
                                     fmaxf(fabsf(f23.x), fabsf(f23.y))));
          }
        }
        int e = 0;  // column scale 2^e
        if constexpr (QBF16) {
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
          if (amax > 0.f)
            e = min(112, max(-112, ((__float_as_int(amax) >> 23) & 0xff) - 127 - 14));
        }
        const float down = __int_as_float((127 - e) << 23);
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
          const float2 f01 = unpack2<QBF16>(raw4[ks].x);
          const float2 f23 = unpack2<QBF16>(raw4[ks].y);
          qf[ks][cg][0] = pack2<false>(f01.x * down, f01.y * down);
          qf[ks][cg][1] = pack2<false>(f23.x * down, f23.y * down);
        }
        // the lane's C-fragment columns 2 c4, 2 c4 + 1 are B-fragment columns
        // of lanes 8 c4 and 8 c4 + 4
        const int ea = __shfl_sync(0xffffffffu, e, 8 * c4);
        const int eb = __shfl_sync(0xffffffffu, e, 8 * c4 + 4);
        float c2 = p.scale_log2;
        if constexpr (CACHE == kCacheE4M3) c2 *= p.k_scale[h];
        c2a[cg] = c2 * __int_as_float((127 + ea) << 23);
        c2b[cg] = c2 * __int_as_float((127 + eb) << 23);
      }
    }
  };

  // ---- S^T[16 tok][8] = K . Q^T for one page and every column group, on
  // two accumulator chains per group
  auto qk_page = [&](uint32_t kt, float (&s)[CW][4]) {
    float s2[CW][4];
#pragma unroll
    for (int cg = 0; cg < CW; ++cg)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[cg][e] = s2[cg][e] = 0.f;
    if constexpr (!kFp8) {
#pragma unroll
      for (int ks = 0; ks < C::kKSteps; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, kt + swz(qk_tok, 2 * ks + qk_chunk_hi));
#pragma unroll
        for (int cg = 0; cg < CW; ++cg) {
          if (ks & 1) mma_16816<kBF>(s2[cg], a, qf[ks][cg][0], qf[ks][cg][1]);
          else mma_16816<kBF>(s[cg], a, qf[ks][cg][0], qf[ks][cg][1]);
        }
      }
    } else {
#pragma unroll
      for (int gi = 0; gi < D / 32; ++gi) {
        uint32_t r[4];
        ldsm_x4(r, kt + swz(qk_tok, 2 * gi + qk_chunk_hi));
        uint32_t a[4];
        a[0] = e4m3x2_to_f16x2(r[0]);
        a[1] = e4m3x2_to_f16x2(r[1]);
        a[2] = e4m3x2_to_f16x2(r[0] >> 16);
        a[3] = e4m3x2_to_f16x2(r[1] >> 16);
#pragma unroll
        for (int cg = 0; cg < CW; ++cg)
          mma_16816<false>(s[cg], a, qf[2 * gi][cg][0], qf[2 * gi][cg][1]);
        a[0] = e4m3x2_to_f16x2(r[2]);
        a[1] = e4m3x2_to_f16x2(r[3]);
        a[2] = e4m3x2_to_f16x2(r[2] >> 16);
        a[3] = e4m3x2_to_f16x2(r[3] >> 16);
#pragma unroll
        for (int cg = 0; cg < CW; ++cg)
          mma_16816<false>(s2[cg], a, qf[2 * gi + 1][cg][0], qf[2 * gi + 1][cg][1]);
      }
    }
#pragma unroll
    for (int cg = 0; cg < CW; ++cg)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[cg][e] += s2[cg][e];
  };

  // ---- O^T += V^T . P^T for one page; V rows of masked tokens are zeroed
  // (they may hold anything, and 0 * NaN would poison the sum)
  auto pv_page = [&](uint32_t vt, int valid, const uint32_t (&bh)[CW][2],
                     const uint32_t (&bl)[CW][2]) {
    uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
    if (valid < kPageSize) {
      const int t0 = 2 * c4;
      mlo = (t0 < valid ? 0x0000ffffu : 0u) | (t0 + 1 < valid ? 0xffff0000u : 0u);
      mhi = (t0 + 8 < valid ? 0x0000ffffu : 0u) | (t0 + 9 < valid ? 0xffff0000u : 0u);
    }
    if constexpr (!kFp8) {
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        uint32_t a[4];
        ldsm_x4_trans(a, vt + swz(pv_tok, 2 * mt + pv_chunk_hi));
        a[0] &= mlo;
        a[1] &= mlo;
        a[2] &= mhi;
        a[3] &= mhi;
#pragma unroll
        for (int cg = 0; cg < CW; ++cg) {
          mma_16816<kBF>(o[mt][cg], a, bh[cg][0], bh[cg][1]);
          mma_16816<kBF>(o[mt][cg], a, bl[cg][0], bl[cg][1]);
        }
      }
    } else {
#pragma unroll
      for (int gi = 0; gi < D / 32; ++gi) {
        uint32_t r[4];
        ldsm_x4_trans(r, vt + swz(pv_tok, 2 * gi + pv_chunk_hi));
        uint32_t a[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) a[e] = e4m3x2_to_f16x2(__byte_perm(r[e], 0, 0x0020));
        a[0] &= mlo;
        a[1] &= mlo;
        a[2] &= mhi;
        a[3] &= mhi;
#pragma unroll
        for (int cg = 0; cg < CW; ++cg) {
          mma_16816<false>(o[2 * gi][cg], a, bh[cg][0], bh[cg][1]);
          mma_16816<false>(o[2 * gi][cg], a, bl[cg][0], bl[cg][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) a[e] = e4m3x2_to_f16x2(__byte_perm(r[e], 0, 0x0031));
        a[0] &= mlo;
        a[1] &= mlo;
        a[2] &= mhi;
        a[3] &= mhi;
#pragma unroll
        for (int cg = 0; cg < CW; ++cg) {
          mma_16816<false>(o[2 * gi + 1][cg], a, bh[cg][0], bh[cg][1]);
          mma_16816<false>(o[2 * gi + 1][cg], a, bl[cg][0], bl[cg][1]);
        }
      }
    }
  };

  // ---- NP (1 or 2) pages of one segment: their scores, one online-
  // softmax update over all their tokens (log2 domain; tokens past the
  // context are masked), then P.V.  Several pages give the warp independent
  // MMA chains and fewer reductions per token.
  auto compute_pages = [&](auto npc, const uint32_t* kt, const int* valids) {
    constexpr int NP = decltype(npc)::value;
    float x[NP][CW][4];
    float ksc[NP][2], vsc[NP][2];  // per-token K and V scales of rows r8, r8 + 8
    if constexpr (kTok) {  // read first: their latency hides under the QK MMAs
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        const uint32_t sp = scl + ((kt[i] - ring) / C::kStageBytes) * C::kScaleBytes;
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(ksc[i][0]) : "r"(sp + r8 * 4));
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(ksc[i][1]) : "r"(sp + (r8 + 8) * 4));
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(vsc[i][0]) : "r"(sp + (kPageSize + r8) * 4));
        asm volatile("ld.shared.f32 %0, [%1];"
                     : "=f"(vsc[i][1]) : "r"(sp + (kPageSize + r8 + 8) * 4));
      }
    }
#pragma unroll
    for (int i = 0; i < NP; ++i) qk_page(kt[i], x[i]);
    float mx[CW][2];
#pragma unroll
    for (int cg = 0; cg < CW; ++cg) mx[cg][0] = mx[cg][1] = -INFINITY;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const int v = valids[i];
      const int rem = v & kRemMask;  // tokens from the page's start to the context's end
      if constexpr (kTok) {
        if (r8 >= rem) vsc[i][0] = 0.f;  // their P is 0; their scale may be anything
        if (r8 + 8 >= rem) vsc[i][1] = 0.f;
      }
#pragma unroll
      for (int cg = 0; cg < CW; ++cg) {
        float (&xx)[4] = x[i][cg];
#pragma unroll
        for (int e = 0; e < 4; ++e) xx[e] *= (e & 1) ? c2b[cg] : c2a[cg];
        if constexpr (kTok) {
          xx[0] *= ksc[i][0];  // rows past the context are masked below
          xx[1] *= ksc[i][0];
          xx[2] *= ksc[i][1];
          xx[3] *= ksc[i][1];
        }
        if constexpr (QC == 1) {
          if (rem < kPageSize) {
            if (r8 >= rem) xx[0] = xx[1] = -INFINITY;
            if (r8 + 8 >= rem) xx[2] = xx[3] = -INFINITY;
          }
          if (v & kWinFlag) {  // rows before the window's start that are no sinks
            const int sr = (v >> 6) & 15, wr = ((v >> 11) & 63) - 8;
            if (r8 < wr && r8 >= sr) xx[0] = xx[1] = -INFINITY;
            if (r8 + 8 < wr && r8 + 8 >= sr) xx[2] = xx[3] = -INFINITY;
          }
        } else {
          const int c0 = col_base(cg) + 2 * c4, c1 = c0 + 1;
          const int j0 = col_real(c0) ? c0 / G : p.qlen - 1;
          const int j1 = col_real(c1) ? c1 / G : p.qlen - 1;
          if (rem < kPageSize + QC - 1) {
            // causal among the new tokens: query token j of the last qlen
            // sees the page's first rem - (qlen - 1 - j) tokens
            const int l0 = rem - (p.qlen - 1 - j0), l1 = rem - (p.qlen - 1 - j1);
            if (r8 >= l0) xx[0] = -INFINITY;
            if (r8 >= l1) xx[1] = -INFINITY;
            if (r8 + 8 >= l0) xx[2] = -INFINITY;
            if (r8 + 8 >= l1) xx[3] = -INFINITY;
          }
          if (v & kWinFlag) {  // query token j's window starts j rows after token 0's
            const int sr = (v >> 6) & 15, wr = ((v >> 11) & 63) - 8;
            const int w0 = wr + j0, w1 = wr + j1;
            if (r8 < w0 && r8 >= sr) xx[0] = -INFINITY;
            if (r8 < w1 && r8 >= sr) xx[1] = -INFINITY;
            if (r8 + 8 < w0 && r8 + 8 >= sr) xx[2] = -INFINITY;
            if (r8 + 8 < w1 && r8 + 8 >= sr) xx[3] = -INFINITY;
          }
        }
        mx[cg][0] = fmaxf(mx[cg][0], fmaxf(xx[0], xx[2]));
        mx[cg][1] = fmaxf(mx[cg][1], fmaxf(xx[1], xx[3]));
      }
    }
    bool grow = false;
#pragma unroll
    for (int cg = 0; cg < CW; ++cg) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx[cg][0] = fmaxf(mx[cg][0], __shfl_xor_sync(0xffffffffu, mx[cg][0], off));
        mx[cg][1] = fmaxf(mx[cg][1], __shfl_xor_sync(0xffffffffu, mx[cg][1], off));
      }
      grow = grow || (mx[cg][0] > m2[cg][0] + kRescaleThreshold) ||
             (mx[cg][1] > m2[cg][1] + kRescaleThreshold);
    }
    if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
      for (int cg = 0; cg < CW; ++cg) {
        const float n0 = fmaxf(m2[cg][0], mx[cg][0]), n1 = fmaxf(m2[cg][1], mx[cg][1]);
        float a0 = exp2f(m2[cg][0] - n0), a1 = exp2f(m2[cg][1] - n1);
        if constexpr (QC > 1) {  // a column that has seen nothing yet stays as it is
          if (n0 == -INFINITY) a0 = 1.f;
          if (n1 == -INFINITY) a1 = 1.f;
        }
        m2[cg][0] = n0;
        m2[cg][1] = n1;
        l2[cg][0] *= a0;
        l2[cg][1] *= a1;
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
          o[mt][cg][0] *= a0;
          o[mt][cg][1] *= a1;
          o[mt][cg][2] *= a0;
          o[mt][cg][3] *= a1;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      uint32_t bh[CW][2], bl[CW][2];
#pragma unroll
      for (int cg = 0; cg < CW; ++cg) {
        // a column every token so far was masked for keeps m = -inf: weigh
        // its (all -inf) scores against 0, not -inf (only with QC > 1)
        float mu0 = m2[cg][0], mu1 = m2[cg][1];
        if constexpr (QC > 1) {
          if (mu0 == -INFINITY) mu0 = 0.f;
          if (mu1 == -INFINITY) mu1 = 0.f;
        }
        float p0 = exp2f(x[i][cg][0] - mu0), p1 = exp2f(x[i][cg][1] - mu1);
        float p2 = exp2f(x[i][cg][2] - mu0), p3 = exp2f(x[i][cg][3] - mu1);
        l2[cg][0] += p0 + p2;
        l2[cg][1] += p1 + p3;
        if constexpr (kTok) {  // P.V weights carry each token's V scale
          p0 *= vsc[i][0];
          p1 *= vsc[i][0];
          p2 *= vsc[i][1];
          p3 *= vsc[i][1];
        }
        // P as hi + lo 16-bit parts, transposed into B fragments
        const uint32_t h01 = pack2<kBF>(p0, p1), h23 = pack2<kBF>(p2, p3);
        const float2 f01 = unpack2<kBF>(h01), f23 = unpack2<kBF>(h23);
        const uint32_t l01 = pack2<kBF>(p0 - f01.x, p1 - f01.y);
        const uint32_t l23 = pack2<kBF>(p2 - f23.x, p3 - f23.y);
        bh[cg][0] = movm_trans(h01);
        bh[cg][1] = movm_trans(h23);
        bl[cg][0] = movm_trans(l01);
        bl[cg][1] = movm_trans(l23);
      }
      const int vrows = valids[i] & kRemMask;
      pv_page(kt[i] + C::kTileBytes, vrows < kPageSize ? vrows : kPageSize, bh, bl);
    }
  };
  auto compute_page = [&](uint32_t kt, int valid) {
    const uint32_t kt1[1] = {kt};
    const int v1[1] = {valid};
    compute_pages(Int<1>{}, kt1, v1);
  };

  // ---- fused append (16-bit caches): the page holding a sequence's newest
  // position gets that token's K and V row from the step's inputs, in the
  // staged copy (so this pass attends to it) and in the cache (for later
  // steps).  The page (b, h) is staged once and read by this warp alone, so
  // nothing else in the grid reads the row.
  auto append_new = [&](uint32_t kt, int tma_row, int r, int b, int h) {
    if (lane < D / 8) {  // 8 elements (16 bytes) per lane
      const int64_t src = ((int64_t)b * p.Hkv + h) * (D / 8) + lane;
      const uint4 kin = reinterpret_cast<const uint4*>(p.k_new)[src];
      const uint4 vin = reinterpret_cast<const uint4*>(p.v_new)[src];
      const int64_t dst = ((int64_t)tma_row + r) * (D / 8) + lane;
      reinterpret_cast<uint4*>(p.k_cache)[dst] = kin;
      reinterpret_cast<uint4*>(p.v_cache)[dst] = vin;
      const uint32_t off = swz(r, lane);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(kt + off), "r"(kin.x),
                   "r"(kin.y), "r"(kin.z), "r"(kin.w) : "memory");
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(kt + C::kTileBytes + off),
                   "r"(vin.x), "r"(vin.y), "r"(vin.z), "r"(vin.w) : "memory");
      // the slot is refilled by the tensor-copy (async) proxy later
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncwarp();
  };

  // ---- merging warp states through shared memory: element i of the lane
  // state (per column group: m[2], l[2], o[MT][4]) at buf[i * S + li]
  auto store_state_at = [&](float* buf, int li, int S) {
#pragma unroll
    for (int cg = 0; cg < CW; ++cg) {
      float* bg = buf + cg * kGS * S;
      bg[0 * S + li] = m2[cg][0];
      bg[1 * S + li] = m2[cg][1];
      bg[2 * S + li] = l2[cg][0];
      bg[3 * S + li] = l2[cg][1];
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) bg[(4 + 4 * mt + e) * S + li] = o[mt][cg][e];
    }
  };
  auto merge_state_at = [&](const float* buf, int li, int S) {
#pragma unroll
    for (int cg = 0; cg < CW; ++cg) {
      const float* bg = buf + cg * kGS * S;
      float a[2], bw[2];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const float mb = bg[cc * S + li];
        const float M = fmaxf(m2[cg][cc], mb);
        if (M == -INFINITY) {
          a[cc] = 1.f;
          bw[cc] = 0.f;
        } else {
          a[cc] = exp2f(m2[cg][cc] - M);
          bw[cc] = exp2f(mb - M);
          m2[cg][cc] = M;
        }
        l2[cg][cc] = a[cc] * l2[cg][cc] + bw[cc] * bg[(2 + cc) * S + li];
      }
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          o[mt][cg][e] = a[e & 1] * o[mt][cg][e] + bw[e & 1] * bg[(4 + 4 * mt + e) * S + li];
    }
  };
  auto store_state = [&](float* buf) { store_state_at(buf, lane, 32); };
  auto merge_state = [&](const float* buf) { merge_state_at(buf, lane, 32); };

  // ---- merging the partials of a completed segment.  Threads t, t+T, ...
  // (T threads: one warp mid-kernel, the whole CTA at exit) take float4
  // columns t, t+T, ...; each column adds its head's partials in slot order
  // (against a running maximum for up to four partials, else against their
  // common maximum), so the result is bitwise the same whichever form runs.
  // No shared memory, no barrier.
  auto merge_cols = [&](int seg, int t, int T) {
    const int b = seg / p.Hkv, h = seg - (seg / p.Hkv) * p.Hkv;
    const int64_t np = pfx[b + 1] - pfx[b];
    const int64_t s0 = (int64_t)p.Hkv * pfx[b] + (int64_t)h * np;
    const int64_t c0 = cta_of(s0, b, h);
    const int count = (int)(cta_of(s0 + np - 1, b, h) - c0 + 1);
    const int64_t slot_base = c0 + seg;  // the partials of CTAs c0 .. c0 + count - 1
    constexpr int kCols = NC * D / 4;
#pragma unroll 1
    for (int col = t; col < kCols; col += T) {
      const int head = col / (D / 4);  // MMA column (query token, head)
      if (!col_real(head)) continue;
      const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + slot_base * PC + head;
      const float4* vo = reinterpret_cast<const float4*>(p.part_o + slot_base * PC * D) + col;
      float M = -INFINITY, lsum = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (count <= 4) {
        // a few partials: one pass in slot order, the running reference
        // moving up to each new maximum and what was summed brought down to
        // it, so all their loads go out at once
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          if (kk < count) {
            const float2 v = __ldcg(ml + (int64_t)kk * PC);
            const float4 x = __ldcg(vo + (int64_t)kk * (PC * D / 4));
            if (v.y > 0.f) {
              if (v.x > M) {
                const float a = exp2f(M - v.x);  // 0 while nothing is summed
                lsum *= a;
                acc.x *= a;
                acc.y *= a;
                acc.z *= a;
                acc.w *= a;
                M = v.x;
              }
              const float w = exp2f(v.x - M);
              lsum += w * v.y;
              acc.x += w * x.x;
              acc.y += w * x.y;
              acc.z += w * x.z;
              acc.w += w * x.w;
            }
          }
        }
      } else {
        // many: the common maximum first, then the weighted sum (the
        // exponentials independent of one another)
#pragma unroll 4
        for (int kk = 0; kk < count; ++kk) {
          const float2 v = __ldcg(ml + (int64_t)kk * PC);
          if (v.y > 0.f) M = fmaxf(M, v.x);
        }
        if (M > -INFINITY) {
#pragma unroll 4
          for (int kk = 0; kk < count; ++kk) {
            const float2 v = __ldcg(ml + (int64_t)kk * PC);
            const float4 x = __ldcg(vo + (int64_t)kk * (PC * D / 4));
            const float w = v.y > 0.f ? exp2f(v.x - M) : 0.f;
            lsum += w * v.y;
            acc.x += w * x.x;
            acc.y += w * x.y;
            acc.z += w * x.z;
            acc.w += w * x.w;
          }
        }
      }
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      const int64_t ob = col_row(b, h, head) * D + (col % (D / 4)) * 4;
      store_out_rt(p.out_dtype, p.out, ob + 0, acc.x * inv);
      store_out_rt(p.out_dtype, p.out, ob + 1, acc.y * inv);
      store_out_rt(p.out_dtype, p.out, ob + 2, acc.z * inv);
      store_out_rt(p.out_dtype, p.out, ob + 3, acc.w * inv);
    }
  };
  auto merge_segment = [&](int seg) {  // all threads
    merge_cols(seg, tid, NW * 32);
    if (tid == 0) p.tickets[seg] = 0;  // ready for the next call
  };
  auto merge_segment_warp = [&](int seg) {  // one warp
    merge_cols(seg, lane, 32);
    if (lane == 0) p.tickets[seg] = 0;
  };

  // A CTA learns it completed a split segment from the page-count ticket
  // (each slice adds the CTA's pages of the segment).  The warp that stored a
  // partial does not fence right away (under full memory load the fence
  // waits microseconds for its stores to land): its lane 0 publishes it
  // (fence, then an atomic add of its pages) at its next segment change, when
  // the stores are long done, and reads the atomic's result one segment
  // change later still (or at exit).
  int pub_seg = -1, pub_add = 0;               // lane 0: partial stored, not yet published
  int iss_seg = -1, iss_old = 0, iss_add = 0;  // lane 0: ticket added, result not yet read
  bool dead = false;   // a bounded wait gave up: skip compute and waits
  auto set_dead = [&]() {
    if (!dead) {
      dead = true;
      if (lane == 0) {
        report_error(p.err_word, PKV_ERR_TIMEOUT);
        st_volatile_s32(&sflag[0], 1);
      }
    }
  };
  auto seg_pages = [&](int seg) -> int {
    const int b = seg / p.Hkv;
    return pfx[b + 1] - pfx[b];
  };
  // lane 0: publish / resolve; m0, m1 get the segments this CTA completed
  // (-1: none); only the final call waits for the atomic it issues
  auto tickets_lane0 = [&](bool final_call, int& m0, int& m1) {
    m0 = -1;
    m1 = -1;
    if (iss_seg >= 0) {
      if (iss_old + iss_add == SL * seg_pages(iss_seg)) m0 = iss_seg;
      iss_seg = -1;
    }
    if (pub_seg >= 0) {
      __threadfence();  // release: this warp's partial before its pages count
      iss_old = atomicAdd(&p.tickets[pub_seg], pub_add);
      iss_seg = pub_seg;
      iss_add = pub_add;
      pub_seg = -1;
      if (final_call) {
        if (iss_old + iss_add == SL * seg_pages(iss_seg)) m1 = iss_seg;
        iss_seg = -1;
      }
    }
  };
  auto tickets_at_flush = [&]() {  // every warp, at each segment change
    int m0 = -1, m1 = -1;
    if (lane == 0) tickets_lane0(false, m0, m1);
    m0 = __shfl_sync(0xffffffffu, m0, 0);
    if (m0 >= 0) {
      __threadfence();  // acquire: the other contributors' partials
      merge_segment_warp(m0);
    }
  };

  // ---- the merged state of a segment: write the output (whole segment in
  // this share) or this CTA's partial of this warp's columns
  auto finish = [&](int b, int h, bool split, int pages_mine) {
    const float vs = (CACHE == kCacheE4M3) ? p.v_scale[h] : 1.f;
    const int64_t part = (int64_t)blockIdx.x + b * p.Hkv + h;
#pragma unroll
    for (int cg = 0; cg < CW; ++cg) {
      const int h0 = col_base(cg) + 2 * c4, h1 = h0 + 1;
      float lt0 = l2[cg][0], lt1 = l2[cg][1];
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        lt0 += __shfl_xor_sync(0xffffffffu, lt0, off);
        lt1 += __shfl_xor_sync(0xffffffffu, lt1, off);
      }
      if (!split) {  // the whole segment was here: normalise and write
        const float i0 = lt0 > 0.f ? vs / lt0 : 0.f;
        const float i1 = lt1 > 0.f ? vs / lt1 : 0.f;
        const bool w0 = col_real(h0), w1 = col_real(h1);
        const int64_t ob0 = (w0 ? col_row(b, h, h0) : 0) * D;
        const int64_t ob1 = (w1 ? col_row(b, h, h1) : 0) * D;
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
          const int dA = d_of(mt, 0), dB = d_of(mt, 1);
          if (w0) {
            store_out_rt(p.out_dtype, p.out, ob0 + dA, o[mt][cg][0] * i0);
            store_out_rt(p.out_dtype, p.out, ob0 + dB, o[mt][cg][2] * i0);
          }
          if (w1) {
            store_out_rt(p.out_dtype, p.out, ob1 + dA, o[mt][cg][1] * i1);
            store_out_rt(p.out_dtype, p.out, ob1 + dB, o[mt][cg][3] * i1);
          }
        }
        continue;
      }
      // partial slot cta + seg is unique: shares are contiguous and ordered,
      // so a later CTA never touches an earlier segment
      float* po = p.part_o + part * PC * D;
      float* pml = p.part_ml + part * PC * 2;
      if (r8 == 0) {
        if (h0 < NC) { pml[2 * h0] = m2[cg][0]; pml[2 * h0 + 1] = lt0; }
        if (h1 < NC) { pml[2 * h1] = m2[cg][1]; pml[2 * h1 + 1] = lt1; }
      }
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        const int dA = d_of(mt, 0), dB = d_of(mt, 1);
        if (h0 < NC) {
          po[h0 * D + dA] = o[mt][cg][0] * vs;
          po[h0 * D + dB] = o[mt][cg][2] * vs;
        }
        if (h1 < NC) {
          po[h1 * D + dA] = o[mt][cg][1] * vs;
          po[h1 * D + dB] = o[mt][cg][3] * vs;
        }
      }
    }
    if (split) {
      __syncwarp();
      if (lane == 0) {
        pub_seg = b * p.Hkv + h;
        pub_add = pages_mine;
      }
    }
  };
  // segment n of the share (gsid g0 + n): its sequence, head, whether other
  // CTAs hold some of its pages, and how many are in this share
  auto finish_seg = [&](int n) {
    const int g = g0 + n;
    const int b = seq_of_gsid(g);
    const int h = g - nzp[b] * p.Hkv;
    const int64_t np = pfx[b + 1] - pfx[b];
    const int64_t start = (int64_t)p.Hkv * pfx[b] + (int64_t)h * np;
    const int64_t end = start + np;
    const bool split = start < sh_lo || end > sh_hi;
    const int mine = (int)((end < sh_hi ? end : sh_hi) - (start > sh_lo ? start : sh_lo));
    finish(b, h, split, mine);
  };

  // ---- end of this CTA's part of segment n, for the warps of this slice.
  // Synchronous form: a barrier tree over the slice's warps; the finisher
  // (merges and writes) rotates from flush to flush.
  const int sbar = kSliceBarrier0 + slice;
  auto flush_sync = [&](int n) {
    if constexpr (PS == 1) {
      finish_seg(n);
    } else {
      float* buf0 = mbuf + (PS == 2 ? slice : 0) * C::kLaneState * 32;
      float* buf1 = mbuf + C::kLaneState * 32;
      const int wr = (sw - n) & (PS - 1);  // this warp's role
      named_barrier(sbar, PS * 32);        // the buffers are free again
      if constexpr (PS == 4) {
        if (wr >= 2) store_state(wr == 2 ? buf0 : buf1);
        named_barrier(sbar, PS * 32);
        if (wr < 2) merge_state(wr == 0 ? buf0 : buf1);
        named_barrier(sbar, PS * 32);
      }
      if (wr == 1) store_state(buf0);
      named_barrier(sbar, PS * 32);
      if (wr != 0) return;
      merge_state(buf0);
      finish_seg(n);
    }
  };
  // Asynchronous form (4 warps, NC <= 4): the three other warps drop the lanes
  // of their state that hold real columns into mbuf slots, arrive on the
  // "full" mbarrier and go on at once; the finisher waits on "full", merges,
  // frees the slots through the "empty" mbarrier and writes.  Flush n uses
  // full[n % 2] (its phase n / 2) and empty (its phase n).  No wait can see a
  // barrier two phases away from the one it tests: the finisher of flush n
  // was a writer at flush n - 1 and waited there for empty phase n - 2, which
  // the finisher of flush n - 2 completed only after full[n % 2] completed
  // its phase for flush n - 2; a writer of flush n waits for empty phase
  // n - 1, and every earlier phase of empty was waited for by the warps whose
  // arrivals complete phase n - 1.
  constexpr int kU = NC >= 4 ? NC / 2 : 1;     // C-fragment column pairs with real columns
  constexpr int kCS = C::kLaneState * 8 * kU;  // floats per compact warp state
  constexpr bool kAsyncFlush =
      CW == 1 && SL == 1 && NC <= 4 && (NW - 1) * kCS <= 2 * C::kLaneState * 32;
  auto flush_async = [&](int n) {
    const int fin = n & (NW - 1);
    const uint32_t bar_full = smem_u32(fbar + (n & 1)), bar_empty = smem_u32(fbar + 2);
    const int li = r8 * kU + c4;
    if (warp != fin) {
      if (n > 0 && !dead && !mbar_wait_bounded(bar_empty, (uint32_t)((n - 1) & 1), kWaitLimitNs))
        set_dead();
      if (c4 < kU) store_state_at(mbuf + ((warp - fin - 1) & (NW - 1)) * kCS, li, 8 * kU);
      mbar_arrive(bar_full);
      return;
    }
    if (!dead && !mbar_wait_bounded(bar_full, (uint32_t)((n >> 1) & 1), kWaitLimitNs)) set_dead();
    if (c4 < kU) {
#pragma unroll 1
      for (int sl = 0; sl < NW - 1; ++sl) merge_state_at(mbuf + sl * kCS, li, 8 * kU);
    }
    mbar_arrive(bar_empty);
    finish_seg(n);
  };
  int nfl = 0;   // segments of the share this warp has flushed
  int cur = -1;  // the segment whose state this warp holds (-1: none)
  auto flush_next = [&]() {
    tickets_at_flush();
    if constexpr (kAsyncFlush) flush_async(nfl);
    else flush_sync(nfl);
    reset_state();
    ++nfl;
  };
  // make segment s (sequence b, head h) this warp's current one: hand over
  // the state of every earlier segment (empty for those it had no page of)
  auto enter = [&](int s, int b, int h) {
    while (nfl < s) flush_next();
    if (cur != s) {
      cur = s;
      load_q(b, h);
    }
  };
  // after reading ordinal oo: the slot's last reader loads ordinal oo + R
  auto release = [&](int oo) {
    if (lane == 0) {
      bool last = true;
      if constexpr (SL > 1) {
        last = atomicSub(&slot_pend[oo % R], 1) == 1;
        if (last) slot_pend[oo % R] = SL;
      }
      if (last && oo + R < N && !ld_volatile_s32(&sflag[0])) {
        if (desc_wait(oo + R)) {
          issue(oo + R);
        } else {
          report_error(p.err_word, PKV_ERR_TIMEOUT);
          st_volatile_s32(&sflag[0], 1);
        }
      }
    }
  };
  // Readers claim ordinals up to about R + 2 NW past the oldest unread one,
  // so the load of ordinal oo may not even be issued yet (its slot still
  // holding or loading oo - R); the barrier's parity test would then see
  // the phase before and pass.  So first wait until oo is the slot's issued
  // ordinal, then for its phase.
  auto wait_slot = [&](int oo) {
    if (dead) return;
    bool ok = true;
    if (lane == 0 && ld_volatile_s32(&slot_ord[oo % R]) != oo) {
      uint64_t t0, t1;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
      while (ld_volatile_s32(&slot_ord[oo % R]) != oo) {
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
        if (t1 - t0 > kWaitLimitNs) {
          ok = false;
          break;
        }
        __nanosleep(32);
      }
    }
    if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) ||
        !mbar_wait_bounded(smem_u32(&bars[oo % R]), (uint32_t)((oo / R) & 1), kWaitLimitNs))
      set_dead();
  };
  auto sidx_of = [&](const int4& d) -> int { return nzp[d.z] * p.Hkv + d.w - g0; };

  reset_state();
  // ---- main loop: claim two ordinals, compute, release their slots
  for (;;) {
    int oc = 0;
    if (lane == 0) oc = ld_volatile_s32(&sflag[0]) ? N : atomicAdd(&claim[slice], 2);
    oc = __shfl_sync(0xffffffffu, oc, 0);
    if (oc >= N) break;
    const int n = (N - oc) < 2 ? 1 : 2;
    // the claimer of a block's first ordinal fills the block kFillAhead ahead
    if (slice == 0 && (oc % kDescBlock) == 0) fill_issue(oc / kDescBlock + kFillAhead);
    bool ok = true;
    if (lane == 0) ok = desc_wait(oc);
    if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) set_dead();
    const int4 d0 = desc[oc % kDescN];
    const int4 d1 = n > 1 ? desc[(oc + 1) % kDescN] : d0;
    const int s0 = sidx_of(d0);
    const int s1 = sidx_of(d1);
    const uint32_t kt0 = ring + (uint32_t)((oc % R) * C::kStageBytes);
    const uint32_t kt1 = ring + (uint32_t)(((oc + 1) % R) * C::kStageBytes);
    enter(s0, d0.z, d0.w);
    if (n == 2 && s1 == s0) {  // two pages of one segment at a time
      wait_slot(oc);
      wait_slot(oc + 1);
      const int v0 = d0.x >= 0 ? d0.y : 0, v1 = d1.x >= 0 ? d1.y : 0;
      if constexpr (kFusedAppend) {
        if (p.k_new != nullptr && !dead) {
          if (v0 > 0 && (v0 & kRemMask) <= kPageSize)
            append_new(kt0, d0.x, (v0 & kRemMask) - 1, d0.z, d0.w);
          if (v1 > 0 && (v1 & kRemMask) <= kPageSize)
            append_new(kt1, d1.x, (v1 & kRemMask) - 1, d1.z, d1.w);
        }
      }
      if (!dead) {
        if (v0 > 0 && v1 > 0) {
          const uint32_t kts[2] = {kt0, kt1};
          const int vs2[2] = {v0, v1};
          compute_pages(Int<2>{}, kts, vs2);
        } else {
          if (v0 > 0) compute_page(kt0, v0);
          if (v1 > 0) compute_page(kt1, v1);
        }
      }
      __syncwarp();
      release(oc);
      release(oc + 1);
    } else {
#pragma unroll 1
      for (int i = 0; i < n; ++i) {
        const int4 d = i == 0 ? d0 : d1;
        const uint32_t kt = i == 0 ? kt0 : kt1;
        if (i == 1) enter(s1, d1.z, d1.w);
        wait_slot(oc + i);
        const int v = d.x >= 0 ? d.y : 0;
        if constexpr (kFusedAppend) {
          if (p.k_new != nullptr && !dead && v > 0 && (v & kRemMask) <= kPageSize)
            append_new(kt, d.x, (v & kRemMask) - 1, d.z, d.w);
        }
        if (!dead && v > 0) compute_page(kt, v);
        __syncwarp();
        release(oc + i);
      }
    }
    fill_commit();
  }
  fill_commit();
  // the rest of the share's segments (this warp's last one, and any after it
  // it had no page of)
  while (nfl < nseg) flush_next();
  if (lane == 0) {
    int m0, m1;
    tickets_lane0(true, m0, m1);
    mflag[2 * warp] = m0;
    mflag[2 * warp + 1] = m1;
  }
  merge_barrier();
#pragma unroll 1
  for (int i = 0; i < 2 * NW; ++i) {  // segments this CTA completed at exit
    const int seg = mflag[i];
    if (seg >= 0) {
      __threadfence();  // acquire: the other contributors' partials
      merge_segment(seg);
    }
  }
  if (ld_volatile_s32(&sflag[0])) {
    // a wait gave up: let the last copy issued into each slot land (bounded)
    // before the CTA's shared memory is released
    for (int s = tid; s < R; s += blockDim.x) {
      const int last = ld_volatile_s32(&slot_ord[s]);
      if (last >= 0)
        mbar_wait_bounded(smem_u32(&bars[s]), (uint32_t)((last / R) & 1), kWaitLimitNs);
    }
  }
}

// ---------------------------------------------------------------------------
// Host-side dispatch over head_dim, group and query tokens for one cache kind.
template <int D, int G, int QC, int CACHE, bool QBF16>
cudaError_t launch_split(const DecodeLaunch& l) {
  auto kern = decode_kernel<D, G, QC, CACHE, QBF16>;
  const size_t smem = mq_smem_bytes(D, (CacheKind)CACHE, l.p.B, G * QC);
  static size_t configured = 0;  // largest dynamic smem size set so far
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)l.ctas);
  cfg.blockDim = dim3(kDecodeWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = l.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, l.p, l.tmap_k, l.tmap_v);
}

// One query token per sequence.
template <int CACHE, bool QBF16>
cudaError_t dispatch_split(const DecodeLaunch& l) {
  const int d = l.p.d;
  const int g = l.group;
#define PKV_CASE(DD, GG) \
  if (d == DD && g == GG) return launch_split<DD, GG, 1, CACHE, QBF16>(l);
  if constexpr (!cache_is_fp8((CacheKind)CACHE)) {
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
  }
  PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
#undef PKV_CASE
  return cudaErrorNotSupported;
}

// Several query tokens per sequence (l.qcap = 2, 4 or 8, group * qcap <= 64)
// for one head_dim.
template <int CACHE, bool QBF16, int D>
cudaError_t dispatch_split_multi_d(const DecodeLaunch& l) {
  const int g = l.group;
  const int qc = l.qcap;
#define PKV_CASE(GG, QQ) \
  if (g == GG && qc == QQ) return launch_split<D, GG, QQ, CACHE, QBF16>(l);
  PKV_CASE(1, 2) PKV_CASE(1, 4) PKV_CASE(1, 8)
  PKV_CASE(2, 2) PKV_CASE(2, 4) PKV_CASE(2, 8)
  PKV_CASE(4, 2) PKV_CASE(4, 4) PKV_CASE(4, 8)
  PKV_CASE(8, 2) PKV_CASE(8, 4) PKV_CASE(8, 8)
#undef PKV_CASE
  return cudaErrorNotSupported;
}

}  // namespace mq
}  // namespace pkv
