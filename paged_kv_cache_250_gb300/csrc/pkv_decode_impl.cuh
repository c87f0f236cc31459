// pkv_decode_impl.cuh -- split-K flash-decoding kernel over a paged KV cache,
// with the split combine fused in.
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
// CTAs per SM), so ragged lengths never leave an SM idle.  A CTA walks its
// share in pieces of at most kRangeMax pages; page j of a piece goes to warp
// j % NW (NW = 4 warps per CTA for 16-bit caches, 6 for E4M3, whose byte
// conversions want more warps to hide their latency), so the warps move
// through the same segment together, each with its own online-softmax state,
// taking one or two of their pages per step.
//
// Segment ends.  The NW warp states are merged when the share leaves a
// segment (the merge is order-independent): for groups of up to 4 query
// heads NW - 1 warps hand their state over through shared memory and an
// mbarrier and keep streaming while a rotating last one merges and writes;
// for groups of 8 a tree of CTA barriers does it.  A segment wholly inside one
// share is normalised and written at once; a segment cut by share boundaries
// gets one partial (m, l, o) per CTA, in slot cta + segment, and a page-count
// ticket; the CTA whose pages complete the segment merges the partials (the
// split combine), in slot order.  Nothing waits on another CTA, and every
// sum is taken in a fixed order, so results are bitwise repeatable.
//
// Data path per warp.  A ring of kStages shared-memory slots, each holding
// one K page and one V page of one (block, KV head).  Lane 0 issues 2-D TMA
// tile loads (128-byte swizzle, evict-first L2 policy) that complete on the
// slot's mbarrier; the warp waits, computes, and refills the slot with its
// page kStages ahead.  Block-table lookups for a piece are done by the
// warp's lanes in parallel into a descriptor ring in shared memory, one piece
// ahead of their use.
//
// Math per page (16 tokens), all on warp-level tensor-core MMAs:
//   S^T[16 tok][8] = K[16][d] . Q^T[d][8]   K via ldmatrix from the swizzled
//                                           page, Q^T resident in registers;
//                                           the 8 columns are the g query
//                                           heads of the group (zero-padded)
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

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per bounded wait
constexpr float kRescaleThreshold = 8.0f;         // log2 units
constexpr int kMergeBarrier = 1;                  // named barrier id (0 = __syncthreads)
// A descriptor holds the tokens from the page's start to the context's end,
// capped here (enough for the causal limits of up to 8 query tokens).
constexpr int kRemCap = 2 * kPageSize;
constexpr int kRemMask = 63;       // descriptor y, bits 0-5: tokens to the context's end
constexpr int kWinFlag = 1 << 17;  // descriptor: a sliding window masks rows of this page

template <int N>
struct Int {  // a compile-time count passed to a generic lambda
  static constexpr int value = N;
};

template <int D, int CACHE, bool DEEP = false>
struct DecodeCfg {
  static constexpr int kElem = cache_is_fp8((CacheKind)CACHE) ? 1 : 2;
  static constexpr int kRowBytes = D * kElem;              // bytes per token row
  static constexpr int kBoxes = kRowBytes / 128;           // 128-byte TMA boxes per row
  static constexpr int kBoxBytes = kPageSize * 128;        // one box of a page
  static constexpr int kTileBytes = kPageSize * kRowBytes; // one K (or V) page
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kScaleBytes = decode_scale_bytes((CacheKind)CACHE);  // per stage
  static constexpr int kKSteps = D / 16;  // k-steps of the QK contraction
  static constexpr int kMTiles = D / 16;  // 16-row tiles of O^T
  static constexpr int kStages =
      DEEP ? decode_stages_deep(D, (CacheKind)CACHE) : decode_stages(D, (CacheKind)CACHE);
  static constexpr int kLaneState = 4 + 4 * kMTiles;  // m[2], l[2], o[MT][4] per lane
  static_assert(kRowBytes % 128 == 0, "rows must be whole 128-byte boxes");
};

// Byte offset of 16-byte chunk `chunk` of token row `tok` inside a page
// loaded as 128-byte-swizzled boxes of 16 rows.
__device__ __forceinline__ uint32_t swz(int tok, int chunk) {
  return (uint32_t)((chunk >> 3) * (kPageSize * 128) + tok * 128 +
                    (((chunk & 7) ^ (tok & 7)) << 4));
}

template <int NW>
__device__ __forceinline__ void merge_barrier() {
  asm volatile("bar.sync %0, %1;" ::"n"(kMergeBarrier), "n"(NW * 32) : "memory");
}

__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
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
// MMA's 8 columns hold the NC = QC * G (query token, head) pairs of a group.
// The library builds it for one query token (QC = 1); several query tokens
// per sequence go to the kernel of pkv_decode_mq.cuh.  DEEP: the deeper ring
// and barrier-tree segment ends of the per-token E4M3 kernel at small batches.
template <int D, int G, int QC, int CACHE, bool QBF16, bool DEEP>
__global__ void __launch_bounds__(decode_warps((CacheKind)CACHE) * 32, kDecodeCtasPerSm)
    decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv) {
  constexpr int NC = G * QC;
  static_assert(NC <= 8, "one MMA column per (query token, head)");
  using C = DecodeCfg<D, CACHE, DEEP>;
  constexpr bool kBF = (CACHE == kCacheBF16);  // mma operand type (else fp16)
  constexpr int kS = C::kStages;
  constexpr int NW = decode_warps((CacheKind)CACHE);
  constexpr int kDescRing = decode_desc_ring(NW);  // page descriptors per warp
  static_assert(2 * ((kRangeMax + NW - 1) / NW) <= kDescRing, "two pieces per ring");
  constexpr int kMbuf = DEEP ? 2 * C::kLaneState * 32 : decode_mbuf_floats(D, NW);
  auto merge_barrier = [] { pkv::merge_barrier<NW>(); };
  constexpr int kMT = C::kMTiles;
  // pages a warp takes per step: 2 on rings of 3+ pages (4 measured slower:
  // longer P.V accumulation chains)
  constexpr int kGroup = kS >= 3 ? 2 : 1;
  // the one-kernel step writes new rows in the main loop for 16-bit caches
  // only (E4M3 steps enqueue the append kernel first)
  constexpr bool kFp8 = cache_is_fp8((CacheKind)CACHE);
  constexpr bool kTok = CACHE == kCacheE4M3Tok;  // one scale per token and KV head
  constexpr bool kFusedAppend = QC == 1 && !kFp8;

  // the next kernel on the stream may launch (a programmatic dependent waits
  // for this one to complete before it reads what this one writes)
  if (p.trigger_next) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if ((threadIdx.x & 31) == 0) {  // the tensor maps are parameters: fetch them at once
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  if (!p.early_prologue) griddep_wait();

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const uint32_t ring = base + (uint32_t)(warp * kS * C::kStageBytes);
  // per-token scales of the staged pages, beside the ring (E4M3 per token)
  const uint32_t scl = base + (uint32_t)(NW * kS * C::kStageBytes + warp * kS * C::kScaleBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      base_ptr + (size_t)NW * kS * (C::kStageBytes + C::kScaleBytes));
  uint64_t* fbar = bars + NW * kS;  // [4] flush: full (even, odd), empty, padding
  // everything after the mbarriers stays 16-byte aligned (float4 in mbuf)
  static_assert((NW * kS * 8) % 16 == 0 && (NW * kDescRing * 8) % 16 == 0, "smem alignment");
  int2* desc_all = reinterpret_cast<int2*>(fbar + 4);    // [NW][kDescRing]
  int2* desc = desc_all + warp * kDescRing;
  float* mbuf = reinterpret_cast<float*>(desc_all + NW * kDescRing);  // [kMbuf]
  int* mflag = reinterpret_cast<int*>(mbuf + kMbuf);                   // [2 NW] merges due
  int32_t* pfx = mflag + 2 * NW;                                      // [B+1] pages
  int32_t* nzp = pfx + (p.B + 1);                                     // [B+1] non-empty seqs
  int32_t* ctxs = nzp + (p.B + 1);                                    // [B]
  int32_t* gns = ctxs + p.B;  // [B] pages before a sliding window's gap (all pages if none)
  int32_t* gsk = gns + p.B;   // [B] pages the gap skips
  const int64_t Gn = gridDim.x;

  // ---- prologue: pages per sequence, prefix sums of pages and of non-empty
  // sequences
  if (tid == 0) {
    pfx[0] = 0;
    nzp[0] = 0;
  }
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
  if (lane == 0) {
    for (int s = 0; s < kS; ++s) mbar_init(smem_u32(&bars[warp * kS + s]), 1);
    if (warp == 0) {
      mbar_init(smem_u32(fbar + 0), (NW - 1) * 32);
      mbar_init(smem_u32(fbar + 1), (NW - 1) * 32);
      mbar_init(smem_u32(fbar + 2), 32);
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
  // Warp-wide search (every lane, the same v): the largest b in [lo, hi)
  // with key(b) <= v, given key(lo) <= v and key nondecreasing.  Each round
  // the 32 lanes probe 32 evenly spaced candidates, so 32 sequences take one
  // round of shared-memory loads and 6000 take three.
  auto warp_search = [&](auto key, int64_t v, int lo, int hi) -> int {
    while (hi - lo > 1) {
      const int step = (hi - lo + 31) >> 5;
      const int b = lo + lane * step;
      const unsigned m = __ballot_sync(0xffffffffu, b < hi && key(b) <= v);
      lo += (31 - __clz(m)) * step;  // lane 0 probes lo itself: m != 0
      hi = min(hi, lo + step);
    }
    return lo;
  };
  // first unit whose cost position is >= P (W when none); every lane, the same P
  auto unit_at_cost = [&](int64_t P) -> int64_t {
    if (P >= Tc) return W;
    const int a = warp_search(seq_cost0, P, 0, p.B);
    const int64_t np = pfx[a + 1] - pfx[a];
    const int64_t r = P - seq_cost0(a);
    const int64_t hh = udiv64(r, np + kSegCost);
    const int64_t off = r - hh * (np + kSegCost) - kSegCost;
    return (int64_t)p.Hkv * pfx[a] + hh * np + (off > 0 ? off : 0);
  };
  const int64_t sh_lo = blockIdx.x < Gs ? unit_at_cost(udiv64(Tc * blockIdx.x + Gs - 1, Gs)) : W;
  const int64_t sh_hi =
      blockIdx.x < Gs ? unit_at_cost(udiv64(Tc * (blockIdx.x + 1) + Gs - 1, Gs)) : W;
  // the CTA whose share holds unit x of sequence b, KV head h
  auto cta_of = [&](int64_t x, int b, int64_t h) -> int64_t {
    const int64_t np = pfx[b + 1] - pfx[b];
    const int64_t start = (int64_t)p.Hkv * pfx[b] + h * np;
    const int64_t X = seq_cost0(b) + h * (np + kSegCost) + kSegCost + (x - start);
    return udiv64(X * Gs, Tc);
  };
  auto piece = [&](int i) -> int2 {
    const int64_t s0 = sh_lo + (int64_t)i * kRangeMax;
    if (s0 >= sh_hi) return make_int2((int)W, (int)W);
    return make_int2((int)s0, (int)(s0 + kRangeMax < sh_hi ? s0 + kRangeMax : sh_hi));
  };
  // the sequence holding unit x: the last b with Hkv pfx[b] <= x (empty
  // sequences before it share its pfx); one lane
  auto seq_of = [&](int64_t x) -> int {
    int a = 0, z = p.B;
    while (z - a > 1) {
      const int mid = (a + z) >> 1;
      if ((int64_t)p.Hkv * pfx[mid] <= x) a = mid; else z = mid;
    }
    return a;
  };
  // The warp's pages of piece [s, e) are s + warp + NW j; ordinals continue
  // across pieces; desc[] holds kDescRing ordinals (at least two pieces of
  // at most ceil(kRangeMax / NW) pages per warp each).
  auto warp_count = [&](int2 r) -> int {
    const int n = r.y - r.x - warp;
    return n > 0 ? (n + NW - 1) / NW : 0;
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
  auto fill_desc = [&](int2 r, int ord0) {  // {tma row or -1, page_info}
    const int cnt = warp_count(r);
    for (int j = lane; j < cnt; j += 32) {
      const int64_t x = (int64_t)r.x + warp + (int64_t)NW * j;
      const int b = seq_of(x);
      const int np = pfx[b + 1] - pfx[b];
      const int64_t rr = x - (int64_t)p.Hkv * pfx[b];
      const int h = (int)udiv64(rr, np);
      const int pgu = (int)(rr - (int64_t)h * np);  // unit within the segment
      const int pg = pgu < gns[b] ? pgu : pgu + gsk[b];
      const int blk = p.block_tables[(int64_t)b * p.MBS + pg];
      int row = -1;
      if (blk >= 0 && blk < p.NB) row = (blk * p.Hkv + h) * kPageSize;
      else report_error(p.err_word, PKV_ERR_BOUNDS);
      desc[(ord0 + j) % kDescRing] = make_int2(row, page_info(b, pg));
      if (j == 0 || pgu == 0) {  // a segment may start here: warm its q rows in L2
        for (int i = 0; i < p.qlen; ++i) {
          const char* qp = reinterpret_cast<const char*>(p.q) +
                           (((int64_t)b * p.qlen + i) * p.Hq + h * G) * D * 2;
          for (int off = 0; off < G * D * 2; off += 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(qp + off));
        }
      }
    }
    __syncwarp();
  };

  // The same for the next piece, in two halves so the table loads never
  // stall the warp: fill_issue starts the loads (one page per lane), and
  // fill_commit, a page later, writes the descriptors.
  int f_blk = -1, f_h = 0, f_valid = 0, f_ord = 0, f_cnt = 0;
  bool f_pending = false;
  auto fill_issue = [&](int2 r, int ord0) {
    f_cnt = warp_count(r);
    f_ord = ord0;
    f_pending = true;
    if (lane < f_cnt) {
      const int64_t x = (int64_t)r.x + warp + (int64_t)NW * lane;
      const int b = seq_of(x);
      const int np = pfx[b + 1] - pfx[b];
      const int64_t rr = x - (int64_t)p.Hkv * pfx[b];
      f_h = (int)udiv64(rr, np);
      const int pgu = (int)(rr - (int64_t)f_h * np);  // unit within the segment
      const int pg = pgu < gns[b] ? pgu : pgu + gsk[b];
      f_blk = p.block_tables[(int64_t)b * p.MBS + pg];
      f_valid = page_info(b, pg);
      if (lane == 0 || pgu == 0) {  // a segment may start here: warm its q rows in L2
        for (int i = 0; i < p.qlen; ++i) {
          const char* qp = reinterpret_cast<const char*>(p.q) +
                           (((int64_t)b * p.qlen + i) * p.Hq + f_h * G) * D * 2;
          for (int off = 0; off < G * D * 2; off += 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(qp + off));
        }
      }
    }
  };
  auto fill_commit = [&]() -> bool {
    if (!f_pending) return false;
    f_pending = false;
    if (lane < f_cnt) {
      int row = -1;
      if (f_blk >= 0 && f_blk < p.NB) row = (f_blk * p.Hkv + f_h) * kPageSize;
      else report_error(p.err_word, PKV_ERR_BOUNDS);
      desc[(f_ord + lane) % kDescRing] = make_int2(row, f_valid);
    }
    __syncwarp();
    return true;
  };

  const uint64_t pol = l2_policy_evict_first();

  // the first piece and its descriptors need nothing the previous kernel
  // writes (lengths and tables only); the second piece's lookups are issued
  // when the first piece starts
  const int2 r0 = piece(0);
  fill_desc(r0, 0);

  // From here on the kernel touches data the previous kernel on the stream may
  // write (cache pages, q, outputs, workspace): wait for it.  The warp's
  // first pages (two ring fills for 16-bit caches, one for E4M3: measured
  // best) start towards L2 before the wait (an L2 prefetch moves no data
  // into the CTA; a row the previous kernel writes meanwhile lands in L2
  // over the prefetched line, where the loads after the wait read it).
  if (p.early_prologue) {
    constexpr int kPrefetch = kFp8 ? kS : 2 * kS;
    static_assert(kPrefetch <= 32, "one page per lane");
    if (lane < kPrefetch && lane < warp_count(r0)) {
      const int2 dsc = desc[lane];
      if (dsc.x >= 0) {
        const int64_t off = (int64_t)dsc.x * C::kRowBytes;
        l2_prefetch_bulk(static_cast<const char*>(p.k_cache) + off, C::kTileBytes);
        l2_prefetch_bulk(static_cast<const char*>(p.v_cache) + off, C::kTileBytes);
      }
    }
    griddep_wait();
  }

  int issued = 0;      // ordinals whose load was issued
  int filled_end = 0;  // ordinals with a descriptor
  auto issue = [&](int i) {
    const int2 dsc = desc[i % kDescRing];
    if (lane == 0) {
      const int slot = i % kS;
      const uint32_t bar = smem_u32(&bars[warp * kS + slot]);
      const uint32_t kt = ring + (uint32_t)(slot * C::kStageBytes);
      const uint32_t vt = kt + C::kTileBytes;
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
    }
  };
  auto top_up = [&](int consumed) {  // keep kS loads in flight
    while (issued < consumed + kS && issued < filled_end) issue(issued++);
  };
  filled_end = warp_count(r0);
  top_up(0);

  // sequences with no tokens get a zero output row (spread over CTAs)
  for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
    if (pfx[b + 1] != pfx[b]) continue;
    const int64_t row0 = (int64_t)b * p.qlen * p.Hq * D;
    for (int i = tid; i < p.qlen * p.Hq * D; i += blockDim.x)
      store_out_rt(p.out_dtype, p.out, row0 + i, 0.f);
  }

  // ---- per-lane fragment coordinates
  const int c4 = lane & 3;   // C-fragment column pair: heads 2*c4, 2*c4+1
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

  uint32_t qf[C::kKSteps][2];
  float o[kMT][4];
  float m2[2], l2[2];
  // score scale in log2 units (E4M3: times the K scale) for the lane's two
  // C-fragment columns 2 c4 and 2 c4 + 1
  float c2a = 0.f, c2b = 0.f;

  auto reset_state = [&]() {
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;
    m2[0] = m2[1] = -INFINITY;
    l2[0] = l2[1] = 0.f;
  };

  // row of q / out for MMA column c of segment (b, h): query token c / G,
  // query head h * G + c % G; the column is real when c < G * p.qlen
  auto col_row = [&](int b, int h, int c) -> int64_t {
    return ((int64_t)b * p.qlen + c / G) * p.Hq + h * G + c % G;
  };
  auto col_real = [&](int c) -> bool { return c < NC && c < G * p.qlen; };

  auto load_q = [&](int b, int h) {
    const int col = r8;  // B-fragment column n = lane / 4
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
        qf[ks][0] = b0;
        qf[ks][1] = b1;
      }
    } else {
      // FP8 pages meet q on the fp16 MMA.  A bf16 q can lie outside fp16's
      // range, so each column is brought to [2^14, 2^15) by a power of two
      // (exact), which the column's score scale undoes (also exact).
      uint2 raw[C::kKSteps];
      float amax = 0.f;
#pragma unroll
      for (int ks = 0; ks < C::kKSteps; ++ks) {
        raw[ks] = make_uint2(0u, 0u);
        if (real) raw[ks] = *reinterpret_cast<const uint2*>(qrow + 16 * ks + 4 * c4);
        if constexpr (QBF16) {
          const float2 f01 = unpack2<true>(raw[ks].x), f23 = unpack2<true>(raw[ks].y);
          amax = fmaxf(amax, fmaxf(fmaxf(fabsf(f01.x), fabsf(f01.y)),
                                   fmaxf(fabsf(f23.x), fabsf(f23.y))));
        }
      }
      int e = 0;  // column scale 2^e
      if constexpr (QBF16) {
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        if (amax > 0.f) e = min(112, max(-112, ((__float_as_int(amax) >> 23) & 0xff) - 127 - 14));
      }
      const float down = __int_as_float((127 - e) << 23);
#pragma unroll
      for (int ks = 0; ks < C::kKSteps; ++ks) {
        const float2 f01 = unpack2<QBF16>(raw[ks].x);
        const float2 f23 = unpack2<QBF16>(raw[ks].y);
        qf[ks][0] = pack2<false>(f01.x * down, f01.y * down);
        qf[ks][1] = pack2<false>(f23.x * down, f23.y * down);
      }
      // the lane's C-fragment columns 2 c4, 2 c4 + 1 are B-fragment columns
      // of lanes 8 c4 and 8 c4 + 4
      const int ea = __shfl_sync(0xffffffffu, e, 8 * c4);
      const int eb = __shfl_sync(0xffffffffu, e, 8 * c4 + 4);
      float c2 = p.scale_log2;
      if constexpr (CACHE == kCacheE4M3) c2 *= p.k_scale[h];
      c2a = c2 * __int_as_float((127 + ea) << 23);
      c2b = c2 * __int_as_float((127 + eb) << 23);
      return;
    }
    c2a = c2b = p.scale_log2;
  };

  // ---- S^T[16 tok][8] = K . Q^T for one page, on two accumulator chains
  auto qk_page = [&](uint32_t kt, float (&s)[4]) {
    float s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 4; ++e) s[e] = 0.f;
    if constexpr (!kFp8) {
#pragma unroll
      for (int ks = 0; ks < C::kKSteps; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, kt + swz(qk_tok, 2 * ks + qk_chunk_hi));
        if (ks & 1) mma_16816<kBF>(s2, a, qf[ks][0], qf[ks][1]);
        else mma_16816<kBF>(s, a, qf[ks][0], qf[ks][1]);
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
        mma_16816<false>(s, a, qf[2 * gi][0], qf[2 * gi][1]);
        a[0] = e4m3x2_to_f16x2(r[2]);
        a[1] = e4m3x2_to_f16x2(r[3]);
        a[2] = e4m3x2_to_f16x2(r[2] >> 16);
        a[3] = e4m3x2_to_f16x2(r[3] >> 16);
        mma_16816<false>(s2, a, qf[2 * gi + 1][0], qf[2 * gi + 1][1]);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) s[e] += s2[e];
  };

  // ---- V rows at and past the context's end may hold anything (a stale or
  // never-written slot, and 0 * NaN would poison P.V): the last page of a
  // segment gets them zeroed in its staged copy, so P.V needs no mask.  The
  // slot is refilled by the tensor-copy (async) proxy later.
  auto zero_tail = [&](uint32_t vt, int rem) {
    const int n = (kPageSize - rem) * C::kBoxes * 8;  // 16-byte chunks: (row, box, chunk)
    for (int i = lane; i < n; i += 32) {
      const int row = rem + i / (C::kBoxes * 8);
      const int bx = (i / 8) % C::kBoxes;
      const uint32_t a = vt + (uint32_t)(bx * C::kBoxBytes + row * 128 + (i % 8) * 16);
      asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
  };

  // ---- O^T += V^T . P^T for one page
  auto pv_page = [&](uint32_t vt, uint32_t bh0, uint32_t bh1, uint32_t bl0, uint32_t bl1) {
    if constexpr (!kFp8) {
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        uint32_t a[4];
        ldsm_x4_trans(a, vt + swz(pv_tok, 2 * mt + pv_chunk_hi));
        mma_16816<kBF>(o[mt], a, bh0, bh1);
        mma_16816<kBF>(o[mt], a, bl0, bl1);
      }
    } else {
#pragma unroll
      for (int gi = 0; gi < D / 32; ++gi) {
        uint32_t r[4];
        ldsm_x4_trans(r, vt + swz(pv_tok, 2 * gi + pv_chunk_hi));
        uint32_t a[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) a[e] = e4m3x2_to_f16x2(__byte_perm(r[e], 0, 0x0020));
        mma_16816<false>(o[2 * gi], a, bh0, bh1);
        mma_16816<false>(o[2 * gi], a, bl0, bl1);
#pragma unroll
        for (int e = 0; e < 4; ++e) a[e] = e4m3x2_to_f16x2(__byte_perm(r[e], 0, 0x0031));
        mma_16816<false>(o[2 * gi + 1], a, bh0, bh1);
        mma_16816<false>(o[2 * gi + 1], a, bl0, bl1);
      }
    }
  };

  // ---- NP (1 or 2) pages of one segment: their scores, one online-
  // softmax update over all their tokens (log2 domain; tokens past the
  // context are masked), then P.V.  Several pages give the warp independent
  // MMA chains and fewer reductions per token.
  auto compute_pages = [&](auto npc, const uint32_t* kt, const int* valids) {
    constexpr int NP = decltype(npc)::value;
    float x[NP][4];
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
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const int v = valids[i];
      const int rem = v & kRemMask;  // tokens from the page's start to the context's end
#pragma unroll
      for (int e = 0; e < 4; ++e) x[i][e] *= (e & 1) ? c2b : c2a;
      if constexpr (kTok) {
        x[i][0] *= ksc[i][0];  // rows past the context are masked below
        x[i][1] *= ksc[i][0];
        x[i][2] *= ksc[i][1];
        x[i][3] *= ksc[i][1];
        if (r8 >= rem) vsc[i][0] = 0.f;  // their P is 0; their scale may be anything
        if (r8 + 8 >= rem) vsc[i][1] = 0.f;
      }
      if constexpr (QC == 1) {
        if (rem < kPageSize) {
          if (r8 >= rem) x[i][0] = x[i][1] = -INFINITY;
          if (r8 + 8 >= rem) x[i][2] = x[i][3] = -INFINITY;
        }
        if (v & kWinFlag) {  // rows before the window's start that are no sinks
          const int sr = (v >> 6) & 15, wr = ((v >> 11) & 63) - 8;
          if (r8 < wr && r8 >= sr) x[i][0] = x[i][1] = -INFINITY;
          if (r8 + 8 < wr && r8 + 8 >= sr) x[i][2] = x[i][3] = -INFINITY;
        }
      } else {
        const int c0 = 2 * c4, c1 = 2 * c4 + 1;
        const int j0 = col_real(c0) ? c0 / G : p.qlen - 1, j1 = col_real(c1) ? c1 / G : p.qlen - 1;
        if (rem < kPageSize + QC - 1) {
          // causal among the new tokens: query token j of the last qlen sees
          // the page's first rem - (qlen - 1 - j) tokens
          const int l0 = rem - (p.qlen - 1 - j0), l1 = rem - (p.qlen - 1 - j1);
          if (r8 >= l0) x[i][0] = -INFINITY;
          if (r8 >= l1) x[i][1] = -INFINITY;
          if (r8 + 8 >= l0) x[i][2] = -INFINITY;
          if (r8 + 8 >= l1) x[i][3] = -INFINITY;
        }
        if (v & kWinFlag) {  // query token j's window starts j rows after token 0's
          const int sr = (v >> 6) & 15, wr = ((v >> 11) & 63) - 8;
          const int w0 = wr + j0, w1 = wr + j1;
          if (r8 < w0 && r8 >= sr) x[i][0] = -INFINITY;
          if (r8 < w1 && r8 >= sr) x[i][1] = -INFINITY;
          if (r8 + 8 < w0 && r8 + 8 >= sr) x[i][2] = -INFINITY;
          if (r8 + 8 < w1 && r8 + 8 >= sr) x[i][3] = -INFINITY;
        }
      }
      mx0 = fmaxf(mx0, fmaxf(x[i][0], x[i][2]));
      mx1 = fmaxf(mx1, fmaxf(x[i][1], x[i][3]));
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const bool grow = (mx0 > m2[0] + kRescaleThreshold) || (mx1 > m2[1] + kRescaleThreshold);
    if (__any_sync(0xffffffffu, grow)) {
      const float n0 = fmaxf(m2[0], mx0), n1 = fmaxf(m2[1], mx1);
      float a0 = exp2f(m2[0] - n0), a1 = exp2f(m2[1] - n1);
      if constexpr (QC > 1) {  // a column that has seen nothing yet stays as it is
        if (n0 == -INFINITY) a0 = 1.f;
        if (n1 == -INFINITY) a1 = 1.f;
      }
      m2[0] = n0;
      m2[1] = n1;
      l2[0] *= a0;
      l2[1] *= a1;
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        o[mt][0] *= a0;
        o[mt][1] *= a1;
        o[mt][2] *= a0;
        o[mt][3] *= a1;
      }
    }
    // a column every token so far was masked for keeps m = -inf: weigh its
    // (all -inf) scores against 0, not -inf (only possible with QC > 1)
    float mu0 = m2[0], mu1 = m2[1];
    if constexpr (QC > 1) {
      if (mu0 == -INFINITY) mu0 = 0.f;
      if (mu1 == -INFINITY) mu1 = 0.f;
    }
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      float p0 = exp2f(x[i][0] - mu0), p1 = exp2f(x[i][1] - mu1);
      float p2 = exp2f(x[i][2] - mu0), p3 = exp2f(x[i][3] - mu1);
      l2[0] += p0 + p2;
      l2[1] += p1 + p3;
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
      const int vrows = valids[i] & kRemMask;
      if (vrows < kPageSize) zero_tail(kt[i] + C::kTileBytes, vrows);
      pv_page(kt[i] + C::kTileBytes, movm_trans(h01), movm_trans(h23), movm_trans(l01),
              movm_trans(l23));
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
  // steps).  The page (b, h) is staged by this warp alone, so nothing else in
  // the grid reads the row.
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
  // state (m[2], l[2], o[MT][4]) at buf[i * S + li]
  auto store_state_at = [&](float* buf, int li, int S) {
    buf[0 * S + li] = m2[0];
    buf[1 * S + li] = m2[1];
    buf[2 * S + li] = l2[0];
    buf[3 * S + li] = l2[1];
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) buf[(4 + 4 * mt + e) * S + li] = o[mt][e];
  };
  auto merge_state_at = [&](const float* buf, int li, int S) {
    float a[2], bw[2];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const float mb = buf[cc * S + li];
      const float M = fmaxf(m2[cc], mb);
      if (M == -INFINITY) {
        a[cc] = 1.f;
        bw[cc] = 0.f;
      } else {
        a[cc] = exp2f(m2[cc] - M);
        bw[cc] = exp2f(mb - M);
        m2[cc] = M;
      }
      l2[cc] = a[cc] * l2[cc] + bw[cc] * buf[(2 + cc) * S + li];
    }
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        o[mt][e] = a[e & 1] * o[mt][e] + bw[e & 1] * buf[(4 + 4 * mt + e) * S + li];
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
      const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + slot_base * NC + head;
      const float4* vo = reinterpret_cast<const float4*>(p.part_o + slot_base * NC * D) + col;
      float M = -INFINITY, lsum = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (count <= 4) {
        // a few partials: one pass in slot order, the running reference
        // moving up to each new maximum and what was summed brought down to
        // it, so all their loads go out at once
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          if (kk < count) {
            const float2 v = __ldcg(ml + (int64_t)kk * NC);
            const float4 x = __ldcg(vo + (int64_t)kk * (NC * D / 4));
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
          const float2 v = __ldcg(ml + (int64_t)kk * NC);
          if (v.y > 0.f) M = fmaxf(M, v.x);
        }
        if (M > -INFINITY) {
#pragma unroll 4
          for (int kk = 0; kk < count; ++kk) {
            const float2 v = __ldcg(ml + (int64_t)kk * NC);
            const float4 x = __ldcg(vo + (int64_t)kk * (NC * D / 4));
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

  // A CTA learns it completed a split segment from the page-count ticket.
  // The warp that stored a partial does not fence right away (under full
  // memory load the fence waits microseconds for its stores to land): its
  // lane 0 publishes it (fence, then an atomic add of its pages) at the CTA's
  // next flush, when the stores are long done, and reads the atomic's result
  // one flush later still (or at exit).
  int pub_seg = -1, pub_add = 0;               // lane 0: partial stored, not yet published
  int iss_seg = -1, iss_old = 0, iss_add = 0;  // lane 0: ticket added, result not yet read
  int nflushes = 0;                            // the same in every warp
  int k = 0;           // next ordinal this warp consumes
  bool dead = false;   // a bounded wait gave up: skip compute and waits, keep the barriers
  int k_dead = -1;     // first ordinal whose copy may still be in flight when dead
  auto set_dead = [&](int from) {
    if (!dead) {
      dead = true;
      k_dead = from;
      if (lane == 0) report_error(p.err_word, PKV_ERR_TIMEOUT);
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
      if (iss_old + iss_add == seg_pages(iss_seg)) m0 = iss_seg;
      iss_seg = -1;
    }
    if (pub_seg >= 0) {
      __threadfence();  // release: this warp's partial before its pages count
      iss_old = atomicAdd(&p.tickets[pub_seg], pub_add);
      iss_seg = pub_seg;
      iss_add = pub_add;
      pub_seg = -1;
      if (final_call) {
        if (iss_old + iss_add == seg_pages(iss_seg)) m1 = iss_seg;
        iss_seg = -1;
      }
    }
  };
  auto tickets_step = [&](bool final_call) {  // every warp, before a CTA barrier
    if (lane != 0) return;
    int m0, m1;
    tickets_lane0(final_call, m0, m1);
    mflag[2 * warp] = m0;
    mflag[2 * warp + 1] = m1;
  };
  auto merge_flagged = [&]() {  // all threads, right after a CTA barrier
#pragma unroll 1
    for (int i = 0; i < 2 * NW; ++i) {
      const int seg = mflag[i];
      if (seg >= 0) {
        __threadfence();  // acquire: the other contributors' partials
        merge_segment(seg);
        merge_barrier();  // mbuf free again
      }
    }
  };

  // ---- the merged state of a segment: write the output (whole segment in
  // this share) or this CTA's partial (published at the next flush or exit)
  auto finish = [&](int b, int h, bool split, int pages_mine) {
    const float vs = (CACHE == kCacheE4M3) ? p.v_scale[h] : 1.f;
    const int h0 = 2 * c4, h1 = 2 * c4 + 1;
    float lt0 = l2[0], lt1 = l2[1];
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
          store_out_rt(p.out_dtype, p.out, ob0 + dA, o[mt][0] * i0);
          store_out_rt(p.out_dtype, p.out, ob0 + dB, o[mt][2] * i0);
        }
        if (w1) {
          store_out_rt(p.out_dtype, p.out, ob1 + dA, o[mt][1] * i1);
          store_out_rt(p.out_dtype, p.out, ob1 + dB, o[mt][3] * i1);
        }
      }
      return;
    }
    // partial slot cta + seg is unique: shares are contiguous and ordered, so
    // a later CTA never touches an earlier segment
    const int64_t part = (int64_t)blockIdx.x + b * p.Hkv + h;
    float* po = p.part_o + part * NC * D;
    float* pml = p.part_ml + part * NC * 2;
    if (r8 == 0) {
      if (h0 < NC) { pml[2 * h0] = m2[0]; pml[2 * h0 + 1] = lt0; }
      if (h1 < NC) { pml[2 * h1] = m2[1]; pml[2 * h1 + 1] = lt1; }
    }
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
      const int dA = d_of(mt, 0), dB = d_of(mt, 1);
      if (h0 < NC) {
        po[h0 * D + dA] = o[mt][0] * vs;
        po[h0 * D + dB] = o[mt][2] * vs;
      }
      if (h1 < NC) {
        po[h1 * D + dA] = o[mt][1] * vs;
        po[h1 * D + dB] = o[mt][3] * vs;
      }
    }
    __syncwarp();
    if (lane == 0) {
      pub_seg = b * p.Hkv + h;
      pub_add = pages_mine;
    }
  };

  // ---- end of this CTA's part of a segment.  The warp that finishes (merges
  // the NW states and writes) rotates from flush to flush.
  // Synchronous form (used when the other warps' compact states do not fit
  // in mbuf): a tree of CTA barriers over two state buffers; each round the
  // m highest of the n roles left (m = 2, or 1 when n is 3) hand their states
  // to roles 0 .. m - 1, until roles 0 and 1 are left.
  auto flush_sync = [&](int b, int h, bool split, int pages_mine) {
    float* buf0 = mbuf;
    float* buf1 = mbuf + C::kLaneState * 32;
    const int wr = (warp + NW - nflushes % NW) % NW;  // this warp's role
    ++nflushes;
    tickets_step(false);
    merge_barrier();
    merge_flagged();  // uses mbuf, before the states go there
#pragma unroll
    for (int n = NW; n > 2; n -= (n >= 4 ? 2 : 1)) {
      const int m = n >= 4 ? 2 : 1;
      if (wr >= n - m && wr < n) store_state(wr == n - m ? buf0 : buf1);
      merge_barrier();
      if (wr < m) merge_state(wr == 0 ? buf0 : buf1);
      merge_barrier();
    }
    if (wr == 1) store_state(buf0);
    merge_barrier();
    if (wr != 0) return;
    merge_state(buf0);
    finish(b, h, split, pages_mine);
  };
  // Asynchronous form (NC <= 4): the NW - 1 other warps drop the lanes of their
  // state that hold real heads into mbuf slots, arrive on the "full"
  // mbarrier and go on with the next segment at once, so their copies keep
  // streaming; the finisher waits on "full", merges, frees the slots through
  // the "empty" mbarrier and writes.  A segment this warp's ticket completed
  // is merged by this warp alone.
  // Flush n uses full[n % 2] (its phase n / 2) and empty (its phase n).  No
  // wait can see a barrier two phases away from the one it tests: the
  // finisher of flush n was a writer at flush n - 1 and waited there for
  // empty phase n - 2, which the finisher of flush n - 2 completed only
  // after full[n % 2] completed its phase for flush n - 2; a writer of flush
  // n waits for empty phase n - 1, and every earlier phase of empty was
  // waited for by the warps whose arrivals complete phase n - 1.
  constexpr int kU = NC >= 4 ? NC / 2 : 1;     // C-fragment column pairs with real columns
  constexpr int kCS = C::kLaneState * 8 * kU;  // floats per compact warp state
  constexpr bool kAsyncFlush = !DEEP && NC <= 4 && (NW - 1) * kCS <= kMbuf;
  auto flush_async = [&](int b, int h, bool split, int pages_mine) {
    const int n = nflushes++;
    const int fin = n % NW;
    const uint32_t bar_full = smem_u32(fbar + (n & 1)), bar_empty = smem_u32(fbar + 2);
    int m0 = -1, m1 = -1;
    if (lane == 0) tickets_lane0(false, m0, m1);
    m0 = __shfl_sync(0xffffffffu, m0, 0);
    if (m0 >= 0) {
      __threadfence();  // acquire: the other contributors' partials
      merge_segment_warp(m0);
    }
    const int li = r8 * kU + c4;
    if (warp != fin) {
      if (n > 0 && !dead && !mbar_wait_bounded(bar_empty, (uint32_t)((n - 1) & 1), kWaitLimitNs))
        set_dead(k);
      if (c4 < kU) store_state_at(mbuf + ((warp - fin - 1 + NW) % NW) * kCS, li, 8 * kU);
      mbar_arrive(bar_full);
      return;
    }
    if (!dead && !mbar_wait_bounded(bar_full, (uint32_t)((n >> 1) & 1), kWaitLimitNs)) set_dead(k);
    if (c4 < kU) {
#pragma unroll 1
      for (int sl = 0; sl < NW - 1; ++sl) merge_state_at(mbuf + sl * kCS, li, 8 * kU);
    }
    mbar_arrive(bar_empty);
    finish(b, h, split, pages_mine);
  };
  auto flush = [&](int b, int h, bool split, int pages_mine) {
    if constexpr (kAsyncFlush) flush_async(b, h, split, pages_mine);
    else flush_sync(b, h, split, pages_mine);
  };

  // ---- main loop over the pieces of this CTA's share
  int ord_base = 0;   // first ordinal of the current piece (this warp)
  int cur_b = -1, cur_h = -1, pages_mine = 0;
  bool split = false;  // the current segment is shared with other CTAs
  bool have_q = false;
  for (int n = 0;; ++n) {
    const int2 R = (n == 0) ? r0 : piece(n);
    if (R.x >= R.y) break;  // no more work (later pieces are empty too)
    fill_issue(piece(n + 1), ord_base + warp_count(R));
    // the (b, h) segments inside piece R, in order
    int64_t x = R.x;
    while (x < R.y) {
      const int b = seq_of(x);
      const int np = pfx[b + 1] - pfx[b];
      const int64_t sb = (int64_t)p.Hkv * pfx[b];
      const int h = (int)udiv64(x - sb, np);
      const int64_t seg_start = sb + (int64_t)h * np;
      const int64_t seg_end = seg_start + np;
      const int64_t pe = seg_end < R.y ? seg_end : R.y;
      if (b != cur_b || h != cur_h) {
        if (cur_b >= 0) flush(cur_b, cur_h, split, pages_mine);
        cur_b = b;
        cur_h = h;
        pages_mine = 0;
        have_q = false;
        reset_state();
        split = x > seg_start || seg_end > sh_hi;
      }
      // this warp's ordinals inside [x, pe)
      const int64_t lo_j = x - R.x - warp + NW - 1;
      const int64_t hi_j = pe - R.x - warp + NW - 1;
      const int j0 = (int)((lo_j > 0 ? lo_j : 0) / NW);
      const int j1 = (int)((hi_j > 0 ? hi_j : 0) / NW);
      for (int j = j0; j < j1; ++j, ++k) {
        if (!have_q) {
          load_q(b, h);
          have_q = true;
        }
        if constexpr (kGroup > 1) {  // several pages of the segment at a time
          const int ng = (j1 - j >= kGroup) ? kGroup : 1;
          if (ng > 1) {
            uint32_t kt[kGroup];
            int vv[kGroup], rw[kGroup];
            bool all_ok = true;
#pragma unroll
            for (int i = 0; i < kGroup; ++i) {
              if (i < ng) {
                const int2 di = desc[(k + i) % kDescRing];
                const int si = (k + i) % kS;
                if (!dead && !mbar_wait_bounded(smem_u32(&bars[warp * kS + si]),
                                                (uint32_t)(((k + i) / kS) & 1), kWaitLimitNs))
                  set_dead(k + i);
                kt[i] = ring + (uint32_t)(si * C::kStageBytes);
                vv[i] = (di.x >= 0) ? di.y : 0;
                rw[i] = di.x;
                all_ok = all_ok && vv[i] > 0;
              }
            }
            if constexpr (kFusedAppend) {
              if (p.k_new != nullptr && !dead) {
#pragma unroll
                for (int i = 0; i < kGroup; ++i)  // rem <= P: the page with the newest token
                  if (i < ng && vv[i] > 0 && (vv[i] & kRemMask) <= kPageSize)
                    append_new(kt[i], rw[i], (vv[i] & kRemMask) - 1, b, h);
              }
            }
            if (!dead) {
              if (all_ok) {
                compute_pages(Int<kGroup>{}, kt, vv);
              } else {
                for (int i = 0; i < ng; ++i)
                  if (vv[i] > 0) compute_page(kt[i], vv[i]);
              }
            }
            __syncwarp();
            if (fill_commit()) filled_end = f_ord + f_cnt;
            if (!dead) top_up(k + ng);
            j += ng - 1;
            k += ng - 1;
            continue;
          }
        }
        const int2 dsc = desc[k % kDescRing];
        const int slot = k % kS;
        if (!dead && !mbar_wait_bounded(smem_u32(&bars[warp * kS + slot]),
                                        (uint32_t)((k / kS) & 1), kWaitLimitNs))
          set_dead(k);
        if constexpr (kFusedAppend) {
          if (p.k_new != nullptr && !dead && dsc.x >= 0 && dsc.y > 0 &&
              (dsc.y & kRemMask) <= kPageSize)
            append_new(ring + (uint32_t)(slot * C::kStageBytes), dsc.x, (dsc.y & kRemMask) - 1,
                       b, h);
        }
        if (!dead && dsc.x >= 0 && dsc.y > 0)
          compute_page(ring + (uint32_t)(slot * C::kStageBytes), dsc.y);
        __syncwarp();
        if (fill_commit()) filled_end = f_ord + f_cnt;
        if (!dead) top_up(k + 1);
      }
      pages_mine += (int)(pe - x);
      x = pe;
    }
    if (fill_commit()) {  // this warp had no page left in piece R
      filled_end = f_ord + f_cnt;
      if (!dead) top_up(k);
    }
    ord_base += warp_count(R);
  }
  if (cur_b >= 0) flush(cur_b, cur_h, split, pages_mine);
  tickets_step(true);
  merge_barrier();
  merge_flagged();
  if (dead) {
    // let the copies this warp still has in flight land (bounded) before exit
    for (int q = k_dead; q < issued; ++q)
      mbar_wait_bounded(smem_u32(&bars[warp * kS + (q % kS)]), (uint32_t)((q / kS) & 1),
                        kWaitLimitNs);
  }
}

// ---------------------------------------------------------------------------
// Host-side dispatch over head_dim, group and query tokens for one cache kind.
template <int D, int G, int QC, int CACHE, bool QBF16, bool DEEP>
cudaError_t launch_split(const DecodeLaunch& l) {
  auto kern = decode_kernel<D, G, QC, CACHE, QBF16, DEEP>;
  const size_t smem = decode_smem_bytes_form(D, (CacheKind)CACHE, l.p.B, DEEP);
  static size_t configured = 0;  // largest dynamic smem size set so far
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)l.ctas);
  cfg.blockDim = dim3(decode_warps((CacheKind)CACHE) * 32);
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
  const bool deep = decode_use_deep(d, (CacheKind)CACHE, l.p.B);
#define PKV_CASE(DD, GG)                                                         \
  if (d == DD && g == GG) {                                                      \
    if constexpr (CACHE == kCacheE4M3Tok)                                        \
      if (deep) return launch_split<DD, GG, 1, CACHE, QBF16, true>(l);           \
    return launch_split<DD, GG, 1, CACHE, QBF16, false>(l);                      \
  }
  if constexpr (!cache_is_fp8((CacheKind)CACHE)) {
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
  }
  PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
#undef PKV_CASE
  return cudaErrorNotSupported;
}

}  // namespace pkv
