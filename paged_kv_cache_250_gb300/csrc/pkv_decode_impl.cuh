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
// then h, then page, and cut into equal contiguous ranges, one per CTA of a
// persistent grid (two CTAs per SM).  Inside a CTA, page j of the range goes
// to warp j % 4, so the four warps move through the same (b, h) "segment"
// together.  When the CTA's range leaves a segment, the four warps' online-
// softmax states are merged in shared memory.  A segment wholly inside one
// CTA is normalised and written at once; otherwise each CTA that touches it
// stores a partial (m, l, o) under chunk id (cta + segment), which is unique,
// and the last CTA to finish the segment (an atomic ticket, no waiting)
// merges the partials and writes the output.  Ragged lengths therefore never
// leave SMs idle and no separate combine launch is needed.
//
// Data path per warp.  A ring of kStages shared-memory slots, each holding
// one K page and one V page of one (block, KV head).  Lane 0 issues 2-D TMA
// tile loads (128-byte swizzle, evict-first L2 policy) that complete on the
// slot's mbarrier; the warp waits, computes, and refills the slot with its
// page kStages ahead.  Block-table lookups are done 32 pages at a time, one
// per lane, into a small descriptor window in shared memory.
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

template <int D, int CACHE>
struct DecodeCfg {
  static constexpr int kElem = CACHE == kCacheE4M3 ? 1 : 2;
  static constexpr int kRowBytes = D * kElem;              // bytes per token row
  static constexpr int kBoxes = kRowBytes / 128;           // 128-byte TMA boxes per row
  static constexpr int kBoxBytes = kPageSize * 128;        // one box of a page
  static constexpr int kTileBytes = kPageSize * kRowBytes; // one K (or V) page
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kKSteps = D / 16;  // k-steps of the QK contraction
  static constexpr int kMTiles = D / 16;  // 16-row tiles of O^T
  static constexpr int kStages = decode_stages(D, (CacheKind)CACHE);
  static constexpr int kLaneState = 4 + 4 * kMTiles;  // m[2], l[2], o[MT][4] per lane
  static_assert(kRowBytes % 128 == 0, "rows must be whole 128-byte boxes");
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

template <int D, int G, int CACHE, bool QBF16>
__global__ void __launch_bounds__(kDecodeWarps * 32, kDecodeCtasPerSm)
    decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv) {
  using C = DecodeCfg<D, CACHE>;
  constexpr bool kBF = (CACHE == kCacheBF16);  // mma operand type (else fp16)
  constexpr int kS = C::kStages;
  constexpr int NW = kDecodeWarps;
  constexpr int kMT = C::kMTiles;

  if (!p.early_prologue) griddep_wait();

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const uint32_t ring = base + (uint32_t)(warp * kS * C::kStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + (size_t)NW * kS * C::kStageBytes);
  int4* win_all = reinterpret_cast<int4*>(bars + NW * kS);
  int4* win = win_all + warp * 64;
  float* mbuf = reinterpret_cast<float*>(win_all + NW * 64);  // [2][kLaneState][32]
  int* flag = reinterpret_cast<int*>(mbuf + 2 * C::kLaneState * 32);
  int32_t* pfx = flag + 4;           // [B+1]
  int32_t* ctxs = pfx + (p.B + 1);   // [B]

  // ---- prologue: pages per sequence and their prefix sums (whole CTA)
  if (tid == 0) pfx[0] = 0;
  for (int b = tid; b < p.B; b += blockDim.x) {
    int c = p.context_lens[b];
    int np = 0;
    if (c < 0 || c > p.MBS * kPageSize) {
      if (blockIdx.x == 0) report_error(p.err_word, PKV_ERR_BOUNDS);
      c = 0;
    } else {
      np = (c + kPageSize - 1) / kPageSize;
    }
    ctxs[b] = c;
    pfx[b + 1] = np;
  }
  if (lane == 0) {
    for (int s = 0; s < kS; ++s) mbar_init(smem_u32(&bars[warp * kS + s]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int idx = b0 + lane + 1;
      int v = (idx <= p.B) ? pfx[idx] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += u;
      }
      if (idx <= p.B) pfx[idx] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();

  // ---- sequences with no tokens get a zero output row (spread over CTAs)
  for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
    if (pfx[b + 1] != pfx[b]) continue;
    const int64_t row0 = (int64_t)b * p.Hq * D;
    for (int i = tid; i < p.Hq * D; i += blockDim.x) store_out_rt(p.out_dtype, p.out, row0 + i, 0.f);
  }

  // ---- this CTA's contiguous range of the (b, h, page) units
  const int64_t W = (int64_t)p.Hkv * pfx[p.B];
  const int64_t Gc = W < (int64_t)gridDim.x ? W : (int64_t)gridDim.x;  // CTAs with work
  const int cta = blockIdx.x;
  if (cta >= Gc) return;
  const int64_t lo = W * cta / Gc;
  const int64_t hi = W * (cta + 1) / Gc;
  const int n = (int)(hi - lo);
  const int nk = n > warp ? (n - warp + NW - 1) / NW : 0;  // pages of this warp
  auto cta_of = [&](int64_t x) -> int64_t { return ((x + 1) * Gc - 1) / W; };
  auto seq_of = [&](int64_t x) -> int {
    int a = 0, z = p.B;
    while (z - a > 1) {
      const int mid = (a + z) >> 1;
      if ((int64_t)p.Hkv * pfx[mid] <= x) a = mid; else z = mid;
    }
    return a;
  };

  if (lane == 0) {
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  const uint64_t pol = l2_policy_evict_first();
  if (p.early_prologue) griddep_wait();  // the cache pages may have just been appended

  // ---- page descriptors: {tma row or -1, segment id, page in sequence, valid tokens}
  auto fill_window = [&](int m) {
    const int k = 32 * m + lane;
    int4 dsc = make_int4(-1, -1, 0, 0);
    if (k < nk) {
      const int64_t x = lo + warp + (int64_t)NW * k;
      const int b = seq_of(x);
      const int np = pfx[b + 1] - pfx[b];
      const int64_t r = x - (int64_t)p.Hkv * pfx[b];
      const int h = (int)(r / np);
      const int pg = (int)(r - (int64_t)h * np);
      const int blk = p.block_tables[(int64_t)b * p.MBS + pg];
      int row = -1;
      if (blk >= 0 && blk < p.NB) row = (blk * p.Hkv + h) * kPageSize;
      else report_error(p.err_word, PKV_ERR_BOUNDS);
      dsc = make_int4(row, b * p.Hkv + h, pg, min(kPageSize, ctxs[b] - pg * kPageSize));
    }
    win[(m & 1) * 32 + lane] = dsc;
    __syncwarp();
  };

  int issued = 0;
  auto issue = [&](int i) {
    issued = i + 1;
    if ((i & 31) == 0) fill_window(i >> 5);
    const int4 dsc = win[((i >> 5) & 1) * 32 + (i & 31)];
    if (lane == 0) {
      const int slot = i % kS;
      const uint32_t bar = smem_u32(&bars[warp * kS + slot]);
      const uint32_t kt = ring + (uint32_t)(slot * C::kStageBytes);
      const uint32_t vt = kt + C::kTileBytes;
      if (dsc.x >= 0) {
        mbar_arrive_expect_tx(bar, C::kStageBytes);
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx) {
          tma_load_2d(kt + bx * C::kBoxBytes, &tmk, bar, bx * (128 / C::kElem), dsc.x, pol);
          tma_load_2d(vt + bx * C::kBoxBytes, &tmv, bar, bx * (128 / C::kElem), dsc.x, pol);
        }
      } else {
        mbar_arrive(bar);  // nothing to load; complete the phase
      }
    }
  };

  // ---- per-lane fragment coordinates
  const int c4 = lane & 3;   // C-fragment column pair: heads 2*c4, 2*c4+1
  const int r8 = lane >> 2;  // C-fragment row: token r8 / r8+8, or O^T row r8 / r8+8
  const int qk_tok = (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix row, K page
  const int qk_chunk_hi = lane >> 4;
  const int pv_tok = (lane & 7) + (lane >> 4) * 8;        // ldmatrix row, V page (trans)
  const int pv_chunk_hi = (lane >> 3) & 1;

  // d of O^T rows r8 and r8 + 8 in m-tile mt
  auto d_of = [&](int mt, int half) -> int {
    if constexpr (CACHE != kCacheE4M3) return 16 * mt + r8 + 8 * half;
    else return 32 * (mt >> 1) + 2 * r8 + (mt & 1) + 16 * half;
  };

  uint32_t qf[C::kKSteps][2];
  float o[kMT][4];
  float m2[2], l2[2];
  float c2 = 0.f;  // score scale in log2 units (E4M3: times the K scale)

  auto reset_state = [&]() {
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;
    m2[0] = m2[1] = -INFINITY;
    l2[0] = l2[1] = 0.f;
  };

  auto load_q = [&](int b, int h) {
    const int head = r8;  // B-fragment column n = lane / 4
    const uint16_t* qrow =
        reinterpret_cast<const uint16_t*>(p.q) + ((int64_t)b * p.Hq + h * G + head) * D;
    if constexpr (CACHE != kCacheE4M3) {
#pragma unroll
      for (int ks = 0; ks < C::kKSteps; ++ks) {
        uint32_t b0 = 0, b1 = 0;
        if (head < G) {
          b0 = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c4);
          b1 = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c4 + 8);
        }
        qf[ks][0] = b0;
        qf[ks][1] = b1;
      }
    } else {
#pragma unroll
      for (int ks = 0; ks < C::kKSteps; ++ks) {
        uint32_t b0 = 0, b1 = 0;
        if (head < G) {
          const uint2 raw4 = *reinterpret_cast<const uint2*>(qrow + 16 * ks + 4 * c4);
          const float2 f01 = unpack2<QBF16>(raw4.x);
          const float2 f23 = unpack2<QBF16>(raw4.y);
          b0 = pack2<false>(f01.x, f01.y);
          b1 = pack2<false>(f23.x, f23.y);
        }
        qf[ks][0] = b0;
        qf[ks][1] = b1;
      }
    }
    c2 = p.scale_log2;
    if constexpr (CACHE == kCacheE4M3) c2 *= p.k_scale[h];
  };

  auto compute_page = [&](uint32_t kt, int valid) {
    const uint32_t vt = kt + C::kTileBytes;
    // ---- S^T = K . Q^T
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (CACHE != kCacheE4M3) {
#pragma unroll
      for (int ks = 0; ks < C::kKSteps; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, kt + swz(qk_tok, 2 * ks + qk_chunk_hi));
        mma_16816<kBF>(s, a, qf[ks][0], qf[ks][1]);
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
        mma_16816<false>(s, a, qf[2 * gi + 1][0], qf[2 * gi + 1][1]);
      }
    }
    // ---- online softmax (log2 domain); tokens past the context are masked
    float x0 = s[0] * c2, x1 = s[1] * c2, x2 = s[2] * c2, x3 = s[3] * c2;
    if (valid < kPageSize) {
      if (r8 >= valid) x0 = x1 = -INFINITY;
      if (r8 + 8 >= valid) x2 = x3 = -INFINITY;
    }
    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const bool grow = (mx0 > m2[0] + kRescaleThreshold) || (mx1 > m2[1] + kRescaleThreshold);
    if (__any_sync(0xffffffffu, grow)) {
      const float n0 = fmaxf(m2[0], mx0), n1 = fmaxf(m2[1], mx1);
      const float a0 = exp2f(m2[0] - n0), a1 = exp2f(m2[1] - n1);
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
    const float p0 = exp2f(x0 - m2[0]), p1 = exp2f(x1 - m2[1]);
    const float p2 = exp2f(x2 - m2[0]), p3 = exp2f(x3 - m2[1]);
    l2[0] += p0 + p2;
    l2[1] += p1 + p3;
    const uint32_t h01 = pack2<kBF>(p0, p1), h23 = pack2<kBF>(p2, p3);
    const float2 f01 = unpack2<kBF>(h01), f23 = unpack2<kBF>(h23);
    const uint32_t l01 = pack2<kBF>(p0 - f01.x, p1 - f01.y);
    const uint32_t l23 = pack2<kBF>(p2 - f23.x, p3 - f23.y);
    const uint32_t bh0 = movm_trans(h01), bh1 = movm_trans(h23);
    const uint32_t bl0 = movm_trans(l01), bl1 = movm_trans(l23);
    // ---- O^T += V^T . P^T ; V rows of masked tokens are zeroed (they may hold
    // anything, and 0 * NaN would poison the sum)
    uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
    if (valid < kPageSize) {
      const int t0 = 2 * c4;
      mlo = (t0 < valid ? 0x0000ffffu : 0u) | (t0 + 1 < valid ? 0xffff0000u : 0u);
      mhi = (t0 + 8 < valid ? 0x0000ffffu : 0u) | (t0 + 9 < valid ? 0xffff0000u : 0u);
    }
    if constexpr (CACHE != kCacheE4M3) {
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        uint32_t a[4];
        ldsm_x4_trans(a, vt + swz(pv_tok, 2 * mt + pv_chunk_hi));
        a[0] &= mlo;
        a[1] &= mlo;
        a[2] &= mhi;
        a[3] &= mhi;
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
        a[0] &= mlo;
        a[1] &= mlo;
        a[2] &= mhi;
        a[3] &= mhi;
        mma_16816<false>(o[2 * gi], a, bh0, bh1);
        mma_16816<false>(o[2 * gi], a, bl0, bl1);
#pragma unroll
        for (int e = 0; e < 4; ++e) a[e] = e4m3x2_to_f16x2(__byte_perm(r[e], 0, 0x0031));
        a[0] &= mlo;
        a[1] &= mlo;
        a[2] &= mhi;
        a[3] &= mhi;
        mma_16816<false>(o[2 * gi + 1], a, bh0, bh1);
        mma_16816<false>(o[2 * gi + 1], a, bl0, bl1);
      }
    }
  };

  // ---- merging warp states through shared memory (per-lane layout)
  auto store_state = [&](float* buf) {
    buf[0 * 32 + lane] = m2[0];
    buf[1 * 32 + lane] = m2[1];
    buf[2 * 32 + lane] = l2[0];
    buf[3 * 32 + lane] = l2[1];
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) buf[(4 + 4 * mt + e) * 32 + lane] = o[mt][e];
  };
  auto merge_state = [&](const float* buf) {
    float a[2], bw[2];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const float mb = buf[cc * 32 + lane];
      const float M = fmaxf(m2[cc], mb);
      if (M == -INFINITY) {
        a[cc] = 1.f;
        bw[cc] = 0.f;
      } else {
        a[cc] = exp2f(m2[cc] - M);
        bw[cc] = exp2f(mb - M);
        m2[cc] = M;
      }
      l2[cc] = a[cc] * l2[cc] + bw[cc] * buf[(2 + cc) * 32 + lane];
    }
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        o[mt][e] = a[e & 1] * o[mt][e] + bw[e & 1] * buf[(4 + 4 * mt + e) * 32 + lane];
  };

  // ---- end of a segment: merge the 4 warps, then write output or a partial
  auto end_segment = [&](int b, int h, int64_t seg_start, int64_t seg_end) {
    const int seg = b * p.Hkv + h;
    float* buf0 = mbuf;
    float* buf1 = mbuf + C::kLaneState * 32;
    if (warp >= 2) store_state(warp == 2 ? buf0 : buf1);
    merge_barrier();
    if (warp < 2) merge_state(warp == 0 ? buf0 : buf1);
    merge_barrier();
    if (warp == 1) store_state(buf0);
    merge_barrier();
    const float vs = (CACHE == kCacheE4M3) ? p.v_scale[h] : 1.f;
    const int64_t c_first = cta_of(seg_start);
    const int64_t count = cta_of(seg_end - 1) - c_first + 1;
    const int h0 = 2 * c4, h1 = 2 * c4 + 1;
    if (warp == 0) {
      merge_state(buf0);
      float lt0 = l2[0], lt1 = l2[1];
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        lt0 += __shfl_xor_sync(0xffffffffu, lt0, off);
        lt1 += __shfl_xor_sync(0xffffffffu, lt1, off);
      }
      if (count == 1) {
        // the whole segment is here: normalise and write the output rows
        const float i0 = lt0 > 0.f ? vs / lt0 : 0.f;
        const float i1 = lt1 > 0.f ? vs / lt1 : 0.f;
        const int64_t ob = ((int64_t)b * p.Hq + h * G) * D;
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
          const int dA = d_of(mt, 0), dB = d_of(mt, 1);
          if (h0 < G) {
            store_out_rt(p.out_dtype, p.out, ob + h0 * D + dA, o[mt][0] * i0);
            store_out_rt(p.out_dtype, p.out, ob + h0 * D + dB, o[mt][2] * i0);
          }
          if (h1 < G) {
            store_out_rt(p.out_dtype, p.out, ob + h1 * D + dA, o[mt][1] * i1);
            store_out_rt(p.out_dtype, p.out, ob + h1 * D + dB, o[mt][3] * i1);
          }
        }
      } else {
        const int64_t chunk = (int64_t)cta + seg;
        float* po = p.part_o + chunk * G * D;
        float* pml = p.part_ml + chunk * G * 2;
        if (r8 == 0) {
          if (h0 < G) { pml[2 * h0] = m2[0]; pml[2 * h0 + 1] = lt0; }
          if (h1 < G) { pml[2 * h1] = m2[1]; pml[2 * h1 + 1] = lt1; }
        }
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
          const int dA = d_of(mt, 0), dB = d_of(mt, 1);
          if (h0 < G) {
            po[h0 * D + dA] = o[mt][0] * vs;
            po[h0 * D + dB] = o[mt][2] * vs;
          }
          if (h1 < G) {
            po[h1 * D + dA] = o[mt][1] * vs;
            po[h1 * D + dB] = o[mt][3] * vs;
          }
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          const int old = atomicAdd(&p.tickets[seg], 1);
          flag[0] = (old == count - 1) ? 1 : 0;
        }
      }
    }
    merge_barrier();
    if (count > 1 && flag[0]) {
      // last CTA of this segment: merge every chunk's partial (all threads)
      __threadfence();
      const int64_t first = c_first + seg;
      constexpr int kCols = G * D / 4;  // float4 columns of the segment's output
      constexpr int kThreads = NW * 32;
      constexpr int kPerPass = kCols < kThreads ? kCols : kThreads;
      constexpr int kGroups = kThreads / kPerPass;  // chunk subsets merged in parallel
      float4* red = reinterpret_cast<float4*>(mbuf);      // [kGroups][kCols]
      float* lred = mbuf + 4 * kGroups * kCols;           // [kGroups][G]
      float* Ms = lred + kGroups * G;                     // [G]
      if (tid < G) {
        float M = -INFINITY;
        for (int64_t kk = 0; kk < count; ++kk) {
          const float2 ml = __ldcg(
              reinterpret_cast<const float2*>(p.part_ml + ((first + kk) * G + tid) * 2));
          if (ml.y > 0.f) M = fmaxf(M, ml.x);
        }
        Ms[tid] = M;
      }
      merge_barrier();
      const int grp = tid / kPerPass;
      for (int col = tid % kPerPass; col < kCols; col += kPerPass) {
        const int head = col / (D / 4);
        const float M = Ms[head];
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float lsum = 0.f;
        if (M > -INFINITY) {
#pragma unroll 4
          for (int64_t kk = grp; kk < count; kk += kGroups) {
            const float2 ml = __ldcg(
                reinterpret_cast<const float2*>(p.part_ml + ((first + kk) * G + head) * 2));
            if (!(ml.y > 0.f)) continue;
            const float w = exp2f(ml.x - M);
            lsum += w * ml.y;
            const float4 v =
                __ldcg(reinterpret_cast<const float4*>(p.part_o + (first + kk) * G * D) + col);
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
          }
        }
        if constexpr (kGroups == 1) {
          const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
          const int64_t ob = ((int64_t)b * p.Hq + h * G + head) * D + (col % (D / 4)) * 4;
          store_out_rt(p.out_dtype, p.out, ob + 0, acc.x * inv);
          store_out_rt(p.out_dtype, p.out, ob + 1, acc.y * inv);
          store_out_rt(p.out_dtype, p.out, ob + 2, acc.z * inv);
          store_out_rt(p.out_dtype, p.out, ob + 3, acc.w * inv);
        } else {
          red[grp * kCols + col] = acc;
          if ((col % (D / 4)) == 0) lred[grp * G + head] = lsum;
        }
      }
      if constexpr (kGroups > 1) {
        merge_barrier();
        if (tid < kCols) {
          const int col = tid;
          const int head = col / (D / 4);
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          float L = 0.f;
#pragma unroll
          for (int g2 = 0; g2 < kGroups; ++g2) {
            const float4 v = red[g2 * kCols + col];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
            L += lred[g2 * G + head];
          }
          const float inv = L > 0.f ? 1.f / L : 0.f;
          const int64_t ob = ((int64_t)b * p.Hq + h * G + head) * D + (col % (D / 4)) * 4;
          store_out_rt(p.out_dtype, p.out, ob + 0, acc.x * inv);
          store_out_rt(p.out_dtype, p.out, ob + 1, acc.y * inv);
          store_out_rt(p.out_dtype, p.out, ob + 2, acc.z * inv);
          store_out_rt(p.out_dtype, p.out, ob + 3, acc.w * inv);
        }
      }
      if (tid == 0) p.tickets[seg] = 0;  // ready for the next call
    }
    merge_barrier();  // buffers and flag free again
  };

  // ---- main loop: segments of this CTA's range in order
  const int pre = nk < kS ? nk : kS;
  for (int i = 0; i < pre; ++i) issue(i);
  bool dead = false;  // a bounded wait gave up: skip compute, keep the barriers
  int k_dead = -1;
  int k = 0;
  int64_t x = lo;
  while (true) {
    const int b = seq_of(x);
    const int np = pfx[b + 1] - pfx[b];
    const int64_t sb = (int64_t)p.Hkv * pfx[b];
    const int h = (int)((x - sb) / np);
    const int64_t seg_start = sb + (int64_t)h * np;
    const int64_t seg_end = seg_start + np;
    reset_state();
    bool have_q = false;
    while (k < nk && lo + warp + (int64_t)NW * k < seg_end) {
      if (!have_q) {
        load_q(b, h);
        have_q = true;
      }
      const int4 dsc = win[((k >> 5) & 1) * 32 + (k & 31)];
      const int slot = k % kS;
      if (!dead && !mbar_wait_bounded(smem_u32(&bars[warp * kS + slot]),
                                      (uint32_t)((k / kS) & 1), kWaitLimitNs)) {
        dead = true;
        k_dead = k;
        if (lane == 0) report_error(p.err_word, PKV_ERR_TIMEOUT);
      }
      if (!dead && dsc.x >= 0 && dsc.w > 0)
        compute_page(ring + (uint32_t)(slot * C::kStageBytes), dsc.w);
      __syncwarp();
      if (!dead && k + kS < nk) issue(k + kS);
      ++k;
    }
    end_segment(b, h, seg_start, seg_end);
    x = seg_end;
    if (x >= hi) break;
  }
  if (dead) {
    // let the copies this warp still has in flight land (bounded) before exit
    for (int q = k_dead + 1; q < issued; ++q)
      mbar_wait_bounded(smem_u32(&bars[warp * kS + (q % kS)]), (uint32_t)((q / kS) & 1),
                        kWaitLimitNs);
  }
}

// ---------------------------------------------------------------------------
// Host-side dispatch over head_dim and group for one cache kind.
template <int D, int G, int CACHE, bool QBF16>
cudaError_t launch_split(const DecodeLaunch& l) {
  auto kern = decode_kernel<D, G, CACHE, QBF16>;
  const size_t smem = decode_smem_bytes(D, (CacheKind)CACHE, l.p.B);
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

template <int CACHE, bool QBF16>
cudaError_t dispatch_split(const DecodeLaunch& l) {
  const int d = l.p.d;
  const int g = l.group;
#define PKV_CASE(DD, GG) \
  if (d == DD && g == GG) return launch_split<DD, GG, CACHE, QBF16>(l);
  if constexpr (CACHE != kCacheE4M3) {
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
  }
  PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
#undef PKV_CASE
  return cudaErrorNotSupported;
}

}  // namespace pkv
