// pkv_decode_impl.cuh -- split-K flash-decoding kernel over a paged KV cache.
//
// What it computes: for each sequence b and KV head h, the unnormalised
// online-softmax state (m, l, o) of the g query heads that share h, over a
// contiguous run of the sequence's pages.  The split-combine kernel merges
// the runs.  Sources: "KV Cache & Flash Attention." (kvcache-7e2.pages.dev),
// Flash Attention and online-softmax sections (running max and sum, rescale
// by exp(m_old - m_new), one division at the end) and PagedAttention section
// (block = table[pos / P], offset = pos % P, gathered at lookup time);
// "KV Cache & FlashAttention" (deepforge.srivtx.xyz), running-summary
// paragraph.
//
// Schedule.  All (b, h, page) units are laid out b-major, then h, then page,
// and cut into equal contiguous shares, one per warp of a persistent grid
// (a few CTAs per SM).  A warp's share may cover the tail of one (b, h)
// segment, whole segments and the head of another; each piece is a "chunk"
// whose partial state goes to the workspace under id (warp + segment), which
// is unique.  Ragged lengths therefore never leave SMs idle.
//
// Data path per warp.  A ring of kStages shared-memory slots, each holding
// one K page and one V page.  Lane 0 issues 2-D TMA tile loads (128-byte
// swizzle, evict-first L2 policy) that complete on the slot's mbarrier; the
// whole warp waits, computes, and refills the slot with the page kStages
// ahead.  The block-table lookups for 32 pages at a time are done by the 32
// lanes in parallel into a small descriptor window in shared memory.
//
// Math per page (16 tokens):
//   S^T[16 tok][8] = K[16][d] . Q^T[d][8]      mma.m16n8k16, K via ldmatrix,
//                                              Q^T resident in registers;
//                                              columns are the g query heads
//   online softmax in registers (log2 domain), column max over the 16
//   tokens with 3 shuffles; the running max is only moved when a tile's max
//   exceeds it by more than 2^8, which keeps every p <= 256 and is exact
//   because the same stale max is used for l and o;
//   O^T[d][8] += V^T[d][16] . P^T[16][8]       V^T via ldmatrix.trans, P^T
//                                              via movmatrix; P is split into
//                                              hi + lo 16-bit parts so the
//                                              weights keep ~16 mantissa bits.
// FP8 (E4M3) pages are converted to fp16 in registers (exact) after the
// ldmatrix; the per-head K scale is folded into the score scale and the V
// scale into the partial output.
#pragma once

#include <cuda.h>
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per bounded wait
constexpr float kRescaleThreshold = 8.0f;         // log2 units

template <int D, int CACHE>
struct DecodeCfg {
  static constexpr int kElem = CACHE == kCacheE4M3 ? 1 : 2;
  static constexpr int kRowBytes = D * kElem;              // bytes per token row
  static constexpr int kBoxes = kRowBytes / 128;           // 128-byte TMA boxes per row
  static constexpr int kBoxBytes = kPageSize * 128;        // one box of a page
  static constexpr int kTileBytes = kPageSize * kRowBytes; // one K (or V) page
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kRingBudget = 96 * 1024;
  static constexpr int kStagesRaw = kRingBudget / (kDecodeWarps * kStageBytes);
  static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
  static constexpr int kKSteps = D / 16;  // k-steps of the QK contraction
  static constexpr int kMTiles = D / 16;  // 16-row tiles of O^T
  static_assert(kRowBytes % 128 == 0, "rows must be whole 128-byte boxes");
};

__host__ __device__ constexpr size_t decode_ring_bytes(int stage_bytes, int stages) {
  return (size_t)kDecodeWarps * stages * stage_bytes;
}

// Byte offset of 16-byte chunk `chunk` of token row `tok` inside a page
// loaded as 128-byte-swizzled boxes of 16 rows.
__device__ __forceinline__ uint32_t swz(int tok, int chunk) {
  return (uint32_t)((chunk >> 3) * (kPageSize * 128) + tok * 128 +
                    (((chunk & 7) ^ (tok & 7)) << 4));
}

template <int D, int G, int CACHE, bool QBF16>
__global__ void __launch_bounds__(kDecodeWarps * 32, kDecodeCtasPerSm)
    decode_split_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv) {
  using C = DecodeCfg<D, CACHE>;
  constexpr bool kBF = (CACHE == kCacheBF16);  // mma operand type (else fp16)
  constexpr int kS = C::kStages;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const size_t ring_bytes = decode_ring_bytes(C::kStageBytes, kS);
  const uint32_t ring = base + (uint32_t)(warp * kS * C::kStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + ring_bytes);
  int4* win_all = reinterpret_cast<int4*>(bars + kDecodeWarps * kS);
  int4* win = win_all + warp * 64;
  int32_t* pfx = reinterpret_cast<int32_t*>(win_all + kDecodeWarps * 64);  // [B+1]
  int32_t* ctxs = pfx + (p.B + 1);                                         // [B]

  // ---- prologue: pages per sequence and their prefix sums (whole CTA)
  if (threadIdx.x == 0) pfx[0] = 0;
  for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
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
      int idx = b0 + lane + 1;
      int v = (idx <= p.B) ? pfx[idx] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += u;
      }
      if (idx <= p.B) pfx[idx] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();

  const int64_t W = (int64_t)p.Hkv * pfx[p.B];
  const int gw = blockIdx.x * kDecodeWarps + warp;
  const int64_t G_w = p.num_warps_total;
  const int64_t lo = W * gw / G_w;
  const int64_t hi = W * (gw + 1) / G_w;
  const int n = (int)(hi - lo);
  if (n <= 0) return;

  if (lane == 0) {
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  const uint64_t pol = l2_policy_evict_first();

  // ---- page descriptors: {tma row or -1, segment id, page in sequence, valid tokens}
  auto fill_window = [&](int k) {
    const int64_t x = lo + 32 * (int64_t)k + lane;
    int4 dsc = make_int4(-1, -1, 0, 0);
    if (x < hi) {
      int a = 0, z = p.B;
      while (z - a > 1) {
        int mid = (a + z) >> 1;
        if ((int64_t)p.Hkv * pfx[mid] <= x) a = mid; else z = mid;
      }
      const int b = a;
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
    win[(k & 1) * 32 + lane] = dsc;
    __syncwarp();
  };

  auto issue = [&](int i) {
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
  const int c4 = lane & 3;   // column pair of the C fragments: heads 2*c4, 2*c4+1
  const int r8 = lane >> 2;  // row of the C fragments: token r8 / r8+8, d row r8 / r8+8
  // QK A operand (K page, row-major): ldmatrix lane -> (token, chunk)
  const int qk_tok = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int qk_chunk_hi = lane >> 4;
  // PV A operand (V page read transposed): ldmatrix lane -> (token, chunk)
  const int pv_tok = (lane & 7) + (lane >> 4) * 8;
  const int pv_chunk_hi = (lane >> 3) & 1;

  uint32_t qf[C::kKSteps][2];
  float o[C::kMTiles][4];
  float m2[2], l2[2];
  float c2 = 0.f;      // score scale in log2 units (FP8: times the K scale)
  float vscale = 1.f;  // FP8: V scale
  int cur_seg = -1;

  auto begin_segment = [&](const int4& dsc) {
    cur_seg = dsc.y;
    const int b = cur_seg / p.Hkv;
    const int h = cur_seg - b * p.Hkv;
    const int head = r8;  // B fragment column n = lane / 4
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
#pragma unroll
    for (int mt = 0; mt < C::kMTiles; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;
    m2[0] = m2[1] = -INFINITY;
    l2[0] = l2[1] = 0.f;
    c2 = p.scale_log2;
    vscale = 1.f;
    if constexpr (CACHE == kCacheE4M3) {
      c2 *= p.k_scale[h];
      vscale = p.v_scale[h];
    }
    if (dsc.z == 0 && lane == 0) {
      // first chunk of this segment: record where the combine finds its chunks
      const int np = pfx[b + 1] - pfx[b];
      const int64_t seg_end = (int64_t)p.Hkv * pfx[b] + (int64_t)(h + 1) * np;  // exclusive
      const int64_t w_last = (seg_end * G_w - 1) / W;
      p.seg_info[2 * cur_seg] = gw + cur_seg;
      p.seg_info[2 * cur_seg + 1] = (int)(w_last - gw + 1);
    }
  };

  auto flush = [&]() {
    float lt0 = l2[0], lt1 = l2[1];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      lt0 += __shfl_xor_sync(0xffffffffu, lt0, off);
      lt1 += __shfl_xor_sync(0xffffffffu, lt1, off);
    }
    const int64_t chunk = (int64_t)gw + cur_seg;
    float* po = p.part_o + chunk * G * D;
    float* pml = p.part_ml + chunk * G * 2;
    const int h0 = 2 * c4, h1 = 2 * c4 + 1;
    if (r8 == 0) {
      if (h0 < G) { pml[2 * h0] = m2[0]; pml[2 * h0 + 1] = lt0; }
      if (h1 < G) { pml[2 * h1] = m2[1]; pml[2 * h1 + 1] = lt1; }
    }
#pragma unroll
    for (int mt = 0; mt < C::kMTiles; ++mt) {
      int dA, dB;  // d of O^T rows r8 and r8 + 8 in this tile
      if constexpr (CACHE != kCacheE4M3) {
        dA = 16 * mt + r8;
        dB = dA + 8;
      } else {
        dA = 32 * (mt >> 1) + 2 * r8 + (mt & 1);
        dB = dA + 16;
      }
      if (h0 < G) {
        po[h0 * D + dA] = o[mt][0] * vscale;
        po[h0 * D + dB] = o[mt][2] * vscale;
      }
      if (h1 < G) {
        po[h1 * D + dA] = o[mt][1] * vscale;
        po[h1 * D + dB] = o[mt][3] * vscale;
      }
    }
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
      for (int mt = 0; mt < C::kMTiles; ++mt) {
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
      for (int mt = 0; mt < C::kMTiles; ++mt) {
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

  // ---- main loop
  const int pre = n < kS ? n : kS;
  for (int i = 0; i < pre; ++i) issue(i);
  bool timed_out = false;
  int j = 0;
  for (; j < n; ++j) {
    const int4 dsc = win[((j >> 5) & 1) * 32 + (j & 31)];
    if (dsc.y != cur_seg) {
      if (cur_seg >= 0) flush();
      begin_segment(dsc);
    }
    const int slot = j % kS;
    if (!mbar_wait_bounded(smem_u32(&bars[warp * kS + slot]), (uint32_t)((j / kS) & 1),
                           kWaitLimitNs)) {
      timed_out = true;
      break;
    }
    if (dsc.x >= 0 && dsc.w > 0) compute_page(ring + (uint32_t)(slot * C::kStageBytes), dsc.w);
    __syncwarp();
    if (j + kS < n) issue(j + kS);
  }
  if (timed_out) {
    if (lane == 0) report_error(p.err_word, PKV_ERR_TIMEOUT);
    // let the copies this warp still has in flight land (bounded) before exit
    const int issued = (j + kS < n) ? j + kS : n;
    for (int k = j + 1; k < issued; ++k)
      mbar_wait_bounded(smem_u32(&bars[warp * kS + (k % kS)]), (uint32_t)((k / kS) & 1),
                        kWaitLimitNs);
    return;
  }
  if (cur_seg >= 0) flush();
}

// ---------------------------------------------------------------------------
// Host-side dispatch over head_dim and group for one cache kind.
template <int D, int G, int CACHE, bool QBF16>
cudaError_t launch_split(const DecodeLaunch& l) {
  using C = DecodeCfg<D, CACHE>;
  auto kern = decode_split_kernel<D, G, CACHE, QBF16>;
  const size_t smem = decode_smem_bytes(D, (CacheKind)CACHE, l.p.B);
  static size_t configured = 0;  // largest dynamic smem size set so far
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  (void)sizeof(C);
  kern<<<l.ctas, kDecodeWarps * 32, smem, l.stream>>>(l.p, l.tmap_k, l.tmap_v);
  return cudaGetLastError();
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
