// Paged prefill attention on the 5th-generation tensor cores (tcgen05).
//
// A chunk of q_len new tokens per sequence, already appended to the cache,
// attends causally over the sequence's whole context through its block table
// ("KV Cache & Flash Attention." (kvcache-7e2.pages.dev): the prefill phase
// processes the prompt in one parallel pass; continuous-batching section:
// chunked prefill reads each sequence's pages through its table).  Token j of
// the chunk sits at position ctx - q_len + j and sees positions 0 .. itself.
//
// One CTA (4 warps) owns 128 query rows: 128 / g new tokens of one sequence
// times the g query heads that share one KV head, so every page it loads
// serves the whole group.  Row r is token r / g, head r % g.  Thread t owns
// row t: TMEM lane t holds its scores and its output accumulator, so the
// online softmax (running max m, sum l, rescale of O) needs no shuffles.
// Per block of 64 cached tokens (4 pages):
//   S = Q K^T    tcgen05.mma, M 128 x N 64 x K 128 (d), both operands K-major
//                128-byte-swizzled tiles as the tensor copies write them;
//   softmax      tcgen05.ld of the thread's row, mask, exp2, P as a bf16 (or
//                fp16) hi + lo pair written to shared memory;
//   O += P V     tcgen05.mma twice (hi and lo), M 128 x N 128 (d) x K 64
//                (tokens); V is used where the copies put it, as an MN-major
//                operand.
// K and V have one buffer each: the next block's K is copied in while this
// block's softmax runs, its V once this block's P.V is done.  About 97 KB of
// shared memory and 256 TMEM columns let two CTAs share an SM, so one CTA's
// MMAs and copies overlap the other's softmax.
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kPfRows = 128;          // query rows per CTA
constexpr int kPfTok = 64;            // cached tokens per block (4 pages)
constexpr int kPfPages = kPfTok / kPageSize;
constexpr int kPfD = 128;             // head dim built
constexpr int kPfThreads = 128;
constexpr uint32_t kQHalf = 16384;    // 128 rows x 128 bytes: d columns 0-63 or 64-127 of Q
constexpr uint32_t kKHalf = 8192;     // 64 rows x 128 bytes: the same of a K or V block
// shared memory plan, offsets from a 1024-byte aligned base
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = 2 * kQHalf;
constexpr uint32_t kOffV = kOffK + 2 * kKHalf;
constexpr uint32_t kOffPh = kOffV + 2 * kKHalf;  // P: 128 rows x 64 tokens, hi then lo
constexpr uint32_t kOffPl = kOffPh + kQHalf;
constexpr uint32_t kOffBar = kOffPl + kQHalf;    // mbarriers q, k, v, s, o; TMEM base; counts
constexpr uint32_t kTmemCols = 256;              // S: columns 0..63, O: 128..255
constexpr uint64_t kPfWaitNs = 1000000000ull;

__device__ __forceinline__ void tma_load_2d_plain(uint32_t dst, const void* tmap, uint32_t bar,
                                                  int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(tmap), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar,
                                            int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(tmap), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// ---- tcgen05 (PTX ISA: tensor memory, matrix descriptors, tcgen05.mma)
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
               ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] . B[smem]^T, kind::f16, issued by one thread
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                     uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}
// arrive once on `bar` when every MMA this thread issued before has completed
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(bar) : "memory");
}
// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor, kind::f16: fp32 accumulator, A and B of one 16-bit
// type, A K-major, B K-major or MN-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, bool b_mn, int M, int N) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ float ex2(float x) {  // 2^x (PTX ex2.approx; -inf gives 0)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// 32 consecutive 32-bit TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
               : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

template <bool BF16>
__global__ void __launch_bounds__(kPfThreads, 2)
    prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmq,
                   const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv) {
  const int b = blockIdx.x / p.tiles_per_seq;
  const int tile = blockIdx.x - b * p.tiles_per_seq;
  const int h = blockIdx.y;                 // KV head
  const int G = p.Hq / p.Hkv;               // query heads per KV head
  const int tpt = kPfRows / G;              // tokens per tile
  const int tid = threadIdx.x, warp = tid >> 5;

  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int q0 = p.q_start[b], qn = p.q_start[b + 1] - q0;  // this sequence's rows
  const int ctx = p.context_lens[b];
  if (qn < 0 || ctx < qn || ctx > p.MBS * kPageSize || q0 < 0 || q0 + qn > p.total_q ||
      qn > p.tiles_per_seq * tpt) {
    if (tid == 0 && tile == 0 && h == 0) report_error(p.err_word, PKV_ERR_BOUNDS);
    return;
  }
  if (tile * tpt >= qn) return;  // no rows of this sequence in the tile

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const uint32_t bar_q = base + kOffBar, bar_k = bar_q + 8, bar_v = bar_q + 16,
                 bar_s = bar_q + 24, bar_o = bar_q + 32;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base_ptr + kOffBar + 40);
  // completions expected on the q, k, v, s, o barriers (thread 0 counts)
  volatile int32_t* issued = reinterpret_cast<volatile int32_t*>(base_ptr + kOffBar + 44);

  if (warp == 0) {
    tmem_alloc(base + kOffBar + 40, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < 5; ++i) issued[i] = 0;
    for (int i = 0; i < 5; ++i) mbar_init(bar_q + 8 * i, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_s = tmem, t_o = tmem + 128;   // column offsets
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

  // row t of the tile: new token j = tile * tpt + t / G (position ctx - qn + j),
  // query head h * G + t % G
  const int row = tile * tpt + tid / G;
  const int hq = h * G + tid % G;
  const bool row_real = row < qn;
  const int pos_q = ctx - qn + row;
  const int vis = min(pos_q, ctx - 1);  // last visible position of this row
  const int last_row = min(qn, (tile + 1) * tpt) - 1;
  const int nblk = (ctx - qn + last_row) / kPfTok + 1;  // causal: blocks any row sees
  const int all_vis = ctx - qn + tile * tpt;            // every row sees positions <= this
  const int np = (ctx + kPageSize - 1) / kPageSize;
  const float c2 = p.scale_log2;
  constexpr uint32_t kIdS = idesc_f16(BF16, false, kPfRows, kPfTok);
  constexpr uint32_t kIdO = idesc_f16(BF16, true, kPfRows, kPfD);

  // Every wait is bounded and its outcome voted on by the whole CTA, so all
  // threads leave the loop together and every barrier is met.
  auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
    const bool bad = !mbar_wait_bounded(bar, parity, kPfWaitNs);
    return __syncthreads_or(bad) == 0;
  };
  // the tensor copies of block j's K (or V) pages; pages past the context are
  // not loaded (their scores are masked, their V rows zeroed)
  auto load_block = [&](int j, bool v) {
    const uint32_t dst = base + (v ? kOffV : kOffK);
    const uint32_t bar = v ? bar_v : bar_k;
    const int pg0 = j * kPfPages;
    const int npg = min(kPfPages, np - pg0);
    issued[v ? 2 : 1] = issued[v ? 2 : 1] + 1;
    mbar_arrive_expect_tx(bar, (uint32_t)npg * 2 * kPageSize * 128);
    for (int i = 0; i < npg; ++i) {
      int blk = p.block_tables[(int64_t)b * p.MBS + pg0 + i];
      if (blk < 0 || blk >= p.NB) {  // the copy reads the fill value (zeros) past the pool
        report_error(p.err_word, PKV_ERR_BOUNDS);
        blk = p.NB;
      }
      const int r = (blk * p.Hkv + h) * kPageSize;
      for (int c = 0; c < 2; ++c)
        tma_load_2d_plain(dst + (uint32_t)c * kKHalf + (uint32_t)i * kPageSize * 128,
                          v ? (const void*)&tmv : (const void*)&tmk, bar, c * 64, r);
    }
  };

  if (tid == 0) {
    prefetch_tmap(&tmq);
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
    issued[0] = 1;
    mbar_arrive_expect_tx(bar_q, 2 * kQHalf);
    for (int c = 0; c < 2; ++c)
      tma_load_3d(base + kOffQ + (uint32_t)c * kQHalf, &tmq, bar_q, c * 64, h * G,
                  q0 + tile * tpt);
    load_block(0, false);
    load_block(0, true);
  }
  bool dead = !wait_all(bar_q, 0);

  float m_ref = -INFINITY, l_sum = 0.f;
  for (int j = 0; j < nblk && !dead; ++j) {
    const uint32_t par = (uint32_t)(j & 1);
    if (!wait_all(bar_k, par)) {
      dead = true;
      break;
    }
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kPfD / 16; ++ks) {  // S = Q K^T over d, 16 at a time
        const uint32_t qoff = (uint32_t)(ks >> 2) * kQHalf + (uint32_t)(ks & 3) * 32;
        const uint32_t koff = (uint32_t)(ks >> 2) * kKHalf + (uint32_t)(ks & 3) * 32;
        umma(t_s, sdesc(base + kOffQ + qoff, 16, 1024), sdesc(base + kOffK + koff, 16, 1024),
             kIdS, ks > 0);
      }
      issued[3] = issued[3] + 1;
      umma_commit(bar_s);
    }
    if (!wait_all(bar_s, par)) {
      dead = true;
      break;
    }
    tc_fence_after();
    if (tid == 0 && j + 1 < nblk) load_block(j + 1, false);  // K is free again

    // ---- softmax of this thread's row (log2 domain), masked past `vis`
    const int tok0 = j * kPfTok;
    const bool full = tok0 + kPfTok - 1 <= all_vis;  // no row masks anything here
    uint32_t r[32];
    float mx = -INFINITY;
#pragma unroll 1
    for (int cc = 0; cc < kPfTok / 32; ++cc) {
      tmem_ld32(t_s + lane_base + (uint32_t)cc * 32, r);
      if (full) {
#pragma unroll
        for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(r[e]) * c2);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (tok0 + cc * 32 + e <= vis) mx = fmaxf(mx, __uint_as_float(r[e]) * c2);
      }
    }
    // lazy rescale: keep the reference max while scores stay within 2^8 of it
    const bool grow = mx > m_ref + 8.f;
    float alpha = 1.f;
    if (grow) {
      alpha = ex2(m_ref - mx);  // 0 on the first block
      m_ref = mx;
      l_sum *= alpha;
    }
    if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        const uint32_t ta = t_o + lane_base + (uint32_t)cc * 32;
        tmem_ld32(ta, r);
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
        tmem_st32(ta, r);
      }
    }
    const float mu = m_ref == -INFINITY ? 0.f : m_ref;
#pragma unroll 1
    for (int cc = 0; cc < kPfTok / 32; ++cc) {
      tmem_ld32(t_s + lane_base + (uint32_t)cc * 32, r);
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        float p0 = ex2(__uint_as_float(r[e]) * c2 - mu);
        float p1 = ex2(__uint_as_float(r[e + 1]) * c2 - mu);
        if (!full) {
          const int t = tok0 + cc * 32 + e;
          if (t > vis) p0 = 0.f;
          if (t + 1 > vis) p1 = 0.f;
        }
        l_sum += p0 + p1;
        hi[e / 2] = pack2<BF16>(p0, p1);
        const float2 f = unpack2<BF16>(hi[e / 2]);
        lo[e / 2] = pack2<BF16>(p0 - f.x, p1 - f.y);
      }
      // row tid, tokens cc*32 .. +31: four 16-byte chunks of the swizzled row
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int chunk = cc * 4 + q;
        const uint32_t off = (uint32_t)tid * 128 + (uint32_t)((chunk ^ (tid & 7)) * 16);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(base + kOffPh + off),
                     "r"(hi[4 * q]), "r"(hi[4 * q + 1]), "r"(hi[4 * q + 2]), "r"(hi[4 * q + 3])
                     : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(base + kOffPl + off),
                     "r"(lo[4 * q]), "r"(lo[4 * q + 1]), "r"(lo[4 * q + 2]), "r"(lo[4 * q + 3])
                     : "memory");
      }
    }
    if (!wait_all(bar_v, par)) {  // block j's V (copied while S and the softmax ran)
      dead = true;
      break;
    }
    // rows of V past the context hold whatever the pool or an older block left:
    // zero them (the MMA multiplies them by P = 0)
    if (tok0 + kPfTok > ctx) {
      const int first = max(0, ctx - tok0);
      for (int i = tid; i < (kPfTok - first) * 16; i += kPfThreads) {
        const int rr = first + i / 16, ch = i % 16;  // row, 16-byte chunk of the row
        const uint32_t a = base + kOffV + (uint32_t)(ch >> 3) * kKHalf + (uint32_t)rr * 128 +
                           (uint32_t)(ch & 7) * 16;
        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
      }
    }
    // P and the zeroed V rows are read by the tensor cores (async proxy)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kPfTok / 16; ++ks) {  // O += P V over tokens, 16 at a time
        const uint64_t bv = sdesc(base + kOffV + (uint32_t)ks * 16 * 128, kKHalf, 1024);
        umma(t_o, sdesc(base + kOffPh + (uint32_t)ks * 32, 16, 1024), bv, kIdO, j > 0 || ks > 0);
        umma(t_o, sdesc(base + kOffPl + (uint32_t)ks * 32, 16, 1024), bv, kIdO, 1);
      }
      issued[4] = issued[4] + 1;
      umma_commit(bar_o);
    }
    if (!wait_all(bar_o, par)) {
      dead = true;
      break;
    }
    tc_fence_after();
    if (tid == 0 && j + 1 < nblk) load_block(j + 1, true);  // V is free again
  }

  // ---- out = O / l for the tile's real rows
  if (!dead) {
    const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
    const int64_t orow = ((int64_t)(q0 + row) * p.Hq + hq) * kPfD;
    uint32_t r[32];
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      tmem_ld32(t_o + lane_base + (uint32_t)cc * 32, r);
      if (row_real) {
        if (p.out_dtype == PKV_F32) {
          float4* o4 = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow + cc * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            o4[e] = make_float4(__uint_as_float(r[4 * e]) * inv, __uint_as_float(r[4 * e + 1]) * inv,
                                __uint_as_float(r[4 * e + 2]) * inv,
                                __uint_as_float(r[4 * e + 3]) * inv);
        } else {
          uint4* o4 = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + orow + cc * 32);
          const bool obf = p.out_dtype == PKV_BF16;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float a = __uint_as_float(r[8 * e + 2 * k]) * inv;
              const float c = __uint_as_float(r[8 * e + 2 * k + 1]) * inv;
              w[k] = obf ? pack2<true>(a, c) : pack2<false>(a, c);
            }
            o4[e] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  } else {
    // a wait gave up: let this CTA's copies and MMAs land (bounded, each
    // barrier's last expected phase) before the tensor memory is released
    if (tid == 0) report_error(p.err_word, PKV_ERR_TIMEOUT);
    for (int i = 0; i < 5; ++i)
      if (issued[i] > 0)
        mbar_wait_bounded(bar_q + 8 * i, (uint32_t)((issued[i] - 1) & 1), kPfWaitNs);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t prefill_smem_bytes() { return 1024 + kOffBar + 64; }

cudaError_t launch_prefill(const PrefillLaunch& l) {
  const size_t smem = prefill_smem_bytes();
  static bool configured[2] = {false, false};
  auto kern = l.bf16 ? prefill_kernel<true> : prefill_kernel<false>;
  if (!configured[l.bf16 ? 1 : 0]) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured[l.bf16 ? 1 : 0] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(l.p.B * l.p.tiles_per_seq), (unsigned)l.p.Hkv, 1);
  cfg.blockDim = dim3(kPfThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = l.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, l.p, l.tmap_q, l.tmap_k, l.tmap_v);
}

}  // namespace pkv
