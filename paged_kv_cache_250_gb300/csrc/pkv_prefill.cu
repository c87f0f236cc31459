// Paged prefill attention on the 5th-generation tensor cores (tcgen05).
//
// A chunk of q_len new tokens per sequence, already appended to the cache,
// attends causally over the sequence's whole context through its block table
// ("KV Cache & Flash Attention." (kvcache-7e2.pages.dev): the prefill phase
// processes the prompt in one parallel pass; continuous-batching section:
// chunked prefill reads each sequence's pages through its table).  Token j of
// the chunk sits at position ctx - q_len + j and sees positions 0 .. itself.
//
// One CTA owns 256 query rows in two tiles of 128: 256 / g new tokens of one
// sequence times the g query heads that share one KV head, so every page it
// loads serves the whole group and both tiles.  In a tile, row r is token
// r / g, head r % g.  The CTA's warps have fixed roles:
//   warps 0-3, 4-7  softmax of tile 0, tile 1: thread t of the group owns row
//                   t, TMEM lane t, so the online softmax (running max m, sum
//                   l, rescale of O) needs no shuffles;
//   warp 8          issues the MMAs (one thread);
//   warp 9          the tensor copies: lane 0 arms the barriers, lanes 0-7
//                   read a block's eight table entries one block ahead and
//                   issue one page's copies each.
// Per block of 128 cached tokens (8 pages), for each tile:
//   S = Q K^T    tcgen05.mma, M 128 x N 128 x K 128 (d), both operands K-major
//                128-byte-swizzled tiles as the tensor copies write them, the
//                scores landing in tensor memory;
//   softmax      the row read from tensor memory 32 columns at a time (the
//                next load in flight under the current quarter's work), its
//                max, then exp2 and P as a bf16 (or fp16) hi + lo pair written
//                back over the row's scores (tcgen05.st); blocks that every
//                row sees whole skip the masking code;
//   O += P V     tcgen05.mma with A read from tensor memory, twice (hi and lo)
//                per 64 tokens, M 128 x N 128 (d) x K 16 per instruction; V is
//                used where the copies put it, as an MN-major operand.
// The MMA thread alternates between the tiles (P.V of one tile, then the next
// block's scores of the same tile, which overwrite its P: MMAs run in issue
// order), so the tensor cores work on one tile while the other tile's softmax
// runs.  K and V blocks are double-buffered.  The roles hand over through
// mbarriers only; tensor memory holds S0/P0, S1/P1, O0 and O1, 128 columns
// each.
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kPfRows = 128;          // query rows per tile; two tiles per CTA
constexpr int kPfTok = 128;           // cached tokens per block (8 pages)
constexpr int kPfPages = kPfTok / kPageSize;
constexpr int kPfThreads = 320;       // 8 softmax warps, the MMA warp, the copy warp
constexpr uint32_t kQHalf = 16384;    // 128 rows x 128 bytes: 64 d columns of a Q tile
constexpr uint32_t kKHalf = 16384;    // 128 rows x 128 bytes: the same of a K or V block
// mbarriers (8 bytes each) from the barrier area
constexpr int kBarQ = 0, kBarKFull = 1, kBarVFull = 3, kBarKFree = 5, kBarVFree = 7,
              kBarSFull = 9, kBarPFull = 11, kBarODone = 13, kNumBars = 15;
constexpr uint32_t kTmemCols = 512;  // S0/P0 0..127, S1/P1 128..255, O0 from 256, O1 after it
// Shared memory plan for head dim D (NH = D / 64 halves of 128-byte rows),
// offsets from a 1024-byte aligned base: Q tile t at t * NH * kQHalf, K and V
// buffer b at b * NH * kKHalf from their areas, then barriers and counts.
template <int D>
struct PfPlan {
  static constexpr int NH = D / 64;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = 2 * NH * kQHalf;
  static constexpr uint32_t kOffV = kOffK + 2 * NH * kKHalf;
  static constexpr uint32_t kOffBar = kOffV + 2 * NH * kKHalf;
  static constexpr uint32_t kOffMisc = kOffBar + 8 * kNumBars;  // TMEM base, abort, counts
  static constexpr size_t kSmem = 1024 + kOffMisc + 8 + 4 * kNumBars;
  static_assert(D == 64 || D == 128, "head dims built");
};
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
// D[tmem] (+)= A[tmem] . B[smem]^T, kind::f16: A is M lanes x K 16-bit values,
// two per 32-bit column
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
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

// The same 32-column load without its wait: r holds the columns only after
// tmem_ld_wait(r).
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}
// Wait for this thread's TMEM loads.  The registers of the last load pass
// through the wait, so no use of them can be scheduled above it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :: "memory");
}
// 16 consecutive 32-bit TMEM columns of this thread's lane, no wait
__device__ __forceinline__ void tmem_st16_issue(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Packed fp32 pairs (PTX f32x2 arithmetic, sm_100 and later): one
// instruction for two lanes' worth of add or fused multiply-add.
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2_split(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// max of three (PTX three-input max.f32, sm_100 and later)
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
template <bool B>
struct Masked {
  static constexpr bool value = B;
};

template <bool BF16, int D>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmq,
                   const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv) {
  const int b = blockIdx.x / p.tiles_per_seq;
  const int ctile = blockIdx.x - b * p.tiles_per_seq;
  const int h = blockIdx.y;                 // KV head
  const int G = p.Hq / p.Hkv;               // query heads per KV head
  const int tpt = kPfRows / G;              // tokens per tile
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  using PL = PfPlan<D>;
  constexpr int NH = PL::NH, kPfD = D;
  constexpr uint32_t kOffQ = PL::kOffQ, kOffK = PL::kOffK, kOffV = PL::kOffV,
                     kOffBar = PL::kOffBar, kOffMisc = PL::kOffMisc;

  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int q0 = p.q_start[b], qn = p.q_start[b + 1] - q0;  // this sequence's rows
  const int ctx = p.context_lens[b];
  if (qn < 0 || ctx < qn || ctx > p.MBS * kPageSize || q0 < 0 || q0 + qn > p.total_q ||
      qn > p.tiles_per_seq * 2 * tpt) {
    if (tid == 0 && ctile == 0 && h == 0) report_error(p.err_word, PKV_ERR_BOUNDS);
    return;
  }
  const int tok_base = ctile * 2 * tpt;  // first new token of the CTA
  if (tok_base >= qn) return;            // no rows of this sequence here

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  auto bar = [&](int i) -> uint32_t { return base + kOffBar + 8u * (uint32_t)i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base_ptr + kOffMisc);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(base_ptr + kOffMisc + 4);
  // completions expected on each barrier (counted by the thread that arms it)
  volatile int32_t* armed = reinterpret_cast<volatile int32_t*>(base_ptr + kOffMisc + 8);

  if (warp == 0) {
    tmem_alloc(base + kOffMisc, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kNumBars; ++i) {
      armed[i] = 0;
      // P full: one arrival per softmax warp of the tile
      mbar_init(bar(i), (i == kBarPFull || i == kBarPFull + 1) ? kPfRows / 32 : 1);
    }
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int last_tok = min(qn, tok_base + 2 * tpt) - 1;
  const int nblk = (ctx - qn + last_tok) / kPfTok + 1;  // causal: blocks any row sees
  const int np = (ctx + kPageSize - 1) / kPageSize;

  // A bounded wait; a wait that gives up raises the CTA's abort flag, and
  // every role stops waiting once the flag is up, so no role can stall the
  // others for more than one bound.
  auto wait = [&](int i, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (mbar_wait_bounded(bar(i), parity, kPfWaitNs)) return true;
    *abort_flag = 1;
    return false;
  };

  if (warp == 9) {
    // ---------------------------------------------------------- copies
    // Lane 0 arms the barriers; lane i < 8 reads the block-table entry of
    // page i of a block (one block ahead, so the lookups' latency hides under
    // the previous block's waits) and issues that page's copies, for K and
    // for V from the same entry.
    if (lane == 0) {
      prefetch_tmap(&tmq);
      prefetch_tmap(&tmk);
      prefetch_tmap(&tmv);
      armed[kBarQ] = 1;
      mbar_arrive_expect_tx(bar(kBarQ), 2 * NH * kQHalf);
      for (int t = 0; t < 2; ++t)
        for (int c = 0; c < NH; ++c)
          tma_load_3d(base + kOffQ + (uint32_t)(t * NH + c) * kQHalf, &tmq, bar(kBarQ), c * 64,
                      h * G, q0 + tok_base + t * tpt);
    }
    const int64_t trow = (int64_t)b * p.MBS;
    auto table_entry = [&](int j) -> int {
      const int pg = j * kPfPages + lane;
      return lane < kPfPages && pg < np ? p.block_tables[trow + pg] : 0;
    };
    int cur = table_entry(0);
    for (int j = 0; j < nblk; ++j) {
      const int bb = j & 1;
      const int npg = min(kPfPages, np - j * kPfPages);
      const int nxt = j + 1 < nblk ? table_entry(j + 1) : 0;
      int blk = cur;
      if (lane < npg && (blk < 0 || blk >= p.NB)) {  // the copy reads the fill value (zeros) past the pool
        report_error(p.err_word, PKV_ERR_BOUNDS);
        blk = p.NB;
      }
      bool ok = true;
      for (int v = 0; v < 2; ++v) {  // K, then V of block j
        const int full = (v ? kBarVFull : kBarKFull) + bb;
        if (j >= 2)
          ok = __all_sync(0xffffffffu, wait((v ? kBarVFree : kBarKFree) + bb,
                                            (uint32_t)(((j - 2) >> 1) & 1)));
        if (!ok) break;
        if (lane == 0) {
          armed[full] = armed[full] + 1;
          mbar_arrive_expect_tx(bar(full), (uint32_t)npg * NH * kPageSize * 128);
        }
        __syncwarp();
        if (lane < npg) {
          const uint32_t dst = base + (v ? kOffV : kOffK) + (uint32_t)bb * NH * kKHalf +
                               (uint32_t)lane * kPageSize * 128;
          const int r = (blk * p.Hkv + h) * kPageSize;
          for (int c = 0; c < NH; ++c)
            tma_load_2d_plain(dst + (uint32_t)c * kKHalf,
                              v ? (const void*)&tmv : (const void*)&tmk, bar(full), c * 64, r);
        }
      }
      if (!ok || __any_sync(0xffffffffu, *abort_flag != 0)) break;
      cur = nxt;
    }
  } else if (warp == 8) {
    // ---------------------------------------------------------- MMAs
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(BF16, false, kPfRows, kPfTok);
      constexpr uint32_t kIdO = idesc_f16(BF16, true, kPfRows, kPfD);
      auto commit = [&](int i) {
        armed[i] = armed[i] + 1;
        umma_commit(bar(i));
      };
      // The descriptors' address field is (address >> 4) in 14 bits and shared
      // memory ends below 256 KB, so a descriptor at address + offset is the
      // base descriptor plus offset >> 4: build the bases once.
      const uint64_t dq = sdesc(base + kOffQ, 16, 1024);
      const uint64_t dk = sdesc(base + kOffK, 16, 1024);
      const uint64_t dv = sdesc(base + kOffV, kKHalf, 1024);
      auto qk = [&](int t, int j) {  // S_t = Q_t K(j)^T over d, 16 at a time
        const uint64_t a0 = dq + ((uint64_t)t * NH * kQHalf >> 4);
        const uint64_t b0 = dk + ((uint64_t)(j & 1) * NH * kKHalf >> 4);
#pragma unroll
        for (int ks = 0; ks < kPfD / 16; ++ks) {
          const uint32_t qoff = (uint32_t)(ks >> 2) * kQHalf + (uint32_t)(ks & 3) * 32;
          const uint32_t koff = (uint32_t)(ks >> 2) * kKHalf + (uint32_t)(ks & 3) * 32;
          umma(tmem + (uint32_t)t * kPfTok, a0 + (qoff >> 4), b0 + (koff >> 4), kIdS, ks > 0);
        }
        commit(kBarSFull + t);
      };
      // O_t += P_t V(j) over tokens, 16 at a time; P_t sits over S_t's
      // columns: per 64 tokens, 32 columns of hi pairs, then 32 of lo pairs
      auto pv = [&](int t, int j) {
        const uint64_t b0 = dv + ((uint64_t)(j & 1) * NH * kKHalf >> 4);
        const uint32_t pt = tmem + (uint32_t)t * kPfTok;
        const uint32_t dt = tmem + 256 + (uint32_t)t * kPfD;
#pragma unroll
        for (int ks = 0; ks < kPfTok / 16; ++ks) {
          const uint64_t bv = b0 + ((uint32_t)ks * 16 * 128 >> 4);
          const uint32_t pa = pt + (uint32_t)(ks >> 2) * 64 + (uint32_t)(ks & 3) * 8;
          umma_ts(dt, pa, bv, kIdO, j > 0 || ks > 0);
          umma_ts(dt, pa + 32, bv, kIdO, 1);
        }
        commit(kBarODone + t);
      };
      bool ok = wait(kBarQ, 0) && wait(kBarKFull, 0);
      if (ok) {
        tc_fence_after();
        qk(0, 0);
        qk(1, 0);
        commit(kBarKFree);
      }
      // Per tile: this block's P.V, then the next block's scores, which
      // overwrite P (the MMAs of one thread run in issue order).
      for (int j = 0; ok && j < nblk; ++j) {
        const int bb = j & 1, nb = (j + 1) & 1;
        const uint32_t par = (uint32_t)(j & 1);
        const bool more = j + 1 < nblk;
        if (!wait(kBarPFull, par)) break;  // P0 written over S0
        if (!wait(kBarVFull + bb, (uint32_t)((j >> 1) & 1))) break;
        tc_fence_after();
        pv(0, j);
        if (more) {
          if (!wait(kBarKFull + nb, (uint32_t)(((j + 1) >> 1) & 1))) break;
          qk(0, j + 1);
        }
        if (!wait(kBarPFull + 1, par)) break;
        tc_fence_after();
        pv(1, j);
        commit(kBarVFree + bb);
        if (more) {
          qk(1, j + 1);
          commit(kBarKFree + nb);
        }
      }
    }
  } else {
    // ---------------------------------------------------------- softmax
    const int t = warp >> 2;             // tile
    const int tt = tid - t * kPfRows;    // row in the tile
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + (uint32_t)t * kPfTok + lane_base;  // S_t, then P_t
    const uint32_t t_o = tmem + 256 + (uint32_t)t * kPfD + lane_base;
    const int row = tok_base + t * tpt + tt / G;  // new token of this row
    const int hq = h * G + tt % G;
    const bool row_real = row < qn;
    const int vis = min(ctx - qn + row, ctx - 1);        // last visible position
    const int all_vis = ctx - qn + tok_base + t * tpt;   // every row of the tile sees <= this
    const float c2 = p.scale_log2;
    float m_ref = -INFINITY, l_sum = 0.f;
    bool ok = true;
    uint32_t r[32];
    for (int j = 0; j < nblk; ++j) {
      const uint32_t par = (uint32_t)(j & 1);
      ok = __all_sync(0xffffffffu, wait(kBarSFull + t, par));
      if (!ok) break;
      tc_fence_after();
      const int tok0 = j * kPfTok;
      const bool full = tok0 + kPfTok - 1 <= all_vis;  // no row masks anything here
      // The row's 128 scores are read in quarters of 32 columns, the next
      // quarter's load in flight while the current one is worked on.
      uint32_t sa[32], sb[32];
      // row max of the raw scores (c2 > 0 commutes with the max): quarters
      // 3, 2, 1, 0, so quarter 0 is still in sb when the P pass starts
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      auto qmax = [&](auto mc, const uint32_t (&sq)[32], int qq) {
        if constexpr (!decltype(mc)::value) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            m4[i & 3] = max3(m4[i & 3], __uint_as_float(sq[2 * i]), __uint_as_float(sq[2 * i + 1]));
        } else {
          const int t0 = tok0 + 32 * qq;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float a = t0 + 2 * i <= vis ? __uint_as_float(sq[2 * i]) : -INFINITY;
            const float c = t0 + 2 * i + 1 <= vis ? __uint_as_float(sq[2 * i + 1]) : -INFINITY;
            m4[i & 3] = max3(m4[i & 3], a, c);
          }
        }
      };
      auto max_pass = [&](auto mc) {
        tmem_ld32_issue(t_s + 96, sa);
        tmem_ld_wait(sa);
        tmem_ld32_issue(t_s + 64, sb);
        qmax(mc, sa, 3);
        tmem_ld_wait(sb);
        tmem_ld32_issue(t_s + 32, sa);
        qmax(mc, sb, 2);
        tmem_ld_wait(sa);
        tmem_ld32_issue(t_s + 0, sb);
        qmax(mc, sa, 1);
        tmem_ld_wait(sb);
        qmax(mc, sb, 0);
      };
      if (full) max_pass(Masked<false>{});
      else max_pass(Masked<true>{});
      const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * c2;
      // lazy rescale: keep the reference max while scores stay within 2^8 of it
      const bool grow = mx > m_ref + 8.f;
      float alpha = 1.f;
      if (grow) {
        alpha = ex2(m_ref - mx);  // 0 on the first block
        m_ref = mx;
        l_sum *= alpha;
      }
      if (j > 0) {  // O_t and P_t are free once the previous block's P.V is done
        ok = __all_sync(0xffffffffu, wait(kBarODone + t, (uint32_t)((j - 1) & 1)));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, grow)) {
#pragma unroll 1
          for (int cc = 0; cc < kPfD / 32; ++cc) {
            const uint32_t ta = t_o + (uint32_t)cc * 32;
            tmem_ld32(ta, r);
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tmem_st32(ta, r);
          }
        }
      }
      const float mu = m_ref == -INFINITY ? 0.f : m_ref;
      // P over S.  Per 64 tokens the hi pairs take 32 columns, then the lo
      // pairs 32: quarter q's pairs go to columns 64 (q / 2) + 16 (q % 2) + i
      // (hi) and 32 more (lo).  An even quarter's lo columns hold the next
      // quarter's scores, so that quarter is in registers before they are
      // written.
      const uint64_t c2x2 = f2(c2, c2), nmu2 = f2(-mu, -mu);
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};  // four independent f32x2 chains
      uint32_t hi[16], lo[16];
      auto qp = [&](auto mc, const uint32_t (&sq)[32], int qq) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 y = f2_split(fma2(f2(__uint_as_float(sq[2 * i]),
                                            __uint_as_float(sq[2 * i + 1])), c2x2, nmu2));
          float p0 = ex2(y.x), p1 = ex2(y.y);
          if constexpr (decltype(mc)::value) {
            const int tk = tok0 + 32 * qq + 2 * i;
            if (tk > vis) p0 = 0.f;
            if (tk + 1 > vis) p1 = 0.f;
          }
          const uint64_t pp = f2(p0, p1);
          acc[i & 3] = add2(acc[i & 3], pp);
          hi[i] = pack2<BF16>(p0, p1);
          const float2 hf = unpack2<BF16>(hi[i]);
          const float2 l = f2_split(sub2(pp, f2(hf.x, hf.y)));
          lo[i] = pack2<BF16>(l.x, l.y);
        }
      };
      auto qst = [&](int qq) {
        const uint32_t c = (uint32_t)(64 * (qq >> 1) + 16 * (qq & 1));
        tmem_st16_issue(t_s + c, hi);
        tmem_st16_issue(t_s + c + 32, lo);
      };
      auto p_pass = [&](auto mc) {
        tmem_ld32_issue(t_s + 32, sa);
        qp(mc, sb, 0);
        tmem_ld_wait(sa);
        qst(0);
        tmem_ld32_issue(t_s + 64, sb);
        qp(mc, sa, 1);
        tmem_ld_wait(sb);
        qst(1);
        tmem_ld32_issue(t_s + 96, sa);
        qp(mc, sb, 2);
        tmem_ld_wait(sa);
        qst(2);
        qp(mc, sa, 3);
        qst(3);
      };
      if (full) p_pass(Masked<false>{});
      else p_pass(Masked<true>{});
      tmem_st_wait();
      {
        const float2 a0 = f2_split(add2(acc[0], acc[1])), a1 = f2_split(add2(acc[2], acc[3]));
        l_sum += (a0.x + a0.y) + (a1.x + a1.y);
      }
      // rows of V past the context hold whatever the pool or an older block
      // left: tile 0 zeroes them before it hands over (the MMA multiplies them
      // by P = 0)
      if (t == 0 && tok0 + kPfTok > ctx) {
        ok = __all_sync(0xffffffffu, wait(kBarVFull + (j & 1), (uint32_t)((j >> 1) & 1)));
        if (!ok) break;
        const int first = max(0, ctx - tok0);
        const uint32_t vb = base + kOffV + (uint32_t)(j & 1) * NH * kKHalf;
        for (int i = tt; i < (kPfTok - first) * 8 * NH; i += kPfRows) {
          const int rr = first + i / (8 * NH), ch = i % (8 * NH);  // row, 16-byte chunk
          const uint32_t a = vb + (uint32_t)(ch >> 3) * kKHalf + (uint32_t)rr * 128 +
                             (uint32_t)(ch & 7) * 16;
          asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
        }
      }
      // zeroed V rows are read by the tensor cores (async proxy); P is in
      // tensor memory
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull + t));
    }
    // ---- out = O / l for the tile's real rows
    if (ok) ok = __all_sync(0xffffffffu, wait(kBarODone + t, (uint32_t)((nblk - 1) & 1)));
    if (ok) {
      tc_fence_after();
      const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
      const int64_t orow = ((int64_t)(q0 + row) * p.Hq + hq) * kPfD;
#pragma unroll 1
      for (int cc = 0; cc < kPfD / 32; ++cc) {
        tmem_ld32(t_o + (uint32_t)cc * 32, r);
        if (row_real) {
          if (p.out_dtype == PKV_F32) {
            float4* o4 = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow + cc * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              o4[e] = make_float4(__uint_as_float(r[4 * e]) * inv,
                                  __uint_as_float(r[4 * e + 1]) * inv,
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
    }
  }

  // ---- every role is done.  After an abort, let this CTA's copies and MMAs
  // land (bounded, each barrier's last armed phase) before the tensor memory
  // is released.
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    if (tid == 0) report_error(p.err_word, PKV_ERR_TIMEOUT);
    if (tid < kNumBars && tid != kBarPFull && tid != kBarPFull + 1 && armed[tid] > 0)
      mbar_wait_bounded(bar(tid), (uint32_t)((armed[tid] - 1) & 1), kPfWaitNs);
    __syncthreads();
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t prefill_smem_bytes(int d) { return d == 64 ? PfPlan<64>::kSmem : PfPlan<128>::kSmem; }

cudaError_t launch_prefill(const PrefillLaunch& l) {
  const int d = l.d;
  if (d != 64 && d != 128) return cudaErrorNotSupported;
  const size_t smem = prefill_smem_bytes(d);
  static bool configured[2][2] = {{false, false}, {false, false}};
  auto kern = l.bf16 ? (d == 64 ? prefill_kernel<true, 64> : prefill_kernel<true, 128>)
                     : (d == 64 ? prefill_kernel<false, 64> : prefill_kernel<false, 128>);
  bool& done = configured[l.bf16 ? 1 : 0][d == 64 ? 0 : 1];
  if (!done) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    done = true;
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
