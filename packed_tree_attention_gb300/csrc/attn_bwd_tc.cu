// Packed DAG attention backward on the tcgen05 tensor cores (sm_103a).
//
// Octopus project page, "Architecture & Co-Design" item 03: the packed pass routes every
// reader's gradient into the producer's KV; shared prefix tokens are owned once, so their
// dK/dV are sums over every reader row.  Two kernels, no atomics:
//
// k_dkdv_tc  one CTA per (page pair, kv head): two consecutive own pages of a segment give
//            128 keys (a lone page fills keys 0-63).  It walks the pair's work items (a
//            query tile against one or both pages, each half with its own entry mask) and,
//            for each item and each of the G query heads of the group, computes in the
//            transposed orientation, keys on the TMEM lanes:
//              S^T = K Q^T,  dP^T = V dO^T                    (M128 keys x N128 rows, K = d)
//              P^T = exp(S^T - LSE),  dS^T = P^T (dP^T - D)   (softmax warps, written back to
//                                                              TMEM as bf16 over S^T / dP^T)
//              dV += P^T dO,  dK += dS^T Q                    (M128 keys x N128 d, K = rows,
//                                                              A operand read from TMEM)
//            Every MMA is 128 x 128 and each Q/dO tile load serves 128 keys.  The pair's
//            dK/dV are written once at the end (dK scaled).
// k_dq_tc    one CTA per (q-tile, query head), tiles heaviest first: the tile's entries two
//            at a time (128 keys), per step
//              S = Q K^T,  dP = dO V^T                        (M128 rows x N128 keys, K = d)
//              P = exp(S - LSE),  dS = P (dP - D)             (softmax warps, dS written back
//                                                              to TMEM as bf16 over dP)
//              dQ += dS K                                     (M128 rows x N128 d, K = keys,
//                                                              A operand read from TMEM)
//
// Shared-memory tiles are 128-byte swizzled.  A 128-key K or V operand is two TMA boxes of
// 64 rows per 64-column d-half, so the two pages need not be adjacent in the pool.  The
// [rows x d] Q / dO tiles and the K tiles serve both as K-major operands and as MN-major B
// operands; P and dS never touch shared memory.  Waits are bounded as in the forward.

#include <cuda_bf16.h>

#include <atomic>
#include <type_traits>

#include "internal.h"
#include "tc_common.cuh"

namespace octo {
namespace {

using namespace tc;

constexpr uint32_t kIdDQ = idesc_bf16(128, 128, 0, 1);   // rows x d, A from TMEM, B MN-major

struct BwdParams {
  const int32_t* tile_off;
  const int32_t* tile_rows;
  const int32_t* tile_row0;
  const int32_t* tile_order;
  const octo_entry* entries;
  const int32_t* csc_perm;
  const int32_t* page_off;
  const int32_t* pair_pages;
  const int32_t* pair_item_off;
  const int32_t* pair_n_items;
  const int32_t* pair_order;
  const PairItem* pair_items;
  const float* lse2t;   // [n_tiles][Hq][128] LSE * log2(e) per tile row (0 past the tile)
  const float* Dt;      // [n_tiles][Hq][128] D = rowsum(dO * O) per tile row
  const uint4* aug;     // [n_tiles][Hq][128 rows] bf16 (-LSE/scale hi, lo, -D hi, lo, 0 x 4)
  float* dq;
  float* dk;
  float* dv;
  int64_t n_rows;
  int32_t Hq, Hkv, G;
  float scale, scale_log2;
  int32_t* status;
};

struct Ctl {
  volatile int32_t abort;
  uint32_t tmem_base;
};

__device__ __forceinline__ bool wait_ab(uint64_t* bar, uint32_t parity, Ctl* C, int32_t* status) {
  if (mbar_test(bar, parity)) return true;
  for (uint32_t i = 0; i < kSpinLimit; i++) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 1023) == 1023 && C->abort) return false;
  }
  C->abort = 1;
  atomicExch(status, OCTO_ETIMEOUT);
  return false;
}
// Barrier traffic of the softmax warps is kept to one lane per warp: while MMAs stream
// their operands from shared memory, every other shared-memory access (mbarrier polls and
// arrivals included) queues behind them.  Lane 0 waits and the warp sync passes the
// acquired state on; for an arrival every lane's TMEM accesses are fenced and ordered before
// the warp sync, and lane 0's arrive releases them.
__device__ __forceinline__ bool warp_wait_ab(uint64_t* bar, uint32_t parity, Ctl* C, int32_t* status) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = wait_ab(bar, parity, C, status);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok;
}
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Row statistics in a tile-padded layout, one CTA per (tile, head): the log2-domain LSE and
// D = rowsum(dO * O) of each tile row at [tile][head][0, 128), zero past the tile, read by
// the dQ softmax; and for the dK/dV MMAs a [128 rows x 8] bf16 block per (tile, head)
// holding -LSE/scale and -D, each as a bf16 pair hi + lo (about 16 significant bits):
// multiplied by a block of ones in one extra K = 16 MMA step, it subtracts them from S^T
// and dP^T inside the accumulator.
__global__ void __launch_bounds__(128) k_pre_tiles(const __nv_bfloat16* __restrict__ o,
                                                   const __nv_bfloat16* __restrict__ dout,
                                                   const float* __restrict__ lse, const int32_t* __restrict__ tile_row0,
                                                   const int32_t* __restrict__ tile_rows, int64_t n_rows, int32_t Hq,
                                                   float inv_scale, float* __restrict__ lse2t, float* __restrict__ Dt,
                                                   uint4* __restrict__ aug) {
  const int32_t tile = blockIdx.x / Hq, h = blockIdx.x % Hq;
  const int32_t row0 = tile_row0[tile], rows = tile_rows[tile];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* lo = lse2t + (size_t)blockIdx.x * 128;
  float* dd = Dt + (size_t)blockIdx.x * 128;
  uint4* ag = aug + (size_t)blockIdx.x * 128;
  for (int r = warp; r < 128; r += 4) {
    float part = 0.f;
    if (r < rows) {
      const size_t base = ((size_t)(row0 + r) * Hq + h) * 128 + lane * 4;
      const uint2 a = *reinterpret_cast<const uint2*>(o + base);
      const uint2 b = *reinterpret_cast<const uint2*>(dout + base);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int i = 0; i < 2; i++) {
        const float2 x = __bfloat1622float2(a2[i]), y = __bfloat1622float2(b2[i]);
        part = fmaf(x.x, y.x, part);
        part = fmaf(x.y, y.y, part);
      }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if (lane == 0) {
      const float L = r < rows ? lse[(int64_t)h * n_rows + row0 + r] : 0.f;
      dd[r] = part;
      lo[r] = L * 1.4426950408889634f;
      const float av = -L * inv_scale, bv = -part;
      const __nv_bfloat16 ah = __float2bfloat16_rn(av), bh = __float2bfloat16_rn(bv);
      const __nv_bfloat16 al = __float2bfloat16_rn(av - __bfloat162float(ah));
      const __nv_bfloat16 bl = __float2bfloat16_rn(bv - __bfloat162float(bh));
      uint4 v;
      v.x = (uint32_t)__bfloat16_as_ushort(ah) | ((uint32_t)__bfloat16_as_ushort(al) << 16);
      v.y = (uint32_t)__bfloat16_as_ushort(bh) | ((uint32_t)__bfloat16_as_ushort(bl) << 16);
      v.z = 0;
      v.w = 0;
      ag[r] = v;
    }
  }
}

// =====================================================================================
// dK / dV
// =====================================================================================
constexpr int kDkThreads = 384;   // warp 0 TMA, warps 1-2 MMA issuers (1 also TMEM), warps 4-11 softmax
// smem: ones blocks 2 x 4KB | 2 stages x row-statistics block 4KB | K pair 32KB | V pair 32KB |
// 2 stages x (Q 32KB + dO 32KB).  The softmax warps read no memory per element: LSE and D
// enter through one more K = 16 MMA step (ones x statistics block) of S^T and dP^T.
// The 4KB blocks are K-major without swizzle: 128 rows x 8 bf16 (16 B per row; K = 0..7),
// then 2KB of zeros for K = 8..15.
constexpr uint32_t kDkOffOnesS = 0;      // rows: 1, 1, 0 ...  (picks -LSE/scale hi + lo)
constexpr uint32_t kDkOffOnesD = 4096;   // rows: 0, 0, 1, 1, 0 ...  (picks -D hi + lo)
constexpr uint32_t kDkOffAug = 8192;     // per stage: the (tile, head) statistics block
constexpr uint32_t kDkOffK = 16384;
constexpr uint32_t kDkOffV = kDkOffK + 32768;
constexpr uint32_t kDkOffQD = kDkOffV + 32768;
constexpr uint32_t kDkStageQD = 65536;
constexpr uint32_t kDkOffBar = kDkOffQD + 2 * kDkStageQD;
constexpr uint32_t kDkSmem = kDkOffBar + 256 + 1024;
constexpr uint32_t kIdKR = idesc_bf16(128, 128, 0, 0);   // keys x rows, both K-major
constexpr uint32_t kIdKD = idesc_bf16(128, 128, 0, 1);   // keys x d, A from TMEM, B MN-major

struct DkBars {
  uint64_t kv_full;
  uint64_t qd_full[2];
  uint64_t qd_free[2];
  uint64_t s_full, dp_full;   // S^T / dP^T of the current step in TMEM
  uint64_t p_full, ds_full;   // P^T / dS^T written back to TMEM
  uint64_t acc_done;          // single use, one arrival per issuer: every accumulation MMA has completed
  uint64_t drain;
  Ctl ctl;
};

// One CTA per (page pair, kv head).  TMEM: S^T [0,128), dP^T [128,256), dV [256,384),
// dK [384,512); lane = key.  Softmax warpgroup c reads columns [64 c, 64 c + 64) of S^T and
// dP^T and writes its 64 rows of P^T / dS^T as bf16 over the first 32 of them, so the A
// operand of the accumulation MMAs sits at columns 0-31 and 64-95 of the region and no
// warpgroup overwrites columns the other still reads.
__global__ void __launch_bounds__(kDkThreads, 1)
    k_dkdv_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
              const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DkBars* B = reinterpret_cast<DkBars*>(smem + kDkOffBar);
  Ctl* C = &B->ctl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t g = blockIdx.x % p.Hkv;
  const int32_t pr = p.pair_order[blockIdx.x / p.Hkv];
  const int32_t pa = p.pair_pages[2 * pr], pb = p.pair_pages[2 * pr + 1];
  const PairItem* items = p.pair_items + p.pair_item_off[pr];
  const int32_t n_items = p.pair_n_items[pr];
  const int32_t G = p.G;
  const int32_t n = n_items * G;   // steps: (item, query head of the group)

  if (threadIdx.x == 0) {
    mbar_init(&B->kv_full, 1);
    for (int s = 0; s < 2; s++) {
      mbar_init(&B->qd_full[s], 1);
      mbar_init(&B->qd_free[s], 2);   // both issuers' MMAs of the item have completed
    }
    mbar_init(&B->s_full, 1);
    mbar_init(&B->dp_full, 1);
    mbar_init(&B->p_full, 8);   // one arrival per softmax warp
    mbar_init(&B->ds_full, 8);
    mbar_init(&B->acc_done, 2);
    mbar_init(&B->drain, 2);
    C->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&C->tmem_base, 512);
    tmem_relinquish();
  }
  {
    // ones blocks (rows 0-127, then the zero K = 8..15 half) and the zero halves of the
    // statistics stages; 16 KB, 1024 x 16 B
    const uint32_t one2 = 0x3F803F80u;   // two bf16 ones
    for (int i = threadIdx.x; i < 1024; i += kDkThreads) {
      const int blk = i >> 8, row = i & 255;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (row < 128 && blk == 0) v.x = one2;
      if (row < 128 && blk == 1) v.y = one2;
      if (row < 128 && blk >= 2) continue;   // statistics rows: written by the TMA
      reinterpret_cast<uint4*>(smem + blk * 4096)[row] = v;
    }
    fence_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = C->tmem_base;
  const uint32_t sK = smem_u32(smem + kDkOffK);
  const uint32_t sV = smem_u32(smem + kDkOffV);
  const uint32_t sQD = smem_u32(smem + kDkOffQD);

  if (warp == 0) {
    if (lane == 0 && n > 0) {
      prefetch_map(&tmQ);
      prefetch_map(&tmDO);
      mbar_expect_tx(&B->kv_full, pb >= 0 ? 65536 : 32768);
      for (int hp = 0; hp < 2; hp++) {
        const int32_t pg = hp ? pb : pa;
        if (pg < 0) continue;
        const int32_t krow = (pg * p.Hkv + g) * 64;
        // keys 64 hp .. 64 hp + 63 of each 128-row d-half
        tma_load_2d(smem + kDkOffK + hp * 8192, &tmK, &B->kv_full, 0, krow);
        tma_load_2d(smem + kDkOffK + 16384 + hp * 8192, &tmK, &B->kv_full, 64, krow);
        tma_load_2d(smem + kDkOffV + hp * 8192, &tmV, &B->kv_full, 0, krow);
        tma_load_2d(smem + kDkOffV + 16384 + hp * 8192, &tmV, &B->kv_full, 64, krow);
      }
      int32_t issued = 0;
      int32_t row0_next = items[0].row0, tile_next = items[0].tile;
      for (int32_t w = 0; w < n; w++) {
        const int st = w & 1;
        const int32_t h = g * G + (w % G);
        const int32_t row0 = row0_next, tile_n = tile_next;
        if (w + 1 < n && (w + 1) % G == 0) {
          row0_next = items[(w + 1) / G].row0;
          tile_next = items[(w + 1) / G].tile;
        }
        if (w >= 2 && !wait_ab(&B->qd_free[st], ((w >> 1) - 1) & 1, C, p.status)) break;
        uint8_t* dst = smem + kDkOffQD + st * kDkStageQD;
        mbar_expect_tx(&B->qd_full[st], 65536 + 2048);
        bulk_load(smem + kDkOffAug + st * 4096, p.aug + ((size_t)tile_n * p.Hq + h) * 128, 2048, &B->qd_full[st]);
        tma_load_3d(dst, &tmQ, &B->qd_full[st], 0, h, row0);
        tma_load_3d(dst + 16384, &tmQ, &B->qd_full[st], 64, h, row0);
        tma_load_3d(dst + 32768, &tmDO, &B->qd_full[st], 0, h, row0);
        tma_load_3d(dst + 49152, &tmDO, &B->qd_full[st], 64, h, row0);
        issued = w + 1;
      }
      mbar_wait(&B->kv_full, 0, p.status, OCTO_ETIMEOUT);
      for (int32_t w = max(0, issued - 2); w < issued; w++)
        mbar_wait(&B->qd_full[w & 1], (w >> 1) & 1, p.status, OCTO_ETIMEOUT);
    }
  } else if (warp == 1 || warp == 2) {
    // Two issuers with disjoint TMEM, so that a full tensor-core queue on one chain does
    // not hold up the other.  A (warp 1): dV += P^T dO, then S^T of the next item over P^T;
    // B (warp 2): dK += dS^T Q, then dP^T of the next item over dS^T.  Each thread's MMAs
    // run in issue order, which orders every overwrite after the MMAs that read the columns.
    const bool isA = warp == 1;
    if (lane == 0 && n > 0) {
      const uint64_t aX = desc_sw128(isA ? sK : sV, 16, 1024);   // K for S^T, V for dP^T
      const uint64_t bX0 = desc_sw128(sQD + (isA ? 0 : 32768), 16, 1024);   // Q / dO, K-major
      // the MN-major B operand of the accumulation: dO for dV, Q for dK
      const uint64_t bY0 = desc_sw128(sQD + (isA ? 32768 : 0), 16384, 1024);
      const uint32_t tX = tbase + (isA ? 0 : 128);     // S^T / dP^T (then P^T / dS^T)
      const uint32_t tAcc = tbase + (isA ? 256 : 384); // dV / dK
      // S'^T = K Q^T - LSE/scale  or  dP'^T = V dO^T - D
      const uint64_t aOnes = desc_noswz(smem_u32(smem + (isA ? kDkOffOnesS : kDkOffOnesD)), 2048, 128);
      const uint64_t bAug0 = desc_noswz(smem_u32(smem + kDkOffAug), 2048, 128);
      uint64_t* x_full = isA ? &B->s_full : &B->dp_full;
      uint64_t* y_full = isA ? &B->p_full : &B->ds_full;
      auto issue_x = [&](int st) {
        const uint64_t so = (uint64_t)(st * (kDkStageQD >> 4));
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          mma_f16_ss(tX, aX + o, bX0 + so + o, kIdKR, kk > 0);
        }
        mma_f16_ss(tX, aOnes, bAug0 + (uint64_t)(st * (4096 >> 4)), kIdKR, 1);
        mma_commit(x_full);
      };
      bool ok = wait_ab(&B->kv_full, 0, C, p.status) && wait_ab(&B->qd_full[0], 0, C, p.status);
      if (ok) {
        tc_fence_after();
        issue_x(0);
      }
      for (int32_t w = 0; ok && w < n; w++) {
        const int st = w & 1;
        const uint64_t so = (uint64_t)(st * (kDkStageQD >> 4));
        if (!(ok = wait_ab(y_full, w & 1, C, p.status))) break;
        tc_fence_after();
        // K = 16 query rows per MMA: 8 TMEM columns of P^T / dS^T (rows 64-127 at +64),
        // 2 swizzle atoms of dO / Q
#pragma unroll
        for (int kk = 0; kk < 8; kk++)
          mma_f16_ts(tAcc, tX + kk * 8 + (kk >= 4 ? 32 : 0), bY0 + so + (uint64_t)(kk * (2048 >> 4)), kIdKD,
                     (w > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&B->qd_free[st]);
        if (w + 1 < n) {
          if (!(ok = wait_ab(&B->qd_full[st ^ 1], ((w + 1) >> 1) & 1, C, p.status))) break;
          tc_fence_after();
          issue_x(st ^ 1);
        }
      }
      if (ok) mma_commit(&B->acc_done);
      mma_commit(&B->drain);
      mbar_wait(&B->drain, 0, p.status, OCTO_ETIMEOUT);
    }
  } else if (warp >= 4) {
    // softmax warps: warpgroup c takes query rows [64 c, 64 c + 64) of every step; a warp
    // reaches the TMEM lanes (keys) of its quadrant warp % 4
    const int c = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int k = wq * 32 + lane;
    const int hk = k >> 6, j = k & 63;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tbase + lane_off, tDP = tS + 128;
    bool ok = true;
    PairItem it{}, it_n{};
    if (n > 0) it_n = items[0];
    for (int32_t w = 0; ok && w < n; w++) {
      if (w % G == 0) {
        it = it_n;
        if (w / G + 1 < n_items) it_n = items[w / G + 1];   // prefetch
      }
      // visible rows of this key: rmin <= r < rmax
      // (selects, not indexing by hk: a dynamic index would put the item in local memory)
      const int lo = hk ? it.lo[1] : it.lo[0], hi = hk ? it.hi[1] : it.hi[0];
      int rmin = hk ? it.qlo[1] : it.qlo[0];
      if ((it.causal >> hk) & 1) rmin = max(rmin, j - (hk ? it.diag[1] : it.diag[0]));
      const int rmax = (j >= lo && j < hi) ? it.rows : 0;
      if (!(ok = warp_wait_ab(&B->s_full, w & 1, C, p.status))) break;
      tc_fence_after();
      uint32_t x0[32], x1[32];
      tmem_ld32(tS + 64 * c, x0);
      tmem_ld32(tS + 64 * c + 32, x1);
      tmem_wait_ld();
      // most steps see all 64 rows of this warpgroup for every key: no per-element mask
      const bool all_vis = __all_sync(0xffffffffu, rmin <= 64 * c && rmax >= 64 * c + 64);
      float P[64];
      auto p_phase = [&](auto masked) {
#pragma unroll
        for (int i = 0; i < 64; i += 4) {
          const uint32_t* xs = i < 32 ? x0 : x1;
          const int ii = i & 31;
          float a0, a1, a2, a3;
          // S'^T already holds S - LSE / scale
          mul2(a0, a1, __uint_as_float(xs[ii]), __uint_as_float(xs[ii + 1]), p.scale_log2, p.scale_log2);
          mul2(a2, a3, __uint_as_float(xs[ii + 2]), __uint_as_float(xs[ii + 3]), p.scale_log2, p.scale_log2);
          // every exponential on MUFU: here the softmax warps' issue slots, shared with the
          // MMA issuers, are scarcer than MUFU throughput (unlike the forward)
          a2 = ex2(a2);
          a3 = ex2(a3);
          a0 = ex2(a0);
          a1 = ex2(a1);
          if constexpr (decltype(masked)::value) {
            const int r = 64 * c + i;
            a0 = (r >= rmin && r < rmax) ? a0 : 0.f;
            a1 = (r + 1 >= rmin && r + 1 < rmax) ? a1 : 0.f;
            a2 = (r + 2 >= rmin && r + 2 < rmax) ? a2 : 0.f;
            a3 = (r + 3 >= rmin && r + 3 < rmax) ? a3 : 0.f;
          }
          P[i] = a0;
          P[i + 1] = a1;
          P[i + 2] = a2;
          P[i + 3] = a3;
        }
      };
      if (all_vis)
        p_phase(std::false_type{});
      else
        p_phase(std::true_type{});
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; i++) pk[i] = pack_bf16(P[2 * i], P[2 * i + 1]);
      tmem_st32(tS + 64 * c, pk);
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(&B->p_full);
      if (!(ok = warp_wait_ab(&B->dp_full, w & 1, C, p.status))) break;
      tc_fence_after();
      auto ds_phase = [&](auto masked) {
#pragma unroll
        for (int half = 0; half < 2; half++) {
          uint32_t x[32];
          tmem_ld32(tDP + 64 * c + 32 * half, x);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const int q = 32 * half + i;
            float d0, d1, d2, d3;
            // dP'^T already holds dP - D
            mul2(d0, d1, __uint_as_float(x[i]), __uint_as_float(x[i + 1]), P[q], P[q + 1]);
            mul2(d2, d3, __uint_as_float(x[i + 2]), __uint_as_float(x[i + 3]), P[q + 2], P[q + 3]);
            if constexpr (decltype(masked)::value) {
              // masked entries: exactly zero even where dP is not finite
              const int r = 64 * c + q;
              d0 = (r >= rmin && r < rmax) ? d0 : 0.f;
              d1 = (r + 1 >= rmin && r + 1 < rmax) ? d1 : 0.f;
              d2 = (r + 2 >= rmin && r + 2 < rmax) ? d2 : 0.f;
              d3 = (r + 3 >= rmin && r + 3 < rmax) ? d3 : 0.f;
            }
            pk[q / 2] = pack_bf16(d0, d1);
            pk[q / 2 + 1] = pack_bf16(d2, d3);
          }
        }
      };
      if (all_vis)
        ds_phase(std::false_type{});
      else
        ds_phase(std::true_type{});
      tmem_st32(tDP + 64 * c, pk);
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(&B->ds_full);
    }
    // epilogue: warpgroup c writes d columns [64 c, 64 c + 64) of this key's dV and dK rows
    if (n > 0) {
      const bool fin = ok && warp_wait_ab(&B->acc_done, 0, C, p.status);
      if (fin) {
        tc_fence_after();
        const int32_t pg = hk ? pb : pa;
        const size_t row = (size_t)(max(pg, 0) * p.Hkv + g) * 64 + j;
#pragma unroll 1
        for (int part = 0; part < 4; part++) {
          // part 0, 1: dV columns; 2, 3: dK columns
          uint32_t v[32];
          tmem_ld32(tbase + lane_off + (part < 2 ? 256 : 384) + 64 * c + 32 * (part & 1), v);
          tmem_wait_ld();
          if (pg >= 0) {
            float* out = (part < 2 ? p.dv : p.dk) + row * 128 + 64 * c + 32 * (part & 1);
            const float sc = part < 2 ? 1.f : p.scale;
#pragma unroll
            for (int q4 = 0; q4 < 8; q4++)
              st_global_v4(out + 4 * q4, __float_as_uint(__uint_as_float(v[4 * q4]) * sc),
                           __float_as_uint(__uint_as_float(v[4 * q4 + 1]) * sc),
                           __float_as_uint(__uint_as_float(v[4 * q4 + 2]) * sc),
                           __float_as_uint(__uint_as_float(v[4 * q4 + 3]) * sc));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

// =====================================================================================
// dQ
// =====================================================================================
constexpr int kDqThreads = 384;   // warp 0 TMA, warp 1 S/dP MMAs + TMEM, warp 2 dQ MMAs, warps 4-11 softmax
constexpr int kDqNK = 3;          // K pairs in flight: step j's K lands while step j - 1 runs
constexpr int kDqNV = 2;
// smem: Q 32KB | dO 32KB | 3 stages x K pair 32KB | 2 stages x V pair 32KB
constexpr uint32_t kDqOffQ = 0;
constexpr uint32_t kDqOffDO = 32768;
constexpr uint32_t kDqOffK = 65536;
constexpr uint32_t kDqOffV = kDqOffK + kDqNK * 32768;
constexpr uint32_t kDqOffBar = kDqOffV + kDqNV * 32768;
constexpr uint32_t kDqSmem = kDqOffBar + 256 + 1024;
constexpr uint32_t kIdRP = idesc_bf16(128, 128, 0, 0);   // rows x keys of an entry pair, both K-major

struct DqBars {
  uint64_t q_full;
  uint64_t k_full[kDqNK], k_empty[kDqNK];
  uint64_t v_full[kDqNV], v_empty[kDqNV];
  uint64_t s_full, s_free;   // S of the current step in TMEM / read by every softmax thread
  uint64_t dp_full[2];
  // dS of that buffer written back by all 8 softmax warps.  One barrier per buffer:
  // warpgroup 0 may finish step j + 1 before warpgroup 1 finishes step j, and its
  // arrivals must not complete step j's phase.
  uint64_t ds_full[2];
  uint64_t dq_done[2];   // dQ of a step has completed: its dS buffer may be rewritten
  uint64_t acc_done;  // single use: every dQ MMA has completed
  uint64_t drain;
  Ctl ctl;
};

// One CTA per (query tile, query head), tiles heaviest first.  The tile's entries go two at
// a time: keys 0-63 of a step from the first entry, 64-127 from the second (an odd last
// entry runs alone; its dQ MMAs stop at key 64).  TMEM: S [0, 128), dP of step j in
// [128 + 128 (j % 2), +128) with dS as bf16 at its columns 0-31 (keys 0-63) and 64-95
// (keys 64-127), dQ [384, 512); lane = row.  Two MMA issuers, so that a full tensor-core queue on one chain does not hold
// up the other: A issues S(j + 1) once the softmax has read S(j) and dP(j + 1) once dQ(j - 1)
// has completed (it read dS(j - 1) from that buffer); B issues dQ(j) once dS(j) is written.
// The softmax finds S(j + 1) and dP(j + 1) ready when it finishes step j.  K and V have
// rings of their own, as V is free once dP has run while K is read again by dQ.
__global__ void __launch_bounds__(kDqThreads, 1)
    k_dq_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
            const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DqBars* B = reinterpret_cast<DqBars*>(smem + kDqOffBar);
  Ctl* C = &B->ctl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t h = blockIdx.x % p.Hq;
  const int32_t g = h / p.G;
  const int32_t tile = p.tile_order[blockIdx.x / p.Hq];
  const int32_t e0 = p.tile_off[tile];
  const int32_t ne = p.tile_off[tile + 1] - e0;
  const int32_t n = (ne + 1) >> 1;   // steps (entry pairs)
  const int32_t rows = p.tile_rows[tile];
  const int32_t row0 = p.tile_row0[tile];

  if (threadIdx.x == 0) {
    mbar_init(&B->q_full, 1);
    for (int s = 0; s < kDqNK; s++) {
      mbar_init(&B->k_full[s], 1);
      mbar_init(&B->k_empty[s], 1);
    }
    for (int s = 0; s < kDqNV; s++) {
      mbar_init(&B->v_full[s], 1);
      mbar_init(&B->v_empty[s], 1);
    }
    mbar_init(&B->s_full, 1);
    mbar_init(&B->s_free, 8);   // one arrival per softmax warp
    for (int b = 0; b < 2; b++) {
      mbar_init(&B->dp_full[b], 1);
    }
    mbar_init(&B->ds_full[0], 8);
    mbar_init(&B->ds_full[1], 8);
    mbar_init(&B->dq_done[0], 1);
    mbar_init(&B->dq_done[1], 1);
    mbar_init(&B->acc_done, 1);
    mbar_init(&B->drain, 2);
    C->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&C->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = C->tmem_base;
  const uint32_t sQ = smem_u32(smem + kDqOffQ);
  const uint32_t sDO = smem_u32(smem + kDqOffDO);
  const uint32_t sK = smem_u32(smem + kDqOffK);
  const uint32_t sV = smem_u32(smem + kDqOffV);

  if (warp == 0) {
    if (lane == 0 && n > 0) {
      prefetch_map(&tmQ);
      prefetch_map(&tmDO);
      prefetch_map(&tmK);
      prefetch_map(&tmV);
      mbar_expect_tx(&B->q_full, 65536);
      for (int c = 0; c < 2; c++) {
        tma_load_3d(smem + kDqOffQ + c * 16384, &tmQ, &B->q_full, c * 64, h, row0);
        tma_load_3d(smem + kDqOffDO + c * 16384, &tmDO, &B->q_full, c * 64, h, row0);
      }
      int32_t issued = 0;
      for (int32_t j = 0; j < n; j++) {
        const int sk = j % kDqNK, sv = j % kDqNV;
        const int32_t ea = e0 + 2 * j;
        const int32_t pa = (int32_t)p.entries[ea].kv_page;
        const int32_t pb = 2 * j + 1 < ne ? (int32_t)p.entries[ea + 1].kv_page : -1;
        const uint32_t bytes = pb >= 0 ? 32768 : 16384;
        if (j >= kDqNK && !wait_ab(&B->k_empty[sk], ((j / kDqNK) - 1) & 1, C, p.status)) break;
        uint8_t* kd = smem + kDqOffK + sk * 32768;
        mbar_expect_tx(&B->k_full[sk], bytes);
        for (int hp = 0; hp < 2; hp++) {
          const int32_t pg = hp ? pb : pa;
          if (pg < 0) continue;
          const int32_t krow = (pg * p.Hkv + g) * 64;
          tma_load_2d(kd + hp * 8192, &tmK, &B->k_full[sk], 0, krow);
          tma_load_2d(kd + 16384 + hp * 8192, &tmK, &B->k_full[sk], 64, krow);
        }
        if (j >= kDqNV && !wait_ab(&B->v_empty[sv], ((j / kDqNV) - 1) & 1, C, p.status)) break;
        uint8_t* vd = smem + kDqOffV + sv * 32768;
        mbar_expect_tx(&B->v_full[sv], bytes);
        for (int hp = 0; hp < 2; hp++) {
          const int32_t pg = hp ? pb : pa;
          if (pg < 0) continue;
          const int32_t krow = (pg * p.Hkv + g) * 64;
          tma_load_2d(vd + hp * 8192, &tmV, &B->v_full[sv], 0, krow);
          tma_load_2d(vd + 16384 + hp * 8192, &tmV, &B->v_full[sv], 64, krow);
        }
        issued = j + 1;
      }
      mbar_wait(&B->q_full, 0, p.status, OCTO_ETIMEOUT);
      // copies still in flight land before the CTA can exit
      for (int32_t j = max(0, issued - kDqNK); j < issued; j++)
        mbar_wait(&B->k_full[j % kDqNK], (j / kDqNK) & 1, p.status, OCTO_ETIMEOUT);
      for (int32_t j = max(0, issued - kDqNV); j < issued; j++)
        mbar_wait(&B->v_full[j % kDqNV], (j / kDqNV) & 1, p.status, OCTO_ETIMEOUT);
    }
  } else if (warp == 1) {
    // issuer A: S and dP (each thread's MMAs run in issue order; the two issuers touch
    // disjoint TMEM, and A rewrites a dS buffer only after B's dQ that read it completed)
    if (lane == 0 && n > 0) {
      const uint64_t aQ = desc_sw128(sQ, 16, 1024), aDO = desc_sw128(sDO, 16, 1024);
      const uint64_t bK0 = desc_sw128(sK, 16, 1024), bV0 = desc_sw128(sV, 16, 1024);
      // S of step j: needs its K pair
      auto issue_s = [&](int32_t j) -> bool {
        const int sk = j % kDqNK;
        if (!wait_ab(&B->k_full[sk], (j / kDqNK) & 1, C, p.status)) return false;
        tc_fence_after();
        const uint64_t so = (uint64_t)(sk * (32768 >> 4));
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          mma_f16_ss(tbase, aQ + o, bK0 + so + o, kIdRP, kk > 0);
        }
        mma_commit(&B->s_full);
        return true;
      };
      // dP of step j: needs its V pair, which it alone reads
      auto issue_dp = [&](int32_t j) -> bool {
        const int sv = j % kDqNV;
        if (!wait_ab(&B->v_full[sv], (j / kDqNV) & 1, C, p.status)) return false;
        tc_fence_after();
        const uint64_t so = (uint64_t)(sv * (32768 >> 4));
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          mma_f16_ss(tbase + 128 + 128 * (j & 1), aDO + o, bV0 + so + o, kIdRP, kk > 0);
        }
        mma_commit(&B->dp_full[j & 1]);
        mma_commit(&B->v_empty[sv]);
        return true;
      };
      bool ok = wait_ab(&B->q_full, 0, C, p.status) && issue_s(0) && issue_dp(0);
      if (ok && n > 1) ok = issue_dp(1);
      for (int32_t j = 0; ok && j + 1 < n; j++) {
        if (!(ok = wait_ab(&B->s_free, j & 1, C, p.status))) break;
        if (!(ok = issue_s(j + 1))) break;
        if (j >= 1) {
          // dP(j + 1) rewrites the buffer dQ(j - 1) read
          if (!(ok = wait_ab(&B->dq_done[(j - 1) & 1], ((j - 1) >> 1) & 1, C, p.status))) break;
          if (!(ok = issue_dp(j + 1))) break;
        }
      }
      mma_commit(&B->drain);
      mbar_wait(&B->drain, 0, p.status, OCTO_ETIMEOUT);
    }
  } else if (warp == 2) {
    // issuer B: dQ += dS K once the softmax has written dS(j)
    if (lane == 0 && n > 0) {
      const uint64_t bKm0 = desc_sw128(sK, 16384, 1024);   // K pair as the MN-major B operand [keys x d]
      const uint32_t tDQ = tbase + 384;
      bool ok = true;
      for (int32_t j = 0; ok && j < n; j++) {
        const int sk = j % kDqNK;
        const uint64_t so = (uint64_t)(sk * (32768 >> 4));
        if (!(ok = wait_ab(&B->ds_full[j & 1], (j >> 1) & 1, C, p.status))) break;
        tc_fence_after();
        // K = 16 keys per MMA: 8 TMEM columns of dS (keys 64-127 at +64), 2 swizzle atoms of
        // K.  S(j), the other reader of this K stage, completed before dS(j) was written.
        const uint32_t tDS = tbase + 128 + 128 * (j & 1);
        const int nk = 2 * j + 1 < ne ? 8 : 4;
#pragma unroll
        for (int kk = 0; kk < 8; kk++)
          if (kk < nk)
            mma_f16_ts(tDQ, tDS + kk * 8 + (kk >= 4 ? 32 : 0), bKm0 + so + (uint64_t)(kk * (2048 >> 4)), kIdDQ,
                       (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&B->k_empty[sk]);
        mma_commit(&B->dq_done[j & 1]);
      }
      if (ok) mma_commit(&B->acc_done);
      mma_commit(&B->drain);
      mbar_wait(&B->drain, 0, p.status, OCTO_ETIMEOUT);
    }
  } else if (warp >= 4) {
    // softmax warps: warpgroup c takes keys [64 c, 64 c + 64) of every step, i.e. the
    // step's entry c; a warp reaches the TMEM lanes (rows) of its quadrant warp % 4
    const int c = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const bool row_ok = r < rows;
    const int64_t row = (int64_t)row0 + r;
    const float lse2 = p.lse2t[((size_t)tile * p.Hq + h) * 128 + r];
    const float Dr = p.Dt[((size_t)tile * p.Hq + h) * 128 + r];
    bool ok = true;
    octo_entry e_next{};
    if (n > 0 && c < ne) e_next = p.entries[e0 + c];
    for (int32_t j = 0; j < n; j++) {
      const bool has = 2 * j + c < ne;
      const octo_entry e = e_next;
      if (2 * (j + 1) + c < ne) e_next = p.entries[e0 + 2 * (j + 1) + c];   // prefetch
      // visible slots [lo, hi) of this row in this entry
      int lo = 64, hi = 0;
      if (has && row_ok && r >= (int)e.q_lo) {
        lo = e.kv_lo;
        hi = e.kv_hi;
        if (e.flags & 1) hi = min(hi, r + e.diag + 1);
      }
      const bool all_vis = __all_sync(0xffffffffu, lo == 0 && hi == 64);
      const int b = j & 1;
      const uint32_t tDP = tbase + lane_off + 128 + 128 * b;
      if (!(ok = warp_wait_ab(&B->s_full, j & 1, C, p.status))) break;
      tc_fence_after();
      uint32_t x0[32], x1[32];
      tmem_ld32(tbase + lane_off + 64 * c, x0);
      tmem_ld32(tbase + lane_off + 64 * c + 32, x1);
      tmem_wait_ld();
      // S may be overwritten by the next step's S from here on
      tc_fence_before();
      warp_arrive(&B->s_free);
      float P[64];
      auto p_phase = [&](auto masked) {
#pragma unroll
        for (int i = 0; i < 64; i += 4) {
          const uint32_t* xs = i < 32 ? x0 : x1;
          const int ii = i & 31;
          float a0, a1, a2, a3;
          fma2(a0, a1, __uint_as_float(xs[ii]), __uint_as_float(xs[ii + 1]), p.scale_log2, -lse2);
          fma2(a2, a3, __uint_as_float(xs[ii + 2]), __uint_as_float(xs[ii + 3]), p.scale_log2, -lse2);
          // every exponential on MUFU: here the softmax warps' issue slots, shared with the
          // MMA issuers, are scarcer than MUFU throughput (unlike the forward)
          a2 = ex2(a2);
          a3 = ex2(a3);
          a0 = ex2(a0);
          a1 = ex2(a1);
          if constexpr (decltype(masked)::value) {
            a0 = (i >= lo && i < hi) ? a0 : 0.f;
            a1 = (i + 1 >= lo && i + 1 < hi) ? a1 : 0.f;
            a2 = (i + 2 >= lo && i + 2 < hi) ? a2 : 0.f;
            a3 = (i + 3 >= lo && i + 3 < hi) ? a3 : 0.f;
          }
          P[i] = a0;
          P[i + 1] = a1;
          P[i + 2] = a2;
          P[i + 3] = a3;
        }
      };
      if (all_vis)
        p_phase(std::false_type{});
      else
        p_phase(std::true_type{});
      if (!(ok = warp_wait_ab(&B->dp_full[b], (j >> 1) & 1, C, p.status))) break;
      tc_fence_after();
      uint32_t pk[32];
      auto ds_phase = [&](auto masked) {
#pragma unroll
        for (int half = 0; half < 2; half++) {
          uint32_t x[32];
          tmem_ld32(tDP + 64 * c + 32 * half, x);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const int q = 32 * half + i;
            float d0, d1;
            add2(d0, d1, __uint_as_float(x[i]), __uint_as_float(x[i + 1]), -Dr, -Dr);
            mul2(d0, d1, d0, d1, P[q], P[q + 1]);
            if constexpr (decltype(masked)::value) {
              // masked entries: exactly zero even where dP is not finite
              d0 = (q >= lo && q < hi) ? d0 : 0.f;
              d1 = (q + 1 >= lo && q + 1 < hi) ? d1 : 0.f;
            }
            pk[q / 2] = pack_bf16(d0, d1);
          }
        }
      };
      if (all_vis)
        ds_phase(std::false_type{});
      else
        ds_phase(std::true_type{});
      // dS of keys [64 c, 64 c + 64) over the first 32 of the dP columns this warpgroup read
      tmem_st32(tDP + 64 * c, pk);
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(&B->ds_full[b]);
    }
    // epilogue: warpgroup c writes d columns [64 c, 64 c + 64) of this row's dQ
    if (n > 0) {
      const bool fin = ok && warp_wait_ab(&B->acc_done, 0, C, p.status);
      if (fin) {
        tc_fence_after();
        float* out = p.dq + (row * p.Hq + h) * 128 + 64 * c;
#pragma unroll 1
        for (int part = 0; part < 2; part++) {
          uint32_t v[32];
          tmem_ld32(tbase + lane_off + 384 + 64 * c + 32 * part, v);
          tmem_wait_ld();
          if (row_ok) {
#pragma unroll
            for (int q4 = 0; q4 < 8; q4++)
              st_global_v4(out + 32 * part + 4 * q4, __float_as_uint(__uint_as_float(v[4 * q4]) * p.scale),
                           __float_as_uint(__uint_as_float(v[4 * q4 + 1]) * p.scale),
                           __float_as_uint(__uint_as_float(v[4 * q4 + 2]) * p.scale),
                           __float_as_uint(__uint_as_float(v[4 * q4 + 3]) * p.scale));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

}  // namespace


bool bwd_tc_supported(const octo_plan_s* p, int32_t Hq) {
  const octo_pool_desc& d = p->pool->desc;
  const int32_t G = Hq / d.n_kv_heads;
  return d.dtype == OCTO_DTYPE_BF16 && d.head_dim == 128 && d.page_size == 64 && p->info.bm == 128 &&
         !p->info.is_decode && (G % 2) == 0 && p->tile_order && (p->n_pairs == 0 || p->pair_order);
}

size_t bwd_tc_workspace(const octo_plan_s* p, int32_t Hq) {
  // LSE and D per tile row (fp32) and the 2 KB statistics block per (tile, head)
  return 2 * align_up((size_t)p->info.n_tiles * Hq * 128 * sizeof(float), 256) + (size_t)p->info.n_tiles * Hq * 2048;
}

int bwd_tc(const octo_plan_s* p, int32_t Hq, const void* q, const void* k, const void* v, const void* o,
           const float* lse, const void* dout, float* dq, float* dk, float* dv, float scale, void* ws,
           cudaStream_t s) {
  const octo_pool_desc& d = p->pool->desc;
  const int64_t N = p->info.n_rows;
  if (N == 0 || p->info.n_tiles == 0) return OCTO_OK;
  if (((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)o | (uintptr_t)dout | (uintptr_t)dq | (uintptr_t)ws) & 15)
    return OCTO_EINVAL;
  const size_t st_bytes = align_up((size_t)p->info.n_tiles * Hq * 128 * sizeof(float), 256);
  float* lse2t = (float*)ws;
  float* Dt = (float*)((char*)ws + st_bytes);
  uint4* aug = (uint4*)((char*)ws + 2 * st_bytes);
  k_pre_tiles<<<(unsigned)(p->info.n_tiles * Hq), 128, 0, s>>>((const __nv_bfloat16*)o, (const __nv_bfloat16*)dout, lse,
                                                                 p->tile_row0, p->tile_rows, N, Hq, 1.f / scale, lse2t,
                                                                 Dt, aug);
  count_launch();
  CUtensorMap mq, mdo, mk, mv;
  {
    uint64_t dims[3] = {128, (uint64_t)Hq, (uint64_t)N};
    uint64_t str[2] = {128 * 2, (uint64_t)Hq * 128 * 2};
    uint32_t box[3] = {64, 1, 128};
    if (int st = encode_tmap(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, str, box,
                             CU_TENSOR_MAP_SWIZZLE_128B))
      return st;
    if (int st = encode_tmap(&mdo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(dout), dims, str, box,
                             CU_TENSOR_MAP_SWIZZLE_128B))
      return st;
  }
  {
    uint64_t dims[2] = {128, (uint64_t)d.num_pages * d.n_kv_heads * 64};
    uint64_t str[1] = {128 * 2};
    uint32_t box[2] = {64, 64};
    if (int st = encode_tmap(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(k), dims, str, box,
                             CU_TENSOR_MAP_SWIZZLE_128B))
      return st;
    if (int st = encode_tmap(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(v), dims, str, box,
                             CU_TENSOR_MAP_SWIZZLE_128B))
      return st;
  }
  BwdParams prm;
  prm.tile_off = p->tile_off;
  prm.tile_rows = p->tile_rows;
  prm.tile_row0 = p->tile_row0;
  prm.tile_order = p->tile_order;
  prm.entries = p->entries;
  prm.csc_perm = p->csc_perm;
  prm.page_off = p->page_off;
  prm.pair_pages = p->pair_pages;
  prm.pair_item_off = p->pair_item_off;
  prm.pair_n_items = p->pair_n_items;
  prm.pair_order = p->pair_order;
  prm.pair_items = p->pair_items;
  prm.lse2t = lse2t;
  prm.Dt = Dt;
  prm.aug = aug;
  prm.dq = dq;
  prm.dk = dk;
  prm.dv = dv;
  prm.n_rows = N;
  prm.Hq = Hq;
  prm.Hkv = d.n_kv_heads;
  prm.G = Hq / d.n_kv_heads;
  prm.scale = scale;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.status = p->pool->d_status;
  if (int st = set_smem_limit((const void*)k_dkdv_tc, (int)kDkSmem)) return st;
  if (int st = set_smem_limit((const void*)k_dq_tc, (int)kDqSmem)) return st;
  // the block sizes must fit the compiled register counts (a property of the binary)
  static std::atomic<int> fits{-1};
  if (fits.load() < 0) {
    cudaFuncAttributes fa, fb;
    OCTO_CUDA(cudaFuncGetAttributes(&fa, k_dkdv_tc));
    OCTO_CUDA(cudaFuncGetAttributes(&fb, k_dq_tc));
    fits.store(fa.maxThreadsPerBlock >= kDkThreads && fb.maxThreadsPerBlock >= kDqThreads ? 1 : 0);
  }
  if (fits.load() == 0) return OCTO_ENOTSUP;
  const int64_t g1 = (int64_t)p->n_pairs * d.n_kv_heads;
  if (g1 > 0) {
    k_dkdv_tc<<<(unsigned)g1, kDkThreads, kDkSmem, s>>>(mq, mdo, mk, mv, prm);
    count_launch();
  }
  const int64_t g2 = p->info.n_tiles * Hq;
  k_dq_tc<<<(unsigned)g2, kDqThreads, kDqSmem, s>>>(mq, mdo, mk, mv, prm);
  count_launch();
  return cuda_status(cudaGetLastError());
}

}  // namespace octo
