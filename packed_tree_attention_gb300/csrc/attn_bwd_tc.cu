// Packed DAG attention backward on the tcgen05 tensor cores (sm_103a).
//
// Octopus project page, "Architecture & Co-Design" item 03: the packed pass routes every
// reader's gradient into the producer's KV; shared prefix tokens are owned once, so their
// dK/dV are sums over every reader row.  Two kernels, no atomics:
//
// k_dkdv_tc  one CTA per (kv page, kv head), pages launched heaviest first.  It walks the
//            page's reader entries (the plan's kv-page-major list, in list order) and, for
//            each reader entry and each of the G query heads of the group:
//              S  = Q K^T,  dP = dO V^T                       (M128 rows x N64 keys, K = d)
//              P  = exp(S - LSE),  dS = P (dP - D)            (softmax warps, entry mask)
//              dV^T += dO^T P,  dK^T += Q^T dS                (M128 d x N64 keys, K = rows)
//            The transposed accumulators keep the MMA at M = 128 with 64-key pages.  The
//            page's dK/dV are written once at the end (dK scaled).
// k_dq_tc    one CTA per (q-tile, kv head, query-head pair), like the forward: per entry
//              S, dP, then dQ += dS K                         (M128 rows x N128 d, K = keys)
//
// Both kernels issue their small (N = 64) MMAs from two threads: issuing, not executing,
// is what a single issuer is limited by at these tile sizes.  In k_dkdv_tc each issuer
// owns one Q/dO stage and its own dV^T/dK^T accumulators; the epilogue adds the two in a
// fixed order, so the sums stay deterministic.
//
// Shared-memory tiles are 128-byte swizzled; a [rows x 64 keys] tile of P or dS written by
// the softmax warps is read as a K-major A operand (dQ) or an MN-major B operand (dK/dV),
// and the TMA-loaded [rows x d] Q / dO tiles serve as K-major A (S, dP) and MN-major A
// (dK^T, dV^T).  Waits are bounded as in the forward.

#include <cuda_bf16.h>

#include "internal.h"
#include "tc_common.cuh"

namespace octo {
namespace {

using namespace tc;

constexpr uint32_t kIdRK = idesc_bf16(128, 64, 0, 0);    // rows x keys, both K-major
constexpr uint32_t kIdDK = idesc_bf16(128, 64, 1, 1);    // d x keys, both MN-major
constexpr uint32_t kIdDQ = idesc_bf16(128, 128, 0, 1);   // rows x d, B MN-major

struct BwdParams {
  const int32_t* tile_off;
  const int32_t* tile_rows;
  const int32_t* tile_row0;
  const int32_t* tile_order;
  const octo_entry* entries;
  const int32_t* csc_perm;
  const int32_t* page_off;
  const int32_t* page_order;
  const float* lse;
  const float* Dv;
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
__device__ __forceinline__ bool warp_wait_ab(uint64_t* bar, uint32_t parity, Ctl* C, int32_t* status) {
  return __all_sync(0xffffffffu, wait_ab(bar, parity, C, status));
}

// Loads this thread's row of S and dP (64 columns each, 32 at a time) from TMEM, applies
// the entry mask, and writes the row of P (if p_row != 0) and of dS, as bf16, into the
// 128-byte-swizzled row tiles at p_row / ds_row (byte addresses of this row).  Half a row
// is live at a time.
__device__ __forceinline__ void p_ds_to_smem(uint32_t tS, uint32_t tP, const octo_entry& e, int r, bool row_ok,
                                             float lse2, float Dr, float scale_log2, uint32_t p_row, uint32_t ds_row) {
  int lo = (int)e.kv_lo, hi = (int)e.kv_hi;
  if (!row_ok || r < (int)e.q_lo) lo = 64;
  if (e.flags & 1) hi = min(hi, r + e.diag + 1);
#pragma unroll
  for (int half = 0; half < 2; half++) {
    uint32_t sv[32], dv[32];
    tmem_ld32(tS + 32 * half, sv);
    tmem_ld32(tP + 32 * half, dv);
    tmem_wait_ld();
    uint32_t pk[16], dk[16];
#pragma unroll
    for (int i = 0; i < 16; i++) {
      const int j0 = 32 * half + 2 * i, j1 = j0 + 1;
      float a0, a1;
      fma2(a0, a1, __uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1]), scale_log2, -lse2);
      // MUFU for 3 of every 4 pairs, the FMA-pipe polynomial for the 4th
      if ((i & 3) == 3) {
        a0 = ex2_poly(a0);
        a1 = ex2_poly(a1);
      } else {
        a0 = ex2(a0);
        a1 = ex2(a1);
      }
      const float p0 = (j0 >= lo && j0 < hi) ? a0 : 0.f;
      const float p1 = (j1 >= lo && j1 < hi) ? a1 : 0.f;
      float d0, d1;
      add2(d0, d1, __uint_as_float(dv[2 * i]), __uint_as_float(dv[2 * i + 1]), -Dr, -Dr);
      mul2(d0, d1, d0, d1, p0, p1);
      pk[i] = pack_bf16(p0, p1);
      dk[i] = pack_bf16(d0, d1);
    }
#pragma unroll
    for (int q = 0; q < 4; q++) {
      const int c = 4 * half + q;
      const uint32_t off = (uint32_t)((c ^ (r & 7)) << 4);
      if (p_row) st_shared_v4(p_row + off, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      st_shared_v4(ds_row + off, dk[4 * q], dk[4 * q + 1], dk[4 * q + 2], dk[4 * q + 3]);
    }
  }
}

// =====================================================================================
// dK / dV
// =====================================================================================
constexpr int kDkThreads = 352;   // warp 0 TMA, warps 1-2 MMA (1 also TMEM), warps 3-10 softmax
// smem: K/V page 32KB | 2 stages x (Q 32KB + dO 32KB) | 2 stages x (P 16KB + dS 16KB)
constexpr uint32_t kDkOffKV = 0;
constexpr uint32_t kDkOffQD = 32768;
constexpr uint32_t kDkStageQD = 65536;
constexpr uint32_t kDkOffPS = kDkOffQD + 2 * kDkStageQD;
constexpr uint32_t kDkStagePS = 32768;
constexpr uint32_t kDkOffBar = kDkOffPS + 2 * kDkStagePS;
constexpr uint32_t kDkSmem = kDkOffBar + 256 + 1024;

struct DkBars {
  uint64_t kv_full;
  uint64_t qd_full[2];
  uint64_t sd_full[2];
  uint64_t sd_free[2];
  uint64_t pd_full[2];
  uint64_t mm_done[2];
  uint64_t acc_done;   // single use, 2 arrivals: every accumulation MMA has completed
  uint64_t drain;
  Ctl ctl;
};

__global__ void __launch_bounds__(kDkThreads, 1)
    k_dkdv_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
              const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DkBars* B = reinterpret_cast<DkBars*>(smem + kDkOffBar);
  Ctl* C = &B->ctl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t g = blockIdx.x % p.Hkv;
  const int32_t page = p.page_order[blockIdx.x / p.Hkv];
  const int32_t c0 = p.page_off[page];
  const int32_t n_ent = p.page_off[page + 1] - c0;
  const int32_t G = p.G;
  const int32_t n = n_ent * G;  // work items: (reader entry, head)

  if (threadIdx.x == 0) {
    mbar_init(&B->kv_full, 1);
    for (int s = 0; s < 2; s++) {
      mbar_init(&B->qd_full[s], 1);
      mbar_init(&B->sd_full[s], 1);
      mbar_init(&B->sd_free[s], 128);
      mbar_init(&B->pd_full[s], 128);
      mbar_init(&B->mm_done[s], 1);
    }
    mbar_init(&B->acc_done, 2);
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
  // TMEM columns: issuer k's dV^T [128 k, +64) and dK^T [128 k + 64, +64);
  // stage s: S [256 + 128 s, +64), dP [320 + 128 s, +64)
  const uint32_t sKV = smem_u32(smem + kDkOffKV);
  const uint32_t sQD = smem_u32(smem + kDkOffQD);
  const uint32_t sPS = smem_u32(smem + kDkOffPS);
  const int32_t krow = (page * p.Hkv + g) * 64;

  if (warp == 0) {
    if (lane == 0 && n > 0) {
      prefetch_map(&tmQ);
      prefetch_map(&tmDO);
      mbar_expect_tx(&B->kv_full, 32768);
      tma_load_2d(smem + kDkOffKV, &tmK, &B->kv_full, 0, krow);
      tma_load_2d(smem + kDkOffKV + 8192, &tmK, &B->kv_full, 64, krow);
      tma_load_2d(smem + kDkOffKV + 16384, &tmV, &B->kv_full, 0, krow);
      tma_load_2d(smem + kDkOffKV + 24576, &tmV, &B->kv_full, 64, krow);
      int32_t issued = 0;
      int32_t row0_next = p.tile_row0[p.entries[p.csc_perm[c0]].q_tile];
      for (int32_t w = 0; w < n; w++) {
        const int st = w & 1;
        const int32_t h = g * G + (w % G);
        const int32_t row0 = row0_next;
        // the next item's tile, looked up before this item's stage wait
        if (w + 1 < n) row0_next = (w + 1) % G ? row0 : p.tile_row0[p.entries[p.csc_perm[c0 + (w + 1) / G]].q_tile];
        if (w >= 2 && !wait_ab(&B->mm_done[st], ((w >> 1) - 1) & 1, C, p.status)) break;
        uint8_t* dst = smem + kDkOffQD + st * kDkStageQD;
        mbar_expect_tx(&B->qd_full[st], 65536);
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
    // issuer k = warp - 1 takes the items w with w % 2 == k (Q/dO stage k)
    const int k = warp - 1;
    if (lane == 0 && n > k) {
      const uint32_t q = sQD + k * kDkStageQD, dO = q + 32768;
      const uint32_t pP = sPS + k * kDkStagePS, pS = pP + 16384;
      const uint64_t dq_k = desc_sw128(q, 16, 1024), ddo_k = desc_sw128(dO, 16, 1024);
      const uint64_t dk_b = desc_sw128(sKV, 16, 1024), dv_b = desc_sw128(sKV + 16384, 16, 1024);
      const uint64_t dqT = desc_sw128(q, 16384, 1024), ddoT = desc_sw128(dO, 16384, 1024);
      const uint64_t dpP = desc_sw128(pP, 16384, 1024), dpS = desc_sw128(pS, 16384, 1024);
      const uint32_t tS = tbase + 256 + 128 * k, tP = tS + 64;
      const uint32_t tdV = tbase + 128 * k, tdK = tdV + 64;
      bool ok = wait_ab(&B->kv_full, 0, C, p.status);
      for (int32_t w = k; ok && w < n; w += 2) {
        const uint32_t ph = (w >> 1) & 1;
        if (!(ok = wait_ab(&B->qd_full[k], ph, C, p.status))) break;
        // S / dP buffer k: the softmax has read item w - 2's
        if (w >= 2 && !(ok = wait_ab(&B->sd_free[k], ph ^ 1, C, p.status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          const uint32_t qo = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          const uint32_t ko = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
          mma_f16_ss(tS, dq_k + qo, dk_b + ko, kIdRK, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          const uint32_t qo = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          const uint32_t vo = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
          mma_f16_ss(tP, ddo_k + qo, dv_b + vo, kIdRK, kk > 0);
        }
        mma_commit(&B->sd_full[k]);
        if (!(ok = wait_ab(&B->pd_full[k], ph, C, p.status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          // dV^T += dO^T P ; dK^T += Q^T dS  (K = 16 rows per step: 2 swizzle atoms)
          const uint32_t acc = (w > k || kk > 0) ? 1u : 0u;
          const uint64_t o = (uint64_t)(kk * (2048 >> 4));
          mma_f16_ss(tdV, ddoT + o, dpP + o, kIdDK, acc);
          mma_f16_ss(tdK, dqT + o, dpS + o, kIdDK, acc);
        }
        mma_commit(&B->mm_done[k]);
      }
      if (ok) mma_commit(&B->acc_done);
      mma_commit(&B->drain);
      mbar_wait(&B->drain, 0, p.status, OCTO_ETIMEOUT);
    } else if (lane == 0 && n > 0) {
      // no item for this issuer: its arrivals only
      mma_commit(&B->acc_done);
      mma_commit(&B->drain);
      mbar_wait(&B->drain, 0, p.status, OCTO_ETIMEOUT);
    }
  } else {
    // warps 3-10: two warpgroups; warpgroup k takes the items w with w % 2 == k (stage k).
    // A warp reaches the TMEM lanes of its quadrant warp % 4.
    const int wg = (warp - 3) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    bool ok = true;
    int32_t w = wg;
    // item metadata, loaded one item ahead (this warpgroup's next item is w + 2)
    octo_entry e_n;
    int32_t rows_n = 0;
    float lse2_n = 0.f, Dr_n = 0.f;
    auto load_item = [](const BwdParams& pp, int32_t c0_, int32_t G_, int32_t g_, int32_t wi, int r_, octo_entry& e,
                        int32_t& rows, float& lse2, float& Dr) {
      e = pp.entries[pp.csc_perm[c0_ + wi / G_]];
      const int32_t h = g_ * G_ + (wi % G_);
      rows = pp.tile_rows[e.q_tile];
      const int64_t row = (int64_t)pp.tile_row0[e.q_tile] + r_;
      const bool ok_ = r_ < rows;
      lse2 = ok_ ? pp.lse[(int64_t)h * pp.n_rows + row] * 1.4426950408889634f : 0.f;
      Dr = ok_ ? pp.Dv[(int64_t)h * pp.n_rows + row] : 0.f;
    };
    if (w < n) load_item(p, c0, G, g, w, r, e_n, rows_n, lse2_n, Dr_n);
    for (; w < n; w += 2) {
      const int st = w & 1;
      const octo_entry e = e_n;
      const bool row_ok = r < rows_n;
      const float lse2 = lse2_n, Dr = Dr_n;
      if (w + 2 < n) load_item(p, c0, G, g, w + 2, r, e_n, rows_n, lse2_n, Dr_n);
      // the accumulation MMAs of item w - 2 read this stage's P / dS buffers
      if (w >= 2) {
        if (!(ok = warp_wait_ab(&B->mm_done[st], ((w >> 1) - 1) & 1, C, p.status))) break;
      }
      if (!(ok = warp_wait_ab(&B->sd_full[st], (w >> 1) & 1, C, p.status))) break;
      tc_fence_after();
      const uint32_t pP = sPS + st * kDkStagePS;
      p_ds_to_smem(tbase + lane_off + 256 + 128 * st, tbase + lane_off + 320 + 128 * st, e, r, row_ok, lse2, Dr,
                   p.scale_log2, pP + r * 128, pP + 16384 + r * 128);
      tc_fence_before();
      mbar_arrive(&B->sd_free[st]);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&B->pd_full[st]);
    }
    // epilogue (warpgroup 0): TMEM lane = d, 64 columns = page slots.  It waits on a
    // single-use barrier: a parity wait on mm_done of the other warpgroup's stage could be
    // one completion short and still pass.
    if (wg == 0 && n > 0) {
      bool fin = ok && warp_wait_ab(&B->acc_done, 0, C, p.status);
      if (fin) {
        tc_fence_after();
        const int dd = r;
        float* dvp = p.dv + (size_t)krow * 128 + dd;
        float* dkp = p.dk + (size_t)krow * 128 + dd;
        const bool two = n > 1;   // the second issuer accumulated something
#pragma unroll 1
        for (int c = 0; c < 4; c++) {
          // c = 0, 1: dV^T columns; c = 2, 3: dK^T columns
          uint32_t v[32];
          tmem_ld32(tbase + lane_off + c * 32, v);
          if (two) {
            uint32_t v1[32];
            tmem_ld32(tbase + lane_off + 128 + c * 32, v1);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; j++) v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(v1[j]));
          } else {
            tmem_wait_ld();
          }
          float* dst = c < 2 ? dvp : dkp;
          const float sc = c < 2 ? 1.f : p.scale;
#pragma unroll
          for (int j = 0; j < 32; j++) dst[(size_t)((c & 1) * 32 + j) * 128] = __uint_as_float(v[j]) * sc;
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
constexpr int kDqThreads = 352;   // warp 0 TMA, warps 1-2 MMA per head (1 also TMEM), warps 3-10 softmax
constexpr int kDqNS = 2;
// smem: Q 64KB (2 heads) | dO 64KB | 2 stages x K/V 32KB | dS 2 heads x 16KB
constexpr uint32_t kDqOffQ = 0;
constexpr uint32_t kDqOffDO = 65536;
constexpr uint32_t kDqOffKV = 131072;
constexpr uint32_t kDqOffDS = kDqOffKV + kDqNS * 32768;
constexpr uint32_t kDqOffBar = kDqOffDS + 32768;
constexpr uint32_t kDqSmem = kDqOffBar + 256 + 1024;

struct DqBars {
  uint64_t q_full;
  uint64_t kv_full[kDqNS];
  uint64_t kv_empty[kDqNS];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t drain;
  Ctl ctl;
};

__global__ void __launch_bounds__(kDqThreads, 1)
    k_dq_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
            const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DqBars* B = reinterpret_cast<DqBars*>(smem + kDqOffBar);
  Ctl* C = &B->ctl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t HP = p.G >> 1;
  const int32_t hp = blockIdx.x % HP;
  const int32_t g = (blockIdx.x / HP) % p.Hkv;
  const int32_t tile = p.tile_order[blockIdx.x / (HP * p.Hkv)];
  const int32_t h0 = g * p.G + 2 * hp;
  const int32_t e0 = p.tile_off[tile];
  const int32_t n = p.tile_off[tile + 1] - e0;
  const int32_t rows = p.tile_rows[tile];
  const int32_t row0 = p.tile_row0[tile];

  if (threadIdx.x == 0) {
    mbar_init(&B->q_full, 1);
    for (int s = 0; s < kDqNS; s++) {
      mbar_init(&B->kv_full[s], 1);
      mbar_init(&B->kv_empty[s], 2);   // released by both heads' dQ MMAs
    }
    for (int h = 0; h < 2; h++) {
      mbar_init(&B->s_full[h], 1);
      mbar_init(&B->s_free[h], 128);
      mbar_init(&B->p_full[h], 128);
      mbar_init(&B->o_done[h], 1);
    }
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
  // TMEM: dQ_h [128 h, +128), S_h [256 + 128 h, +64), dP_h [320 + 128 h, +64)
  const uint32_t sQ = smem_u32(smem + kDqOffQ);
  const uint32_t sDO = smem_u32(smem + kDqOffDO);
  const uint32_t sKV = smem_u32(smem + kDqOffKV);
  const uint32_t sDS = smem_u32(smem + kDqOffDS);

  if (warp == 0) {
    if (lane == 0 && n > 0) {
      prefetch_map(&tmQ);
      prefetch_map(&tmDO);
      prefetch_map(&tmK);
      prefetch_map(&tmV);
      mbar_expect_tx(&B->q_full, 131072);
      for (int hh = 0; hh < 2; hh++)
        for (int c = 0; c < 2; c++) {
          tma_load_3d(smem + kDqOffQ + (hh * 2 + c) * 16384, &tmQ, &B->q_full, c * 64, h0 + hh, row0);
          tma_load_3d(smem + kDqOffDO + (hh * 2 + c) * 16384, &tmDO, &B->q_full, c * 64, h0 + hh, row0);
        }
      int32_t issued = 0;
      uint32_t page_next = p.entries[e0].kv_page;
      for (int32_t j = 0; j < n; j++) {
        const int st = j % kDqNS;
        const uint32_t page = page_next;
        if (j + 1 < n) page_next = p.entries[e0 + j + 1].kv_page;   // off the critical path
        if (j >= kDqNS && !wait_ab(&B->kv_empty[st], ((j / kDqNS) - 1) & 1, C, p.status)) break;
        const int32_t krow = (int32_t)((page * (uint32_t)p.Hkv + (uint32_t)g) * 64u);
        uint8_t* kd = smem + kDqOffKV + st * 32768;
        mbar_expect_tx(&B->kv_full[st], 32768);
        tma_load_2d(kd, &tmK, &B->kv_full[st], 0, krow);
        tma_load_2d(kd + 8192, &tmK, &B->kv_full[st], 64, krow);
        tma_load_2d(kd + 16384, &tmV, &B->kv_full[st], 0, krow);
        tma_load_2d(kd + 24576, &tmV, &B->kv_full[st], 64, krow);
        issued = j + 1;
      }
      mbar_wait(&B->q_full, 0, p.status, OCTO_ETIMEOUT);
      for (int32_t j = max(0, issued - kDqNS); j < issued; j++)
        mbar_wait(&B->kv_full[j % kDqNS], (j / kDqNS) & 1, p.status, OCTO_ETIMEOUT);
    }
  } else if (warp == 1 || warp == 2) {
    // MMA issuer for head hh = warp - 1
    const int hh = warp - 1;
    if (lane == 0 && n > 0) {
      const uint32_t tS = tbase + 256 + 128 * hh, tP = tS + 64, tQ = tbase + 128 * hh;
      const uint64_t dq_h = desc_sw128(sQ + hh * 32768, 16, 1024), ddo_h = desc_sw128(sDO + hh * 32768, 16, 1024);
      const uint64_t dk0 = desc_sw128(sKV, 16, 1024), dv0 = desc_sw128(sKV + 16384, 16, 1024);
      const uint64_t dkmn = desc_sw128(sKV, 8192, 1024);   // K page as the MN-major B operand [keys x d]
      const uint64_t dds = desc_sw128(sDS + hh * 16384, 16, 1024);
      auto issue_sd = [&](int st) {
        const uint64_t ko_st = (uint64_t)(st * (32768 >> 4));
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          const uint32_t qo = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          const uint32_t ko = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
          mma_f16_ss(tS, dq_h + qo, dk0 + ko_st + ko, kIdRK, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          const uint32_t qo = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          const uint32_t vo = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
          mma_f16_ss(tP, ddo_h + qo, dv0 + ko_st + vo, kIdRK, kk > 0);
        }
        mma_commit(&B->s_full[hh]);
      };
      auto issue_dq = [&](int st, bool first) {
        const uint64_t kb = dkmn + (uint64_t)(st * (32768 >> 4));
#pragma unroll
        for (int kk = 0; kk < 4; kk++)
          mma_f16_ss(tQ, dds + (uint64_t)(kk * 2), kb + (uint64_t)(kk * (2048 >> 4)), kIdDQ, (!first || kk > 0) ? 1u : 0u);
        mma_commit(&B->o_done[hh]);
      };
      bool ok = wait_ab(&B->q_full, 0, C, p.status) && wait_ab(&B->kv_full[0], 0, C, p.status);
      if (ok) {
        tc_fence_after();
        issue_sd(0);
      }
      for (int32_t j = 0; ok && j < n; j++) {
        const int st = j % kDqNS, st2 = (j + 1) % kDqNS;
        if (!(ok = wait_ab(&B->p_full[hh], j & 1, C, p.status))) break;
        tc_fence_after();
        issue_dq(st, j == 0);
        mma_commit(&B->kv_empty[st]);
        if (j + 1 < n) {
          if (!(ok = wait_ab(&B->kv_full[st2], ((j + 1) / kDqNS) & 1, C, p.status))) break;
          if (!(ok = wait_ab(&B->s_free[hh], j & 1, C, p.status))) break;
          tc_fence_after();
          issue_sd(st2);
        }
      }
      mma_commit(&B->drain);
      mbar_wait(&B->drain, 0, p.status, OCTO_ETIMEOUT);
    }
  } else {
    // warps 3-10: warpgroup hh handles head h0 + hh; a warp reaches TMEM quadrant warp % 4
    const int hh = (warp - 3) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int h = h0 + hh;
    const bool row_ok = r < rows;
    const int64_t row = (int64_t)row0 + r;
    const float lse2 = row_ok ? p.lse[(int64_t)h * p.n_rows + row] * 1.4426950408889634f : 0.f;
    const float Dr = row_ok ? p.Dv[(int64_t)h * p.n_rows + row] : 0.f;
    const uint32_t tS = tbase + lane_off + 256 + 128 * hh;
    const uint32_t dsrow = sDS + hh * 16384;
    bool ok = true;
    octo_entry e_next = p.entries[e0];
    for (int32_t j = 0; j < n; j++) {
      const octo_entry e = e_next;
      if (j + 1 < n) e_next = p.entries[e0 + j + 1];   // prefetch
      if (!(ok = warp_wait_ab(&B->s_full[hh], j & 1, C, p.status))) break;
      tc_fence_after();
      if (j > 0) {
        if (!(ok = warp_wait_ab(&B->o_done[hh], (j - 1) & 1, C, p.status))) break;
      }
      p_ds_to_smem(tS, tS + 64, e, r, row_ok, lse2, Dr, p.scale_log2, 0u, dsrow + r * 128);
      tc_fence_before();
      mbar_arrive(&B->s_free[hh]);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&B->p_full[hh]);
    }
    if (ok && n > 0 && warp_wait_ab(&B->o_done[hh], (n - 1) & 1, C, p.status)) {
      tc_fence_after();
      float* out = p.dq + (row * p.Hq + h) * 128;
#pragma unroll 1
      for (int c = 0; c < 4; c++) {
        uint32_t v[32];
        tmem_ld32(tbase + lane_off + 128 * hh + c * 32, v);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int q4 = 0; q4 < 8; q4++)
            st_global_v4(out + c * 32 + q4 * 4, __float_as_uint(__uint_as_float(v[4 * q4]) * p.scale),
                         __float_as_uint(__uint_as_float(v[4 * q4 + 1]) * p.scale),
                         __float_as_uint(__uint_as_float(v[4 * q4 + 2]) * p.scale),
                         __float_as_uint(__uint_as_float(v[4 * q4 + 3]) * p.scale));
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

int bwd_pre_launch(const octo_plan_s* p, int32_t Hq, const void* o, const void* dout, float* Dv, cudaStream_t s);

bool bwd_tc_supported(const octo_plan_s* p, int32_t Hq) {
  const octo_pool_desc& d = p->pool->desc;
  const int32_t G = Hq / d.n_kv_heads;
  return d.dtype == OCTO_DTYPE_BF16 && d.head_dim == 128 && d.page_size == 64 && p->info.bm == 128 &&
         !p->info.is_decode && (G % 2) == 0 && p->tile_order && p->page_order;
}

size_t bwd_tc_workspace(const octo_plan_s* p, int32_t Hq) {
  return align_up((size_t)p->info.n_rows * Hq * sizeof(float), 256);
}

int bwd_tc(const octo_plan_s* p, int32_t Hq, const void* q, const void* k, const void* v, const void* o,
           const float* lse, const void* dout, float* dq, float* dk, float* dv, float scale, void* ws,
           cudaStream_t s) {
  const octo_pool_desc& d = p->pool->desc;
  const int64_t N = p->info.n_rows;
  if (N == 0 || p->info.n_tiles == 0) return OCTO_OK;
  if (((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)dout | (uintptr_t)dq) & 15) return OCTO_EINVAL;
  float* Dv = (float*)ws;
  if (int st = bwd_pre_launch(p, Hq, o, dout, Dv, s)) return st;
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
  prm.page_order = p->page_order;
  prm.lse = lse;
  prm.Dv = Dv;
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
  static bool attr = false;
  if (!attr) {
    OCTO_CUDA(cudaFuncSetAttribute(k_dkdv_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDkSmem));
    OCTO_CUDA(cudaFuncSetAttribute(k_dq_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDqSmem));
    // the block sizes must fit the compiled register counts
    cudaFuncAttributes fa;
    OCTO_CUDA(cudaFuncGetAttributes(&fa, k_dkdv_tc));
    if (fa.maxThreadsPerBlock < kDkThreads) return OCTO_ENOTSUP;
    OCTO_CUDA(cudaFuncGetAttributes(&fa, k_dq_tc));
    if (fa.maxThreadsPerBlock < kDqThreads) return OCTO_ENOTSUP;
    attr = true;
  }
  const int64_t g1 = (int64_t)p->info.n_touched_pages * d.n_kv_heads;
  if (g1 > 0) {
    k_dkdv_tc<<<(unsigned)g1, kDkThreads, kDkSmem, s>>>(mq, mdo, mk, mv, prm);
    count_launch();
  }
  const int64_t g2 = p->info.n_tiles * d.n_kv_heads * (prm.G / 2);
  k_dq_tc<<<(unsigned)g2, kDqThreads, kDqSmem, s>>>(mq, mdo, mk, mv, prm);
  count_launch();
  return cuda_status(cudaGetLastError());
}

}  // namespace octo
