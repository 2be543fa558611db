// Packed DAG attention forward on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// Octopus project page, "Architecture & Co-Design" item 03: one unpadded 1D pass over
// the packed tree; every row attends to its ancestor path and its mounted spans.  The
// compiled plan lists, per 128-row q-tile, the (page, source) blocks of visible keys;
// this kernel runs them as a block-sparse flash-attention forward.
//
// One CTA = one q-tile x two query heads of one kv-head group (GQA: the pair shares each
// K/V page it loads).  Warp roles (384 threads):
//   warp 0      TMA producer: Q once (2 heads x 128 rows x 128 d), then K and V of each
//               entry's page through a 5-stage ring (a page load takes ~1.3 us, several
//               entries' worth of tensor work, so it has to start well ahead)
//   warps 1, 3  MMA issuers, one thread each, one per head: S_h = Q_h K^T (M128 N64
//               K16 x8) and O_h += P_h V (M128 N128 K16 x4), accumulators in TMEM.  Each
//               head's chain S -> softmax -> P V waits on its own warpgroup; one thread
//               issuing both heads' MMAs in turn made each wait behind the other (45%
//               slower, measured)
//   warp 2      TMEM allocator (512 columns: O_0, O_1, and two S buffers per head)
//   warps 4-7   softmax of head 0, warps 8-11 softmax of head 1: one row per thread,
//               S read with tcgen05.ld, mask from the entry rectangle, online softmax
//               in the log2 domain with lazy rescaling (no maximum per entry: O is
//               rescaled in TMEM only when an entry's probabilities relative to the
//               running max sum past 2^16), P written back to TMEM as bf16
//               over the S it came from; P V takes its A operand from TMEM
// S (and the P that replaces it) is double-buffered per head: the MMA issuer runs S two
// entries ahead, so a softmax warpgroup starts entry j+1 while the tensor core still runs
// P V of entry j, and the two heads' warpgroups keep the tensor core alternating between
// them.  MMAs of one issuer execute in order, so S of entry j+2 overwrites a buffer only
// after P V of entry j has read the P in it.  Each buffer has its own barriers, so no
// wait can see a barrier two phases ahead.  Every
// mbarrier wait is bounded; on expiry the kernel records OCTO_ETIMEOUT, drains its own
// copies and MMAs, frees TMEM and returns.

#include <cuda_bf16.h>

#include "internal.h"
#include "tc_common.cuh"

namespace octo {
namespace {

using namespace tc;

constexpr int kNS = 5;
constexpr int kThreads = 384;
constexpr uint32_t kQBytes = 2 * 2 * 128 * 128;     // 2 heads x 2 chunks x 128 rows x 128 B
constexpr uint32_t kKVStage = 2 * 2 * 64 * 128;     // K + V, 2 chunks x 64 rows x 128 B each
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = kOffQ + kQBytes;
constexpr uint32_t kOffBar = kOffKV + kNS * kKVStage;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;

constexpr uint32_t kIdS = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t kIdO = idesc_bf16(128, 128, 0, 1);

struct FwdTcParams {
  const int32_t* tile_off;
  const int32_t* tile_rows;
  const int32_t* tile_row0;
  const int32_t* tile_order;
  const octo_entry* entries;
  __nv_bfloat16* o;
  float* lse;
  int64_t n_rows;
  int32_t Hq, Hkv, G;
  float scale_log2;
  int32_t* status;
};

struct Bars {
  uint64_t q_full;
  uint64_t kv_full[kNS];
  uint64_t kv_empty[kNS];
  uint64_t s_full[2][2];   // [head][buffer]
  uint64_t p_full[2][2];
  uint64_t o_done[2][2];
  uint64_t drain;
  uint32_t tmem_base;
  volatile int32_t abort;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Bars* B, int32_t* status) {
  if (mbar_test(bar, parity)) return true;
  for (uint32_t i = 0; i < kSpinLimit; i++) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 1023) == 1023 && B->abort) return false;
  }
  B->abort = 1;
  atomicExch(status, OCTO_ETIMEOUT);
  return false;
}

// the same wait in every lane of a warp, with a warp-uniform result (the tcgen05
// .sync.aligned loads and stores that follow need the whole warp)
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, Bars* B, int32_t* status) {
  return __all_sync(0xffffffffu, wait_or_abort(bar, parity, B, status));
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kThreads, 1)
    k_fwd_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
             const __grid_constant__ CUtensorMap tmV, FwdTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* B = reinterpret_cast<Bars*>(smem + kOffBar);
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
    for (int s = 0; s < kNS; s++) {
      mbar_init(&B->kv_full[s], 1);
      mbar_init(&B->kv_empty[s], 2);   // released by both heads' P V
    }
    for (int h = 0; h < 2; h++)
      for (int b = 0; b < 2; b++) {
        mbar_init(&B->s_full[h][b], 1);
        mbar_init(&B->p_full[h][b], 128);
        mbar_init(&B->o_done[h][b], 1);
      }
    mbar_init(&B->drain, 2);
    B->abort = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&B->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = B->tmem_base;

  const uint32_t sQ = smem_u32(smem + kOffQ);
  const uint32_t sKV = smem_u32(smem + kOffKV);

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && n > 0) {
      prefetch_map(&tmQ);
      prefetch_map(&tmK);
      prefetch_map(&tmV);
      mbar_expect_tx(&B->q_full, kQBytes);
      for (int hh = 0; hh < 2; hh++)
        for (int c = 0; c < 2; c++)
          tma_load_3d(smem + kOffQ + (hh * 2 + c) * 16384, &tmQ, &B->q_full, c * 64, h0 + hh, row0);
      int32_t issued = 0;
      uint32_t page_next = p.entries[e0].kv_page;
      for (int32_t j = 0; j < n; j++) {
        const int st = j % kNS;
        const uint32_t page = page_next;
        if (j + 1 < n) page_next = p.entries[e0 + j + 1].kv_page;   // off the critical path
        if (j >= kNS && !wait_or_abort(&B->kv_empty[st], ((j / kNS) - 1) & 1, B, p.status)) break;
        const int32_t krow = (int32_t)((page * (uint32_t)p.Hkv + (uint32_t)g) * 64u);
        uint8_t* kd = smem + kOffKV + st * kKVStage;
        mbar_expect_tx(&B->kv_full[st], kKVStage);
        tma_load_2d(kd, &tmK, &B->kv_full[st], 0, krow);
        tma_load_2d(kd + 8192, &tmK, &B->kv_full[st], 64, krow);
        tma_load_2d(kd + 16384, &tmV, &B->kv_full[st], 0, krow);
        tma_load_2d(kd + 24576, &tmV, &B->kv_full[st], 64, krow);
        issued = j + 1;
      }
      // drain: every copy this thread started has landed before the CTA may exit
      mbar_wait(&B->q_full, 0, p.status, OCTO_ETIMEOUT);
      for (int32_t j = max(0, issued - kNS); j < issued; j++)
        mbar_wait(&B->kv_full[j % kNS], (j / kNS) & 1, p.status, OCTO_ETIMEOUT);
    }
  } else if (warp == 1 || warp == 3) {
    // ---------------- MMA issuers: warp 1 for head 0, warp 3 for head 1 ----------------
    const int hh = warp == 1 ? 0 : 1;
    if (lane == 0 && n > 0) {
      // Descriptors are built once; per MMA only the start-address field moves (all smem
      // offsets here stay inside the 14-bit field), so each issue is an add and the MMA.
      const uint64_t dq0 = desc_sw128(sQ + hh * 32768, 16, 1024);
      const uint64_t dk0 = desc_sw128(sKV, 16, 1024);
      const uint64_t dv0 = desc_sw128(sKV + 16384, 8192, 1024);
      const uint32_t dO_ = tbase + hh * 128;
      const uint32_t dS_ = tbase + 256 + hh * 128;
      auto issue_S = [&](int st, int b) {
        const uint64_t kb = dk0 + (uint64_t)(st * (kKVStage >> 4));
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          const uint32_t qo = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          const uint32_t ko = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
          mma_f16_ss(dS_ + b * 64, dq0 + qo, kb + ko, kIdS, kk > 0);
        }
        mma_commit(&B->s_full[hh][b]);
      };
      auto issue_PV = [&](int st, int b, bool first) {
        const uint32_t pa = dS_ + b * 64;   // P (bf16 pairs) over S
        const uint64_t vb = dv0 + (uint64_t)(st * (kKVStage >> 4));
#pragma unroll
        for (int kk = 0; kk < 4; kk++)
          mma_f16_ts(dO_, pa + kk * 8, vb + (uint64_t)(kk * (2048 >> 4)), kIdO, (!first || kk > 0) ? 1u : 0u);
        mma_commit(&B->o_done[hh][b]);
      };
      // S runs two entries ahead of P V
      bool ok = wait_or_abort(&B->q_full, 0, B, p.status);
      for (int32_t j = 0; ok && j < min(n, 2); j++) {
        if (!(ok = wait_or_abort(&B->kv_full[j], 0, B, p.status))) break;
        tc_fence_after();
        issue_S(j, j);
      }
      for (int32_t j = 0; ok && j < n; j++) {
        const int st = j % kNS;
        const int b = j & 1;
        const int32_t j2 = j + 2;
        if (!(ok = wait_or_abort(&B->p_full[hh][b], (j >> 1) & 1, B, p.status))) break;
        tc_fence_after();
        issue_PV(st, b, j == 0);
        mma_commit(&B->kv_empty[st]);
        if (j2 < n) {
          // buffer b held P of entry j, which P V above has read (in-order MMAs)
          if (!(ok = wait_or_abort(&B->kv_full[j2 % kNS], (j2 / kNS) & 1, B, p.status))) break;
          tc_fence_after();
          issue_S(j2 % kNS, b);
        }
      }
      // drain: all MMAs this thread issued are complete before TMEM is released
      mma_commit(&B->drain);
      mbar_wait(&B->drain, 0, p.status, OCTO_ETIMEOUT);
    }
  } else if (warp >= 4) {
    // ---------------- softmax warpgroups ----------------
    const int hh = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS0 = tbase + lane_off + 256 + hh * 128;
    const uint32_t tO = tbase + lane_off + hh * 128;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    octo_entry e_next = p.entries[e0];
    for (int32_t j = 0; j < n; j++) {
      const octo_entry e = e_next;
      if (j + 1 < n) e_next = p.entries[e0 + j + 1];   // prefetch, off the critical path
      const int b = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (!(ok = warp_wait(&B->s_full[hh][b], ph, B, p.status))) break;
      tc_fence_after();
      uint32_t s0[32], s1[32];
      tmem_ld32(tS0 + b * 64, s0);
      tmem_ld32(tS0 + b * 64 + 32, s1);
      tmem_wait_ld();
      // raw scores; the scale is folded into the exponent below
      float x[64];
#pragma unroll
      for (int i = 0; i < 32; i++) {
        x[i] = __uint_as_float(s0[i]);
        x[32 + i] = __uint_as_float(s1[i]);
      }
      const bool full = e.q_lo == 0 && e.kv_lo == 0 && e.kv_hi == 64 && !(e.flags & 1);
      if (!full) {
        const int lo = r < (int)e.q_lo ? 64 : (int)e.kv_lo;
        int hi = e.kv_hi;
        if (e.flags & 1) hi = min(hi, r + e.diag + 1);
#pragma unroll
        for (int i = 0; i < 64; i++)
          if (i < lo || i >= hi) x[i] = -INFINITY;
      }
      bool need = false;
      float factor = 1.f;
      // nothing visible to this row yet: start from the entry's exact maximum
      if (m_used == -INFINITY) m_used = max64(x) * p.scale_log2;
      float msub = (m_used == -INFINITY) ? 0.f : m_used;
      // p = 2^(s * scale_log2 - msub), every exponential on MUFU; eight running partial sums
      uint32_t pk[32];
      auto pass = [&]() -> float {
        float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 32; i++) {
          float a, c;
          fma2(a, c, x[2 * i], x[2 * i + 1], p.scale_log2, -msub);
          a = ex2(a);
          c = ex2(c);
          add2(ps[2 * (i & 3)], ps[2 * (i & 3) + 1], ps[2 * (i & 3)], ps[2 * (i & 3) + 1], a, c);
          pk[i] = pack_bf16(a, c);
        }
        return ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      };
      // Lazy rescaling without a maximum per entry: the running maximum stays while every
      // p of the entry is at most 2^16, which holds whenever their sum is; an entry whose
      // sum is larger (or not finite) is redone from its exact maximum.
      float le = pass();
      const bool over = !(le <= 65536.f);
      if (__any_sync(0xffffffffu, over)) {
        if (over) {
          const float mc = max64(x) * p.scale_log2;
          factor = ex2(m_used - mc);
          l *= factor;
          m_used = mc;
          msub = mc;
          need = true;
        }
        le = pass();
      }
      l += le;
      if (__any_sync(0xffffffffu, need)) {
        // O must hold every P V so far before it is rescaled
        if (!(ok = warp_wait(&B->o_done[hh][(j - 1) & 1], ((j - 1) >> 1) & 1, B, p.status))) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 4; c++) {
          uint32_t ov[32];
          tmem_ld32(tO + c * 32, ov);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i++) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * factor);
          tmem_st32(tO + c * 32, ov);
        }
        tmem_wait_st();
      }
      // P over the first 32 columns of this S buffer (its S is no longer needed)
      tmem_st32(tS0 + b * 64, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&B->p_full[hh][b]);
    }
    // ---------------- epilogue ----------------
    if (ok && n > 0 && warp_wait(&B->o_done[hh][(n - 1) & 1], ((n - 1) >> 1) & 1, B, p.status)) {
      tc_fence_after();
      const float inv = 1.f / l;
      const int h = h0 + hh;
      const int64_t row = (int64_t)row0 + r;
      __nv_bfloat16* orow = p.o + (row * p.Hq + h) * 128;
#pragma unroll 1
      for (int c = 0; c < 4; c++) {
        uint32_t ov[32];
        tmem_ld32(tO + c * 32, ov);
        tmem_wait_ld();
        if (r < rows) {
#pragma unroll
          for (int q4 = 0; q4 < 4; q4++) {
            uint32_t w[4];
#pragma unroll
            for (int t = 0; t < 4; t++)
              w[t] = pack_bf16(__uint_as_float(ov[q4 * 8 + 2 * t]) * inv, __uint_as_float(ov[q4 * 8 + 2 * t + 1]) * inv);
            st_global_v4(orow + c * 32 + q4 * 8, w[0], w[1], w[2], w[3]);
          }
        }
      }
      if (r < rows) {
        const float msub = (m_used == -INFINITY) ? 0.f : m_used;
        p.lse[(int64_t)h * p.n_rows + row] = (msub + lg2(l)) * 0.69314718055994531f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tbase, 512);
}

}  // namespace

// ---- host ----
int encode_tmap(CUtensorMap* map, CUtensorMapDataType dt, uint32_t rank, void* base, const uint64_t* dims,
                const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swz) {
  using Fn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*, const cuuint64_t*,
                          const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                          CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static Fn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !ptr)
      return OCTO_ECUDA;
    fn = reinterpret_cast<Fn>(ptr);
  }
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, dt, rank, base, dims, strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? OCTO_OK : OCTO_EINVAL;
}

bool fwd_tc_supported(const octo_plan_s* p, int32_t Hq) {
  const octo_pool_desc& d = p->pool->desc;
  const int32_t G = Hq / d.n_kv_heads;
  return d.dtype == OCTO_DTYPE_BF16 && d.head_dim == 128 && d.page_size == 64 && p->info.bm == 128 &&
         !p->info.is_decode && (G % 2) == 0 && p->tile_order;
}

int fwd_tc(const octo_plan_s* p, int32_t Hq, const void* q, const void* k, const void* v, void* o, float* lse,
           float scale, cudaStream_t s) {
  const octo_pool_desc& d = p->pool->desc;
  const int64_t N = p->info.n_rows;
  if (N == 0 || p->info.n_tiles == 0) return OCTO_OK;
  if (((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)o) & 15) return OCTO_EINVAL;
  CUtensorMap mq, mk, mv;
  {
    uint64_t dims[3] = {128, (uint64_t)Hq, (uint64_t)N};
    uint64_t str[2] = {128 * 2, (uint64_t)Hq * 128 * 2};
    uint32_t box[3] = {64, 1, 128};
    if (int st = encode_tmap(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, str, box,
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
  FwdTcParams prm;
  prm.tile_off = p->tile_off;
  prm.tile_rows = p->tile_rows;
  prm.tile_row0 = p->tile_row0;
  prm.tile_order = p->tile_order;
  prm.entries = p->entries;
  prm.o = (__nv_bfloat16*)o;
  prm.lse = lse;
  prm.n_rows = N;
  prm.Hq = Hq;
  prm.Hkv = d.n_kv_heads;
  prm.G = Hq / d.n_kv_heads;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.status = p->pool->d_status;
  if (int st = set_smem_limit((const void*)k_fwd_tc, (int)kSmemBytes)) return st;
  const int64_t grid = p->info.n_tiles * d.n_kv_heads * (prm.G / 2);
  if (grid > INT32_MAX) return OCTO_EINVAL;
  k_fwd_tc<<<(unsigned)grid, kThreads, kSmemBytes, s>>>(mq, mk, mv, prm);
  count_launch();
  return cuda_status(cudaGetLastError());
}

}  // namespace octo
