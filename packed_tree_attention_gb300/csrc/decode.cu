// Paged single-token decode over cursors (split-KV), bf16 pools, head_dim 128.
//
// Octopus project page, "Architecture & Co-Design" item 01: completed turns persist as
// radix cursors over shared KV pages; item 02: mounted sibling spans are read in place
// (0 new pages).  A decode step attends from each cursor's newest token over its whole
// context: shared prefix pages, its own pages and the mounted spans -- exactly the entry
// list of a one-row tile in the compiled decode plan.
//
// HBM-bound, so the kernel is built around bytes in flight and few instructions per byte:
//   k_decode_split   one CTA (4 warps) per (split, kv head): a split is a run of up to
//                    kSplitEntries consecutive entries of one cursor, staged in shared
//                    memory when the CTA starts.  One thread streams each entry's visible
//                    K and V rows (contiguous in the pool: one bulk copy each, completing on
//                    the stage's mbarrier) into a 2- or 3-stage ring.  Warp w takes keys
//                    [16 w, 16 w + 16) of every page and all G query heads of the group at
//                    once, so each K and V element is converted once and feeds G fused
//                    multiply-adds (packed f32x2):
//                      scores  L lanes per key, each a fixed 128/L slice of d for all G
//                              heads (query slices in registers; the slice's chunk order
//                              rotates with the key, so the unswizzled rows are read
//                              without bank conflicts); a reduce-scatter over the L lanes
//                              leaves each lane one head's score;
//                      softmax online, per warp and head (its own max and sum);
//                      P.V     lane = 4 columns of d for all G heads; P of the warp's keys
//                              is passed through shared memory as (p, p) pairs.
//                    At the end the four warps' (m, l, acc) are merged in warp order and
//                    written as the split's partial.
//   k_decode_combine one warp per (cursor, head): merges the cursor's split partials in
//                    split order (deterministic) into out and lse.
// Splits launch in the order of the first page they read, so the CTAs reading the same
// pages (a shared prefix, a mounted span and its owner's run) run together and the
// repeated reads come from L2.

#include <cuda_bf16.h>

#include <mutex>
#include <utility>
#include <vector>

#include "internal.h"
#include "tc_common.cuh"

namespace octo {
namespace {

constexpr int kD = 128;
constexpr int kP = 64;
constexpr int kStageBytes = 2 * kP * kD * 2;  // K + V rows of one page and kv head, bf16
constexpr int kWarps = 4;                     // 16 keys of each page per warp
constexpr int kRec = 4 + kD;                  // floats per (split, head) partial, 16-byte aligned

struct DecParams {
  const octo_entry* entries;
  const int32_t* split_order;  // launch order (by first page read)
  const int32_t* split_tile;   // cursor of each split
  const int32_t* split_e0;     // first entry (global index)
  const int32_t* split_e1;
  const __nv_bfloat16* q;
  const __nv_bfloat16* kp;
  const __nv_bfloat16* vp;
  float* part;                 // [n_splits][Hq][kRec]: m, l, 2 pad, acc[128]
  int32_t* status;             // device status word: OCTO_ETIMEOUT if a bounded wait gave up
  int32_t n_splits, Hq, Hkv, G;
  float scale_log2;
};

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// packed fp32 pairs (sm_100 f32x2 arithmetic), kept in 64-bit registers
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 up2(uint64_t v) {
  float2 f;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(v));
  return f;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// the two bf16 of a 32-bit word as an fp32 pair (low element first)
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) {
  return pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Bounded wait on a stage's full barrier; false once the wait gave up (status set).
__device__ __forceinline__ bool wait_full(uint64_t* bar, uint32_t parity, int32_t* status) {
  if (tc::mbar_test(bar, parity)) return true;
  for (uint32_t i = 0; i < tc::kSpinLimit; i++)
    if (tc::mbar_try(bar, parity)) return true;
  atomicExch(status, OCTO_ETIMEOUT);
  return false;
}

// GP = query heads per kv head rounded up to a power of two (heads >= G are zero queries
// whose results are dropped).  Eight lanes per key keep the query slices at 16 d per head
// (64 registers for GP = 4), so three CTAs fit on an SM with a 2-stage ring (12 warps: the
// kernel is latency-bound, and more warps beat a deeper ring, measured); GP = 8 keeps two
// CTAs with 3 stages.
template <int GP>
struct DecShape {
  static constexpr int L = 8;             // lanes per key in the score pass
  static constexpr int NC = 16 / L;       // 16-byte chunks of d per lane (d slice 8 NC)
  static constexpr int KPP = 32 / L;      // keys per score pass
  static constexpr int NPASS = 16 / KPP;  // passes over the warp's 16 keys
  static constexpr int SPREAD = L / GP;   // lanes that end with the same head
  static constexpr int ST = GP <= 4 ? 2 : 3;          // ring stages
  static constexpr int MIN_CTAS = GP <= 4 ? 3 : 2;    // CTAs per SM the registers allow
  static constexpr int SMEM = ST * kStageBytes + kWarps * 16 * GP * 8 + kSplitEntries * (int)sizeof(octo_entry) + ST * 8;
};

template <int GP>
__global__ void __launch_bounds__(kWarps * 32, DecShape<GP>::MIN_CTAS) k_decode_split(DecParams p) {
  using S = DecShape<GP>;
  extern __shared__ __align__(128) uint8_t sm[];
  // shared memory: stages | (p, p) pairs [warp][16 keys][GP] | the split's entries | full barriers
  uint64_t* pbuf = reinterpret_cast<uint64_t*>(sm + S::ST * kStageBytes) + (threadIdx.x >> 5) * 16 * GP;
  octo_entry* ents = reinterpret_cast<octo_entry*>(sm + S::ST * kStageBytes + kWarps * 16 * GP * 8);
  uint64_t* full = reinterpret_cast<uint64_t*>(ents + kSplitEntries);

  const int split = p.split_order[blockIdx.x / p.Hkv];
  const int g = blockIdx.x % p.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cur = p.split_tile[split];
  const int e0 = p.split_e0[split];
  const int n = min(p.split_e1[split] - e0, kSplitEntries);  // splits hold at most kSplitEntries

  {
    const int32_t* src = reinterpret_cast<const int32_t*>(p.entries + e0);
    int32_t* dst = reinterpret_cast<int32_t*>(ents);
    for (int i = threadIdx.x; i < n * (int)(sizeof(octo_entry) / 4); i += blockDim.x) dst[i] = src[i];
  }
  if (threadIdx.x == 0) {
    for (int st = 0; st < S::ST; st++) tc::mbar_init(&full[st], 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  // entry jj's visible rows [lo, hi) of K and V: one bulk copy each, rows at their slot
  auto issue = [&](int jj) {
    const octo_entry& e = ents[jj];
    const int st = jj % S::ST;
    const uint32_t rows = e.kv_hi - e.kv_lo;
    const size_t off = (((size_t)e.kv_page * p.Hkv + g) * kP + e.kv_lo) * kD;
    uint8_t* dk = sm + st * kStageBytes + e.kv_lo * 256;
    tc::mbar_expect_tx(&full[st], rows * 512);
    tc::bulk_load(dk, p.kp + off, rows * 256, &full[st]);
    tc::bulk_load(dk + kP * 256, p.vp + off, rows * 256, &full[st]);
  };
  if (threadIdx.x == 0)
    for (int jj = 0; jj < S::ST - 1 && jj < n; jj++) issue(jj);

  // score-pass lane roles: key kk of the pass, d slice s; the head this lane ends with.
  // The lane's i-th 16-byte chunk of d is L ((i + kk) % NC) + s: the keys of a pass start
  // at different chunk columns, so the unswizzled rows are read without bank conflicts.
  const int s = lane % S::L, kk = lane / S::L;
  const int hs = s / S::SPREAD;
  uint32_t coff[S::NC];
#pragma unroll
  for (int i = 0; i < S::NC; i++) coff[i] = (S::L * ((i + kk) % S::NC) + s) * 16;
  // query slices of all GP heads, pre-scaled into the log2 domain
  uint64_t q2[GP][S::NC * 4];
#pragma unroll
  for (int h = 0; h < GP; h++) {
    const bool real = h < p.G;
    const __nv_bfloat16* qp = p.q + ((size_t)cur * p.Hq + g * p.G + (real ? h : 0)) * kD;
#pragma unroll
    for (int i = 0; i < S::NC; i++) {
      uint4 w = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(qp) + coff[i]);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int t = 0; t < 4; t++) {
        const float a = real ? __uint_as_float(ws[t] << 16) * p.scale_log2 : 0.f;
        const float b = real ? __uint_as_float(ws[t] & 0xffff0000u) * p.scale_log2 : 0.f;
        q2[h][i * 4 + t] = pk2(a, b);
      }
    }
  }

  float m = -INFINITY, l = 0.f;  // online softmax state of head hs over this warp's keys
  uint64_t acc[GP][2];           // P.V columns 4 lane .. 4 lane + 3 of every head
#pragma unroll
  for (int h = 0; h < GP; h++) acc[h][0] = acc[h][1] = 0;

  int j = 0;
  for (; j < n; j++) {
    const bool ok = wait_full(&full[j % S::ST], (j / S::ST) & 1, p.status);
    // every thread has entry j; every warp is done with entry j - 1, whose stage is refilled
    if (!__syncthreads_and(ok)) break;
    if (threadIdx.x == 0 && j + S::ST - 1 < n) issue(j + S::ST - 1);
    const uint8_t* stk = sm + (j % S::ST) * kStageBytes;
    const uint8_t* stv = stk + kP * 256;
    const int lo = ents[j].kv_lo, hi = ents[j].kv_hi;

    // scores of the warp's keys: pass ps covers keys 16 warp + KPP ps + kk
    float sc[S::NPASS];
#pragma unroll
    for (int ps = 0; ps < S::NPASS; ps++) {
      const int key = 16 * warp + S::KPP * ps + kk;
      const uint8_t* row = stk + key * 256;
      uint64_t a2[GP];
#pragma unroll
      for (int h = 0; h < GP; h++) a2[h] = 0;
#pragma unroll
      for (int i = 0; i < S::NC; i++) {
        const uint4 w = *reinterpret_cast<const uint4*>(row + coff[i]);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int t = 0; t < 4; t++) {
          const uint64_t k2 = bf2_to_f2(ws[t]);
#pragma unroll
          for (int h = 0; h < GP; h++) a2[h] = fma2(q2[h][i * 4 + t], k2, a2[h]);
        }
      }
      float v[GP];
#pragma unroll
      for (int h = 0; h < GP; h++) {
        const float2 f = up2(a2[h]);
        v[h] = f.x + f.y;
      }
      // reduce-scatter over the L lanes of the key: halve the head set on each lane bit
      // from the top; once one head is left, plain butterfly sums
#pragma unroll
      for (int b = 0; (S::L >> (b + 1)) >= 1; b++) {
        const int mask = S::L >> (b + 1);
        const int nv = GP >> b;
        if (nv >= 2) {
          const bool up = (lane & mask) != 0;
#pragma unroll
          for (int t = 0; t < nv / 2; t++) {
            const float send = up ? v[t] : v[t + nv / 2];
            const float keep = up ? v[t + nv / 2] : v[t];
            v[t] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
          }
        } else {
          v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
        }
      }
      sc[ps] = (key >= lo && key < hi) ? v[0] : -INFINITY;
    }

    // online softmax of head hs over the warp's 16 keys (reduce across the kk lanes)
    float mx = sc[0];
#pragma unroll
    for (int ps = 1; ps < S::NPASS; ps++) mx = fmaxf(mx, sc[ps]);
#pragma unroll
    for (int o = S::L; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float mn = fmaxf(m, mx);
    const float msub = mn == -INFINITY ? 0.f : mn;
    const float corr = ex2f(m - msub);
    float psum = 0.f;
#pragma unroll
    for (int ps = 0; ps < S::NPASS; ps++) {
      const float pv = ex2f(sc[ps] - msub);
      psum += pv;
      if (s % S::SPREAD == 0) pbuf[(S::KPP * ps + kk) * GP + hs] = pk2(pv, pv);
    }
#pragma unroll
    for (int o = S::L; o < 32; o <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
    l = l * corr + psum;
    m = mn;
    // rescale every head's accumulator by its correction (held by lane h SPREAD)
#pragma unroll
    for (int h = 0; h < GP; h++) {
      const float ch = __shfl_sync(0xffffffffu, corr, h * S::SPREAD);
      const uint64_t c2 = pk2(ch, ch);
      acc[h][0] = fma2(acc[h][0], c2, 0);
      acc[h][1] = fma2(acc[h][1], c2, 0);
    }
    __syncwarp();

    // P.V over the warp's visible keys; lane = columns 4 lane .. 4 lane + 3
    const int k0 = max(lo, 16 * warp), k1 = min(hi, 16 * warp + 16);
    for (int key = k0; key < k1; key++) {
      const uint2 w = *reinterpret_cast<const uint2*>(stv + key * 256 + lane * 8);
      const uint64_t v01 = bf2_to_f2(w.x), v23 = bf2_to_f2(w.y);
      const uint64_t* pp = pbuf + (key - 16 * warp) * GP;
#pragma unroll
      for (int h = 0; h < GP; h++) {
        const uint64_t p2 = pp[h];
        acc[h][0] = fma2(p2, v01, acc[h][0]);
        acc[h][1] = fma2(p2, v23, acc[h][1]);
      }
    }
  }
  if (j < n) {
    // a wait gave up: let the copies already issued land before the CTA exits
    if (threadIdx.x == 0)
      for (int jj = j; jj < n && jj < j + S::ST - 1; jj++)
        wait_full(&full[jj % S::ST], (jj / S::ST) & 1, p.status);
    return;
  }
  __syncthreads();  // stages free: reuse stage 0 for the merge of the four warps

  // merge: ml[warp][GP][2] then accs[warp][GP][128] (fp32)
  float* ml = reinterpret_cast<float*>(sm);
  float* accs = ml + kWarps * GP * 2;
  if (kk == 0 && s % S::SPREAD == 0) {
    ml[(warp * GP + hs) * 2] = m;
    ml[(warp * GP + hs) * 2 + 1] = l;
  }
#pragma unroll
  for (int h = 0; h < GP; h++) {
    const float2 a = up2(acc[h][0]), b = up2(acc[h][1]);
    *reinterpret_cast<float4*>(accs + (warp * GP + h) * kD + 4 * lane) = make_float4(a.x, a.y, b.x, b.y);
  }
  __syncthreads();
  const int col = threadIdx.x;  // kWarps * 32 == kD
  for (int h = 0; h < p.G; h++) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; w++) M = fmaxf(M, ml[(w * GP + h) * 2]);
    const float msub = M == -INFINITY ? 0.f : M;
    float L = 0.f, a = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; w++) {
      const float f = ex2f(ml[(w * GP + h) * 2] - msub);
      L += ml[(w * GP + h) * 2 + 1] * f;
      a += accs[(w * GP + h) * kD + col] * f;
    }
    float* out = p.part + ((size_t)split * p.Hq + g * p.G + h) * kRec;
    if (col == 0) {
      out[0] = M;
      out[1] = L;
    }
    out[4 + col] = a;
  }
}

__global__ void k_decode_combine(const float* __restrict__ part, const int32_t* __restrict__ cur_split0,
                                 int32_t n, int32_t Hq, __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (w >= n * Hq) return;
  const int cur = w / Hq, h = w % Hq;
  const int s0 = cur_split0[cur], s1 = cur_split0[cur + 1];
  float M = -INFINITY;
  for (int s = s0; s < s1; s++) M = fmaxf(M, part[((size_t)s * Hq + h) * kRec]);
  const float msub = M == -INFINITY ? 0.f : M;
  float L = 0.f, a[4] = {0.f, 0.f, 0.f, 0.f};
  for (int s = s0; s < s1; s++) {
    const float* pp = part + ((size_t)s * Hq + h) * kRec;
    const float f = ex2f(pp[0] - msub);
    L += pp[1] * f;
    const float4 v = *reinterpret_cast<const float4*>(pp + 4 + 4 * lane);
    a[0] += v.x * f;
    a[1] += v.y * f;
    a[2] += v.z * f;
    a[3] += v.w * f;
  }
  const float inv = 1.f / L;
  __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(out + ((size_t)cur * Hq + h) * kD + 4 * lane);
  o[0] = __floats2bfloat162_rn(a[0] * inv, a[1] * inv);
  o[1] = __floats2bfloat162_rn(a[2] * inv, a[3] * inv);
  if (lane == 0 && lse) {
    float lg;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(L));
    lse[(size_t)cur * Hq + h] = (msub + lg) * 0.69314718055994531f;
  }
}

template <int GP>
int launch_split(const DecParams& prm, dim3 grid, cudaStream_t s) {
  const int smem = DecShape<GP>::SMEM;
  if (int st = set_smem_limit((const void*)k_decode_split<GP>, smem)) return st;
  k_decode_split<GP><<<grid, kWarps * 32, smem, s>>>(prm);
  count_launch();
  return OCTO_OK;
}

}  // namespace

bool decode_split_supported(const octo_plan_s* p, int32_t Hq) {
  const octo_pool_desc& d = p->pool->desc;
  const int32_t G = Hq / d.n_kv_heads;
  return p->info.is_decode && d.dtype == OCTO_DTYPE_BF16 && d.head_dim == 128 && d.page_size == 64 && G >= 1 &&
         G <= 8 && p->split_tile;
}

size_t decode_split_workspace(const octo_plan_s* p, int32_t Hq) {
  return align_up((size_t)p->n_splits * Hq * kRec * sizeof(float), 256);
}

int decode_split(const octo_plan_s* p, int32_t Hq, const void* q, const void* k, const void* v, void* out, float* lse,
                 float scale, void* ws, cudaStream_t s) {
  const octo_pool_desc& d = p->pool->desc;
  if (p->info.n_rows == 0) return OCTO_OK;
  if (((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)out | (uintptr_t)ws) & 15) return OCTO_EINVAL;
  DecParams prm;
  prm.entries = p->entries;
  prm.split_order = p->split_order;
  prm.split_tile = p->split_tile;
  prm.split_e0 = p->split_e0;
  prm.split_e1 = p->split_e1;
  prm.q = (const __nv_bfloat16*)q;
  prm.kp = (const __nv_bfloat16*)k;
  prm.vp = (const __nv_bfloat16*)v;
  prm.part = (float*)ws;
  prm.status = p->pool->d_status;
  prm.n_splits = p->n_splits;
  prm.Hq = Hq;
  prm.Hkv = d.n_kv_heads;
  prm.G = Hq / d.n_kv_heads;
  prm.scale_log2 = scale * 1.4426950408889634f;
  if (p->n_splits > 0) {
    const int gp = prm.G <= 1 ? 1 : prm.G <= 2 ? 2 : prm.G <= 4 ? 4 : 8;
    const dim3 grid((unsigned)(p->n_splits * d.n_kv_heads));
    int st = OCTO_OK;
    switch (gp) {
      case 1: st = launch_split<1>(prm, grid, s); break;
      case 2: st = launch_split<2>(prm, grid, s); break;
      case 4: st = launch_split<4>(prm, grid, s); break;
      default: st = launch_split<8>(prm, grid, s); break;
    }
    if (st != OCTO_OK) return st;
  }
  const int64_t warps = p->info.n_rows * Hq;
  k_decode_combine<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, s>>>(
      (const float*)ws, p->cur_split0, (int32_t)p->info.n_rows, Hq, (__nv_bfloat16*)out, lse);
  count_launch();
  return cuda_status(cudaGetLastError());
}

}  // namespace octo

// ---------------------------------------------------------------------------------------
// Allocation-free decode: the same split-KV kernels with their partials in a static device
// array instead of a caller workspace.
// ---------------------------------------------------------------------------------------
namespace octo {
namespace {

// One per device that loads the library, alive until the process exits.
static __device__ __align__(256) unsigned char g_decode_scratch[OCTO_NOALLOC_SCRATCH_BYTES];

// Scratch addresses already looked up, keyed by the unique id of the CUDA context that was
// current (cuCtxGetId): a device address belongs to one context, and a context destroyed
// and made again (cudaDeviceReset, or another context made current on the same device)
// loads the module afresh, so an address cached per device ordinal could be stale.
std::mutex g_scratch_mu;
std::vector<std::pair<unsigned long long, void*>> g_scratch_by_ctx;

int current_context_id(unsigned long long* id) {
  using GetCur = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCur get_cur = nullptr;
  static GetId get_id = nullptr;
  if (!get_cur || !get_id) {
    void *a = nullptr, *b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) != cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) != cudaSuccess ||
        qa != cudaDriverEntryPointSuccess || qb != cudaDriverEntryPointSuccess || !a || !b)
      return OCTO_ECUDA;
    get_cur = reinterpret_cast<GetCur>(a);
    get_id = reinterpret_cast<GetId>(b);
  }
  CUcontext ctx = nullptr;
  if (get_cur(&ctx) != CUDA_SUCCESS) return OCTO_ECUDA;
  if (!ctx) {
    // no context current yet: cudaSetDevice makes the device's primary context current
    int dev = 0;
    OCTO_CUDA(cudaGetDevice(&dev));
    OCTO_CUDA(cudaSetDevice(dev));
    if (get_cur(&ctx) != CUDA_SUCCESS || !ctx) return OCTO_ECUDA;
  }
  return get_id(ctx, id) == CUDA_SUCCESS ? OCTO_OK : OCTO_ECUDA;
}

// Device address of the scratch array in the current context, looked up once per context
// (cudaGetSymbolAddress with that context's device current).
int scratch_for_current_device(void** out) {
  unsigned long long id = 0;
  if (int st = current_context_id(&id)) return st;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  for (const auto& e : g_scratch_by_ctx)
    if (e.first == id) {
      *out = e.second;
      return OCTO_OK;
    }
  void* ptr = nullptr;
  OCTO_CUDA(cudaGetSymbolAddress(&ptr, g_decode_scratch));
  if (!ptr) return OCTO_ECUDA;
  g_scratch_by_ctx.emplace_back(id, ptr);
  *out = ptr;
  return OCTO_OK;
}

}  // namespace
}  // namespace octo

extern "C" int octo_decode_noalloc(octo_plan_t plan, int32_t Hq, const void* q, const void* k_pool,
                                   const void* v_pool, void* out, float* lse, float scale, void* stream) {
  if (!plan || !plan->info.is_decode) return OCTO_EINVAL;
  const int32_t Hkv = plan->pool->desc.n_kv_heads;
  if (Hq <= 0 || Hq % Hkv != 0) return OCTO_EINVAL;
  if (plan->info.n_rows > 0 && (!q || !out)) return OCTO_EINVAL;
  if (!octo::decode_split_supported(plan, Hq)) return OCTO_ENOTSUP;
  if (octo::decode_split_workspace(plan, Hq) > (size_t)OCTO_NOALLOC_SCRATCH_BYTES) return OCTO_ESCRATCH;
  const void* k = k_pool ? k_pool : plan->pool->desc.k_pool;
  const void* v = v_pool ? v_pool : plan->pool->desc.v_pool;
  if (plan->info.n_entries > 0 && (!k || !v)) return OCTO_EINVAL;
  void* scratch = nullptr;
  if (int st = octo::scratch_for_current_device(&scratch)) return st;
  plan->last_stream = (cudaStream_t)stream;
  return octo::decode_split(plan, Hq, q, k, v, out, lse, scale, scratch, (cudaStream_t)stream);
}
