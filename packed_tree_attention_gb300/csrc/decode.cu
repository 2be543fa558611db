// Paged single-token decode over cursors (split-KV), bf16 pools, head_dim 128.
//
// Octopus project page, "Architecture & Co-Design" item 01: completed turns persist as
// radix cursors over shared KV pages; item 02: mounted sibling spans are read in place
// (0 new pages).  A decode step attends from each cursor's newest token over its whole
// context: shared prefix pages, its own pages and the mounted spans -- exactly the entry
// list of a one-row tile in the compiled decode plan.
//
// HBM-bound, so the kernel is built around bytes in flight, not FLOPs:
//   k_decode_split   one CTA per (split, kv head): a split is a run of up to
//                    kSplitEntries consecutive entries of one cursor.  The CTA streams each
//                    entry's visible K/V rows into shared memory with 16-byte cp.async
//                    (two stages, rows XOR-swizzled by 16-byte chunk so that per-key reads
//                    are conflict-free), and each of its G warps (one per query head of the
//                    group) computes scores on CUDA cores (lane = key), an online softmax,
//                    and P.V (lane = 4 columns of d).  Partials (m, l, acc) go to the
//                    workspace.
//   k_decode_combine one warp per (cursor, head): merges the cursor's split partials in
//                    split order (deterministic) into out and lse.
// Splits are ordered split-index-major, so the CTAs reading the same shared prefix pages
// of an episode's cursors run together and the repeats come from L2.

#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"

namespace octo {
namespace {

constexpr int kD = 128;
constexpr int kP = 64;
constexpr int kStageBytes = 2 * kP * kD * 2;  // K + V page, bf16
constexpr int kRec = 4 + kD;                    // floats per (split, head) partial, 16-byte aligned

struct DecParams {
  const octo_entry* entries;
  const int32_t* split_order;  // launch order (split-index-major)
  const int32_t* split_tile;   // cursor of each split
  const int32_t* split_e0;     // first entry (global index)
  const int32_t* split_e1;
  const __nv_bfloat16* q;
  const __nv_bfloat16* kp;
  const __nv_bfloat16* vp;
  float* part;                 // [n_splits][Hq][kRec]: m, l, 2 pad, acc[128]
  int32_t n_splits, Hq, Hkv, G;
  float scale_log2;
};

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// byte offset of (row, 16-byte chunk) inside a [64 rows][256 B] tile, chunk XOR-swizzled
__device__ __forceinline__ uint32_t swz(int row, int chunk) { return row * 256 + ((chunk ^ (row & 15)) << 4); }

// Issues the copies of one entry's visible rows [lo, hi) of K and V into a stage.
__device__ __forceinline__ void load_entry(const DecParams& p, const octo_entry& e, int g, uint32_t sbase) {
  const size_t base = (((size_t)e.kv_page * p.Hkv + g) * kP) * kD;
  const int lo = e.kv_lo, n16 = (e.kv_hi - e.kv_lo) * 16;  // 16 chunks of 16 B per row
  for (int i = threadIdx.x; i < n16; i += blockDim.x) {
    const int row = lo + (i >> 4), c = i & 15;
    cp_async16(sbase + swz(row, c), p.kp + base + (size_t)row * kD + c * 8);
    cp_async16(sbase + kP * 256 + swz(row, c), p.vp + base + (size_t)row * kD + c * 8);
  }
}

__global__ void __launch_bounds__(256) k_decode_split(DecParams p) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int split = p.split_order[blockIdx.x / p.Hkv];
  const int g = blockIdx.x % p.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cur = p.split_tile[split];
  const int e0 = p.split_e0[split], e1 = p.split_e1[split];
  const int h = g * p.G + warp;
  const uint32_t s0 = (uint32_t)__cvta_generic_to_shared(sm);

  // this warp's query, pre-scaled into the log2 domain, as fp32 in registers
  float q[kD];
  {
    const __nv_bfloat16* qp = p.q + ((size_t)cur * p.Hq + h) * kD;
#pragma unroll
    for (int i = 0; i < kD; i += 8) {
      uint4 w = *reinterpret_cast<const uint4*>(qp + i);
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
      for (int t = 0; t < 4; t++) {
        float2 f = __bfloat1622float2(b[t]);
        q[i + 2 * t] = f.x * p.scale_log2;
        q[i + 2 * t + 1] = f.y * p.scale_log2;
      }
    }
  }
  float m = -INFINITY, l = 0.f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};  // columns 4*lane .. 4*lane+3

  const int n = e1 - e0;
  if (n > 0) load_entry(p, p.entries[e0], g, s0);
  cp_commit();
  for (int j = 0; j < n; j++) {
    const octo_entry e = p.entries[e0 + j];
    if (j + 1 < n) load_entry(p, p.entries[e0 + j + 1], g, s0 + ((j + 1) & 1) * kStageBytes);
    cp_commit();
    cp_wait<1>();
    __syncthreads();
    const uint32_t st = s0 + (j & 1) * kStageBytes;
    const uint8_t* stp = sm + (j & 1) * kStageBytes;
    // scores: lane handles keys lane and lane + 32
    float sc[2];
#pragma unroll
    for (int kk = 0; kk < 2; kk++) {
      const int key = lane + 32 * kk;
      float a = 0.f;
      if (key >= e.kv_lo && key < e.kv_hi) {
#pragma unroll
        for (int c = 0; c < 16; c++) {
          uint4 w = *reinterpret_cast<const uint4*>(stp + swz(key, c));
          const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
          for (int t = 0; t < 4; t++) {
            float2 f = __bfloat1622float2(b[t]);
            a = fmaf(q[c * 8 + 2 * t], f.x, a);
            a = fmaf(q[c * 8 + 2 * t + 1], f.y, a);
          }
        }
      } else {
        a = -INFINITY;
      }
      sc[kk] = a;
    }
    float mx = fmaxf(sc[0], sc[1]);
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float mn = fmaxf(m, mx);
    const float msub = mn == -INFINITY ? 0.f : mn;
    const float corr = ex2f(m - msub);
    const float p0 = ex2f(sc[0] - msub), p1 = ex2f(sc[1] - msub);
    float ps = p0 + p1;
#pragma unroll
    for (int o = 16; o; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
    l = l * corr + ps;
    m = mn;
#pragma unroll
    for (int t = 0; t < 4; t++) acc[t] *= corr;
    // P.V: lane owns columns 4*lane .. 4*lane + 3 (chunk lane/2, half lane&1)
    const int c = lane >> 1, half = lane & 1;
    for (int key = e.kv_lo; key < e.kv_hi; key++) {
      const float pk = __shfl_sync(0xffffffffu, key < 32 ? p0 : p1, key & 31);
      const uint2 w = *reinterpret_cast<const uint2*>(stp + kP * 256 + swz(key, c) + half * 8);
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&w);
      float2 f0 = __bfloat1622float2(b[0]), f1 = __bfloat1622float2(b[1]);
      acc[0] = fmaf(pk, f0.x, acc[0]);
      acc[1] = fmaf(pk, f0.y, acc[1]);
      acc[2] = fmaf(pk, f1.x, acc[2]);
      acc[3] = fmaf(pk, f1.y, acc[3]);
    }
    (void)st;
    __syncthreads();  // the stage is refilled next iteration
  }
  cp_wait<0>();
  float* out = p.part + ((size_t)split * p.Hq + h) * kRec;
  if (lane == 0) {
    out[0] = m;
    out[1] = l;
  }
  *reinterpret_cast<float4*>(out + 4 + 4 * lane) = make_float4(acc[0], acc[1], acc[2], acc[3]);
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
  prm.n_splits = p->n_splits;
  prm.Hq = Hq;
  prm.Hkv = d.n_kv_heads;
  prm.G = Hq / d.n_kv_heads;
  prm.scale_log2 = scale * 1.4426950408889634f;
  const int smem = 2 * kStageBytes;
  static bool attr = false;
  if (!attr) {
    OCTO_CUDA(cudaFuncSetAttribute(k_decode_split, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    attr = true;
  }
  if (p->n_splits > 0) {
    k_decode_split<<<(unsigned)(p->n_splits * d.n_kv_heads), 32 * prm.G, smem, s>>>(prm);
    count_launch();
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

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device
// (cudaGetSymbolAddress with that device current).
int scratch_for_current_device(void** out) {
  int dev = 0;
  OCTO_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return OCTO_ENOTSUP;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    OCTO_CUDA(cudaGetSymbolAddress(&ptr, g_decode_scratch));
    if (!ptr) return OCTO_ECUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
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
