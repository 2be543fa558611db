// Per-token log-probability and loss over the packed rows of a plan, with its gradient.
//
// Octopus project page, "Architecture & Co-Design" item 03 (1D packed DAG-GRPO): all
// branches of an episode train in one unpadded packed pass and single-ownership masking
// counts a shared prefix once; the five-primitives table, row done, makes the close
// reminder untrainable (mask m = 0), which the caller folds into a per-token weight.
//
// Every owned token t is one packed row.  Its term is the log-probability of its token id
// under the logits of pred(t), the row of the token before it on its path (the previous
// own token, or for a segment's first token the parent's token at the fork point minus
// one; none for a root's first token).  Mounted spans are context only and change no
// predecessor.  A row feeds the terms of all its successors: the next own row and the
// first rows of the segments that continue from it (children of a fork at that point, the
// continuation of a rewind), which the pack stores per row as a sorted list.
//
//   logp[t]         = x[pred t, id t] - lse(pred t)
//   loss            = - sum_t w_t logp[t]
//   dloss/dx[r, v]  = W_r softmax(x[r])_v - sum over successors t of r with id t = v of w_t,
//                     W_r = sum over successors t of r of w_t
//
// k_token_logprob  one CTA per row: pass 1 streams the row once (16-byte loads, cached)
//                  for its max and sum of exponentials (log2 domain); the successors'
//                  logits are gathered; pass 2 streams the row again -- its first
//                  vectors from shared memory, where pass 1 left them, the rest from L2
//                  (the CTA read them microseconds earlier; loaded evict-first as their
//                  last use) -- and writes the gradient, rounded once, possibly over the
//                  logits themselves.  HBM-bound: the algorithmic bytes
//                  are one read of the logits plus one write of the gradient.
// k_loss_sum       the rows' loss partials summed in a fixed order (deterministic).

#include <cuda_bf16.h>

#include "internal.h"

namespace octo {
namespace {

constexpr int kThreads = 512;
constexpr int kMaxSucc = 64;  // successors of one row (checked when the plan is packed)
// 16-byte vectors per thread kept in shared memory from pass 1 to pass 2 (96 KB per CTA,
// two CTAs per SM): a third of a 151,936-entry bf16 row never goes back to L2, so the
// rows in flight fit it better
constexpr int kKeep = 12;
constexpr int kKeepBytes = kKeep * kThreads * 16;

struct LpParams {
  const void* logits;
  void* dlogits;
  int64_t ld;  // elements between rows
  int32_t V;
  const int32_t* ids;  // [plan rows]
  const float* w;      // [plan rows] or null (ones)
  float* logp;         // [plan rows]
  float* row_lse;      // [n] or null
  float* row_loss;     // [n] workspace
  float gs;
  const int32_t* seg_row_base;
  const int32_t* seg_pred;
  int32_t n_segs, n_rows_total;
  const int32_t* ex_pred;  // extra successors, sorted by predecessor row
  const int32_t* ex_row;
  int32_t n_ex;
  int32_t row0, n;
  int32_t* status;
};

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2f(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 16-byte vector loads: cached (pass 1) or evict-first (pass 2, the last use)
template <bool kLast>
__device__ __forceinline__ uint4 ld16(const void* p) {
  return kLast ? __ldcs(reinterpret_cast<const uint4*>(p)) : *reinterpret_cast<const uint4*>(p);
}

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int E = 8;
  __device__ static void cvt(const uint4 w, float (&x)[E]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
      x[2 * i] = __uint_as_float(u[i] << 16);
      x[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
  }
  __device__ static void store(void* p, const float (&g)[E]) {
    uint32_t u[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
      __nv_bfloat162 b = __floats2bfloat162_rn(g[2 * i], g[2 * i + 1]);
      u[i] = *reinterpret_cast<uint32_t*>(&b);
    }
    __stcs(reinterpret_cast<uint4*>(p), make_uint4(u[0], u[1], u[2], u[3]));
  }
  __device__ static float scalar(const void* p) { return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p)); }
  __device__ static void put(void* p, float g) { *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(g); }
};
template <>
struct Vec<float> {
  static constexpr int E = 4;
  __device__ static void cvt(const uint4 w, float (&x)[E]) {
    x[0] = __uint_as_float(w.x), x[1] = __uint_as_float(w.y), x[2] = __uint_as_float(w.z), x[3] = __uint_as_float(w.w);
  }
  __device__ static void store(void* p, const float (&g)[E]) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(g[0], g[1], g[2], g[3]));
  }
  __device__ static float scalar(const void* p) { return *reinterpret_cast<const float*>(p); }
  __device__ static void put(void* p, float g) { *reinterpret_cast<float*>(p) = g; }
};

// (m, s) of a sum of 2^y terms, s relative to 2^m; merged without overflow
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  s = s * ex2f(m - mn) + s2 * ex2f(m2 - mn);
  m = mn;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 2) k_token_logprob(LpParams p) {
  using VT = Vec<T>;
  constexpr int E = VT::E;
  constexpr float kL2E = 1.4426950408889634f;
  __shared__ int32_t s_t[kMaxSucc], s_id[kMaxSucc];
  __shared__ float s_w[kMaxSucc];
  __shared__ int32_t s_n, s_idlo, s_idhi;
  __shared__ float s_W, s_lse2;
  __shared__ float red_m[kThreads / 32], red_s[kThreads / 32];

  extern __shared__ uint4 keep_smem[];
  const int rl = blockIdx.x;
  const int r = p.row0 + rl;
  const char* row = reinterpret_cast<const char*>(p.logits) + (size_t)rl * p.ld * sizeof(T);
  char* grow = p.dlogits ? reinterpret_cast<char*>(p.dlogits) + (size_t)rl * p.ld * sizeof(T) : nullptr;
  uint4* keep = grow ? keep_smem : nullptr;  // launched with kKeepBytes only with a gradient

  if (threadIdx.x == 0) {
    // the packed segment of r: the last one whose first row is <= r (empty segments
    // before it share its first row, empty ones after it start past r)
    int lo = 0, hi = p.n_segs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.seg_row_base[mid] <= r) lo = mid;
      else hi = mid - 1;
    }
    const int k = lo;
    const int end = k + 1 < p.n_segs ? p.seg_row_base[k + 1] : p.n_rows_total;
    if (r == p.seg_row_base[k] && p.seg_pred[k] < 0) p.logp[r] = 0.f;  // a path start: no term
    int n = 0;
    if (r + 1 < end) s_t[n++] = r + 1;
    int a = 0, b = p.n_ex;  // first extra with predecessor >= r
    while (a < b) {
      const int mid = (a + b) >> 1;
      if (p.ex_pred[mid] < r) a = mid + 1;
      else b = mid;
    }
    for (; a < p.n_ex && p.ex_pred[a] == r && n < kMaxSucc; a++) s_t[n++] = p.ex_row[a];
    float W = 0.f;
    int idlo = p.V, idhi = -1;
    for (int i = 0; i < n; i++) {
      const int t = s_t[i];
      int id = p.ids[t];
      const float wt = p.w ? p.w[t] : 1.f;
      if (id < 0 || id >= p.V) {
        atomicExch(p.status, OCTO_EINVAL);
        p.logp[t] = __int_as_float(0x7fc00000);
        id = -1;  // no gather, no gradient term
      } else {
        idlo = min(idlo, id);
        idhi = max(idhi, id);
        W += wt;
      }
      s_id[i] = id;
      s_w[i] = wt;
    }
    s_n = n;
    s_W = W;
    s_idlo = idlo;
    s_idhi = idhi;
  }
  __syncthreads();
  const int n = s_n;
  const int nv = p.V / E;  // full vectors; the ragged tail goes element by element
  const int tail0 = nv * E;

  if (n > 0 || p.row_lse) {
    // pass 1: max and sum of exponentials, log2 domain
    float m = -INFINITY, s = 0.f;
#pragma unroll 4
    for (int i = threadIdx.x, j = 0; i < nv; i += kThreads, j++) {
      float x[E];
      const uint4 raw = ld16<false>(row + (size_t)i * E * sizeof(T));
      if (keep && j < kKeep) keep[j * kThreads + threadIdx.x] = raw;
      VT::cvt(raw, x);
      float mx = x[0];
#pragma unroll
      for (int e = 1; e < E; e++) mx = fmaxf(mx, x[e]);
      const float m2 = mx * kL2E;
      if (m2 > m) {
        s *= ex2f(m - m2);
        m = m2;
      }
      const float msub = m == -INFINITY ? 0.f : m;  // all -inf so far: every term is 0
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < E; e++) acc += ex2f(fmaf(x[e], kL2E, -msub));
      s += acc;
    }
    for (int v = tail0 + threadIdx.x; v < p.V; v += kThreads) {
      const float y = VT::scalar(row + (size_t)v * sizeof(T)) * kL2E;
      if (y > m) {
        s *= ex2f(m - y);
        m = y;
      }
      s += ex2f(y - (m == -INFINITY ? 0.f : m));
    }
    // block reduction in a fixed shape
#pragma unroll
    for (int o = 16; o; o >>= 1) lse_merge(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
    if ((threadIdx.x & 31) == 0) {
      red_m[threadIdx.x >> 5] = m;
      red_s[threadIdx.x >> 5] = s;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      m = threadIdx.x < kThreads / 32 ? red_m[threadIdx.x] : -INFINITY;
      s = threadIdx.x < kThreads / 32 ? red_s[threadIdx.x] : 0.f;
#pragma unroll
      for (int o = 16; o; o >>= 1)
        lse_merge(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
      if (threadIdx.x == 0) {
        const float l2 = m + lg2f(s);
        s_lse2 = l2;
        if (p.row_lse) p.row_lse[rl] = l2 * 0.69314718055994531f;
        // gather the successors' logits: their terms, and the row's share of the loss
        float part = 0.f;
        for (int i = 0; i < n; i++) {
          if (s_id[i] < 0) continue;
          const float lp = VT::scalar(row + (size_t)s_id[i] * sizeof(T)) - l2 * 0.69314718055994531f;
          p.logp[s_t[i]] = lp;
          part -= s_w[i] * lp;
        }
        p.row_loss[rl] = part;
      }
    }
    __syncthreads();  // the gathered elements are read before pass 2 may overwrite them
  } else if (threadIdx.x == 0) {
    p.row_loss[rl] = 0.f;
  }

  if (!grow) return;
  if (n == 0) {
    // no successor: the row's gradient is zero (written without reading the logits)
    float z[E];
#pragma unroll
    for (int e = 0; e < E; e++) z[e] = 0.f;
    for (int i = threadIdx.x; i < nv; i += kThreads) VT::store(grow + (size_t)i * E * sizeof(T), z);
    for (int v = tail0 + threadIdx.x; v < p.V; v += kThreads) VT::put(grow + (size_t)v * sizeof(T), 0.f);
    return;
  }
  // pass 2: gs (W 2^(y - lse2) - sum of the matching successors' weights)
  const float l2 = s_lse2, Wg = s_W * p.gs;
  const int idlo = s_idlo, idhi = s_idhi;
  auto onehot = [&](int v) {
    float sub = 0.f;
    for (int i = 0; i < n; i++)
      if (s_id[i] == v) sub += s_w[i];
    return sub * p.gs;
  };
#pragma unroll 4
  for (int i = threadIdx.x, j = 0; i < nv; i += kThreads, j++) {
    float x[E], g[E];
    VT::cvt(keep && j < kKeep ? keep[j * kThreads + threadIdx.x] : ld16<true>(row + (size_t)i * E * sizeof(T)), x);
#pragma unroll
    for (int e = 0; e < E; e++) g[e] = Wg * ex2f(fmaf(x[e], kL2E, -l2));
    if (i * E <= idhi && i * E + E - 1 >= idlo) {
#pragma unroll
      for (int e = 0; e < E; e++) g[e] -= onehot(i * E + e);
    }
    VT::store(grow + (size_t)i * E * sizeof(T), g);
  }
  for (int v = tail0 + threadIdx.x; v < p.V; v += kThreads) {
    const float y = VT::scalar(row + (size_t)v * sizeof(T));
    VT::put(grow + (size_t)v * sizeof(T), Wg * ex2f(fmaf(y, kL2E, -l2)) - onehot(v));
  }
}

__global__ void __launch_bounds__(1024) k_loss_sum(const float* __restrict__ part, int32_t n, float* __restrict__ loss) {
  __shared__ float red[32];
  float s = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) s += part[i];
#pragma unroll
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    s = threadIdx.x < (int)(blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (threadIdx.x == 0) *loss = s;
  }
}

}  // namespace
}  // namespace octo

extern "C" {

int octo_token_logprob_workspace_size(int32_t n_rows, size_t* bytes) {
  if (n_rows < 0 || !bytes) return OCTO_EINVAL;
  *bytes = octo::align_up((size_t)n_rows * sizeof(float), 256);
  return OCTO_OK;
}

int octo_token_logprob(octo_plan_t plan, int32_t row0, int32_t n_rows, const void* logits, int32_t dtype,
                       int64_t ld, int32_t vocab, const int32_t* ids, const float* weight, float* logp,
                       float* row_lse, void* dlogits, float grad_scale, float* loss, void* ws, size_t ws_bytes,
                       void* stream) {
  using namespace octo;
  if (!plan || plan->info.is_decode) return OCTO_EINVAL;
  const int64_t N = plan->info.n_rows;
  if (row0 < 0 || n_rows < 0 || (int64_t)row0 + n_rows > N || vocab < 1 || ld < vocab) return OCTO_EINVAL;
  if (dtype != OCTO_DTYPE_BF16 && dtype != OCTO_DTYPE_F32) return OCTO_EINVAL;
  if (plan->max_succ > kMaxSucc) return OCTO_ENOTSUP;
  if (n_rows == 0) {
    if (loss) OCTO_CUDA(cudaMemsetAsync(loss, 0, sizeof(float), (cudaStream_t)stream));
    return OCTO_OK;
  }
  size_t need = 0;
  octo_token_logprob_workspace_size(n_rows, &need);
  if (!logits || !ids || !logp || !ws || ws_bytes < need) return OCTO_EINVAL;
  const size_t es = dtype == OCTO_DTYPE_BF16 ? 2 : 4;
  if ((((uintptr_t)logits | (uintptr_t)dlogits) & 15) || ((size_t)ld * es) % 16) return OCTO_EINVAL;
  LpParams p;
  p.logits = logits;
  p.dlogits = dlogits;
  p.ld = ld;
  p.V = vocab;
  p.ids = ids;
  p.w = weight;
  p.logp = logp;
  p.row_lse = row_lse;
  p.row_loss = (float*)ws;
  p.gs = grad_scale;
  p.seg_row_base = plan->seg_row_base;
  p.seg_pred = plan->seg_pred;
  p.n_segs = plan->info.n_segments;
  p.n_rows_total = (int32_t)N;
  p.ex_pred = plan->succ_pred;
  p.ex_row = plan->succ_row;
  p.n_ex = plan->n_succ_extra;
  p.row0 = row0;
  p.n = n_rows;
  p.status = plan->pool->d_status;
  cudaStream_t s = (cudaStream_t)stream;
  plan->last_stream = s;
  const int smem = dlogits ? kKeepBytes : 0;
  if (smem) {
    const void* f = dtype == OCTO_DTYPE_BF16 ? (const void*)k_token_logprob<__nv_bfloat16> : (const void*)k_token_logprob<float>;
    if (int st = set_smem_limit(f, smem)) return st;
  }
  if (dtype == OCTO_DTYPE_BF16)
    k_token_logprob<__nv_bfloat16><<<n_rows, kThreads, smem, s>>>(p);
  else
    k_token_logprob<float><<<n_rows, kThreads, smem, s>>>(p);
  count_launch();
  if (loss) {
    k_loss_sum<<<1, 1024, 0, s>>>((const float*)ws, n_rows, loss);
    count_launch();
  }
  return cuda_status(cudaGetLastError());
}

}  // extern "C"
