// CUDA-core (SIMT) attention over a compiled plan: the fp32 path and the generic path
// for shapes the tensor-core kernels do not cover (head_dim 64, any page size, any
// q-tile size, fp32 pools).
//
// Octopus project page, "Architecture & Co-Design" item 03: each packed row attends to
// its tree-ancestor path plus the spans mounted into it; shared prefix tokens are stored
// once and their dK/dV collect the gradient of every reader.  Per row and query head h
// (kv head g = h / G):
//   s_j = scale * q . k_j over visible j,  O = softmax(s) V,  LSE = ln sum_j exp(s_j)
//   D = dO . O,  P_j = exp(s_j - LSE),  dS_j = P_j (dO . v_j - D)
//   dQ = scale sum_j dS_j k_j,  dK_j = scale sum dS_j q,  dV_j = sum P_j dO
// the dK/dV sums running over every reader row of the key's page (kv-page-major walk of
// the plan's CSC lists, in list order) and over the G query heads of the group: no
// atomics, a fixed summation order.
//
// One warp per (row, head); each lane holds head_dim/32 elements.  exp/log are the
// accurate expf/logf so the fp32 path meets a 1e-5 relative bound.

#include <cuda_bf16.h>

#include "internal.h"

namespace octo {
namespace {

template <typename T>
__device__ __forceinline__ float ld(const T* p);
template <>
__device__ __forceinline__ float ld<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }
template <typename T>
__device__ __forceinline__ void st(T* p, float v);
template <>
__device__ __forceinline__ void st<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16* p, float v) { *p = __float2bfloat16(v); }

__device__ __forceinline__ float warp_sum(float v) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

struct SimtPlan {
  const int32_t* tile_off;
  const int32_t* tile_rows;
  const int32_t* tile_row0;
  const octo_entry* entries;
  const int32_t* csc_perm;
  const int32_t* page_off;
  const int32_t* touched;
  int32_t P, Hkv, Hq;
};

__device__ __forceinline__ bool visible(const octo_entry& e, int32_t r, int32_t j) {
  return r >= e.q_lo && j >= e.kv_lo && j < e.kv_hi && (!(e.flags & 1) || j <= r + e.diag);
}

// grid: (tiles, Hq); block: 32 * warps; lse index = h * lse_h + row * lse_r
template <typename T, int D>
__global__ void k_fwd_simt(SimtPlan pl, const T* __restrict__ q, const T* __restrict__ kp, const T* __restrict__ vp,
                           T* __restrict__ o, float* __restrict__ lse, int64_t lse_h, int64_t lse_r, float scale) {
  constexpr int E = D / 32;
  const int32_t tile = blockIdx.x, h = blockIdx.y;
  const int32_t g = h / (pl.Hq / pl.Hkv);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int32_t rows = pl.tile_rows[tile], row0 = pl.tile_row0[tile];
  const int32_t e0 = pl.tile_off[tile], e1 = pl.tile_off[tile + 1];
  for (int32_t r = warp; r < rows; r += nwarps) {
    const int64_t row = row0 + r;
    float qv[E], acc[E];
    const T* qp = q + (row * pl.Hq + h) * D;
#pragma unroll
    for (int i = 0; i < E; i++) {
      qv[i] = ld(qp + lane + 32 * i) * scale;
      acc[i] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int32_t ei = e0; ei < e1; ei++) {
      const octo_entry e = pl.entries[ei];
      if (r < e.q_lo) continue;
      int32_t hi = e.kv_hi;
      if (e.flags & 1) hi = min(hi, r + e.diag + 1);
      const size_t base = (((size_t)e.kv_page * pl.Hkv + g) * pl.P) * D;
      for (int32_t j = e.kv_lo; j < hi; j++) {
        const T* kr = kp + base + (size_t)j * D;
        float part = 0.f;
#pragma unroll
        for (int i = 0; i < E; i++) part += qv[i] * ld(kr + lane + 32 * i);
        float s = warp_sum(part);
        float mn = fmaxf(m, s);
        float c = expf(m - mn);  // 0 when m = -inf
        float p = expf(s - mn);
        l = l * c + p;
        const T* vr = vp + base + (size_t)j * D;
#pragma unroll
        for (int i = 0; i < E; i++) acc[i] = acc[i] * c + p * ld(vr + lane + 32 * i);
        m = mn;
      }
    }
    float inv = 1.f / l;
    T* op = o + (row * pl.Hq + h) * D;
#pragma unroll
    for (int i = 0; i < E; i++) st(op + lane + 32 * i, acc[i] * inv);
    if (lane == 0 && lse) lse[h * lse_h + row * lse_r] = m + logf(l);
  }
}

// D[h][row] = dO . O
template <typename T, int D>
__global__ void k_bwd_pre(const T* __restrict__ o, const T* __restrict__ dout, float* __restrict__ Dv, int64_t n_rows,
                          int32_t Hq) {
  constexpr int E = D / 32;
  int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= n_rows * Hq) return;
  int64_t row = w / Hq;
  int32_t h = (int32_t)(w % Hq);
  const T* a = o + w * D;
  const T* b = dout + w * D;
  float part = 0.f;
#pragma unroll
  for (int i = 0; i < E; i++) part += ld(a + lane + 32 * i) * ld(b + lane + 32 * i);
  part = warp_sum(part);
  if (lane == 0) Dv[(int64_t)h * n_rows + row] = part;
}

// dQ: grid (tiles, Hq), warp per row
template <typename T, int D>
__global__ void k_bwd_dq_simt(SimtPlan pl, const T* __restrict__ q, const T* __restrict__ kp, const T* __restrict__ vp,
                              const T* __restrict__ dout, const float* __restrict__ lse, const float* __restrict__ Dv,
                              int64_t n_rows, float* __restrict__ dq, float scale) {
  constexpr int E = D / 32;
  const int32_t tile = blockIdx.x, h = blockIdx.y;
  const int32_t g = h / (pl.Hq / pl.Hkv);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int32_t rows = pl.tile_rows[tile], row0 = pl.tile_row0[tile];
  const int32_t e0 = pl.tile_off[tile], e1 = pl.tile_off[tile + 1];
  for (int32_t r = warp; r < rows; r += nwarps) {
    const int64_t row = row0 + r;
    float qv[E], dov[E], acc[E];
    const T* qp = q + (row * pl.Hq + h) * D;
    const T* dp = dout + (row * pl.Hq + h) * D;
#pragma unroll
    for (int i = 0; i < E; i++) {
      qv[i] = ld(qp + lane + 32 * i);
      dov[i] = ld(dp + lane + 32 * i);
      acc[i] = 0.f;
    }
    const float L = lse[(int64_t)h * n_rows + row];
    const float Dr = Dv[(int64_t)h * n_rows + row];
    for (int32_t ei = e0; ei < e1; ei++) {
      const octo_entry e = pl.entries[ei];
      if (r < e.q_lo) continue;
      int32_t hi = e.kv_hi;
      if (e.flags & 1) hi = min(hi, r + e.diag + 1);
      const size_t base = (((size_t)e.kv_page * pl.Hkv + g) * pl.P) * D;
      for (int32_t j = e.kv_lo; j < hi; j++) {
        const T* kr = kp + base + (size_t)j * D;
        const T* vr = vp + base + (size_t)j * D;
        float ps = 0.f, pd = 0.f;
        float kv[E];
#pragma unroll
        for (int i = 0; i < E; i++) {
          kv[i] = ld(kr + lane + 32 * i);
          ps += qv[i] * kv[i];
          pd += dov[i] * ld(vr + lane + 32 * i);
        }
        ps = warp_sum(ps);
        pd = warp_sum(pd);
        float p = expf(ps * scale - L);
        float ds = p * (pd - Dr);
#pragma unroll
        for (int i = 0; i < E; i++) acc[i] += ds * kv[i];
      }
    }
    float* out = dq + (row * pl.Hq + h) * D;
#pragma unroll
    for (int i = 0; i < E; i++) out[lane + 32 * i] = acc[i] * scale;
  }
}

// dK, dV: grid (touched pages, Hkv), warp per page slot; walks the page's CSC list
template <typename T, int D>
__global__ void k_bwd_dkdv_simt(SimtPlan pl, const T* __restrict__ q, const T* __restrict__ kp,
                                const T* __restrict__ vp, const T* __restrict__ dout, const float* __restrict__ lse,
                                const float* __restrict__ Dv, int64_t n_rows, float* __restrict__ dk,
                                float* __restrict__ dv, float scale) {
  constexpr int E = D / 32;
  const int32_t page = pl.touched[blockIdx.x], g = blockIdx.y;
  const int32_t G = pl.Hq / pl.Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int32_t c0 = pl.page_off[page], c1 = pl.page_off[page + 1];
  const size_t base = (((size_t)page * pl.Hkv + g) * pl.P) * D;
  for (int32_t j = warp; j < pl.P; j += nwarps) {
    float kv[E], vv[E], ak[E], av[E];
#pragma unroll
    for (int i = 0; i < E; i++) {
      kv[i] = ld(kp + base + (size_t)j * D + lane + 32 * i);
      vv[i] = ld(vp + base + (size_t)j * D + lane + 32 * i);
      ak[i] = av[i] = 0.f;
    }
    for (int32_t ci = c0; ci < c1; ci++) {
      const octo_entry e = pl.entries[pl.csc_perm[ci]];
      if (j < e.kv_lo || j >= e.kv_hi) continue;
      const int32_t rows = pl.tile_rows[e.q_tile], row0 = pl.tile_row0[e.q_tile];
      int32_t rlo = e.q_lo;
      if (e.flags & 1) rlo = max(rlo, j - e.diag);
      for (int32_t r = rlo; r < rows; r++) {
        const int64_t row = row0 + r;
        for (int32_t hh = 0; hh < G; hh++) {
          const int32_t h = g * G + hh;
          const T* qp = q + (row * pl.Hq + h) * D;
          const T* dp = dout + (row * pl.Hq + h) * D;
          float qv[E], dov[E];
          float ps = 0.f, pd = 0.f;
#pragma unroll
          for (int i = 0; i < E; i++) {
            qv[i] = ld(qp + lane + 32 * i);
            dov[i] = ld(dp + lane + 32 * i);
            ps += qv[i] * kv[i];
            pd += dov[i] * vv[i];
          }
          ps = warp_sum(ps);
          pd = warp_sum(pd);
          float p = expf(ps * scale - lse[(int64_t)h * n_rows + row]);
          float ds = p * (pd - Dv[(int64_t)h * n_rows + row]);
#pragma unroll
          for (int i = 0; i < E; i++) {
            ak[i] += ds * qv[i];
            av[i] += p * dov[i];
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < E; i++) {
      dk[base + (size_t)j * D + lane + 32 * i] = ak[i] * scale;
      dv[base + (size_t)j * D + lane + 32 * i] = av[i];
    }
  }
}

SimtPlan make_simt_plan(const octo_plan_s* p, int32_t Hq) {
  SimtPlan s;
  s.tile_off = p->tile_off;
  s.tile_rows = p->tile_rows;
  s.tile_row0 = p->tile_row0;
  s.entries = p->entries;
  s.csc_perm = p->csc_perm;
  s.page_off = p->page_off;
  s.touched = p->touched;
  s.P = p->pool->desc.page_size;
  s.Hkv = p->pool->desc.n_kv_heads;
  s.Hq = Hq;
  return s;
}

template <typename T, int D>
int fwd_simt_t(const octo_plan_s* p, int32_t Hq, const void* q, const void* k, const void* v, void* o, float* lse,
               float scale, bool decode, cudaStream_t s) {
  SimtPlan sp = make_simt_plan(p, Hq);
  const int64_t T_ = p->info.n_tiles, N = p->info.n_rows;
  if (T_ == 0) return OCTO_OK;
  dim3 grid((unsigned)T_, (unsigned)Hq);
  int warps = decode ? 1 : 4;
  int64_t lse_h = decode ? 1 : N, lse_r = decode ? Hq : 1;
  k_fwd_simt<T, D><<<grid, 32 * warps, 0, s>>>(sp, (const T*)q, (const T*)k, (const T*)v, (T*)o, lse, lse_h, lse_r,
                                               scale);
  count_launch();
  return cuda_status(cudaGetLastError());
}

template <typename T, int D>
int bwd_simt_t(const octo_plan_s* p, int32_t Hq, const void* q, const void* k, const void* v, const void* o,
               const float* lse, const void* dout, float* dq, float* dk, float* dv, float scale, void* ws,
               cudaStream_t s) {
  SimtPlan sp = make_simt_plan(p, Hq);
  const int64_t N = p->info.n_rows;
  float* Dv = (float*)ws;
  if (N > 0) {
    int64_t warps = N * Hq;
    k_bwd_pre<T, D><<<(unsigned)((warps * 32 + 255) / 256), 256, 0, s>>>((const T*)o, (const T*)dout, Dv, N, Hq);
    count_launch();
    dim3 grid((unsigned)p->info.n_tiles, (unsigned)Hq);
    k_bwd_dq_simt<T, D><<<grid, 128, 0, s>>>(sp, (const T*)q, (const T*)k, (const T*)v, (const T*)dout, lse, Dv, N,
                                             dq, scale);
    count_launch();
  }
  if (p->info.n_touched_pages > 0) {
    dim3 grid2((unsigned)p->info.n_touched_pages, (unsigned)p->pool->desc.n_kv_heads);
    k_bwd_dkdv_simt<T, D><<<grid2, 128, 0, s>>>(sp, (const T*)q, (const T*)k, (const T*)v, (const T*)dout, lse, Dv, N,
                                                dk, dv, scale);
    count_launch();
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace

int fwd_simt(const octo_plan_s* p, int32_t Hq, const void* q, const void* k, const void* v, void* o, float* lse,
             float scale, bool decode, cudaStream_t s) {
  const octo_pool_desc& d = p->pool->desc;
  if (d.dtype == OCTO_DTYPE_F32)
    return d.head_dim == 64 ? fwd_simt_t<float, 64>(p, Hq, q, k, v, o, lse, scale, decode, s)
                            : fwd_simt_t<float, 128>(p, Hq, q, k, v, o, lse, scale, decode, s);
  return d.head_dim == 64 ? fwd_simt_t<__nv_bfloat16, 64>(p, Hq, q, k, v, o, lse, scale, decode, s)
                          : fwd_simt_t<__nv_bfloat16, 128>(p, Hq, q, k, v, o, lse, scale, decode, s);
}

int bwd_simt(const octo_plan_s* p, int32_t Hq, const void* q, const void* k, const void* v, const void* o,
             const float* lse, const void* dout, float* dq, float* dk, float* dv, float scale, void* ws,
             cudaStream_t s) {
  const octo_pool_desc& d = p->pool->desc;
  if (d.dtype == OCTO_DTYPE_F32)
    return d.head_dim == 64 ? bwd_simt_t<float, 64>(p, Hq, q, k, v, o, lse, dout, dq, dk, dv, scale, ws, s)
                            : bwd_simt_t<float, 128>(p, Hq, q, k, v, o, lse, dout, dq, dk, dv, scale, ws, s);
  return d.head_dim == 64 ? bwd_simt_t<__nv_bfloat16, 64>(p, Hq, q, k, v, o, lse, dout, dq, dk, dv, scale, ws, s)
                          : bwd_simt_t<__nv_bfloat16, 128>(p, Hq, q, k, v, o, lse, dout, dq, dk, dv, scale, ws, s);
}

}  // namespace octo
