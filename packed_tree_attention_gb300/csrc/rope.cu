// Rotary position embedding at the packed positions.
//
// Octopus project page, "Architecture & Co-Design" item 02: mounted sibling KV is read
// "rotation-free" under the monotonic position offset s = max(p_B, e_A + 1).  Keys are
// rotated once, at the position the pool gives each token when it is appended, and a
// mount reads them as stored; a query is rotated at its own row's position.  The reader's
// position jump therefore shows up in every query-key angle, and without it a longer
// sibling's keys would sit at or after the reader's queries (the results table's "RoPE
// flip" for unshifted zero-copy KV).
//
// Rotation: the usual half-split form.  For head vector x (dimension d) at position p and
// i < d/2, (x_i, x_{i+d/2}) turns by the angle p * base^(-2i/d).  The angle is formed and
// reduced modulo 2 pi in double precision (positions reach the hundreds of thousands, where
// a float product loses the angle), then its sine and cosine are taken in float.
//
// Entry points (see include/octopus.h): rows of a plan in place (queries forward, their
// gradients with the inverse rotation), keys while they are appended, and key gradients in
// the pool's layout (inverse rotation at each slot's token position).

#include <cuda_bf16.h>

#include <cmath>
#include <vector>

#include "internal.h"

namespace octo {

struct RopeFreq {
  double inv[64];   // base^(-2i/d), i < d/2
  int32_t half;     // d / 2
};

int rope_validate(int32_t d, float base) {
  return (d < 2 || d > 128 || (d & 1) || !(base > 0.f) || !std::isfinite(base)) ? OCTO_EINVAL : OCTO_OK;
}

int rope_freq(int32_t d, float base, RopeFreq* f) {
  if (int st = rope_validate(d, base)) return st;
  f->half = d / 2;
  for (int i = 0; i < 64; i++) f->inv[i] = i < f->half ? std::pow((double)base, -2.0 * i / d) : 0.0;
  return OCTO_OK;
}

namespace {

__device__ __forceinline__ void rope_cs(int32_t pos, double inv, float& c, float& s) {
  const double ang = (double)pos * inv;
  const double r = ang - 6.283185307179586476925 * rint(ang * 0.15915494309189533576888);
  sincosf((float)r, &s, &c);
}

__device__ __forceinline__ float ld(const float* p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st(float* p, float v) { *p = v; }
__device__ __forceinline__ void st(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Four rows per block: the rows' d/2 (cos, sin) pairs once (one thread per pair), then
// every head of the rows.  sgn = -1 turns the other way (the inverse rotation, for
// gradients).  When d/2 is a multiple of the 16-byte vector width and x is 16-byte aligned,
// each thread takes a 16-byte vector from both halves (8 bf16 or 4 fp32 pairs).
constexpr int kRopeRows = 4;

template <typename T>
struct Vec16;
template <>
struct Vec16<float> {
  static constexpr int W = 4;
  __device__ static void unpack(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y); f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  __device__ static uint4 pack(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
};
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int W = 8;
  __device__ static void unpack(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      f[2 * i] = a.x;
      f[2 * i + 1] = a.y;
    }
  }
  __device__ static uint4 pack(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const __nv_bfloat162 a = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&a);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <typename T>
__global__ void __launch_bounds__(256) k_rope_rows(T* __restrict__ x, const int32_t* __restrict__ row_pos,
                                                   int64_t n_rows, int32_t H, RopeFreq f, float sgn, bool vec) {
  __shared__ float cs[kRopeRows][64][2];
  const int64_t row0 = (int64_t)blockIdx.x * kRopeRows;
  const int32_t half = f.half, d = 2 * half;
  const int nr = (int)min((int64_t)kRopeRows, n_rows - row0);
  {
    const int r = threadIdx.x / 64, i = threadIdx.x % 64;
    if (r < nr && i < half) rope_cs(row_pos[row0 + r], f.inv[i], cs[r][i][0], cs[r][i][1]);
  }
  __syncthreads();
  if (vec) {
    constexpr int W = Vec16<T>::W;
    const int32_t qv = half / W;        // vectors per half head
    const int32_t per_row = H * qv;
    for (int32_t e = threadIdx.x; e < nr * per_row; e += blockDim.x) {
      const int r = e / per_row, h = (e % per_row) / qv, i0 = (e % qv) * W;
      T* xr = x + (row0 + r) * H * d + (size_t)h * d;
      uint4* pa = reinterpret_cast<uint4*>(xr + i0);
      uint4* pb = reinterpret_cast<uint4*>(xr + i0 + half);
      float a[W], b[W], ya[W], yb[W];
      Vec16<T>::unpack(*pa, a);
      Vec16<T>::unpack(*pb, b);
#pragma unroll
      for (int t = 0; t < W; t++) {
        const float c = cs[r][i0 + t][0], sn = sgn * cs[r][i0 + t][1];
        ya[t] = a[t] * c - b[t] * sn;
        yb[t] = b[t] * c + a[t] * sn;
      }
      *pa = Vec16<T>::pack(ya);
      *pb = Vec16<T>::pack(yb);
    }
    return;
  }
  for (int32_t e = threadIdx.x; e < nr * H * half; e += blockDim.x) {
    const int r = e / (H * half), h = (e % (H * half)) / half, i = e % half;
    T* p = x + (row0 + r) * H * d + (size_t)h * d + i;
    const float a = ld(p), b = ld(p + half);
    const float c = cs[r][i][0], sn = sgn * cs[r][i][1];
    st(p, a * c - b * sn);
    st(p + half, b * c + a * sn);
  }
}

// One block per appended token: V copied, K rotated at the token's position.
template <typename T>
__global__ void k_append_rope(T* __restrict__ kp, T* __restrict__ vp, const T* __restrict__ k,
                              const T* __restrict__ v, const int32_t* __restrict__ dst,
                              const int32_t* __restrict__ pos, int32_t Hkv, int32_t P, RopeFreq f) {
  __shared__ float cs[64][2];
  const int32_t i = blockIdx.x;
  const int32_t half = f.half, d = 2 * half;
  if (threadIdx.x < half) rope_cs(pos[i], f.inv[threadIdx.x], cs[threadIdx.x][0], cs[threadIdx.x][1]);
  __syncthreads();
  const int32_t page = dst[i] / P, slot = dst[i] % P;
  for (int32_t e = threadIdx.x; e < Hkv * half; e += blockDim.x) {
    const int32_t g = e / half, j = e % half;
    const size_t o = (((size_t)page * Hkv + g) * P + slot) * d + j;
    const size_t src = ((size_t)i * Hkv + g) * d + j;
    const float a = ld(k + src), b = ld(k + src + half);
    st(kp + o, a * cs[j][0] - b * cs[j][1]);
    st(kp + o + half, b * cs[j][0] + a * cs[j][1]);
    vp[o] = v[src];
    vp[o + half] = v[src + half];
  }
}

// One block per (touched page, slot): every kv head's key gradient at that slot turns back
// by the slot's token position (slots holding no token are left as they are).
__global__ void k_rope_pool_grad(float* __restrict__ dk, const int32_t* __restrict__ touched,
                                 const int32_t* __restrict__ slot_pos, int32_t Hkv, int32_t P, RopeFreq f) {
  __shared__ float cs[64][2];
  const int32_t page = touched[blockIdx.x / P], slot = blockIdx.x % P;
  const int32_t pos = slot_pos[(size_t)page * P + slot];
  if (pos < 0) return;
  const int32_t half = f.half, d = 2 * half;
  if (threadIdx.x < half) rope_cs(pos, f.inv[threadIdx.x], cs[threadIdx.x][0], cs[threadIdx.x][1]);
  __syncthreads();
  for (int32_t e = threadIdx.x; e < Hkv * half; e += blockDim.x) {
    const int32_t g = e / half, j = e % half;
    float* p = dk + (((size_t)page * Hkv + g) * P + slot) * d + j;
    const float a = p[0], b = p[half];
    p[0] = a * cs[j][0] + b * cs[j][1];
    p[half] = b * cs[j][0] - a * cs[j][1];
  }
}

}  // namespace

int launch_append_rope(const octo_pool_desc& d, const int32_t* d_dst, const int32_t* d_pos, int32_t n,
                       const void* k, const void* v, float base, cudaStream_t s) {
  if (n <= 0) return OCTO_OK;
  RopeFreq f;
  if (int st = rope_freq(d.head_dim, base, &f)) return st;
  if (d.dtype == OCTO_DTYPE_F32)
    k_append_rope<float><<<n, 128, 0, s>>>((float*)d.k_pool, (float*)d.v_pool, (const float*)k, (const float*)v,
                                           d_dst, d_pos, d.n_kv_heads, d.page_size, f);
  else
    k_append_rope<__nv_bfloat16><<<n, 128, 0, s>>>((__nv_bfloat16*)d.k_pool, (__nv_bfloat16*)d.v_pool,
                                                   (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, d_dst, d_pos,
                                                   d.n_kv_heads, d.page_size, f);
  count_launch();
  return cuda_status(cudaGetLastError());
}

}  // namespace octo

extern "C" {

int octo_rope_rows(octo_plan_t plan, int32_t n_heads, void* x, int32_t dtype, float base, int32_t inverse,
                   void* stream) {
  if (!plan || n_heads <= 0 || n_heads > 65535) return OCTO_EINVAL;
  if (dtype != OCTO_DTYPE_F32 && dtype != OCTO_DTYPE_BF16) return OCTO_EINVAL;
  octo::RopeFreq f;
  if (int st = octo::rope_freq(plan->pool->desc.head_dim, base, &f)) return st;
  const int64_t N = plan->info.n_rows;
  if (N == 0) return OCTO_OK;
  if (!x) return OCTO_EINVAL;
  cudaStream_t s = (cudaStream_t)stream;
  plan->last_stream = s;
  const float sgn = inverse ? -1.f : 1.f;
  const unsigned grid = (unsigned)((N + octo::kRopeRows - 1) / octo::kRopeRows);
  if (dtype == OCTO_DTYPE_F32) {
    const bool vec = (f.half % 4) == 0 && ((uintptr_t)x % 16) == 0;
    octo::k_rope_rows<float><<<grid, 256, 0, s>>>((float*)x, plan->row_pos, N, n_heads, f, sgn, vec);
  } else {
    const bool vec = (f.half % 8) == 0 && ((uintptr_t)x % 16) == 0;
    octo::k_rope_rows<__nv_bfloat16><<<grid, 256, 0, s>>>((__nv_bfloat16*)x, plan->row_pos, N, n_heads, f, sgn,
                                                          vec);
  }
  octo::count_launch();
  return octo::cuda_status(cudaGetLastError());
}

int octo_rope_pool_grad(octo_plan_t plan, float* dk_pool, float base, void* stream) {
  if (!plan || plan->info.is_decode) return OCTO_EINVAL;
  const octo_pool_desc& d = plan->pool->desc;
  octo::RopeFreq f;
  if (int st = octo::rope_freq(d.head_dim, base, &f)) return st;
  const int32_t n_touched = plan->info.n_touched_pages;
  if (n_touched == 0) return OCTO_OK;
  if (!dk_pool) return OCTO_EINVAL;
  // token position of every slot of every page a live segment owns (-1: no token)
  const int32_t P = d.page_size;
  std::vector<int32_t> slot_pos((size_t)d.num_pages * P, -1);
  for (const octo::Segment& g : plan->pool->segs) {
    if (g.freed) continue;
    for (int32_t t = 0; t < g.len; t++) slot_pos[(size_t)g.pages[t / P] * P + t % P] = g.pos[t];
  }
  cudaStream_t s = (cudaStream_t)stream;
  plan->last_stream = s;
  int32_t* d_pos = nullptr;
  OCTO_CUDA(cudaMallocAsync((void**)&d_pos, slot_pos.size() * sizeof(int32_t), s));
  OCTO_CUDA(cudaMemcpyAsync(d_pos, slot_pos.data(), slot_pos.size() * sizeof(int32_t), cudaMemcpyHostToDevice, s));
  octo::k_rope_pool_grad<<<(unsigned)((int64_t)n_touched * P), 128, 0, s>>>(dk_pool, plan->touched, d_pos,
                                                                             d.n_kv_heads, P, f);
  octo::count_launch();
  const int st = octo::cuda_status(cudaGetLastError());
  OCTO_CUDA(cudaFreeAsync(d_pos, s));
  // the host vector is pageable: make sure the copy has consumed it
  OCTO_CUDA(cudaStreamSynchronize(s));
  return st;
}

}  // extern "C"
