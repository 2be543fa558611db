// Tree-packed recurrent layer: the gated delta rule over the packed episode DAG.
//
// ia.com.br summary, associative versus working memory: the hybrid model's linear-recurrent
// layers (Gated DeltaNet / Mamba-2) keep the branch's working memory as a state h.  Octopus
// project page, five-primitives table: fork clones the recurrent checkpoint at the fork
// point, rewind restores the exact state of step k, and read_thread mounts a sibling's KV
// into the attention layers only -- the recurrent layers skip the span; "Architecture &
// Co-Design" item 03: the packed pass compiles the trees together with the recurrent
// boundary checkpoints.
//
// Per head, with state S [D x D] (rows: value dimension, columns: key dimension):
//     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,    o_t = S_t q_t,
// where S_{t-1} is the state after the row before t on its path (mounted spans never
// enter), and a path start begins from S = 0.  The plan cuts the packed rows into runs (a
// run starts from one row's state and no row inside it feeds another run) and the runs
// into chunks of C = 64 rows.  Within a chunk, with lg the running sum of log alpha,
// g = exp(lg), G_ts = exp(lg_t - lg_s), A = strict lower part of G o K K^T,
// Minv = (I + diag(beta) A)^-1 and T = Minv diag(beta):
//     W = T diag(g) K,  U = T V,  Delta = U - W S0^T,
//     O = diag(g) Q S0^T + tril(G o Q K^T) Delta,
//     S_end = g_C S0 + Delta^T diag(g_C / g) K.
// The backward runs the same way in reverse: the gradient G_C with respect to a chunk's end
// state gives the one at its start as
//     G_0 = g_C G_C - (G_C K^T diag(g_C / g)) W + dO^T E,   E = diag(g) Q - tril(G o Q K^T) W,
// and, per chunk, the gradients of q, k, v, alpha, beta follow from S0, G_C and the chunk's
// rows (k_rec_grad_a / k_rec_grad_b).  A run's end gradient is the sum, in run order, of the
// start gradients of the runs continuing from its last row: a fork or rewind point feeds
// several.  The sequential parts (chunk to chunk inside a run) go one launch per run level,
// every run of a level, head and 32-row block of the state in parallel.
//
// Everything is fp32 on the CUDA cores: each CTA does its chunk's products from shared
// memory with 256 threads, a thread owning an 8-row x (D / 32)-column tile of a C x D result.

#include <algorithm>
#include <cmath>

#include "internal.h"

namespace octo {
namespace {

constexpr int kC = kRecChunk;     // 64 rows per chunk
constexpr int kT = 256;           // threads per CTA
constexpr int kLC = kC + 4;       // row length of C x C matrices in shared memory
constexpr int kL32 = 36;          // row length of C x 32 column blocks in shared memory

struct RecParams {
  const float *q, *k, *v, *alpha, *beta, *dout;
  float *o, *dq, *dk, *dv, *dalpha, *dbeta;
  const int32_t* run_info;   // [n_runs][4] r0, r1, predecessor run, first chunk
  const int32_t* child_off;
  const int32_t* child;
  const int32_t* level_runs;
  const int32_t* chunk_info;   // [n_chunks][2] first row, rows
  int32_t H;
  // workspace: saved by the forward for the backward
  float* S0;       // [chunk][h][D][D] state at the chunk's start
  float* Wb;       // [chunk][h][C][D]
  float* Db;       // [chunk][h][C][D] Delta
  float* Mb;       // [chunk][h][C][C] Minv
  float* Lb;       // [chunk][h][C] lg
  float* run_end;  // [run][h][D][D] state after the run's last row
  // workspace: temporaries
  float* Ub;       // [chunk][h][C][D] U (forward), E (backward)
  float* Gb;       // [chunk][h][D][D] gradient with respect to the chunk's end state
  float* Yb;       // [chunk][h][C][D]
  float* Sc;       // [chunk][h][3][C] per-row dlg parts g * dg and r, then <G_C, S0> at [2][0]
  float* run_grad; // [run][h][D][D] gradient with respect to the run's start state
};

// Shared-memory tiles keep rows 16-byte aligned with a length of 4 mod 32 floats: 16-byte
// reads along a row are then free of bank conflicts both when every lane reads the same
// row (a broadcast) and when the lanes read 32 different rows at the same column.
template <int D>
struct Lay {
  static constexpr int LD = D + 4;   // row length of C x D and 32 x D tiles
  static constexpr int NC = D / 32;  // columns per thread of a C x D result
};

__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// 16-byte global -> shared copy without the registers (zero-filled when !valid)
__device__ __forceinline__ void cp16(float* dst, const float* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr(dst)), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
}
// closes the group of this thread's copies issued since the last commit
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// waits until at most N of this thread's committed groups are still in flight
template <int N>
__device__ __forceinline__ void cp_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// rows [row0, row0 + rows) of x [N][H][D] at head h into dst [C][LD]; zeros past `rows`
template <int D>
__device__ __forceinline__ void cp_rows(float* dst, const float* __restrict__ x, int64_t row0, int rows, int H, int h) {
  constexpr int Q = D / 4;
  for (int i = threadIdx.x; i < kC * Q; i += kT) {
    const int t = i / Q, c = (i % Q) * 4;
    const bool ok = t < rows;
    cp16(dst + t * Lay<D>::LD + c, ok ? x + ((row0 + t) * H + h) * D + c : x, ok);
  }
}
// columns [j0, j0 + 32) of the same rows into dst [C][kL32]
template <int D>
__device__ __forceinline__ void cp_rows32(float* dst, const float* __restrict__ x, int64_t row0, int rows, int H,
                                          int h, int j0) {
  for (int i = threadIdx.x; i < kC * 8; i += kT) {
    const int t = i >> 3, c = (i & 7) * 4;
    const bool ok = t < rows;
    cp16(dst + t * kL32 + c, ok ? x + ((row0 + t) * H + h) * D + j0 + c : x, ok);
  }
}
// a dense [R][D] block into dst [R][LD] (R = C, or 32 rows j0.. of a [D][D] state)
template <int D, int R = kC>
__device__ __forceinline__ void cp_blk(float* dst, const float* __restrict__ src) {
  constexpr int Q = D / 4;
  for (int i = threadIdx.x; i < R * Q; i += kT) cp16(dst + (i / Q) * Lay<D>::LD + (i % Q) * 4, src + i * 4, true);
}
// columns [j0, j0 + 32) of a dense [R][D] block into dst [R][kL32] (R = C, or all D rows
// of a [D][D] state)
template <int D, int R = kC>
__device__ __forceinline__ void cp_blk32(float* dst, const float* __restrict__ src, int j0) {
  for (int i = threadIdx.x; i < R * 8; i += kT) cp16(dst + (i >> 3) * kL32 + (i & 7) * 4, src + (i >> 3) * D + j0 + (i & 7) * 4, true);
}
// a dense [C][C] block into dst [C][kLC]
__device__ __forceinline__ void cp_cc(float* dst, const float* __restrict__ src) {
  for (int i = threadIdx.x; i < kC * kC / 4; i += kT) cp16(dst + (i / 16) * kLC + (i % 16) * 4, src + i * 4, true);
}

// acc[r][c] += sum_k A[i0 + r][k] B[k][j0 + 32 c]      (A, B row-major; K % 4 == 0)
template <int R, int NC>
__device__ __forceinline__ void mm_nn(float (&acc)[R][NC], const float* A, int lda, const float* B, int ldb, int K,
                                      int i0, int j0) {
#pragma unroll 2
  for (int k = 0; k < K; k += 4) {
    float4 a[R];
#pragma unroll
    for (int r = 0; r < R; r++) a[r] = *reinterpret_cast<const float4*>(A + (i0 + r) * lda + k);
#pragma unroll
    for (int kk = 0; kk < 4; kk++) {
      float b[NC];
#pragma unroll
      for (int c = 0; c < NC; c++) b[c] = B[(k + kk) * ldb + j0 + 32 * c];
#pragma unroll
      for (int r = 0; r < R; r++) {
        const float av = kk == 0 ? a[r].x : kk == 1 ? a[r].y : kk == 2 ? a[r].z : a[r].w;
#pragma unroll
        for (int c = 0; c < NC; c++) acc[r][c] = fmaf(av, b[c], acc[r][c]);
      }
    }
  }
}

// component kk of a float4 (kk a compile-time constant after unrolling)
__device__ __forceinline__ float f4c(const float4& v, int kk) {
  return kk == 0 ? v.x : kk == 1 ? v.y : kk == 2 ? v.z : v.w;
}

// acc[r][c] += sum_k A[i0 + SI r][k] B[j0 + SJ c][k]      (B read by rows: a product with B^T)
template <int R, int NC, int SI = 1, int SJ = 32>
__device__ __forceinline__ void mm_nt(float (&acc)[R][NC], const float* A, int lda, const float* B, int ldb, int K,
                                      int i0, int j0) {
#pragma unroll 2
  for (int k = 0; k < K; k += 4) {
    float4 a[R], b[NC];
#pragma unroll
    for (int r = 0; r < R; r++) a[r] = *reinterpret_cast<const float4*>(A + (i0 + SI * r) * lda + k);
#pragma unroll
    for (int c = 0; c < NC; c++) b[c] = *reinterpret_cast<const float4*>(B + (j0 + SJ * c) * ldb + k);
    // one component of the 4-step at a time: consecutive FMAs update different accumulators
#pragma unroll
    for (int kk = 0; kk < 4; kk++)
#pragma unroll
      for (int r = 0; r < R; r++)
#pragma unroll
        for (int c = 0; c < NC; c++) acc[r][c] = fmaf(f4c(a[r], kk), f4c(b[c], kk), acc[r][c]);
  }
}

// acc[r][c] += sum_k A[k][i0 + r] B[k][j0 + 32 c]      (A read by columns: a product with A^T;
// i0 % 4 == 0)
template <int R, int NC>
__device__ __forceinline__ void mm_tn(float (&acc)[R][NC], const float* A, int lda, const float* B, int ldb, int K,
                                      int i0, int j0) {
#pragma unroll 4
  for (int k = 0; k < K; k++) {
    float a[R], b[NC];
#pragma unroll
    for (int r = 0; r < R; r += 4) {
      const float4 x = *reinterpret_cast<const float4*>(A + k * lda + i0 + r);
      a[r] = x.x;
      a[r + 1] = x.y;
      a[r + 2] = x.z;
      a[r + 3] = x.w;
    }
#pragma unroll
    for (int c = 0; c < NC; c++) b[c] = B[k * ldb + j0 + 32 * c];
#pragma unroll
    for (int r = 0; r < R; r++)
#pragma unroll
      for (int c = 0; c < NC; c++) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
  }
}

// N consecutive floats (N = 2 or 4, 8- or 16-byte aligned) in one shared-memory read
template <int N>
__device__ __forceinline__ void ldv(float (&x)[N], const float* p) {
  static_assert(N == 2 || N == 4, "vector width");
  if constexpr (N == 4) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
  } else {
    const float2 v = *reinterpret_cast<const float2*>(p);
    x[0] = v.x, x[1] = v.y;
  }
}

// acc[r][c] += sum_k A[k][i0 + r] B[k][j0 + c]: a thread's rows and columns are consecutive,
// each read as one vector (a 2-D warp tile: lanes split both rows and columns)
template <int R, int NC>
__device__ __forceinline__ void mm_tn_v(float (&acc)[R][NC], const float* A, int lda, const float* B, int ldb, int K,
                                        int i0, int j0) {
#pragma unroll 4
  for (int k = 0; k < K; k++) {
    float a[R], b[NC];
    ldv<R>(a, A + k * lda + i0);
    ldv<NC>(b, B + k * ldb + j0);
#pragma unroll
    for (int r = 0; r < R; r++)
#pragma unroll
      for (int c = 0; c < NC; c++) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
  }
}

// Two products that share one operand, which is then read from shared memory once for
// both (half the shared-memory reads of that operand):
// acc1 += A1 B^T and acc2 += A2 B^T, as mm_nt
template <int R, int NC>
__device__ __forceinline__ void mm_nt2(float (&acc1)[R][NC], float (&acc2)[R][NC], const float* A1, const float* A2,
                                       int lda, const float* B, int ldb, int K, int i0, int j0) {
#pragma unroll 1
  for (int k = 0; k < K; k += 4) {
    float4 b[NC];
#pragma unroll
    for (int c = 0; c < NC; c++) b[c] = *reinterpret_cast<const float4*>(B + (j0 + 32 * c) * ldb + k);
#pragma unroll
    for (int u = 0; u < 2; u++) {
      const float* A = u ? A2 : A1;
      float(&acc)[R][NC] = u ? acc2 : acc1;
      float4 a[R];
#pragma unroll
      for (int r = 0; r < R; r++) a[r] = *reinterpret_cast<const float4*>(A + (i0 + r) * lda + k);
#pragma unroll
      for (int kk = 0; kk < 4; kk++)
#pragma unroll
        for (int r = 0; r < R; r++)
#pragma unroll
          for (int c = 0; c < NC; c++) acc[r][c] = fmaf(f4c(a[r], kk), f4c(b[c], kk), acc[r][c]);
    }
  }
}

// acc1 += A1 B and acc2 += A2 B, as mm_nn
template <int R, int NC>
__device__ __forceinline__ void mm_nn2(float (&acc1)[R][NC], float (&acc2)[R][NC], const float* A1, const float* A2,
                                       int lda, const float* B, int ldb, int K, int i0, int j0) {
#pragma unroll 1
  for (int k = 0; k < K; k += 4) {
    float4 a1[R], a2[R];
#pragma unroll
    for (int r = 0; r < R; r++) {
      a1[r] = *reinterpret_cast<const float4*>(A1 + (i0 + r) * lda + k);
      a2[r] = *reinterpret_cast<const float4*>(A2 + (i0 + r) * lda + k);
    }
#pragma unroll
    for (int kk = 0; kk < 4; kk++) {
      float b[NC];
#pragma unroll
      for (int c = 0; c < NC; c++) b[c] = B[(k + kk) * ldb + j0 + 32 * c];
#pragma unroll
      for (int r = 0; r < R; r++) {
        const float x1 = kk == 0 ? a1[r].x : kk == 1 ? a1[r].y : kk == 2 ? a1[r].z : a1[r].w;
        const float x2 = kk == 0 ? a2[r].x : kk == 1 ? a2[r].y : kk == 2 ? a2[r].z : a2[r].w;
#pragma unroll
        for (int c = 0; c < NC; c++) {
          acc1[r][c] = fmaf(x1, b[c], acc1[r][c]);
          acc2[r][c] = fmaf(x2, b[c], acc2[r][c]);
        }
      }
    }
  }
}

// acc1 += A B1 and acc2 += A B2, as mm_nn
template <int R, int NC>
__device__ __forceinline__ void mm_nn_b2(float (&acc1)[R][NC], float (&acc2)[R][NC], const float* A, int lda,
                                         const float* B1, const float* B2, int ldb, int K, int i0, int j0) {
#pragma unroll 1
  for (int k = 0; k < K; k += 4) {
    float4 a[R];
#pragma unroll
    for (int r = 0; r < R; r++) a[r] = *reinterpret_cast<const float4*>(A + (i0 + r) * lda + k);
#pragma unroll
    for (int kk = 0; kk < 4; kk++) {
      float b1[NC], b2[NC];
#pragma unroll
      for (int c = 0; c < NC; c++) {
        b1[c] = B1[(k + kk) * ldb + j0 + 32 * c];
        b2[c] = B2[(k + kk) * ldb + j0 + 32 * c];
      }
#pragma unroll
      for (int r = 0; r < R; r++) {
        const float x = kk == 0 ? a[r].x : kk == 1 ? a[r].y : kk == 2 ? a[r].z : a[r].w;
#pragma unroll
        for (int c = 0; c < NC; c++) {
          acc1[r][c] = fmaf(x, b1[c], acc1[r][c]);
          acc2[r][c] = fmaf(x, b2[c], acc2[r][c]);
        }
      }
    }
  }
}

template <int R, int NC>
__device__ __forceinline__ void zero(float (&acc)[R][NC]) {
#pragma unroll
  for (int r = 0; r < R; r++)
#pragma unroll
    for (int c = 0; c < NC; c++) acc[r][c] = 0.f;
}

// per-row gate values of one chunk: lg (running sum of log alpha), beta, rows past the end
// get alpha = 1, beta = 0 (no effect).  Ends with a block barrier.
__device__ __forceinline__ void load_gates(float* lg, float* be, float* al, const float* __restrict__ alpha,
                                           const float* __restrict__ beta, int64_t row0, int rows, int H, int h) {
  __shared__ float warp_tot;
  const int t = threadIdx.x;
  float x = 0.f;
  if (t < kC) {
    const float a = t < rows ? alpha[(row0 + t) * H + h] : 1.f;
    al[t] = a;
    be[t] = t < rows ? beta[(row0 + t) * H + h] : 0.f;
    x = logf(a);
    // inclusive running sum within the warp (rows 0-31, 32-63)
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if ((t & 31) >= o) x += y;
    }
    if (t == 31) warp_tot = x;
  }
  __syncthreads();
  if (t < kC) lg[t] = t >= 32 ? x + warp_tot : x;
  __syncthreads();
}

// C x C product into registers: acc (8 rows x 2 columns per thread) = sum_k X[i][k] Y[j][k]
template <int D>
__device__ __forceinline__ void gram(float (&acc)[8][2], const float* X, const float* Y) {
  zero(acc);
  mm_nt(acc, X, Lay<D>::LD, Y, Lay<D>::LD, D, (threadIdx.x >> 5) * 8, threadIdx.x & 31);
}
// The same product with a 2-D warp tile: warp w a 16 x 32 block of the C x C result, the
// thread rows gram_row(r) and columns gram_col(c) (a quarter of the operand reads of gram)
__device__ __forceinline__ int gram_row(int r) { return 16 * (threadIdx.x >> 6) + ((threadIdx.x >> 3) & 3) + 4 * r; }
__device__ __forceinline__ int gram_col(int c) { return 32 * ((threadIdx.x >> 5) & 1) + (threadIdx.x & 7) + 8 * c; }
template <int D>
__device__ __forceinline__ void gram_w(float (&acc)[4][4], const float* X, const float* Y) {
  zero(acc);
  mm_nt<4, 4, 4, 8>(acc, X, Lay<D>::LD, Y, Lay<D>::LD, D, gram_row(0), gram_col(0));
}
// two of them with the same Y
template <int D>
__device__ __forceinline__ void gram2(float (&acc1)[8][2], float (&acc2)[8][2], const float* X1, const float* X2,
                                      const float* Y) {
  zero(acc1);
  zero(acc2);
  mm_nt2(acc1, acc2, X1, X2, Lay<D>::LD, Y, Lay<D>::LD, D, (threadIdx.x >> 5) * 8, threadIdx.x & 31);
}

// =====================================================================================
// forward
// =====================================================================================

// Per chunk and head: lg, Minv = (I + diag(beta) A)^-1, W = Minv diag(beta g) K and
// U = Minv diag(beta) V.
template <int D>
__global__ void __launch_bounds__(kT) k_rec_prep(RecParams p) {
  constexpr int LD = Lay<D>::LD, NC = Lay<D>::NC;
  extern __shared__ __align__(16) float sm[];
  float* sK = sm;
  float* sV = sK + kC * LD;
  float* sA = sV + kC * LD;
  float* sMi = sA + kC * kLC;
  float* lg = sMi + kC * kLC;
  float* be = lg + kC;
  float* al = be + kC;
  const int ch = blockIdx.x / p.H, h = blockIdx.x % p.H;
  const int64_t row0 = p.chunk_info[2 * ch];
  const int rows = p.chunk_info[2 * ch + 1];
  const size_t blk = (size_t)ch * p.H + h;
  const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
  cp_rows<D>(sK, p.k, row0, rows, p.H, h);
  cp_rows<D>(sV, p.v, row0, rows, p.H, h);
  for (int i = threadIdx.x; i < kC * kLC; i += kT) sMi[i] = 0.f;
  load_gates(lg, be, al, p.alpha, p.beta, row0, rows, p.H, h);
  cp_wait();
  __syncthreads();
  {
    float acc[4][4];
    gram_w<D>(acc, sK, sK);
#pragma unroll
    for (int r = 0; r < 4; r++)
#pragma unroll
      for (int c = 0; c < 4; c++) {
        const int t = gram_row(r), s = gram_col(c);
        sA[t * kLC + s] = s < t ? expf(lg[t] - lg[s]) * acc[r][c] : 0.f;
      }
  }
  __syncthreads();
  // forward substitution, a column of Minv per thread (columns are independent):
  //   Minv[t][s] = [t == s] - beta_t sum_{u < t} A[t][u] Minv[u][s], Minv[u][s] = 0 for u < s;
  // every lane walks the same t and u, so the reads of A are broadcasts
  if (threadIdx.x < kC) {
    const int s = threadIdx.x;
    for (int t = 0; t < kC; t++) {
      float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;   // four chains for the FMA latency
      int u = 0;
      for (; u + 4 <= t; u += 4) {
        x0 = fmaf(sA[t * kLC + u], sMi[u * kLC + s], x0);
        x1 = fmaf(sA[t * kLC + u + 1], sMi[(u + 1) * kLC + s], x1);
        x2 = fmaf(sA[t * kLC + u + 2], sMi[(u + 2) * kLC + s], x2);
        x3 = fmaf(sA[t * kLC + u + 3], sMi[(u + 3) * kLC + s], x3);
      }
      for (; u < t; u++) x0 = fmaf(sA[t * kLC + u], sMi[u * kLC + s], x0);
      const float x = (x0 + x1) + (x2 + x3);
      sMi[t * kLC + s] = (s == t ? 1.f : 0.f) - (t > s ? be[t] * x : 0.f);
    }
  }
  __syncthreads();
  // rows of K scaled by beta g, of V by beta
  if (threadIdx.x < kC) al[threadIdx.x] = be[threadIdx.x] * expf(lg[threadIdx.x]);   // alpha is not needed here
  __syncthreads();
  for (int i = threadIdx.x; i < kC * D; i += kT) {
    const int t = i / D, c = i % D;
    sK[t * LD + c] *= al[t];
    sV[t * LD + c] *= be[t];
  }
  __syncthreads();
  float w[8][NC], u[8][NC];
  zero(w);
  zero(u);
  mm_nn_b2(w, u, sMi, kLC, sK, sV, LD, kC, ty * 8, tx);
  float* Wg = p.Wb + blk * kC * D;
  float* Ug = p.Ub + blk * kC * D;
#pragma unroll
  for (int r = 0; r < 8; r++)
#pragma unroll
    for (int c = 0; c < NC; c++) {
      Wg[(ty * 8 + r) * D + tx + 32 * c] = w[r][c];
      Ug[(ty * 8 + r) * D + tx + 32 * c] = u[r][c];
    }
  float* Mg = p.Mb + blk * kC * kC;
  for (int i = threadIdx.x; i < kC * kC; i += kT) Mg[i] = sMi[(i / kC) * kLC + i % kC];
  if (threadIdx.x < kC) p.Lb[blk * kC + threadIdx.x] = lg[threadIdx.x];
}

// The state passed chunk to chunk along the runs of one level: one CTA per (run, head,
// 32-row block of S).  Per chunk: S0 saved, Delta = U - W S0^T (saved),
// S = g_C S0 + Delta^T diag(g_C / g) K; at the run's end S is saved for the runs that
// continue from it.  Both products use 2-D warp tiles (lanes split rows and columns, so a
// warp reads a 16 x 16 or 16 x d/4 block of operands, not all columns of one of them).
template <int D>
__global__ void __launch_bounds__(kT) k_rec_scan_fwd(RecParams p, int32_t lvl0) {
  // single buffers (94 KB of shared memory: two CTAs share an SM), filled ahead all the
  // same: the next chunk's W arrives during this chunk's second product, its U, lg and K
  // during the next first product
  constexpr int LD = Lay<D>::LD, NB = D / 32, NV = D / 32;
  extern __shared__ __align__(16) float sm[];
  float* sW = sm;
  float* sK = sW + kC * LD;
  float* sS = sK + kC * LD;          // [32][LD]
  float* sU = sS + 32 * LD;          // [C][kL32]: U, then Delta (scaled by g_C / g)
  float* lg = sU + kC * kL32;
  const int li = blockIdx.x / (p.H * NB), h = (blockIdx.x / NB) % p.H, jb = blockIdx.x % NB;
  const int run = p.level_runs[lvl0 + li];
  const int32_t r0 = p.run_info[4 * run], r1 = p.run_info[4 * run + 1];
  const int32_t pr = p.run_info[4 * run + 2], c0 = p.run_info[4 * run + 3];
  const int nch = (r1 - r0 + kC - 1) / kC;
  const int w = threadIdx.x >> 5, ly = (threadIdx.x >> 3) & 3, lx = threadIdx.x & 7;
  const int j0 = jb * 32;
  // first product, Delta [C x 32]: warp (w >> 1, w & 1) a 16 x 16 block, rows 16 (w >> 1) +
  // ly + 4 r, columns 16 (w & 1) + lx + 8 c
  const int t1 = 16 * (w >> 1) + ly, s1 = 16 * (w & 1) + lx;
  // second product, S [32 x D]: warp (w >> 2, w & 3) a 16 x D/4 block, rows 16 (w >> 2) +
  // 4 ly + r, columns (D / 4) (w & 3) + NV lx + c
  const int j2 = 16 * (w >> 2) + 4 * ly, k2 = (D / 4) * (w & 3) + NV * lx;
  auto issue_w = [&](int ci) {
    cp_blk<D>(sW, p.Wb + ((size_t)(c0 + ci) * p.H + h) * kC * D);
    cp_commit();
  };
  auto issue_uk = [&](int ci) {
    const int ch = c0 + ci;
    const size_t blk = (size_t)ch * p.H + h;
    cp_blk32<D>(sU, p.Ub + blk * kC * D, j0);
    if (threadIdx.x < kC / 4) cp16(lg + threadIdx.x * 4, p.Lb + blk * kC + threadIdx.x * 4, true);
    cp_rows<D>(sK, p.k, p.chunk_info[2 * ch], p.chunk_info[2 * ch + 1], p.H, h);
    cp_commit();
  };
  if (pr >= 0)
    cp_blk<D, 32>(sS, p.run_end + ((size_t)pr * p.H + h) * D * D + (size_t)j0 * D);
  else
    for (int i = threadIdx.x; i < 32 * LD; i += kT) sS[i] = 0.f;
  if (nch > 0) {
    issue_w(0);   // with the start state
    issue_uk(0);
  } else {
    cp_commit();
  }
  for (int ci = 0; ci < nch; ci++) {
    const size_t blk = (size_t)(c0 + ci) * p.H + h;
    cp_wait_group<1>();   // W (and the start state)
    __syncthreads();
    float* S0g = p.S0 + blk * D * D + (size_t)j0 * D;
    for (int i = threadIdx.x; i < 32 * D / 4; i += kT)
      *reinterpret_cast<float4*>(S0g + i * 4) = *reinterpret_cast<const float4*>(sS + (i / (D / 4)) * LD + (i % (D / 4)) * 4);
    float acc[4][2];
    zero(acc);
    mm_nt<4, 2, 4, 8>(acc, sW, LD, sS, LD, D, t1, s1);   // (W S0^T)[t][j]
    cp_wait_group<0>();   // U, lg, K
    __syncthreads();      // every warp is past its reads of W
    if (ci + 1 < nch) issue_w(ci + 1);
    else cp_commit();
    {
      const float gC = lg[kC - 1];
      float* Dg = p.Db + blk * kC * D;
#pragma unroll
      for (int r = 0; r < 4; r++) {
        const int t = t1 + 4 * r;
        const float sc = expf(gC - lg[t]);
#pragma unroll
        for (int c = 0; c < 2; c++) {
          const int j = s1 + 8 * c;
          const float dl = sU[t * kL32 + j] - acc[r][c];
          Dg[t * D + j0 + j] = dl;
          sU[t * kL32 + j] = dl * sc;
        }
      }
    }
    __syncthreads();
    {
      float acc2[4][NV];
      zero(acc2);
      mm_tn_v(acc2, sU, kL32, sK, LD, kC, j2, k2);   // (Delta^T diag(g_C/g) K)[j][k]
      const float gC = expf(lg[kC - 1]);
#pragma unroll
      for (int r = 0; r < 4; r++)
#pragma unroll
        for (int c = 0; c < NV; c++) {
          float& x = sS[(j2 + r) * LD + k2 + c];
          x = fmaf(gC, x, acc2[r][c]);
        }
    }
    __syncthreads();      // U, lg, K read; S updated
    if (ci + 1 < nch) issue_uk(ci + 1);
    else cp_commit();
  }
  cp_wait_group<0>();
  __syncthreads();
  float* Eg = p.run_end + ((size_t)run * p.H + h) * D * D + (size_t)j0 * D;
  for (int i = threadIdx.x; i < 32 * D / 4; i += kT)
    *reinterpret_cast<float4*>(Eg + i * 4) = *reinterpret_cast<const float4*>(sS + (i / (D / 4)) * LD + (i % (D / 4)) * 4);
}

// Outputs per chunk and head: O = diag(g) Q S0^T + tril(G o Q K^T) Delta.  K's buffer takes
// Delta once the Q K^T block is formed.
template <int D>
__global__ void __launch_bounds__(kT) k_rec_out(RecParams p) {
  constexpr int LD = Lay<D>::LD, NC = Lay<D>::NC;
  extern __shared__ __align__(16) float sm[];
  float* sQ = sm;
  float* sKD = sQ + kC * LD;   // K, then Delta
  float* sS = sKD + kC * LD;   // [D][kL32] a 32-column block of S0
  float* sB = sS + D * kL32;   // [C][kLC]
  float* lg = sB + kC * kLC;
  const int ch = blockIdx.x / p.H, h = blockIdx.x % p.H;
  const int64_t row0 = p.chunk_info[2 * ch];
  const int rows = p.chunk_info[2 * ch + 1];
  const size_t blk = (size_t)ch * p.H + h;
  const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
  cp_rows<D>(sQ, p.q, row0, rows, p.H, h);
  cp_rows<D>(sKD, p.k, row0, rows, p.H, h);
  if (threadIdx.x < kC) lg[threadIdx.x] = p.Lb[blk * kC + threadIdx.x];
  cp_wait();
  __syncthreads();
  {
    float acc[4][4];
    gram_w<D>(acc, sQ, sKD);
#pragma unroll
    for (int r = 0; r < 4; r++)
#pragma unroll
      for (int c = 0; c < 4; c++) {
        const int t = gram_row(r), s = gram_col(c);
        sB[t * kLC + s] = s <= t ? expf(lg[t] - lg[s]) * acc[r][c] : 0.f;
      }
  }
  __syncthreads();
  cp_blk<D>(sKD, p.Db + blk * kC * D);
  const float* S0g = p.S0 + blk * D * D;
  // Q S0^T by 32-column blocks of the contraction, every block adding to all of out
  // (single-buffered: two CTAs share an SM)
  float out[8][NC];
  zero(out);
#pragma unroll 1
  for (int jd = 0; jd < NC; jd++) {
    if (jd) __syncthreads();
    cp_blk32<D, D>(sS, S0g, 32 * jd);
    cp_wait();
    __syncthreads();
    mm_nt(out, sQ + 32 * jd, LD, sS, kL32, 32, ty * 8, tx);
  }
#pragma unroll
  for (int r = 0; r < 8; r++) {
    const float g = expf(lg[ty * 8 + r]);
#pragma unroll
    for (int c = 0; c < NC; c++) out[r][c] *= g;
  }
  mm_nn(out, sB, kLC, sKD, LD, kC, ty * 8, tx);
#pragma unroll
  for (int r = 0; r < 8; r++) {
    const int t = ty * 8 + r;
    if (t < rows)
#pragma unroll
      for (int c = 0; c < NC; c++) p.o[((row0 + t) * p.H + h) * D + tx + 32 * c] = out[r][c];
  }
}

// =====================================================================================
// backward
// =====================================================================================

// E = diag(g) Q - tril(G o Q K^T) W per chunk and head (K's buffer then holds W).
template <int D>
__global__ void __launch_bounds__(kT) k_rec_prep_bwd(RecParams p) {
  constexpr int LD = Lay<D>::LD, NC = Lay<D>::NC;
  extern __shared__ __align__(16) float sm[];
  float* sQ = sm;
  float* sKW = sQ + kC * LD;
  float* sB = sKW + kC * LD;
  float* lg = sB + kC * kLC;
  const int ch = blockIdx.x / p.H, h = blockIdx.x % p.H;
  const int64_t row0 = p.chunk_info[2 * ch];
  const int rows = p.chunk_info[2 * ch + 1];
  const size_t blk = (size_t)ch * p.H + h;
  const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
  cp_rows<D>(sQ, p.q, row0, rows, p.H, h);
  cp_rows<D>(sKW, p.k, row0, rows, p.H, h);
  if (threadIdx.x < kC) lg[threadIdx.x] = p.Lb[blk * kC + threadIdx.x];
  cp_wait();
  __syncthreads();
  {
    float acc[4][4];
    gram_w<D>(acc, sQ, sKW);
#pragma unroll
    for (int r = 0; r < 4; r++)
#pragma unroll
      for (int c = 0; c < 4; c++) {
        const int t = gram_row(r), s = gram_col(c);
        sB[t * kLC + s] = s <= t ? -expf(lg[t] - lg[s]) * acc[r][c] : 0.f;
      }
  }
  __syncthreads();
  cp_blk<D>(sKW, p.Wb + blk * kC * D);
  cp_wait();
  __syncthreads();
  float e[8][NC];
#pragma unroll
  for (int r = 0; r < 8; r++) {
    const float g = expf(lg[ty * 8 + r]);
#pragma unroll
    for (int c = 0; c < NC; c++) e[r][c] = g * sQ[(ty * 8 + r) * LD + tx + 32 * c];
  }
  mm_nn(e, sB, kLC, sKW, LD, kC, ty * 8, tx);
  float* Eg = p.Ub + blk * kC * D;
#pragma unroll
  for (int r = 0; r < 8; r++)
#pragma unroll
    for (int c = 0; c < NC; c++) Eg[(ty * 8 + r) * D + tx + 32 * c] = e[r][c];
}

// The state gradient passed back chunk to chunk along the runs of one level (levels in
// decreasing order): one CTA per (run, head, 32-row block).  It starts from the sum of
// the start gradients of the runs continuing from the run's last row (in run order) and,
// per chunk from the last: saves it as the chunk's end gradient, then
// G = g_C G - (G K^T diag(g_C / g)) W + dO^T E.  The run's start gradient is saved.
template <int D>
__global__ void __launch_bounds__(kT) k_rec_scan_bwd(RecParams p, int32_t lvl0) {
  // 104 KB of shared memory, so two CTAs share an SM (the levels of many runs take two
  // rounds of CTAs, not three): one K buffer, refilled with the next chunk's K once this
  // chunk's G K^T is formed, and W and E brought in one column half at a time
  constexpr int LD = Lay<D>::LD, NB = D / 32, NH = D / 2, HL = NH + 4, NCH = NH / 32;
  extern __shared__ __align__(16) float sm[];
  float* sK = sm;                    // [C][LD] K
  float* lg = sK + kC * LD;          // [C]
  float* sW = lg + kC;               // [C][HL] a column half of W
  float* sE = sW + kC * HL;          // [C][HL] the same half of E
  float* sG = sE + kC * HL;          // [32][LD]
  float* sX = sG + 32 * LD;          // [32][kLC]
  float* sO = sX + 32 * kLC;         // [C][kL32] rows of dO, this block's columns
  const int li = blockIdx.x / (p.H * NB), h = (blockIdx.x / NB) % p.H, jb = blockIdx.x % NB;
  const int run = p.level_runs[lvl0 + li];
  const int32_t r0 = p.run_info[4 * run], r1 = p.run_info[4 * run + 1], c0 = p.run_info[4 * run + 3];
  const int nch = (r1 - r0 + kC - 1) / kC;
  const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
  const int j0 = jb * 32;
  auto issue_k = [&](int ci) {
    const int ch = c0 + ci;
    const size_t blk = (size_t)ch * p.H + h;
    cp_rows<D>(sK, p.k, p.chunk_info[2 * ch], p.chunk_info[2 * ch + 1], p.H, h);
    if (threadIdx.x < kC / 4) cp16(lg + threadIdx.x * 4, p.Lb + blk * kC + threadIdx.x * 4, true);
    cp_commit();
  };
  // columns [NH hf, NH hf + NH) of the chunk's W and E (not committed)
  auto issue_we = [&](size_t blk, int hf) {
    const float* w = p.Wb + blk * kC * D + NH * hf;
    const float* e = p.Ub + blk * kC * D + NH * hf;
    for (int i = threadIdx.x; i < kC * NH / 4; i += kT) {
      const int t = i / (NH / 4), cc = (i % (NH / 4)) * 4;
      cp16(sW + t * HL + cc, w + t * D + cc, true);
      cp16(sE + t * HL + cc, e + t * D + cc, true);
    }
  };
  if (nch > 0) issue_k(nch - 1);
  for (int i = threadIdx.x; i < 32 * D; i += kT) {
    float x = 0.f;
    for (int c = p.child_off[run]; c < p.child_off[run + 1]; c++)
      x += p.run_grad[((size_t)p.child[c] * p.H + h) * D * D + (j0 + i / D) * D + i % D];
    sG[(i / D) * LD + i % D] = x;
  }
  for (int ci = nch - 1; ci >= 0; ci--) {
    const int ch = c0 + ci;
    const size_t blk = (size_t)ch * p.H + h;
    const int64_t row0 = p.chunk_info[2 * ch];
    const int rows = p.chunk_info[2 * ch + 1];
    issue_we(blk, 0);
    cp_rows32<D>(sO, p.dout, row0, rows, p.H, h, j0);
    cp_commit();
    cp_wait_group<1>();   // this chunk's K and lg
    __syncthreads();
    const float lgC = lg[kC - 1];   // kept: K's buffer takes the next chunk's K below
    float* Gg = p.Gb + blk * D * D + (size_t)j0 * D;
    for (int i = threadIdx.x; i < 32 * D / 4; i += kT)
      *reinterpret_cast<float4*>(Gg + i * 4) = *reinterpret_cast<const float4*>(sG + (i / (D / 4)) * LD + (i % (D / 4)) * 4);
    {
      float acc[4][2];
      zero(acc);
      mm_nt(acc, sG, LD, sK, LD, D, ty * 4, tx);   // (G K^T)[j][t]
#pragma unroll
      for (int r = 0; r < 4; r++)
#pragma unroll
        for (int c = 0; c < 2; c++) {
          const int t = tx + 32 * c;
          sX[(ty * 4 + r) * kLC + t] = acc[r][c] * expf(lgC - lg[t]);
        }
    }
    cp_wait_group<0>();   // W and E, first half; dO
    __syncthreads();      // every warp is past its reads of K and lg
    if (ci > 0) issue_k(ci - 1);
    const float gC = expf(lgC);
#pragma unroll 1
    for (int hf = 0; hf < 2; hf++) {
      if (hf) {
        __syncthreads();   // the first halves of W and E are read
        issue_we(blk, 1);
        cp_commit();
        cp_wait_group<0>();
        __syncthreads();
      }
      float acc[4][NCH], acc2[4][NCH];
      zero(acc);
      zero(acc2);
      mm_nn(acc, sX, kLC, sW, HL, kC, ty * 4, tx);
      mm_tn(acc2, sO, kL32, sE, HL, kC, ty * 4, tx);
#pragma unroll
      for (int r = 0; r < 4; r++)
#pragma unroll
        for (int c = 0; c < NCH; c++) {
          float& x = sG[(ty * 4 + r) * LD + NH * hf + tx + 32 * c];
          x = gC * x - acc[r][c] + acc2[r][c];
        }
    }
    __syncthreads();
  }
  float* Rg = p.run_grad + ((size_t)run * p.H + h) * D * D + (size_t)j0 * D;
  for (int i = threadIdx.x; i < 32 * D / 4; i += kT)
    *reinterpret_cast<float4*>(Rg + i * 4) = *reinterpret_cast<const float4*>(sG + (i / (D / 4)) * LD + (i % (D / 4)) * 4);
}

// sum over the 32 lanes of a warp
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Gradients, part a, per chunk and head: X = V - diag(g) K S0^T;
// Gbar = diag(g_C / g) K G_C^T + tril(G o Q K^T)^T dO (gradient of Delta);
// Y = Minv^T Gbar; dv = diag(beta) Y; dbeta_t = Y_t . (X_t - (A Delta)_t); and the row
// parts of the gate gradient: g_t dg_t = -dv_t . (g_t K S0^T)_t + g_t dO_t . (Q S0^T)_t and
// r_t = (g_C / g_t) Delta_t . (K G_C^T)_t, and <G_C, S0>.  Y goes to the workspace for part b.
template <int D>
__global__ void __launch_bounds__(kT) k_rec_grad_a(RecParams p) {
  constexpr int LD = Lay<D>::LD, NC = Lay<D>::NC;
  extern __shared__ __align__(16) float sm[];
  float* sK = sm;
  float* sQ = sK + kC * LD;      // Q, later Delta
  float* sO = sQ + kC * LD;      // dO
  float* sX = sO + kC * LD;      // V, then X
  float* sY = sX + kC * LD;      // Gbar, then Y
  float* sS = sY + kC * LD;      // [D][kL32] a 32-column block of S0
  float* sT = sS + D * kL32;     // [D][kL32] the same columns of G_C
  float* sB = sT + D * kL32;     // [C][kLC]: tril(G o Q K^T), then Minv, then A
  float* lg = sB + kC * kLC;
  float* be = lg + kC;
  float* al = be + kC;
  const int ch = blockIdx.x / p.H, h = blockIdx.x % p.H;
  const int64_t row0 = p.chunk_info[2 * ch];
  const int rows = p.chunk_info[2 * ch + 1];
  const size_t blk = (size_t)ch * p.H + h;
  const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
  const float* S0g = p.S0 + blk * D * D;
  const float* GCg = p.Gb + blk * D * D;
  cp_rows<D>(sK, p.k, row0, rows, p.H, h);
  cp_rows<D>(sQ, p.q, row0, rows, p.H, h);
  cp_rows<D>(sO, p.dout, row0, rows, p.H, h);
  cp_rows<D>(sX, p.v, row0, rows, p.H, h);
  cp_commit();
  cp_blk32<D, D>(sS, S0g, 0);
  cp_commit();
  cp_blk32<D, D>(sT, GCg, 0);
  cp_commit();
  load_gates(lg, be, al, p.alpha, p.beta, row0, rows, p.H, h);
  cp_wait_group<2>();
  __syncthreads();
  {
    float acc[4][4];
    gram_w<D>(acc, sQ, sK);
#pragma unroll
    for (int r = 0; r < 4; r++)
#pragma unroll
      for (int c = 0; c < 4; c++) {
        const int t = gram_row(r), s = gram_col(c);
        sB[t * kLC + s] = s <= t ? expf(lg[t] - lg[s]) * acc[r][c] : 0.f;
      }
  }
  float pq[8], pr[8], pdb[8], gsum = 0.f;
#pragma unroll
  for (int r = 0; r < 8; r++) pq[r] = pr[r] = pdb[r] = 0.f;
  const float* Dg = p.Db + blk * kC * D;
  const float lgC = lg[kC - 1];
  // K S0^T, Q S0^T and K G_C^T by 32-column blocks jd of the contraction (column block jd
  // of S0 in sS, of G_C in sT); block jd + 1 of S0 is fetched while G_C's block jd is used,
  // and of G_C while S0's block jd + 1 is used
  float ks[8][NC], qs[8][NC], kg[8][NC];
  zero(ks);
  zero(qs);
  zero(kg);
#pragma unroll 1
  for (int jd = 0; jd < NC; jd++) {
    cp_wait_group<1>();   // S0 columns of block jd
    __syncthreads();
    mm_nt2(ks, qs, sK + 32 * jd, sQ + 32 * jd, LD, sS, kL32, 32, ty * 8, tx);
    cp_wait_group<0>();   // G_C columns of block jd
    __syncthreads();
    for (int i = threadIdx.x; i < D * 32; i += kT)   // <G_C, S0> over these columns
      gsum = fmaf(sS[(i >> 5) * kL32 + (i & 31)], sT[(i >> 5) * kL32 + (i & 31)], gsum);
    __syncthreads();
    if (jd + 1 < NC) cp_blk32<D, D>(sS, S0g, 32 * (jd + 1));
    cp_commit();
    mm_nt(kg, sK + 32 * jd, LD, sT, kL32, 32, ty * 8, tx);
    __syncthreads();
    if (jd + 1 < NC) cp_blk32<D, D>(sT, GCg, 32 * (jd + 1));
    cp_commit();
  }
#pragma unroll
  for (int r = 0; r < 8; r++) {
    const int t = ty * 8 + r;
    const float g = expf(lg[t]), rcf = expf(lgC - lg[t]);
#pragma unroll
    for (int c = 0; c < NC; c++) {
      const int j = tx + 32 * c;
      sX[t * LD + j] -= g * ks[r][c];
      pq[r] = fmaf(sO[t * LD + j], g * qs[r][c], pq[r]);
      const float rc = rcf * kg[r][c];
      sY[t * LD + j] = rc;
      pr[r] = fmaf(Dg[t * D + j], rc, pr[r]);
    }
  }
  cp_wait_group<0>();
  __syncthreads();
  {
    float acc[8][NC];
    zero(acc);
    mm_tn(acc, sB, kLC, sO, LD, kC, ty * 8, tx);   // tril(G o Q K^T)^T dO
#pragma unroll
    for (int r = 0; r < 8; r++)
#pragma unroll
      for (int c = 0; c < NC; c++) sY[(ty * 8 + r) * LD + tx + 32 * c] += acc[r][c];
  }
  __syncthreads();
  cp_cc(sB, p.Mb + blk * kC * kC);
  cp_wait();
  __syncthreads();
  float y[8][NC];
  zero(y);
  mm_tn(y, sB, kLC, sY, LD, kC, ty * 8, tx);     // Minv^T Gbar
  __syncthreads();
  float* Yg = p.Yb + blk * kC * D;
#pragma unroll
  for (int r = 0; r < 8; r++) {
    const int t = ty * 8 + r;
#pragma unroll
    for (int c = 0; c < NC; c++) {
      const int j = tx + 32 * c;
      sY[t * LD + j] = y[r][c];
      Yg[t * D + j] = y[r][c];
      const float dx = be[t] * y[r][c];
      if (t < rows) {
        p.dv[((row0 + t) * p.H + h) * D + j] = dx;
        // g_t (K S0^T)_t = V_t - X_t
        pq[r] = fmaf(-dx, p.v[((row0 + t) * p.H + h) * D + j] - sX[t * LD + j], pq[r]);
      }
    }
  }
  // A = strict lower G o K K^T, and Delta into Q's place
  {
    float acc[4][4];
    gram_w<D>(acc, sK, sK);
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 4; r++)
#pragma unroll
      for (int c = 0; c < 4; c++) {
        const int t = gram_row(r), s = gram_col(c);
        sB[t * kLC + s] = s < t ? expf(lg[t] - lg[s]) * acc[r][c] : 0.f;
      }
    cp_blk<D>(sQ, Dg);
    cp_wait();
  }
  __syncthreads();
  {
    float ad[8][NC];
    zero(ad);
    mm_nn(ad, sB, kLC, sQ, LD, kC, ty * 8, tx);
#pragma unroll
    for (int r = 0; r < 8; r++) {
      const int t = ty * 8 + r;
#pragma unroll
      for (int c = 0; c < NC; c++) {
        const int j = tx + 32 * c;
        pdb[r] = fmaf(sY[t * LD + j], sX[t * LD + j] - ad[r][c], pdb[r]);
      }
    }
  }
  float* Sg = p.Sc + blk * 3 * kC;
#pragma unroll
  for (int r = 0; r < 8; r++) {
    const int t = ty * 8 + r;
    const float a = warp_sum(pq[r]), b = warp_sum(pr[r]), c = warp_sum(pdb[r]);
    if (tx == 0) {
      Sg[t] = a;
      Sg[kC + t] = b;
      if (t < rows) p.dbeta[(row0 + t) * p.H + h] = c;
    }
  }
  // <G_C, S0>: warp sums, then the warps in order (the slice buffer is free by now)
  gsum = warp_sum(gsum);
  __syncthreads();
  if (tx == 0) sS[ty] = gsum;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int w = 0; w < kT / 32; w++) tot += sS[w];
    Sg[2 * kC] = tot;
  }
}

// Gradients, part b, per chunk and head, with DoD = dO Delta^T, L = tril(G) o DoD,
// dA = -strict lower of diag(beta) Y Delta^T, DA = G o dA:
//   dq = diag(g) dO S0 + L K,
//   dk = diag(g_C / g) Delta G_C + L^T Q + (DA + DA^T) K - diag(g beta) Y S0,
//   dlg_t = g_t dg_t + sum_s Z_ts - sum_s Z_st - r_t (+ sum r + g_C <G_C, S0> at the last
//   row), Z = G o (tril(Q K^T o DoD) + strict lower (dA o K K^T)), and
//   dalpha_j = (sum_{t >= j} dlg_t) / alpha_j.
template <int D>
__global__ void __launch_bounds__(kT) k_rec_grad_b(RecParams p) {
  constexpr int LD = Lay<D>::LD, NC = Lay<D>::NC;
  extern __shared__ __align__(16) float sm[];
  float* sK = sm;
  float* sQ = sK + kC * LD;
  float* sO = sQ + kC * LD;
  float* sD = sO + kC * LD;      // Delta
  float* sY = sD + kC * LD;
  float* sL = sY + kC * LD;      // [C][kLC]: L; before that, with sA, two [32][LD] row blocks of S0 / G_C
  float* sA = sL + kC * kLC;     // [C][kLC]: DA + DA^T
  float* lg = sA + kC * kLC;
  float* be = lg + kC;
  float* al = be + kC;
  float* dlg = al + kC;          // [C]
  float* cs = dlg + kC;          // [8][C] column sums of Z per warp
  static_assert(2 * 32 * Lay<D>::LD <= 2 * kC * kLC, "row blocks fit the C x C buffers");
  const int ch = blockIdx.x / p.H, h = blockIdx.x % p.H;
  const int64_t row0 = p.chunk_info[2 * ch];
  const int rows = p.chunk_info[2 * ch + 1];
  const size_t blk = (size_t)ch * p.H + h;
  const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
  const float* S0g = p.S0 + blk * D * D;
  const float* GCg = p.Gb + blk * D * D;
  float* slot[2] = {sL, sL + 32 * LD};
  // row blocks 0 .. NC-1 of S0, then of G_C; block i in slot i % 2
  auto issue = [&](int i) {
    if (i < 2 * NC) cp_blk<D, 32>(slot[i & 1], (i < NC ? S0g : GCg) + (size_t)32 * (i % NC) * D);
    cp_commit();
  };
  cp_rows<D>(sK, p.k, row0, rows, p.H, h);
  cp_rows<D>(sQ, p.q, row0, rows, p.H, h);
  cp_rows<D>(sO, p.dout, row0, rows, p.H, h);
  cp_blk<D>(sD, p.Db + blk * kC * D);
  cp_blk<D>(sY, p.Yb + blk * kC * D);
  cp_commit();
  issue(0);
  load_gates(lg, be, al, p.alpha, p.beta, row0, rows, p.H, h);
  const float lgC = lg[kC - 1];
  // dq = diag(g) dO S0 + L K;  dk = diag(g_C/g) Delta G_C - diag(g beta) Y S0 + L^T Q + (DA + DA^T) K
  float gq[8][NC], gk[8][NC], t1[8][NC];
  zero(gq);
  zero(t1);
#pragma unroll 1
  for (int i = 0; i < 2 * NC; i++) {
    issue(i + 1);
    cp_wait_group<1>();
    __syncthreads();
    const float* blkp = slot[i & 1];
    const int js = i % NC;
    if (i < NC) {
      mm_nn2(gq, t1, sO + 32 * js, sY + 32 * js, LD, blkp, LD, 32, ty * 8, tx);
    } else {
      mm_nn(t1, sD + 32 * js, LD, blkp, LD, 32, ty * 8, tx);
    }
    if (i == NC - 1) {   // Y S0 complete: fold it in, then collect Delta G_C in t1
#pragma unroll
      for (int r = 0; r < 8; r++) {
        const int t = ty * 8 + r;
        const float g = expf(lg[t]);
#pragma unroll
        for (int c = 0; c < NC; c++) {
          gq[r][c] *= g;
          gk[r][c] = -g * be[t] * t1[r][c];
          t1[r][c] = 0.f;
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 8; r++) {
    const float rc = expf(lgC - lg[ty * 8 + r]);
#pragma unroll
    for (int c = 0; c < NC; c++) gk[r][c] = fmaf(rc, t1[r][c], gk[r][c]);
  }
  {
    float dod[8][2], yd[8][2], qk[8][2], kk[8][2];
    gram2<D>(dod, yd, sO, sY, sD);
    gram2<D>(qk, kk, sQ, sK, sK);
    float csum[2] = {0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 8; r++) {
      const int t = ty * 8 + r;
      float rsum = 0.f;
#pragma unroll
      for (int c = 0; c < 2; c++) {
        const int s = tx + 32 * c;
        const float G = s <= t ? expf(lg[t] - lg[s]) : 0.f;
        const float da = s < t ? -be[t] * yd[r][c] : 0.f;
        const float z = G * (qk[r][c] * dod[r][c] + da * kk[r][c]);
        rsum += z;
        csum[c] += z;
        sL[t * kLC + s] = G * dod[r][c];   // L = tril(G) o DoD
        // DA + DA^T (DA is strictly lower triangular)
        if (s < t) {
          sA[t * kLC + s] = G * da;
          sA[s * kLC + t] = G * da;
        } else if (s == t) {
          sA[t * kLC + t] = 0.f;
        }
      }
      rsum = warp_sum(rsum);
      if (tx == 0) dlg[t] = rsum;
    }
    cs[ty * kC + tx] = csum[0];
    cs[ty * kC + tx + 32] = csum[1];
  }
  __syncthreads();
  if (threadIdx.x < kC) {
    float c = 0.f;
    for (int w = 0; w < kT / 32; w++) c += cs[w * kC + threadIdx.x];
    dlg[threadIdx.x] -= c;
  }
  mm_nn2(gq, gk, sL, sA, kLC, sK, LD, kC, ty * 8, tx);   // L K, (DA + DA^T) K
  mm_tn(gk, sL, kLC, sQ, LD, kC, ty * 8, tx);
#pragma unroll
  for (int r = 0; r < 8; r++) {
    const int t = ty * 8 + r;
    if (t < rows)
#pragma unroll
      for (int c = 0; c < NC; c++) {
        p.dq[((row0 + t) * p.H + h) * D + tx + 32 * c] = gq[r][c];
        p.dk[((row0 + t) * p.H + h) * D + tx + 32 * c] = gk[r][c];
      }
  }
  // dalpha_j = (sum_{t >= j} dlg_t) / alpha_j: two warps, suffix sums by shuffles
  __syncthreads();
  if (threadIdx.x < kC) {
    const int t = threadIdx.x;
    const float* Sg = p.Sc + blk * 3 * kC;
    const float r = Sg[kC + t];
    float x = dlg[t] + Sg[t] - r;
    const float rsum = warp_sum(r);
    cs[t] = rsum;   // the column-sum scratch is free: per-warp totals of r
    // suffix sum within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_down_sync(0xffffffffu, x, o);
      if ((t & 31) + o < 32) x += y;
    }
    dlg[t] = x;
  }
  __syncthreads();
  if (threadIdx.x < kC) {
    const int t = threadIdx.x;
    // the last row's extra terms (all r, and g_C <G_C, S0>) reach every row's suffix sum,
    // and rows of the first warp also take the second warp's total
    const float extra = cs[0] + cs[32] + expf(lgC) * p.Sc[blk * 3 * kC + 2 * kC];
    const float x = dlg[t] + extra + (t < 32 ? dlg[32] : 0.f);
    if (t < rows) p.dalpha[(row0 + t) * p.H + h] = x / al[t];
  }
}

template <int D>
constexpr size_t smem_prep() { return (size_t)(2 * kC * Lay<D>::LD + 2 * kC * kLC + 3 * kC) * 4; }
template <int D>
constexpr size_t smem_scan_fwd() { return (size_t)(2 * kC * Lay<D>::LD + 32 * Lay<D>::LD + kC * kL32 + kC) * 4; }
template <int D>
constexpr size_t smem_out() { return (size_t)(2 * kC * Lay<D>::LD + D * kL32 + kC * kLC + kC) * 4; }
template <int D>
constexpr size_t smem_prep_bwd() { return (size_t)(2 * kC * Lay<D>::LD + kC * kLC + kC) * 4; }
template <int D>
constexpr size_t smem_scan_bwd() {
  return (size_t)(kC * Lay<D>::LD + kC + 2 * kC * (D / 2 + 4) + 32 * Lay<D>::LD + 32 * kLC + kC * kL32) * 4;
}
template <int D>
constexpr size_t smem_grad_a() { return (size_t)(5 * kC * Lay<D>::LD + 2 * D * kL32 + kC * kLC + 3 * kC) * 4; }
template <int D>
constexpr size_t smem_grad_b() {
  return (size_t)(5 * kC * Lay<D>::LD + 2 * kC * kLC + 4 * kC + (kT / 32) * kC) * 4;
}
static_assert(smem_grad_b<128>() <= 232448 && smem_grad_a<128>() <= 232448, "shared memory per CTA");

}  // namespace
}  // namespace octo

namespace octo {
namespace {

// Workspace layout (floats, each array 256-byte aligned).  The first part holds what the
// forward saves for the backward; the second part is scratch.
struct RecLayout {
  size_t S0, Wb, Db, Mb, Lb, run_end, Ub, Gb, Yb, Sc, run_grad, total;
};

RecLayout rec_layout(const octo_plan_s* p, int32_t H, int32_t D) {
  const size_t nc = (size_t)p->n_chunks * H, nr = (size_t)p->n_runs * H;
  RecLayout L{};
  size_t off = 0;
  auto put = [&](size_t& f, size_t n) {
    f = off;
    off += align_up(std::max<size_t>(n, 1), 64);
  };
  put(L.S0, nc * D * D);
  put(L.Wb, nc * kC * D);
  put(L.Db, nc * kC * D);
  put(L.Mb, nc * kC * kC);
  put(L.Lb, nc * kC);
  put(L.run_end, nr * D * D);
  put(L.Ub, nc * kC * D);
  put(L.Gb, nc * D * D);
  put(L.Yb, nc * kC * D);
  put(L.Sc, nc * 3 * kC);
  put(L.run_grad, nr * D * D);
  L.total = off;
  return L;
}

RecParams rec_params(const octo_plan_s* p, int32_t H, int32_t D, void* ws) {
  const RecLayout L = rec_layout(p, H, D);
  float* w = (float*)ws;
  RecParams r{};
  r.run_info = p->run_info;
  r.child_off = p->run_child_off;
  r.child = p->run_child;
  r.level_runs = p->level_runs;
  r.chunk_info = p->chunk_info;
  r.H = H;
  r.S0 = w + L.S0;
  r.Wb = w + L.Wb;
  r.Db = w + L.Db;
  r.Mb = w + L.Mb;
  r.Lb = w + L.Lb;
  r.run_end = w + L.run_end;
  r.Ub = w + L.Ub;
  r.Gb = w + L.Gb;
  r.Yb = w + L.Yb;
  r.Sc = w + L.Sc;
  r.run_grad = w + L.run_grad;
  return r;
}

int rec_check(const octo_plan_s* p, int32_t H, int32_t D, void* ws, size_t ws_bytes) {
  if (!p || p->info.is_decode || H <= 0 || H > 65535 || (D != 64 && D != 128)) return OCTO_EINVAL;
  if (!p->run_info && p->info.n_rows > 0) return OCTO_EINVAL;
  if (p->info.n_rows > 0 && (!ws || ws_bytes < rec_layout(p, H, D).total * sizeof(float))) return OCTO_EINVAL;
  return OCTO_OK;
}

template <int D>
int rec_fwd(const octo_plan_s* p, RecParams r, cudaStream_t s) {
  constexpr int NB = D / 32;
  const unsigned ng = (unsigned)((size_t)p->n_chunks * r.H);
  if (int st = set_smem_limit((const void*)k_rec_prep<D>, (int)smem_prep<D>())) return st;
  if (int st = set_smem_limit((const void*)k_rec_scan_fwd<D>, (int)smem_scan_fwd<D>())) return st;
  if (int st = set_smem_limit((const void*)k_rec_out<D>, (int)smem_out<D>())) return st;
  k_rec_prep<D><<<ng, kT, smem_prep<D>(), s>>>(r);
  count_launch();
  for (int l = 0; l < p->n_levels; l++) {
    const int32_t a = p->h_level_off[l], b = p->h_level_off[l + 1];
    k_rec_scan_fwd<D><<<(unsigned)((size_t)(b - a) * r.H * NB), kT, smem_scan_fwd<D>(), s>>>(r, a);
    count_launch();
  }
  k_rec_out<D><<<ng, kT, smem_out<D>(), s>>>(r);
  count_launch();
  return cuda_status(cudaGetLastError());
}

template <int D>
int rec_bwd(const octo_plan_s* p, RecParams r, cudaStream_t s) {
  constexpr int NB = D / 32;
  const unsigned ng = (unsigned)((size_t)p->n_chunks * r.H);
  if (int st = set_smem_limit((const void*)k_rec_prep_bwd<D>, (int)smem_prep_bwd<D>())) return st;
  if (int st = set_smem_limit((const void*)k_rec_scan_bwd<D>, (int)smem_scan_bwd<D>())) return st;
  if (int st = set_smem_limit((const void*)k_rec_grad_a<D>, (int)smem_grad_a<D>())) return st;
  if (int st = set_smem_limit((const void*)k_rec_grad_b<D>, (int)smem_grad_b<D>())) return st;
  k_rec_prep_bwd<D><<<ng, kT, smem_prep_bwd<D>(), s>>>(r);
  count_launch();
  for (int l = p->n_levels - 1; l >= 0; l--) {
    const int32_t a = p->h_level_off[l], b = p->h_level_off[l + 1];
    k_rec_scan_bwd<D><<<(unsigned)((size_t)(b - a) * r.H * NB), kT, smem_scan_bwd<D>(), s>>>(r, a);
    count_launch();
  }
  k_rec_grad_a<D><<<ng, kT, smem_grad_a<D>(), s>>>(r);
  k_rec_grad_b<D><<<ng, kT, smem_grad_b<D>(), s>>>(r);
  count_launch(2);
  return cuda_status(cudaGetLastError());
}

}  // namespace
}  // namespace octo

extern "C" {

size_t octo_recurrent_workspace_size(octo_plan_t plan, int32_t n_heads, int32_t head_dim) {
  if (!plan || plan->info.is_decode || n_heads <= 0 || (head_dim != 64 && head_dim != 128)) return 0;
  return octo::rec_layout(plan, n_heads, head_dim).total * sizeof(float);
}

int octo_recurrent_fwd(octo_plan_t plan, int32_t n_heads, int32_t head_dim, const float* q, const float* k,
                       const float* v, const float* alpha, const float* beta, float* o, void* ws, size_t ws_bytes,
                       void* stream) {
  using namespace octo;
  if (int st = rec_check(plan, n_heads, head_dim, ws, ws_bytes)) return st;
  if (plan->info.n_rows == 0) return OCTO_OK;
  if (!q || !k || !v || !alpha || !beta || !o) return OCTO_EINVAL;
  plan->last_stream = (cudaStream_t)stream;
  NvtxRange nv("octo_recurrent_fwd");
  RecParams r = rec_params(plan, n_heads, head_dim, ws);
  r.q = q;
  r.k = k;
  r.v = v;
  r.alpha = alpha;
  r.beta = beta;
  r.o = o;
  return head_dim == 128 ? rec_fwd<128>(plan, r, (cudaStream_t)stream) : rec_fwd<64>(plan, r, (cudaStream_t)stream);
}

int octo_recurrent_bwd(octo_plan_t plan, int32_t n_heads, int32_t head_dim, const float* q, const float* k,
                       const float* v, const float* alpha, const float* beta, const float* dout, float* dq, float* dk,
                       float* dv, float* dalpha, float* dbeta, void* ws, size_t ws_bytes, void* stream) {
  using namespace octo;
  if (int st = rec_check(plan, n_heads, head_dim, ws, ws_bytes)) return st;
  if (plan->info.n_rows == 0) return OCTO_OK;
  if (!q || !k || !v || !alpha || !beta || !dout || !dq || !dk || !dv || !dalpha || !dbeta) return OCTO_EINVAL;
  plan->last_stream = (cudaStream_t)stream;
  NvtxRange nv("octo_recurrent_bwd");
  RecParams r = rec_params(plan, n_heads, head_dim, ws);
  r.q = q;
  r.k = k;
  r.v = v;
  r.alpha = alpha;
  r.beta = beta;
  r.dout = dout;
  r.dq = dq;
  r.dk = dk;
  r.dv = dv;
  r.dalpha = dalpha;
  r.dbeta = dbeta;
  return head_dim == 128 ? rec_bwd<128>(plan, r, (cudaStream_t)stream) : rec_bwd<64>(plan, r, (cudaStream_t)stream);
}

}  // extern "C"
