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
constexpr int kLC = kC + 1;       // padded row length of C x C matrices in shared memory

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

template <int D>
struct Lay {
  static constexpr int LD = D + 1;   // padded row length of C x D and 32 x D tiles
  static constexpr int NC = D / 32;  // columns per thread of a C x D tile
};

// acc[r][c] += sum_k A[(i0 + r) sai + k sak] * B[k sbk + (j0 + 32 c) sbj], k < K
template <int R, int NC>
__device__ __forceinline__ void mm(float (&acc)[R][NC], const float* A, int sai, int sak, const float* B, int sbk,
                                   int sbj, int K, int i0, int j0) {
#pragma unroll 4
  for (int k = 0; k < K; k++) {
    float a[R], b[NC];
#pragma unroll
    for (int r = 0; r < R; r++) a[r] = A[(i0 + r) * sai + k * sak];
#pragma unroll
    for (int c = 0; c < NC; c++) b[c] = B[k * sbk + (j0 + 32 * c) * sbj];
#pragma unroll
    for (int r = 0; r < R; r++)
#pragma unroll
      for (int c = 0; c < NC; c++) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
  }
}

template <int R, int NC>
__device__ __forceinline__ void zero(float (&acc)[R][NC]) {
#pragma unroll
  for (int r = 0; r < R; r++)
#pragma unroll
    for (int c = 0; c < NC; c++) acc[r][c] = 0.f;
}

// rows [row0, row0 + rows) of x [N][H][D] at head h into dst [C][LD]; zeros past `rows`
template <int D>
__device__ __forceinline__ void load_rows(float* dst, const float* __restrict__ x, int64_t row0, int rows, int H,
                                          int h) {
  for (int i = threadIdx.x; i < kC * D; i += kT) {
    const int t = i / D, c = i % D;
    dst[t * Lay<D>::LD + c] = t < rows ? x[((row0 + t) * H + h) * D + c] : 0.f;
  }
}
// a dense [C][D] block of the workspace into dst [C][LD]
template <int D>
__device__ __forceinline__ void load_blk(float* dst, const float* __restrict__ src) {
  for (int i = threadIdx.x; i < kC * D; i += kT) dst[(i / D) * Lay<D>::LD + i % D] = src[i];
}
// rows [j0, j0 + 32) of a dense [D][D] state into dst [32][LD]
template <int D>
__device__ __forceinline__ void load_state_rows(float* dst, const float* __restrict__ src, int j0) {
  for (int i = threadIdx.x; i < 32 * D; i += kT) dst[(i / D) * Lay<D>::LD + i % D] = src[(j0 + i / D) * D + i % D];
}

// per-row gate values of one chunk: lg (running sum of log alpha), beta, rows past the end
// get alpha = 1, beta = 0 (no effect)
__device__ __forceinline__ void load_gates(float* lg, float* be, float* al, const float* __restrict__ alpha,
                                           const float* __restrict__ beta, int64_t row0, int rows, int H, int h) {
  if (threadIdx.x < kC) {
    const int t = threadIdx.x;
    al[t] = t < rows ? alpha[(row0 + t) * H + h] : 1.f;
    be[t] = t < rows ? beta[(row0 + t) * H + h] : 0.f;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int t = 0; t < kC; t++) {
      s += logf(al[t]);
      lg[t] = s;
    }
  }
  __syncthreads();
}

// C x C product into registers: acc (8 rows x 2 columns per thread) = sum_k X[i][k] Y[j][k]
template <int D>
__device__ __forceinline__ void gram(float (&acc)[8][2], const float* X, const float* Y) {
  zero(acc);
  const int i0 = (threadIdx.x >> 5) * 8, j0 = threadIdx.x & 31;
  mm(acc, X, Lay<D>::LD, 1, Y, 1, Lay<D>::LD, D, i0, j0);
}

// =====================================================================================
// forward
// =====================================================================================

// Per chunk and head: lg, Minv = (I + diag(beta) A)^-1, W = Minv diag(beta g) K and
// U = Minv diag(beta) V.
template <int D>
__global__ void __launch_bounds__(kT) k_rec_prep(RecParams p) {
  constexpr int LD = Lay<D>::LD;
  extern __shared__ float sm[];
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
  load_rows<D>(sK, p.k, row0, rows, p.H, h);
  load_rows<D>(sV, p.v, row0, rows, p.H, h);
  load_gates(lg, be, al, p.alpha, p.beta, row0, rows, p.H, h);
  const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
  {
    float acc[8][2];
    gram<D>(acc, sK, sK);
#pragma unroll
    for (int r = 0; r < 8; r++)
#pragma unroll
      for (int c = 0; c < 2; c++) {
        const int t = ty * 8 + r, s = tx + 32 * c;
        sA[t * kLC + s] = s < t ? expf(lg[t] - lg[s]) * acc[r][c] : 0.f;
      }
  }
  // forward substitution, one row of Minv at a time: Minv[t][s] = [t == s]
  //   - beta_t sum_{s <= u < t} A[t][u] Minv[u][s]
  for (int i = threadIdx.x; i < kC * kLC; i += kT) sMi[i] = 0.f;
  __syncthreads();
  for (int t = 0; t < kC; t++) {
    if (threadIdx.x <= t) {
      const int s = threadIdx.x;
      float x = 0.f;
      for (int u = s; u < t; u++) x = fmaf(sA[t * kLC + u], sMi[u * kLC + s], x);
      sMi[t * kLC + s] = (s == t ? 1.f : 0.f) - be[t] * x;
    }
    __syncthreads();
  }
  // rows of K scaled by beta g, of V by beta
  for (int i = threadIdx.x; i < kC * D; i += kT) {
    const int t = i / D, c = i % D;
    sK[t * LD + c] *= be[t] * expf(lg[t]);
    sV[t * LD + c] *= be[t];
  }
  __syncthreads();
  constexpr int NC = Lay<D>::NC;
  float w[8][NC], u[8][NC];
  zero(w);
  zero(u);
  mm(w, sMi, kLC, 1, sK, LD, 1, kC, ty * 8, tx);
  mm(u, sMi, kLC, 1, sV, LD, 1, kC, ty * 8, tx);
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
// continue from it.
template <int D>
__global__ void __launch_bounds__(kT) k_rec_scan_fwd(RecParams p, int32_t lvl0) {
  constexpr int LD = Lay<D>::LD, NC = Lay<D>::NC, NB = D / 32;
  extern __shared__ float sm[];
  float* sW = sm;
  float* sK = sW + kC * LD;
  float* sS = sK + kC * LD;          // [32][LD]
  float* sU = sS + 32 * LD;          // [C][33]: U, then Delta (scaled by g_C / g)
  float* lg = sU + kC * 33;
  const int li = blockIdx.x / (p.H * NB), h = (blockIdx.x / NB) % p.H, jb = blockIdx.x % NB;
  const int run = p.level_runs[lvl0 + li];
  const int32_t r0 = p.run_info[4 * run], r1 = p.run_info[4 * run + 1];
  const int32_t pr = p.run_info[4 * run + 2], c0 = p.run_info[4 * run + 3];
  const int nch = (r1 - r0 + kC - 1) / kC;
  const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
  const int j0 = jb * 32;
  if (pr >= 0)
    load_state_rows<D>(sS, p.run_end + ((size_t)pr * p.H + h) * D * D, j0);
  else
    for (int i = threadIdx.x; i < 32 * LD; i += kT) sS[i] = 0.f;
  __syncthreads();
  for (int ci = 0; ci < nch; ci++) {
    const int ch = c0 + ci;
    const size_t blk = (size_t)ch * p.H + h;
    float* S0g = p.S0 + blk * D * D;
    for (int i = threadIdx.x; i < 32 * D; i += kT) S0g[(j0 + i / D) * D + i % D] = sS[(i / D) * LD + i % D];
    const int64_t row0 = p.chunk_info[2 * ch];
    const int rows = p.chunk_info[2 * ch + 1];
    load_blk<D>(sW, p.Wb + blk * kC * D);
    load_rows<D>(sK, p.k, row0, rows, p.H, h);
    const float* Ug = p.Ub + blk * kC * D;
    for (int i = threadIdx.x; i < kC * 32; i += kT) sU[(i >> 5) * 33 + (i & 31)] = Ug[(i >> 5) * D + j0 + (i & 31)];
    if (threadIdx.x < kC) lg[threadIdx.x] = p.Lb[blk * kC + threadIdx.x];
    __syncthreads();
    {
      float acc[8][1];
      zero(acc);
      mm(acc, sW, LD, 1, sS, 1, LD, D, ty * 8, tx);   // (W S0^T)[t][j]
      const float gC = lg[kC - 1];
      float* Dg = p.Db + blk * kC * D;
      __syncthreads();
#pragma unroll
      for (int r = 0; r < 8; r++) {
        const int t = ty * 8 + r;
        const float dl = sU[t * 33 + tx] - acc[r][0];
        Dg[t * D + j0 + tx] = dl;
        sU[t * 33 + tx] = dl * expf(gC - lg[t]);
      }
    }
    __syncthreads();
    {
      float acc[4][NC];
      zero(acc);
      mm(acc, sU, 1, 33, sK, LD, 1, kC, ty * 4, tx);   // (Delta^T diag(g_C/g) K)[j][k]
      const float gC = expf(lg[kC - 1]);
#pragma unroll
      for (int r = 0; r < 4; r++)
#pragma unroll
        for (int c = 0; c < NC; c++) {
          float& x = sS[(ty * 4 + r) * LD + tx + 32 * c];
          x = fmaf(gC, x, acc[r][c]);
        }
    }
    __syncthreads();
  }
  float* Eg = p.run_end + ((size_t)run * p.H + h) * D * D;
  for (int i = threadIdx.x; i < 32 * D; i += kT) Eg[(j0 + i / D) * D + i % D] = sS[(i / D) * LD + i % D];
}

// Outputs per chunk and head: O = diag(g) Q S0^T + tril(G o Q K^T) Delta.
template <int D>
__global__ void __launch_bounds__(kT) k_rec_out(RecParams p) {
  constexpr int LD = Lay<D>::LD, NC = Lay<D>::NC;
  extern __shared__ float sm[];
  float* sQ = sm;
  float* sK = sQ + kC * LD;
  float* sD = sK + kC * LD;
  float* sS = sD + kC * LD;    // [32][LD] slice of S0
  float* sB = sS + 32 * LD;    // [C][kLC]
  float* lg = sB + kC * kLC;
  const int ch = blockIdx.x / p.H, h = blockIdx.x % p.H;
  const int64_t row0 = p.chunk_info[2 * ch];
  const int rows = p.chunk_info[2 * ch + 1];
  const size_t blk = (size_t)ch * p.H + h;
  const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
  load_rows<D>(sQ, p.q, row0, rows, p.H, h);
  load_rows<D>(sK, p.k, row0, rows, p.H, h);
  load_blk<D>(sD, p.Db + blk * kC * D);
  if (threadIdx.x < kC) lg[threadIdx.x] = p.Lb[blk * kC + threadIdx.x];
  __syncthreads();
  {
    float acc[8][2];
    gram<D>(acc, sQ, sK);
#pragma unroll
    for (int r = 0; r < 8; r++)
#pragma unroll
      for (int c = 0; c < 2; c++) {
        const int t = ty * 8 + r, s = tx + 32 * c;
        sB[t * kLC + s] = s <= t ? expf(lg[t] - lg[s]) * acc[r][c] : 0.f;
      }
  }
  float out[8][NC];
  zero(out);
  const float* S0g = p.S0 + blk * D * D;
#pragma unroll
  for (int js = 0; js < NC; js++) {
    __syncthreads();
    load_state_rows<D>(sS, S0g, 32 * js);
    __syncthreads();
    float acc[8][1];
    zero(acc);
    mm(acc, sQ, LD, 1, sS, 1, LD, D, ty * 8, tx);
#pragma unroll
    for (int r = 0; r < 8; r++) out[r][js] = acc[r][0] * expf(lg[ty * 8 + r]);
  }
  mm(out, sB, kLC, 1, sD, LD, 1, kC, ty * 8, tx);
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

// E = diag(g) Q - tril(G o Q K^T) W per chunk and head.
template <int D>
__global__ void __launch_bounds__(kT) k_rec_prep_bwd(RecParams p) {
  constexpr int LD = Lay<D>::LD, NC = Lay<D>::NC;
  extern __shared__ float sm[];
  float* sQ = sm;
  float* sK = sQ + kC * LD;
  float* sW = sK + kC * LD;
  float* sB = sW + kC * LD;
  float* lg = sB + kC * kLC;
  const int ch = blockIdx.x / p.H, h = blockIdx.x % p.H;
  const int64_t row0 = p.chunk_info[2 * ch];
  const int rows = p.chunk_info[2 * ch + 1];
  const size_t blk = (size_t)ch * p.H + h;
  const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
  load_rows<D>(sQ, p.q, row0, rows, p.H, h);
  load_rows<D>(sK, p.k, row0, rows, p.H, h);
  load_blk<D>(sW, p.Wb + blk * kC * D);
  if (threadIdx.x < kC) lg[threadIdx.x] = p.Lb[blk * kC + threadIdx.x];
  __syncthreads();
  {
    float acc[8][2];
    gram<D>(acc, sQ, sK);
#pragma unroll
    for (int r = 0; r < 8; r++)
#pragma unroll
      for (int c = 0; c < 2; c++) {
        const int t = ty * 8 + r, s = tx + 32 * c;
        sB[t * kLC + s] = s <= t ? -expf(lg[t] - lg[s]) * acc[r][c] : 0.f;
      }
  }
  __syncthreads();
  float e[8][NC];
#pragma unroll
  for (int r = 0; r < 8; r++) {
    const float g = expf(lg[ty * 8 + r]);
#pragma unroll
    for (int c = 0; c < NC; c++) e[r][c] = g * sQ[(ty * 8 + r) * LD + tx + 32 * c];
  }
  mm(e, sB, kLC, 1, sW, LD, 1, kC, ty * 8, tx);
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
  constexpr int LD = Lay<D>::LD, NC = Lay<D>::NC, NB = D / 32;
  extern __shared__ float sm[];
  float* sK = sm;
  float* sW = sK + kC * LD;
  float* sE = sW + kC * LD;
  float* sG = sE + kC * LD;          // [32][LD]
  float* sX = sG + 32 * LD;          // [32][kLC]
  float* sO = sX + 32 * kLC;         // [C][33] rows of dO, this block's columns
  float* lg = sO + kC * 33;
  const int li = blockIdx.x / (p.H * NB), h = (blockIdx.x / NB) % p.H, jb = blockIdx.x % NB;
  const int run = p.level_runs[lvl0 + li];
  const int32_t r0 = p.run_info[4 * run], r1 = p.run_info[4 * run + 1], c0 = p.run_info[4 * run + 3];
  const int nch = (r1 - r0 + kC - 1) / kC;
  const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
  const int j0 = jb * 32;
  for (int i = threadIdx.x; i < 32 * D; i += kT) {
    float x = 0.f;
    for (int c = p.child_off[run]; c < p.child_off[run + 1]; c++)
      x += p.run_grad[((size_t)p.child[c] * p.H + h) * D * D + (j0 + i / D) * D + i % D];
    sG[(i / D) * LD + i % D] = x;
  }
  __syncthreads();
  for (int ci = nch - 1; ci >= 0; ci--) {
    const int ch = c0 + ci;
    const size_t blk = (size_t)ch * p.H + h;
    float* Gg = p.Gb + blk * D * D;
    for (int i = threadIdx.x; i < 32 * D; i += kT) Gg[(j0 + i / D) * D + i % D] = sG[(i / D) * LD + i % D];
    const int64_t row0 = p.chunk_info[2 * ch];
    const int rows = p.chunk_info[2 * ch + 1];
    load_rows<D>(sK, p.k, row0, rows, p.H, h);
    load_blk<D>(sW, p.Wb + blk * kC * D);
    load_blk<D>(sE, p.Ub + blk * kC * D);
    for (int i = threadIdx.x; i < kC * 32; i += kT) {
      const int t = i >> 5;
      sO[t * 33 + (i & 31)] = t < rows ? p.dout[((row0 + t) * p.H + h) * D + j0 + (i & 31)] : 0.f;
    }
    if (threadIdx.x < kC) lg[threadIdx.x] = p.Lb[blk * kC + threadIdx.x];
    __syncthreads();
    {
      float acc[4][2];
      zero(acc);
      mm(acc, sG, LD, 1, sK, 1, LD, D, ty * 4, tx);   // (G K^T)[j][t]
      const float gC = lg[kC - 1];
#pragma unroll
      for (int r = 0; r < 4; r++)
#pragma unroll
        for (int c = 0; c < 2; c++) {
          const int t = tx + 32 * c;
          sX[(ty * 4 + r) * kLC + t] = acc[r][c] * expf(gC - lg[t]);
        }
    }
    __syncthreads();
    {
      float acc[4][NC], acc2[4][NC];
      zero(acc);
      zero(acc2);
      mm(acc, sX, kLC, 1, sW, LD, 1, kC, ty * 4, tx);
      mm(acc2, sO, 1, 33, sE, LD, 1, kC, ty * 4, tx);
      const float gC = expf(lg[kC - 1]);
#pragma unroll
      for (int r = 0; r < 4; r++)
#pragma unroll
        for (int c = 0; c < NC; c++) {
          float& x = sG[(ty * 4 + r) * LD + tx + 32 * c];
          x = gC * x - acc[r][c] + acc2[r][c];
        }
    }
    __syncthreads();
  }
  float* Rg = p.run_grad + ((size_t)run * p.H + h) * D * D;
  for (int i = threadIdx.x; i < 32 * D; i += kT) Rg[(j0 + i / D) * D + i % D] = sG[(i / D) * LD + i % D];
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
// r_t = (g_C / g_t) Delta_t . (K G_C^T)_t.  Y goes to the workspace for part b.
template <int D>
__global__ void __launch_bounds__(kT) k_rec_grad_a(RecParams p) {
  constexpr int LD = Lay<D>::LD, NC = Lay<D>::NC;
  extern __shared__ float sm[];
  float* sK = sm;
  float* sQ = sK + kC * LD;      // Q, later Delta
  float* sO = sQ + kC * LD;      // dO
  float* sX = sO + kC * LD;      // V, then X
  float* sY = sX + kC * LD;      // Gbar, then Y
  float* sS = sY + kC * LD;      // [32][LD] slice of S0 or G_C
  float* sB = sS + 32 * LD;      // [C][kLC]: tril(G o Q K^T), then Minv, then A
  float* lg = sB + kC * kLC;
  float* be = lg + kC;
  float* al = be + kC;
  const int ch = blockIdx.x / p.H, h = blockIdx.x % p.H;
  const int64_t row0 = p.chunk_info[2 * ch];
  const int rows = p.chunk_info[2 * ch + 1];
  const size_t blk = (size_t)ch * p.H + h;
  const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
  load_rows<D>(sK, p.k, row0, rows, p.H, h);
  load_rows<D>(sQ, p.q, row0, rows, p.H, h);
  load_rows<D>(sO, p.dout, row0, rows, p.H, h);
  load_rows<D>(sX, p.v, row0, rows, p.H, h);
  load_gates(lg, be, al, p.alpha, p.beta, row0, rows, p.H, h);
  {
    float acc[8][2];
    gram<D>(acc, sQ, sK);
#pragma unroll
    for (int r = 0; r < 8; r++)
#pragma unroll
      for (int c = 0; c < 2; c++) {
        const int t = ty * 8 + r, s = tx + 32 * c;
        sB[t * kLC + s] = s <= t ? expf(lg[t] - lg[s]) * acc[r][c] : 0.f;
      }
  }
  float pq[8], pr[8], pdb[8], gsum = 0.f;
#pragma unroll
  for (int r = 0; r < 8; r++) pq[r] = pr[r] = pdb[r] = 0.f;
  const float* S0g = p.S0 + blk * D * D;
  const float* GCg = p.Gb + blk * D * D;
  const float* Dg = p.Db + blk * kC * D;
  const float lgC = lg[kC - 1];
#pragma unroll
  for (int js = 0; js < NC; js++) {
    const int j = 32 * js + tx;
    __syncthreads();
    load_state_rows<D>(sS, S0g, 32 * js);
    __syncthreads();
    float ks[8][1], qs[8][1];
    zero(ks);
    zero(qs);
    mm(ks, sK, LD, 1, sS, 1, LD, D, ty * 8, tx);
    mm(qs, sQ, LD, 1, sS, 1, LD, D, ty * 8, tx);
#pragma unroll
    for (int r = 0; r < 8; r++) {
      const int t = ty * 8 + r;
      const float g = expf(lg[t]);
      sX[t * LD + j] -= g * ks[r][0];
      pq[r] = fmaf(sO[t * LD + j], g * qs[r][0], pq[r]);
    }
    __syncthreads();
    load_state_rows<D>(sS, GCg, 32 * js);
    __syncthreads();
    for (int i = threadIdx.x; i < 32 * D; i += kT)   // <G_C, S0> over these rows
      gsum = fmaf(sS[(i / D) * LD + i % D], S0g[(32 * js + i / D) * D + i % D], gsum);
    float kg[8][1];
    zero(kg);
    mm(kg, sK, LD, 1, sS, 1, LD, D, ty * 8, tx);
#pragma unroll
    for (int r = 0; r < 8; r++) {
      const int t = ty * 8 + r;
      const float rc = expf(lgC - lg[t]) * kg[r][0];
      sY[t * LD + j] = rc;
      pr[r] = fmaf(Dg[t * D + j], rc, pr[r]);
    }
  }
  __syncthreads();
  {
    float acc[8][NC];
    zero(acc);
    mm(acc, sB, 1, kLC, sO, LD, 1, kC, ty * 8, tx);   // tril(G o Q K^T)^T dO
#pragma unroll
    for (int r = 0; r < 8; r++)
#pragma unroll
      for (int c = 0; c < NC; c++) sY[(ty * 8 + r) * LD + tx + 32 * c] += acc[r][c];
  }
  __syncthreads();
  const float* Mg = p.Mb + blk * kC * kC;
  for (int i = threadIdx.x; i < kC * kC; i += kT) sB[(i / kC) * kLC + i % kC] = Mg[i];
  __syncthreads();
  float y[8][NC];
  zero(y);
  mm(y, sB, 1, kLC, sY, LD, 1, kC, ty * 8, tx);     // Minv^T Gbar
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
    float acc[8][2];
    gram<D>(acc, sK, sK);
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 8; r++)
#pragma unroll
      for (int c = 0; c < 2; c++) {
        const int t = ty * 8 + r, s = tx + 32 * c;
        sB[t * kLC + s] = s < t ? expf(lg[t] - lg[s]) * acc[r][c] : 0.f;
      }
    load_blk<D>(sQ, Dg);
  }
  __syncthreads();
  {
    float ad[8][NC];
    zero(ad);
    mm(ad, sB, kLC, 1, sQ, LD, 1, kC, ty * 8, tx);
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
  extern __shared__ float sm[];
  float* sK = sm;
  float* sQ = sK + kC * LD;
  float* sO = sQ + kC * LD;
  float* sD = sO + kC * LD;      // Delta
  float* sY = sD + kC * LD;
  float* sS = sY + kC * LD;      // [32][LD] slice of S0 or G_C
  float* sL = sS + 32 * LD;      // [C][kLC]: DoD, then L
  float* sA = sL + kC * kLC;     // [C][kLC]: dA, then DA
  float* lg = sA + kC * kLC;
  float* be = lg + kC;
  float* al = be + kC;
  float* dlg = al + kC;          // [C]
  float* cs = dlg + kC;          // [8][C] column sums of Z per warp
  const int ch = blockIdx.x / p.H, h = blockIdx.x % p.H;
  const int64_t row0 = p.chunk_info[2 * ch];
  const int rows = p.chunk_info[2 * ch + 1];
  const size_t blk = (size_t)ch * p.H + h;
  const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
  load_rows<D>(sK, p.k, row0, rows, p.H, h);
  load_rows<D>(sQ, p.q, row0, rows, p.H, h);
  load_rows<D>(sO, p.dout, row0, rows, p.H, h);
  load_blk<D>(sD, p.Db + blk * kC * D);
  load_blk<D>(sY, p.Yb + blk * kC * D);
  load_gates(lg, be, al, p.alpha, p.beta, row0, rows, p.H, h);
  const float lgC = lg[kC - 1];
  {
    float dod[8][2], yd[8][2], qk[8][2], kk[8][2];
    gram<D>(dod, sO, sD);
    gram<D>(yd, sY, sD);
    gram<D>(qk, sQ, sK);
    gram<D>(kk, sK, sK);
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
        sA[t * kLC + s] = G * da;          // DA
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
  // dq = diag(g) dO S0 + L K;  dk = diag(g_C/g) Delta G_C - diag(g beta) Y S0 + L^T Q + (DA + DA^T) K
  float gq[8][NC], gk[8][NC];
  zero(gq);
  zero(gk);
  const float* S0g = p.S0 + blk * D * D;
  const float* GCg = p.Gb + blk * D * D;
  {
    float ys[8][NC];
    zero(ys);
#pragma unroll 1
    for (int js = 0; js < NC; js++) {
      __syncthreads();
      load_state_rows<D>(sS, S0g, 32 * js);
      __syncthreads();
      mm(gq, sO + 32 * js, LD, 1, sS, LD, 1, 32, ty * 8, tx);
      mm(ys, sY + 32 * js, LD, 1, sS, LD, 1, 32, ty * 8, tx);
    }
#pragma unroll
    for (int r = 0; r < 8; r++) {
      const int t = ty * 8 + r;
      const float g = expf(lg[t]);
#pragma unroll
      for (int c = 0; c < NC; c++) {
        gq[r][c] *= g;
        gk[r][c] = -g * be[t] * ys[r][c];
      }
    }
  }
  {
    float dg[8][NC];
    zero(dg);
#pragma unroll 1
    for (int js = 0; js < NC; js++) {
      __syncthreads();
      load_state_rows<D>(sS, GCg, 32 * js);
      __syncthreads();
      mm(dg, sD + 32 * js, LD, 1, sS, LD, 1, 32, ty * 8, tx);
    }
#pragma unroll
    for (int r = 0; r < 8; r++) {
      const float rc = expf(lgC - lg[ty * 8 + r]);
#pragma unroll
      for (int c = 0; c < NC; c++) gk[r][c] = fmaf(rc, dg[r][c], gk[r][c]);
    }
  }
  mm(gq, sL, kLC, 1, sK, LD, 1, kC, ty * 8, tx);
  mm(gk, sL, 1, kLC, sQ, LD, 1, kC, ty * 8, tx);
  mm(gk, sA, kLC, 1, sK, LD, 1, kC, ty * 8, tx);
  mm(gk, sA, 1, kLC, sK, LD, 1, kC, ty * 8, tx);
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
  __syncthreads();
  if (threadIdx.x == 0) {
    const float* Sg = p.Sc + blk * 3 * kC;
    float rsum = 0.f;
    for (int t = 0; t < kC; t++) {
      dlg[t] += Sg[t] - Sg[kC + t];
      rsum += Sg[kC + t];
    }
    dlg[kC - 1] += rsum + expf(lgC) * Sg[2 * kC];
    float acc = 0.f;
    for (int t = kC - 1; t >= 0; t--) {
      acc += dlg[t];
      if (t < rows) p.dalpha[(row0 + t) * p.H + h] = acc / al[t];
    }
  }
}

template <int D>
constexpr size_t smem_prep() { return (size_t)(2 * kC * Lay<D>::LD + 2 * kC * kLC + 3 * kC) * 4; }
template <int D>
constexpr size_t smem_scan_fwd() { return (size_t)(2 * kC * Lay<D>::LD + 32 * Lay<D>::LD + kC * 33 + kC) * 4; }
template <int D>
constexpr size_t smem_out() { return (size_t)(3 * kC * Lay<D>::LD + 32 * Lay<D>::LD + kC * kLC + kC) * 4; }
template <int D>
constexpr size_t smem_prep_bwd() { return (size_t)(3 * kC * Lay<D>::LD + kC * kLC + kC) * 4; }
template <int D>
constexpr size_t smem_scan_bwd() {
  return (size_t)(3 * kC * Lay<D>::LD + 32 * Lay<D>::LD + 32 * kLC + kC * 33 + kC) * 4;
}
template <int D>
constexpr size_t smem_grad_a() { return (size_t)(5 * kC * Lay<D>::LD + 32 * Lay<D>::LD + kC * kLC + 3 * kC) * 4; }
template <int D>
constexpr size_t smem_grad_b() {
  return (size_t)(5 * kC * Lay<D>::LD + 32 * Lay<D>::LD + 2 * kC * kLC + 4 * kC + (kT / 32) * kC) * 4;
}

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
