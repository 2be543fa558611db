// Attention entry points: argument checks and dispatch between the tensor-core kernels
// (bf16, head_dim 128, page 64, q-tile 128) and the CUDA-core kernels (everything else).

#include <algorithm>
#include <cmath>

#include "internal.h"
#include "tc_common.cuh"

namespace octo {
int fwd_simt(const octo_plan_s* p, int32_t Hq, const void* q, const void* k, const void* v, void* o, float* lse,
             float scale, bool decode, cudaStream_t s);
int bwd_simt(const octo_plan_s* p, int32_t Hq, const void* q, const void* k, const void* v, const void* o,
             const float* lse, const void* dout, float* dq, float* dk, float* dv, float scale, void* ws,
             cudaStream_t s);
bool fwd_tc_supported(const octo_plan_s* p, int32_t Hq);
bool bwd_tc_supported(const octo_plan_s* p, int32_t Hq);
size_t bwd_tc_workspace(const octo_plan_s* p, int32_t Hq);
bool decode_split_supported(const octo_plan_s* p, int32_t Hq);
size_t decode_split_workspace(const octo_plan_s* p, int32_t Hq);
int decode_split(const octo_plan_s* p, int32_t Hq, const void* q, const void* k, const void* v, void* out, float* lse,
                 float scale, void* ws, cudaStream_t s);
int bwd_tc(const octo_plan_s* p, int32_t Hq, const void* q, const void* k, const void* v, const void* o,
           const float* lse, const void* dout, float* dq, float* dk, float* dv, float scale, void* ws,
           cudaStream_t s);
int fwd_tc(const octo_plan_s* p, int32_t Hq, const void* q, const void* k, const void* v, void* o, float* lse,
           float scale, cudaStream_t s);
}  // namespace octo

namespace {

// A library built with -DOCTO_SIMT_ONLY sends every attention call to the CUDA-core
// kernels (a diagnostic build for comparing the two kernel families on the same shapes;
// octo_kernel_path reports 0 there).  The regular build has no switch that changes kernels
// at run time.
constexpr bool tc_disabled() {
#ifdef OCTO_SIMT_ONLY
  return true;
#else
  return false;
#endif
}

int check_heads(const octo_plan_s* p, int32_t Hq) {
  const int32_t Hkv = p->pool->desc.n_kv_heads;
  if (Hq <= 0 || Hq % Hkv != 0 || Hq > 65535) return OCTO_EINVAL;
  return OCTO_OK;
}

}  // namespace

// One CTA waits, through the bounded mbarrier wait of the tensor-core and decode kernels,
// on a phase of a barrier that no thread arrives on and no copy completes: after
// max_polls polls it records OCTO_ETIMEOUT and returns.  Nothing is in flight meanwhile.
__global__ void k_wait_selftest(int32_t* status, uint32_t max_polls) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    octo::tc::mbar_init(&bar, 1);
    octo::tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) octo::tc::mbar_wait_n(&bar, 0, status, OCTO_ETIMEOUT, max_polls);
  __syncthreads();
}

extern "C" {

int octo_kernel_path(octo_plan_t plan, int32_t n_q_heads, int32_t which) {
  if (!plan || check_heads(plan, n_q_heads)) return -1;
  if (which == 2) return octo::decode_split_supported(plan, n_q_heads) ? 2 : 0;
  if (tc_disabled()) return 0;
  if (which == 0) return octo::fwd_tc_supported(plan, n_q_heads) ? 1 : 0;
  if (which == 1) return octo::bwd_tc_supported(plan, n_q_heads) ? 1 : 0;
  return 0;
}

int octo_attn_fwd(octo_plan_t plan, int32_t Hq, const void* q, const void* k_pool, const void* v_pool, void* o,
                  float* lse, float scale, void* stream) {
  if (!plan || plan->info.is_decode) return OCTO_EINVAL;
  if (int st = check_heads(plan, Hq)) return st;
  if (plan->info.n_rows > 0 && (!q || !o || !lse)) return OCTO_EINVAL;
  const void* k = k_pool ? k_pool : plan->pool->desc.k_pool;
  const void* v = v_pool ? v_pool : plan->pool->desc.v_pool;
  if (plan->info.n_entries > 0 && (!k || !v)) return OCTO_EINVAL;
  plan->last_stream = (cudaStream_t)stream;
  octo::NvtxRange nv("octo_attn_fwd");
  if (!tc_disabled() && octo::fwd_tc_supported(plan, Hq))
    return octo::fwd_tc(plan, Hq, q, k, v, o, lse, scale, (cudaStream_t)stream);
  return octo::fwd_simt(plan, Hq, q, k, v, o, lse, scale, false, (cudaStream_t)stream);
}

size_t octo_attn_bwd_workspace_size(octo_plan_t plan, int32_t Hq) {
  if (!plan || Hq <= 0) return 0;
  const size_t simt = octo::align_up((size_t)plan->info.n_rows * Hq * sizeof(float), 256);
  if (plan->info.is_decode || check_heads(plan, Hq) != OCTO_OK || !octo::bwd_tc_supported(plan, Hq)) return simt;
  return std::max(simt, octo::bwd_tc_workspace(plan, Hq));
}

int octo_attn_bwd(octo_plan_t plan, int32_t Hq, const void* q, const void* k_pool, const void* v_pool, const void* o,
                  const float* lse, const void* dout, float* dq, float* dk_pool, float* dv_pool, float scale,
                  void* ws, size_t ws_bytes, void* stream) {
  if (!plan || plan->info.is_decode) return OCTO_EINVAL;
  if (int st = check_heads(plan, Hq)) return st;
  if (plan->info.n_rows > 0 && (!q || !o || !lse || !dout || !dq)) return OCTO_EINVAL;
  if (plan->info.n_touched_pages > 0 && (!dk_pool || !dv_pool)) return OCTO_EINVAL;
  if (ws_bytes < octo_attn_bwd_workspace_size(plan, Hq) || (ws_bytes > 0 && !ws && plan->info.n_rows > 0))
    return OCTO_EINVAL;
  const void* k = k_pool ? k_pool : plan->pool->desc.k_pool;
  const void* v = v_pool ? v_pool : plan->pool->desc.v_pool;
  if (plan->info.n_entries > 0 && (!k || !v)) return OCTO_EINVAL;
  plan->last_stream = (cudaStream_t)stream;
  octo::NvtxRange nv("octo_attn_bwd");
  // the tensor-core backward folds LSE / scale into its MMAs: it needs a finite 1 / scale
  if (!tc_disabled() && octo::bwd_tc_supported(plan, Hq) && scale != 0.f && std::isfinite(1.f / scale))
    return octo::bwd_tc(plan, Hq, q, k, v, o, lse, dout, dq, dk_pool, dv_pool, scale, ws, (cudaStream_t)stream);
  return octo::bwd_simt(plan, Hq, q, k, v, o, lse, dout, dq, dk_pool, dv_pool, scale, ws, (cudaStream_t)stream);
}

size_t octo_decode_workspace_size(octo_plan_t plan, int32_t Hq) {
  if (!plan || check_heads(plan, Hq)) return 0;
  return octo::decode_split_supported(plan, Hq) ? octo::decode_split_workspace(plan, Hq) : 0;
}

int octo_decode(octo_plan_t plan, int32_t Hq, const void* q, const void* k_pool, const void* v_pool, void* out,
                float* lse, float scale, void* ws, size_t ws_bytes, void* stream) {
  if (!plan || !plan->info.is_decode) return OCTO_EINVAL;
  if (int st = check_heads(plan, Hq)) return st;
  if (plan->info.n_rows > 0 && (!q || !out)) return OCTO_EINVAL;
  if (ws_bytes < octo_decode_workspace_size(plan, Hq)) return OCTO_EINVAL;
  const void* k = k_pool ? k_pool : plan->pool->desc.k_pool;
  const void* v = v_pool ? v_pool : plan->pool->desc.v_pool;
  if (plan->info.n_entries > 0 && (!k || !v)) return OCTO_EINVAL;
  plan->last_stream = (cudaStream_t)stream;
  octo::NvtxRange nv("octo_decode");
  if (octo::decode_split_supported(plan, Hq)) {
    if (!ws && plan->info.n_rows > 0) return OCTO_EINVAL;
    return octo::decode_split(plan, Hq, q, k, v, out, lse, scale, ws, (cudaStream_t)stream);
  }
  return octo::fwd_simt(plan, Hq, q, k, v, out, lse, scale, true, (cudaStream_t)stream);
}

int octo_decode_cursors(octo_pool_t pool, const octo_cursor_t* cursors, int32_t n, int32_t Hq, const void* q,
                        const void* k_pool, const void* v_pool, void* out, float* lse, float scale, void* ws,
                        size_t ws_bytes, void* stream) {
  if (!pool) return OCTO_EINVAL;
  octo_plan_t plan = nullptr;
  if (int st = octo_decode_plan(pool, cursors, n, stream, &plan)) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t need = octo_decode_workspace_size(plan, Hq);
  void* own = nullptr;
  int st = OCTO_OK;
  if (!ws && need > 0) {
    // stream-ordered workspace of the library's own, released after the decode
    st = octo::cuda_status(cudaMallocAsync(&own, need, s));
    ws = own;
    ws_bytes = need;
  }
  if (st == OCTO_OK) st = octo_decode(plan, Hq, q, k_pool, v_pool, out, lse, scale, ws, ws_bytes, stream);
  if (own) cudaFreeAsync(own, s);
  plan->last_stream = s;
  octo_plan_destroy(plan);   // stream-ordered: after the decode
  return st;
}

int octo_wait_selftest(octo_plan_t plan, uint32_t max_polls, void* stream) {
  if (!plan || max_polls == 0 || max_polls > octo::tc::kSpinLimit) return OCTO_EINVAL;
  plan->last_stream = (cudaStream_t)stream;
  k_wait_selftest<<<1, 32, 0, (cudaStream_t)stream>>>(plan->pool->d_status, max_polls);
  octo::count_launch();
  return octo::cuda_status(cudaGetLastError());
}

int octo_sync(octo_plan_t plan, void* stream) {
  if (!plan) return OCTO_EINVAL;
  OCTO_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  int32_t st = 0;
  OCTO_CUDA(cudaMemcpy(&st, plan->pool->d_status, 4, cudaMemcpyDeviceToHost));
  if (st != 0) OCTO_CUDA(cudaMemset(plan->pool->d_status, 0, 4));
  return st;
}

}  // extern "C"
