// Attention entry points: argument checks and dispatch between the tensor-core kernels
// (bf16, head_dim 128, page 64, q-tile 128) and the CUDA-core kernels (everything else).

#include <algorithm>
#include <cmath>
#include <cstdlib>

#include "internal.h"

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

// OCTO_DISABLE_TC=1 routes every call to the CUDA-core kernels (a diagnostic for
// comparing the two kernel families on the same shapes).
bool tc_disabled() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("OCTO_DISABLE_TC");
    v = (e && *e && *e != '0') ? 1 : 0;
  }
  return v == 1;
}

int check_heads(const octo_plan_s* p, int32_t Hq) {
  const int32_t Hkv = p->pool->desc.n_kv_heads;
  if (Hq <= 0 || Hq % Hkv != 0 || Hq > 65535) return OCTO_EINVAL;
  return OCTO_OK;
}

}  // namespace

extern "C" {

int octo_kernel_path(octo_plan_t plan, int32_t n_q_heads, int32_t which) {
  if (!plan || check_heads(plan, n_q_heads)) return -1;
  if (which == 2) return octo::decode_split_supported(plan, n_q_heads) ? 2 : 0;
  if (tc_disabled()) return 0;
  if (which == 0) return octo::fwd_tc_supported(plan, n_q_heads) ? 1 : 0;
  if (which == 1) return octo::bwd_tc_supported(plan, n_q_heads) ? 1 : 0;
  if (which == 2) return octo::decode_split_supported(plan, n_q_heads) ? 2 : 0;
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
  if (octo::decode_split_supported(plan, Hq)) {
    if (!ws && plan->info.n_rows > 0) return OCTO_EINVAL;
    return octo::decode_split(plan, Hq, q, k, v, out, lse, scale, ws, (cudaStream_t)stream);
  }
  return octo::fwd_simt(plan, Hq, q, k, v, out, lse, scale, true, (cudaStream_t)stream);
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
