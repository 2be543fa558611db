// Pool primitives: root / append / fork / mount / rewind / done / unpin / release.
//
// Octopus project page, primitives table: fork shares the parent's KV prefix by
// reference count (+K) without copying; read_thread mounts a sibling span c_A[s_A:e_A)
// into attention with the monotonic jump s = max(p_B, e_A + 1) ("Architecture &
// Co-Design", item 02) and consumes no KV page; rewind restores step k and keeps the
// pruned leaf; done freezes the cursor and pins its pages for parent/peer mounts.
//
// All of this is host metadata.  The only device work is the copy of appended K/V rows
// into their page slots.

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <set>
#include <tuple>

#include "internal.h"

namespace octo {

thread_local int g_last_cuda_error = 0;
static std::atomic<int64_t> g_launches{0};
void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int set_smem_limit(const void* func, int bytes) {
  int dev = 0;
  OCTO_CUDA(cudaGetDevice(&dev));
  static std::mutex mu;
  static std::set<std::tuple<uintptr_t, int, int>> done;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(reinterpret_cast<uintptr_t>(func), dev, bytes);
  if (done.count(key)) return OCTO_OK;
  OCTO_CUDA(cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
  done.insert(key);
  return OCTO_OK;
}

namespace {

template <typename T>
__global__ void append_rows_kernel(T* __restrict__ kp, T* __restrict__ vp, const T* __restrict__ k,
                                   const T* __restrict__ v, const int32_t* __restrict__ dst, int32_t n,
                                   int32_t Hkv, int32_t P, int32_t d) {
  // one block per appended token; dst[i] = page * P + slot
  int32_t i = blockIdx.x;
  if (i >= n) return;
  int32_t page = dst[i] / P, slot = dst[i] % P;
  for (int32_t e = threadIdx.x; e < Hkv * d; e += blockDim.x) {
    int32_t g = e / d, c = e % d;
    size_t o = (((size_t)page * Hkv + g) * P + slot) * d + c;
    size_t src = ((size_t)i * Hkv + g) * d + c;
    if (k) kp[o] = k[src];
    if (v) vp[o] = v[src];
  }
}

// one block per (page, K or V): zero the page's slots for every kv head
template <typename T>
__global__ void zero_pages_kernel(T* __restrict__ kp, T* __restrict__ vp, const int32_t* __restrict__ pages,
                                  int32_t n, size_t page_elems) {
  const int32_t i = blockIdx.x >> 1;
  if (i >= n) return;
  T* base = ((blockIdx.x & 1) ? vp : kp) + (size_t)pages[i] * page_elems;
  for (size_t e = threadIdx.x; e < page_elems; e += blockDim.x) base[e] = T(0);
}

}  // namespace

int launch_zero_pages(const octo_pool_desc& d, const int32_t* d_pages, int32_t n, cudaStream_t s) {
  if (n <= 0 || !d.k_pool || !d.v_pool) return OCTO_OK;
  const size_t pe = (size_t)d.n_kv_heads * d.page_size * d.head_dim;
  if (d.dtype == OCTO_DTYPE_F32)
    zero_pages_kernel<float><<<2 * n, 256, 0, s>>>((float*)d.k_pool, (float*)d.v_pool, d_pages, n, pe);
  else
    zero_pages_kernel<uint16_t><<<2 * n, 256, 0, s>>>((uint16_t*)d.k_pool, (uint16_t*)d.v_pool, d_pages, n, pe);
  count_launch();
  return cuda_status(cudaGetLastError());
}

int launch_append_rows(const octo_pool_desc& d, const int32_t* d_dst, int32_t n, const void* k, const void* v,
                       cudaStream_t s) {
  if (n <= 0) return OCTO_OK;
  int threads = std::min(256, d.n_kv_heads * d.head_dim);
  if (d.dtype == OCTO_DTYPE_F32)
    append_rows_kernel<float><<<n, threads, 0, s>>>((float*)d.k_pool, (float*)d.v_pool, (const float*)k,
                                                    (const float*)v, d_dst, n, d.n_kv_heads, d.page_size,
                                                    d.head_dim);
  else
    append_rows_kernel<uint16_t><<<n, threads, 0, s>>>((uint16_t*)d.k_pool, (uint16_t*)d.v_pool,
                                                       (const uint16_t*)k, (const uint16_t*)v, d_dst, n,
                                                       d.n_kv_heads, d.page_size, d.head_dim);
  count_launch();
  return cuda_status(cudaGetLastError());
}

}  // namespace octo

using octo::MountRec;
using octo::Segment;

static bool seg_ok(octo_pool_t p, octo_cursor_t c) {
  return p && c >= 0 && c < (int32_t)p->segs.size() && !p->segs[c].freed;
}
static bool writable(octo_pool_t p, octo_cursor_t c) {
  if (!seg_ok(p, c)) return false;
  const Segment& s = p->segs[c];
  return s.cursor && !s.frozen && !s.dead;
}

// Frees every segment that no live cursor or pin still needs.  A segment needs its
// parent (the prefix it sees) and the producers of the spans it mounted.  Freeing goes by
// reachability rather than by the counts alone because a reader may mount a span of its
// own descendant (a parent reading a child's result), which makes the two need each
// other; the refcount field stays the number of live holders.
static void collect(octo_pool_t p) {
  const int32_t n = (int32_t)p->segs.size();
  std::vector<char> live(n, 0);
  std::vector<int32_t> stack;
  for (int32_t s = 0; s < n; s++) {
    const Segment& g = p->segs[s];
    if (!g.freed && (g.cursor || g.pinned)) {
      live[s] = 1;
      stack.push_back(s);
    }
  }
  while (!stack.empty()) {
    int32_t s = stack.back();
    stack.pop_back();
    const Segment& g = p->segs[s];
    auto visit = [&](int32_t x) {
      if (x >= 0 && !live[x] && !p->segs[x].freed) {
        live[x] = 1;
        stack.push_back(x);
      }
    };
    visit(g.parent);
    for (int32_t mid : g.mounts) visit(p->mounts[mid].producer);
  }
  std::vector<int32_t> dead;
  for (int32_t s = 0; s < n; s++)
    if (!p->segs[s].freed && !live[s]) dead.push_back(s);
  for (int32_t s : dead) {
    Segment& g = p->segs[s];
    g.freed = true;
    g.refcount = 0;
    for (int32_t pg : g.pages) p->free_pages.insert(pg);
  }
  // the freed segments no longer hold their parent or their producers
  for (int32_t s : dead) {
    const Segment& g = p->segs[s];
    if (g.parent >= 0 && !p->segs[g.parent].freed) p->segs[g.parent].refcount -= 1;
    for (int32_t mid : g.mounts) {
      int32_t a = p->mounts[mid].producer;
      if (!p->segs[a].freed) p->segs[a].refcount -= 1;
    }
  }
}

static int32_t new_segment(octo_pool_t p, int32_t parent, int32_t fork, int32_t p0) {
  Segment g;
  g.parent = parent;
  g.fork = fork;
  g.created = ++p->seq;
  g.p0 = p0;
  g.p_next = p0;
  p->segs.push_back(std::move(g));
  return (int32_t)p->segs.size() - 1;
}

extern "C" {

const char* octo_strerror(int st) {
  switch (st) {
    case OCTO_OK: return "ok";
    case OCTO_EINVAL: return "invalid argument";
    case OCTO_ENOMEM: return "pool has no free page";
    case OCTO_ESTATE: return "cursor state does not allow this operation";
    case OCTO_ECUDA: return "CUDA error";
    case OCTO_ETIMEOUT: return "bounded device wait expired";
    case OCTO_ENOTSUP: return "unsupported shape or dtype";
    case OCTO_ESCRATCH: return "request exceeds the built-in scratch of the allocation-free decode";
  }
  return "unknown status";
}

int octo_last_cuda_error(void) { return octo::g_last_cuda_error; }

int64_t octo_launch_count(void) { return octo::g_launches.load(); }

int octo_pool_create(const octo_pool_desc* desc, octo_pool_t* out) {
  if (!desc || !out) return OCTO_EINVAL;
  const octo_pool_desc& d = *desc;
  if (d.num_pages <= 0 || d.page_size <= 0 || d.page_size > 128 || d.n_kv_heads <= 0 ||
      (d.head_dim != 64 && d.head_dim != 128) || (d.dtype != OCTO_DTYPE_F32 && d.dtype != OCTO_DTYPE_BF16))
    return OCTO_EINVAL;
  octo_pool_s* p = new (std::nothrow) octo_pool_s();
  if (!p) return OCTO_ENOMEM;
  p->desc = d;
  for (int32_t i = 0; i < d.num_pages; i++) p->free_pages.insert(p->free_pages.end(), i);
  // the device status word is allocated on first device use, so that host-only
  // pool work needs no GPU
  *out = p;
  return OCTO_OK;
}

int octo_pool_destroy(octo_pool_t p) {
  if (!p) return OCTO_EINVAL;
  if (p->d_status) {
    cudaDeviceSynchronize();   // no kernel of this pool may still use the status word
    cudaFree(p->d_status);
  }
  delete p;
  return OCTO_OK;
}

int octo_root(octo_pool_t p, octo_cursor_t* out) {
  if (!p || !out) return OCTO_EINVAL;
  *out = new_segment(p, -1, 0, 0);
  return OCTO_OK;
}

// Appends n tokens; with `rope` the K rows are rotated at their positions on the way in.
static int append_impl(octo_pool_t p, octo_cursor_t c, int32_t n, const void* k, const void* v, void* stream,
                       int32_t* pos_out, bool rope, float base) {
  if (!p || n < 0 || c < 0 || c >= (int32_t)p->segs.size()) return OCTO_EINVAL;
  if (!writable(p, c)) return OCTO_ESTATE;
  if ((k == nullptr) != (v == nullptr)) return OCTO_EINVAL;
  if (rope && octo::rope_validate(p->desc.head_dim, base)) return OCTO_EINVAL;
  Segment& g = p->segs[c];
  const int32_t P = p->desc.page_size;
  int64_t need = ((int64_t)g.len + n + P - 1) / P - (int64_t)g.pages.size();
  if (need < 0) need = 0;
  if (need > (int64_t)p->free_pages.size()) return OCTO_ENOMEM;
  if ((int64_t)g.len + n > INT32_MAX / 2) return OCTO_EINVAL;
  for (int64_t i = 0; i < need; i++) {
    auto it = p->free_pages.begin();
    g.pages.push_back(*it);
    p->free_pages.erase(it);
  }
  std::vector<int32_t> newp(g.pages.end() - need, g.pages.end());
  std::vector<int32_t> dst, pos;
  if (k) {
    dst.resize(n);
    pos.resize(n);
  }
  for (int32_t i = 0; i < n; i++) {
    int32_t idx = g.len + i;
    if (k) {
      dst[i] = g.pages[idx / P] * P + idx % P;
      pos[i] = g.p_next;
    }
    if (pos_out) pos_out[i] = g.p_next;
    g.pos.push_back(g.p_next++);
  }
  g.len += n;
  p->seq++;
  // Device work: pages new to the segment are zeroed in the pool arrays (the attention
  // kernels read whole pages and mask, so slots past a segment's end must hold finite
  // values), then the given K/V rows are copied into their slots.
  const bool zero = !newp.empty() && p->desc.k_pool && p->desc.v_pool;
  if (zero || (k && n > 0)) {
    cudaStream_t s = (cudaStream_t)stream;
    std::vector<int32_t> host(newp);
    host.insert(host.end(), dst.begin(), dst.end());
    if (rope) host.insert(host.end(), pos.begin(), pos.end());
    int32_t* d_buf = nullptr;
    OCTO_CUDA(cudaMallocAsync((void**)&d_buf, sizeof(int32_t) * host.size(), s));
    OCTO_CUDA(cudaMemcpyAsync(d_buf, host.data(), sizeof(int32_t) * host.size(), cudaMemcpyHostToDevice, s));
    int st = zero ? octo::launch_zero_pages(p->desc, d_buf, (int32_t)newp.size(), s) : OCTO_OK;
    if (st == OCTO_OK && k && n > 0)
      st = rope ? octo::launch_append_rope(p->desc, d_buf + newp.size(), d_buf + newp.size() + n, n, k, v, base, s)
                : octo::launch_append_rows(p->desc, d_buf + newp.size(), n, k, v, s);
    OCTO_CUDA(cudaFreeAsync(d_buf, s));
    // the host vector is pageable: make sure the copy has consumed it
    OCTO_CUDA(cudaStreamSynchronize(s));
    if (st != OCTO_OK) return st;
  }
  return OCTO_OK;
}

int octo_append(octo_pool_t p, octo_cursor_t c, int32_t n, const void* k, const void* v, void* stream,
                int32_t* pos_out) {
  return append_impl(p, c, n, k, v, stream, pos_out, false, 0.f);
}

int octo_append_rope(octo_pool_t p, octo_cursor_t c, int32_t n, const void* k, const void* v, float base,
                     void* stream, int32_t* pos_out) {
  return append_impl(p, c, n, k, v, stream, pos_out, true, base);
}

int octo_append_step(octo_pool_t p, const octo_cursor_t* cursors, int32_t n, const void* k, const void* v,
                     float rope_base, void* stream, int32_t* pos_out) {
  octo::NvtxRange nv("octo_append_step");
  if (!p || n < 0 || (n > 0 && !cursors)) return OCTO_EINVAL;
  if ((k == nullptr) != (v == nullptr)) return OCTO_EINVAL;
  const bool rope = rope_base != 0.f;
  if (rope && octo::rope_validate(p->desc.head_dim, rope_base)) return OCTO_EINVAL;
  const int32_t P = p->desc.page_size;
  // checks first, so that a refused call changes nothing
  std::vector<int32_t> sorted(cursors, cursors + n);
  std::sort(sorted.begin(), sorted.end());
  if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end()) return OCTO_EINVAL;
  int64_t need = 0;
  for (int32_t i = 0; i < n; i++) {
    const int32_t c = cursors[i];
    if (c < 0 || c >= (int32_t)p->segs.size()) return OCTO_EINVAL;
    if (!writable(p, c)) return OCTO_ESTATE;
    const Segment& g = p->segs[c];
    if ((int64_t)g.len + 1 > INT32_MAX / 2) return OCTO_EINVAL;
    if ((int64_t)g.len / P >= (int64_t)g.pages.size()) need++;
  }
  if (need > (int64_t)p->free_pages.size()) return OCTO_ENOMEM;
  // host arrays for the device: fresh pages | destination slots | positions
  std::vector<int32_t> host;
  host.reserve((size_t)need + 2 * (size_t)n);
  std::vector<int32_t> dst(n), pos(n);
  for (int32_t i = 0; i < n; i++) {
    Segment& g = p->segs[cursors[i]];
    if (g.len / P >= (int32_t)g.pages.size()) {
      auto it = p->free_pages.begin();
      g.pages.push_back(*it);
      host.push_back(*it);
      p->free_pages.erase(it);
    }
    dst[i] = g.pages[g.len / P] * P + g.len % P;
    pos[i] = g.p_next;
    if (pos_out) pos_out[i] = g.p_next;
    g.pos.push_back(g.p_next++);
    g.len += 1;
  }
  p->seq++;
  const int32_t n_fresh = (int32_t)host.size();
  const bool zero = n_fresh > 0 && p->desc.k_pool && p->desc.v_pool;
  if (!zero && !(k && n > 0)) return OCTO_OK;
  host.insert(host.end(), dst.begin(), dst.end());
  host.insert(host.end(), pos.begin(), pos.end());
  cudaStream_t s = (cudaStream_t)stream;
  int32_t* d_buf = nullptr;
  OCTO_CUDA(cudaMallocAsync((void**)&d_buf, sizeof(int32_t) * host.size(), s));
  // pageable source: staged by the runtime before the call returns, so `host` may go
  OCTO_CUDA(cudaMemcpyAsync(d_buf, host.data(), sizeof(int32_t) * host.size(), cudaMemcpyHostToDevice, s));
  int st = zero ? octo::launch_zero_pages(p->desc, d_buf, n_fresh, s) : OCTO_OK;
  if (st == OCTO_OK && k && n > 0)
    st = rope ? octo::launch_append_rope(p->desc, d_buf + n_fresh, d_buf + n_fresh + n, n, k, v, rope_base, s)
              : octo::launch_append_rows(p->desc, d_buf + n_fresh, n, k, v, s);
  OCTO_CUDA(cudaFreeAsync(d_buf, s));
  return st;
}

int octo_fork(octo_pool_t p, octo_cursor_t c, int32_t n, octo_cursor_t* out) {
  if (!p || !out || n < 1 || c < 0 || c >= (int32_t)p->segs.size()) return OCTO_EINVAL;
  if (!writable(p, c)) return OCTO_ESTATE;
  int32_t f = p->segs[c].len, pn = p->segs[c].p_next;
  for (int32_t i = 0; i < n; i++) out[i] = new_segment(p, c, f, pn);
  p->segs[c].refcount += n;
  return OCTO_OK;
}

// True if producer tokens [a, b) already appear in the context the reader's next row
// would see: the producer lies on the reader's lineage below the cut-off, or a mount
// of the same producer visible on that lineage overlaps the span.
static bool span_visible(octo_pool_t p, int32_t r, int32_t A, int32_t a, int32_t b) {
  // own mounts (all of them precede the next row)
  for (int32_t mid : p->segs[r].mounts) {
    const MountRec& m = p->mounts[mid];
    if (m.producer == A && m.a < b && a < m.b) return true;
  }
  int32_t x = r, cutoff = p->segs[r].len;
  if (x == A && a < cutoff) return true;
  while (p->segs[x].parent >= 0) {
    const Segment& child = p->segs[x];
    int32_t par = child.parent;
    cutoff = child.fork;
    if (par == A && a < cutoff) return true;
    for (int32_t mid : p->segs[par].mounts) {
      const MountRec& m = p->mounts[mid];
      if (m.m <= child.fork && m.created < child.created && m.producer == A && m.a < b && a < m.b) return true;
    }
    x = par;
  }
  return false;
}

int octo_mount(octo_pool_t p, octo_cursor_t r, octo_cursor_t A, int32_t a, int32_t b, int32_t* new_pos) {
  if (!p || r < 0 || r >= (int32_t)p->segs.size()) return OCTO_EINVAL;
  if (!writable(p, r)) return OCTO_ESTATE;
  if (!seg_ok(p, A)) return OCTO_EINVAL;
  if (a < 0 || a >= b || b > p->segs[A].len) return OCTO_EINVAL;
  if (span_visible(p, r, A, a, b)) return OCTO_EINVAL;
  Segment& R = p->segs[r];
  int32_t e_A = p->segs[A].pos[b - 1] + 1;
  int32_t np = std::max(R.p_next, e_A + 1);
  MountRec m{r, R.len, A, a, b, np - R.p_next, ++p->seq};
  R.p_next = np;
  R.mounts.push_back((int32_t)p->mounts.size());
  p->mounts.push_back(m);
  p->segs[A].refcount += 1;
  if (new_pos) *new_pos = np;
  return OCTO_OK;
}

int octo_rewind(octo_pool_t p, octo_cursor_t c, int32_t k, octo_cursor_t* out) {
  if (!p || !out || c < 0 || c >= (int32_t)p->segs.size()) return OCTO_EINVAL;
  if (!writable(p, c)) return OCTO_ESTATE;
  Segment& g = p->segs[c];
  if (k < 0 || k > g.len) return OCTO_EINVAL;
  int32_t p0 = k < g.len ? g.pos[k] : g.p_next;
  g.dead = true;
  g.cursor = false;   // the cursor reference moves to the continuation ...
  // ... and the continuation's parent reference replaces it: refcount unchanged
  *out = new_segment(p, c, k, p0);
  return OCTO_OK;
}

int octo_done(octo_pool_t p, octo_cursor_t c) {
  if (!p || c < 0 || c >= (int32_t)p->segs.size()) return OCTO_EINVAL;
  if (!writable(p, c)) return OCTO_ESTATE;
  Segment& g = p->segs[c];
  g.frozen = true;
  g.pinned = true;
  g.refcount += 1;
  p->seq++;
  return OCTO_OK;
}

int octo_unpin(octo_pool_t p, octo_cursor_t c) {
  if (!p || c < 0 || c >= (int32_t)p->segs.size()) return OCTO_EINVAL;
  if (!seg_ok(p, c) || !p->segs[c].pinned) return OCTO_ESTATE;
  p->segs[c].pinned = false;
  p->segs[c].refcount -= 1;
  p->seq++;
  collect(p);
  return OCTO_OK;
}

int octo_release(octo_pool_t p, octo_cursor_t c) {
  if (!p || c < 0 || c >= (int32_t)p->segs.size()) return OCTO_EINVAL;
  if (!seg_ok(p, c) || !p->segs[c].cursor) return OCTO_ESTATE;
  p->segs[c].cursor = false;
  p->segs[c].refcount -= 1;
  p->seq++;
  collect(p);
  return OCTO_OK;
}

int octo_pool_info(octo_pool_t p, int32_t* n_segments, int32_t* free_pages, int32_t* n_mounts) {
  if (!p) return OCTO_EINVAL;
  if (n_segments) *n_segments = (int32_t)p->segs.size();
  if (free_pages) *free_pages = (int32_t)p->free_pages.size();
  if (n_mounts) *n_mounts = (int32_t)p->mounts.size();
  return OCTO_OK;
}

int octo_pool_query(octo_pool_t p, octo_pool_state* st) {
  if (!p || !st || st->seg_capacity < 0) return OCTO_EINVAL;
  const int32_t ns = (int32_t)p->segs.size(), np = p->desc.num_pages;
  if ((st->refcount || st->n_pages) && st->seg_capacity < ns) return OCTO_EINVAL;
  for (int32_t s = 0; s < ns; s++) {
    const Segment& g = p->segs[s];
    if (st->refcount) st->refcount[s] = g.freed ? 0 : g.refcount;
    if (st->n_pages) st->n_pages[s] = (int32_t)g.pages.size();
  }
  if (st->page_owner) {
    std::fill(st->page_owner, st->page_owner + np, -1);
    for (int32_t s = 0; s < ns; s++) {
      const Segment& g = p->segs[s];
      if (g.freed) continue;
      for (int32_t pg : g.pages) st->page_owner[pg] = s;
    }
  }
  st->n_segments = ns;
  st->free_pages = (int32_t)p->free_pages.size();
  st->n_mounts = (int32_t)p->mounts.size();
  st->num_pages = np;
  return OCTO_OK;
}

int octo_seg_query(octo_pool_t p, octo_cursor_t c, octo_seg_info* info, int32_t* pos, int32_t* pages) {
  if (!p || c < 0 || c >= (int32_t)p->segs.size()) return OCTO_EINVAL;
  const Segment& g = p->segs[c];
  if (info) {
    info->parent = g.parent;
    info->fork = g.fork;
    info->len = g.len;
    info->n_pages = (int32_t)g.pages.size();
    info->refcount = g.freed ? 0 : g.refcount;
    info->p_next = g.p_next;
    info->flags = (g.cursor ? 1 : 0) | (g.pinned ? 2 : 0) | (g.frozen ? 4 : 0) | (g.dead ? 8 : 0) |
                  (g.freed ? 16 : 0);
  }
  if (pos) std::copy(g.pos.begin(), g.pos.end(), pos);
  if (pages) std::copy(g.pages.begin(), g.pages.end(), pages);
  return OCTO_OK;
}

}  // extern "C"
