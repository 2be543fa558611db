// DAG -> block-sparse tile list compiler (K0).
//
// Octopus project page, "Architecture & Co-Design" item 03: the trainer compiles the
// branched tree and its live KV mount edges into one unpadded 1D forward/backward pass.
// Here that compilation runs on the GPU:
//
//   layout   packed segments -> row_base (exclusive scan of lengths), q-tiles of bm rows
//            per segment, and the position id of every packed row (the segment's start
//            position plus its index plus the jumps of its own mounts at m <= index;
//            item 02's s = max(p_B, e_A + 1) is applied on the host when mounting)
//   count    one warp per q-tile walks the tile's tree path from the root down and
//            counts (page, source) blocks
//   scan     entries per tile -> tile_off
//   fill     the same walk writes the entries, in the order their keys first appear in
//            the context of the tile's last row
//   csc      entries grouped by kv page, each page's list in entry order
//
// Order of a segment X's contribution to a context (tokens [0, L) of X, mounts of X with
// point m <= mcap): a mount at point m is placed right before X's token m, so its pages
// come after X's pages [0, ceil(m/P)) and before the rest.  An ancestor contributes its
// first f tokens and the mounts it held when the child on the path was created with
// m <= f; the tile's own segment contributes tokens [0, t1) and its mounts with m <= t1-1.

#include <algorithm>
#include <cstring>
#include <numeric>

#include "internal.h"

namespace octo {
namespace {

constexpr int kMaxDepth = 64;
constexpr int kSortCap = 32768;   // max entries per kv page the CSC sort handles

struct WalkArgs {
  const DevSeg* segs;
  const int32_t* pages;
  const DevMount* mounts;
  int32_t P;
};

__device__ __forceinline__ int32_t cdiv(int32_t a, int32_t b) { return (a + b - 1) / b; }

// Walks one tile [t0, t1) of segment S.  In count mode returns the number of entries;
// in fill mode writes them to out[0..n).  All 32 lanes call it with the same arguments.
template <bool FILL>
__device__ int32_t walk_tile(const WalkArgs& w, int32_t tile, int32_t S, int32_t t0, int32_t t1,
                             octo_entry* out, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int32_t P = w.P;
  int32_t chain[kMaxDepth];
  int depth = 0;
  for (int32_t x = S; x >= 0; x = w.segs[x].parent) {
    if (depth == kMaxDepth) {
      if (lane == 0) atomicExch(status, OCTO_ENOTSUP);
      return 0;
    }
    chain[depth++] = x;
  }
  int32_t n = 0;  // entries emitted so far (uniform across lanes)
  for (int lvl = depth - 1; lvl >= 0; lvl--) {
    const int32_t X = chain[lvl];
    const DevSeg sx = w.segs[X];
    const bool own = (lvl == 0);
    int32_t L, mcap, before;
    if (own) {
      L = t1;
      mcap = t1 - 1;
      before = 0x7fffffff;
    } else {
      const DevSeg& child = w.segs[chain[lvl - 1]];
      L = child.fork;
      mcap = child.fork;
      before = child.created_lo;
    }
    const int32_t npages = cdiv(L, P);
    int32_t next_page = 0;
    // path pages [lo, hi) of X
    auto emit_pages = [&](int32_t lo, int32_t hi) {
      int32_t cnt = hi - lo;
      if (cnt <= 0) return;
      if (FILL) {
        for (int32_t k = lane; k < cnt; k += 32) {
          int32_t pi = lo + k;
          int32_t ps = pi * P;
          octo_entry e;
          e.q_tile = (uint32_t)tile;
          e.kv_page = (uint32_t)w.pages[sx.page_off + pi];
          e.kv_lo = 0;
          e.src = -1;
          if (own) {
            int32_t kv_hi = min(P, t1 - ps);
            int32_t q_lo = max(0, ps - t0);
            int32_t dv = t0 - ps;
            bool causal = (q_lo + dv) < (kv_hi - 1);
            e.kv_hi = (uint16_t)kv_hi;
            e.q_lo = (uint16_t)q_lo;
            e.flags = causal ? 1 : 0;
            e.diag = causal ? dv : 0;
          } else {
            e.kv_hi = (uint16_t)min(P, L - ps);
            e.q_lo = 0;
            e.flags = 0;
            e.diag = 0;
          }
          out[n + k] = e;
        }
      }
      n += cnt;
    };
    for (int32_t mi = 0; mi < sx.mount_cnt; mi++) {
      const DevMount M = w.mounts[sx.mount_off + mi];
      if (M.m > mcap || (!own && M.created >= before)) continue;
      int32_t upto = cdiv(M.m, P);
      if (upto > next_page) {
        emit_pages(next_page, upto);
        next_page = upto;
      }
      const DevSeg sa = w.segs[M.producer];
      int32_t pa = M.a / P, pb = (M.b - 1) / P;
      int32_t cnt = pb - pa + 1;
      if (FILL) {
        int32_t q_lo = (own && M.m > t0) ? M.m - t0 : 0;
        for (int32_t k = lane; k < cnt; k += 32) {
          int32_t pj = pa + k;
          octo_entry e;
          e.q_tile = (uint32_t)tile;
          e.kv_page = (uint32_t)w.pages[sa.page_off + pj];
          e.kv_lo = (uint16_t)(max(M.a, pj * P) - pj * P);
          e.kv_hi = (uint16_t)(min(M.b, (pj + 1) * P) - pj * P);
          e.q_lo = (uint16_t)q_lo;
          e.flags = 0;
          e.diag = 0;
          e.src = M.id;
          out[n + k] = e;
        }
      }
      n += cnt;
    }
    emit_pages(next_page, npages);
  }
  return n;
}

__global__ void k_layout(const DevSeg* __restrict__ segs, const int32_t* __restrict__ seg_order, int32_t n_segs,
                         int32_t bm, int32_t* __restrict__ seg_row_base, int32_t* __restrict__ seg_tile_base) {
  // single block: exclusive scans of segment lengths and tile counts
  __shared__ int32_t warp_a[32], warp_b[32];
  __shared__ int32_t carry_a, carry_b;
  if (threadIdx.x == 0) carry_a = carry_b = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int32_t base = 0; base < n_segs; base += blockDim.x) {
    int32_t i = base + threadIdx.x;
    int32_t a = 0, b = 0;
    if (i < n_segs) {
      a = segs[seg_order[i]].len;
      b = cdiv(a, bm);
    }
    int32_t sa = a, sb = b;
    for (int o = 1; o < 32; o <<= 1) {
      int32_t ya = __shfl_up_sync(0xffffffffu, sa, o), yb = __shfl_up_sync(0xffffffffu, sb, o);
      if (lane >= o) sa += ya, sb += yb;
    }
    if (lane == 31) warp_a[wid] = sa, warp_b[wid] = sb;
    __syncthreads();
    if (wid == 0) {
      int32_t va = lane < (int)(blockDim.x >> 5) ? warp_a[lane] : 0;
      int32_t vb = lane < (int)(blockDim.x >> 5) ? warp_b[lane] : 0;
      for (int o = 1; o < 32; o <<= 1) {
        int32_t ya = __shfl_up_sync(0xffffffffu, va, o), yb = __shfl_up_sync(0xffffffffu, vb, o);
        if (lane >= o) va += ya, vb += yb;
      }
      warp_a[lane] = va;
      warp_b[lane] = vb;
    }
    __syncthreads();
    int32_t pa = (wid ? warp_a[wid - 1] : 0) + sa - a + carry_a;
    int32_t pb = (wid ? warp_b[wid - 1] : 0) + sb - b + carry_b;
    if (i < n_segs) {
      seg_row_base[i] = pa;
      seg_tile_base[i] = pb;
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) {
      carry_a = pa + a;
      carry_b = pb + b;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) seg_tile_base[n_segs] = carry_b;
}

// one block per packed segment: tile table and row positions
__global__ void k_tiles(const DevSeg* __restrict__ segs, const DevMount* __restrict__ mounts,
                        const int32_t* __restrict__ seg_order, const int32_t* __restrict__ seg_row_base,
                        const int32_t* __restrict__ seg_tile_base, int32_t bm, int32_t* __restrict__ tile_seg,
                        int32_t* __restrict__ tile_t0, int32_t* __restrict__ tile_rows,
                        int32_t* __restrict__ tile_row0, int32_t* __restrict__ row_pos) {
  const int32_t si = blockIdx.x;
  const int32_t S = seg_order[si];
  const DevSeg s = segs[S];
  const int32_t r0 = seg_row_base[si], tb = seg_tile_base[si];
  for (int32_t t = threadIdx.x; t < cdiv(s.len, bm); t += blockDim.x) {
    tile_seg[tb + t] = S;
    tile_t0[tb + t] = t * bm;
    tile_rows[tb + t] = min(bm, s.len - t * bm);
    tile_row0[tb + t] = r0 + t * bm;
  }
  for (int32_t i = threadIdx.x; i < s.len; i += blockDim.x) {
    int32_t p = s.p0 + i;
    for (int32_t k = 0; k < s.mount_cnt; k++) {
      const DevMount& M = mounts[s.mount_off + k];
      if (M.m <= i) p += M.jump;
    }
    row_pos[r0 + i] = p;
  }
}

// decode: one single-row tile per cursor (its last token)
__global__ void k_decode_tiles(const DevSeg* __restrict__ segs, const DevMount* __restrict__ mounts,
                               const int32_t* __restrict__ cursors, int32_t n, int32_t* __restrict__ tile_seg,
                               int32_t* __restrict__ tile_t0, int32_t* __restrict__ tile_rows,
                               int32_t* __restrict__ tile_row0, int32_t* __restrict__ row_pos,
                               int32_t* __restrict__ seg_row_base) {
  int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const DevSeg s = segs[cursors[i]];
  int32_t last = s.len - 1;
  tile_seg[i] = cursors[i];
  tile_t0[i] = last;
  tile_rows[i] = 1;
  tile_row0[i] = i;
  seg_row_base[i] = i;
  int32_t p = s.p0 + last;
  for (int32_t k = 0; k < s.mount_cnt; k++) {
    const DevMount& M = mounts[s.mount_off + k];
    if (M.m <= last) p += M.jump;
  }
  row_pos[i] = p;
}

__global__ void k_count(WalkArgs w, const int32_t* __restrict__ tile_seg, const int32_t* __restrict__ tile_t0,
                        const int32_t* __restrict__ tile_rows, int32_t n_tiles, int32_t* __restrict__ cnt,
                        int32_t* status) {
  int32_t tile = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (tile >= n_tiles) return;
  int32_t t0 = tile_t0[tile];
  int32_t c = walk_tile<false>(w, tile, tile_seg[tile], t0, t0 + tile_rows[tile], nullptr, status);
  if ((threadIdx.x & 31) == 0) cnt[tile] = c;
}

__global__ void k_fill(WalkArgs w, const int32_t* __restrict__ tile_seg, const int32_t* __restrict__ tile_t0,
                       const int32_t* __restrict__ tile_rows, int32_t n_tiles, const int32_t* __restrict__ tile_off,
                       octo_entry* __restrict__ entries, int32_t* status) {
  int32_t tile = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (tile >= n_tiles) return;
  int32_t t0 = tile_t0[tile];
  walk_tile<true>(w, tile, tile_seg[tile], t0, t0 + tile_rows[tile], entries + tile_off[tile], status);
}

// exclusive scan of in[0..n) into out[0..n], out[n] = total; optional max of in
__global__ void k_scan(const int32_t* __restrict__ in, int32_t n, int32_t* __restrict__ out,
                       int32_t* __restrict__ max_out) {
  __shared__ int32_t warp_s[32], warp_m[32];
  __shared__ int32_t carry, mx;
  if (threadIdx.x == 0) carry = 0, mx = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int32_t base = 0; base < n; base += blockDim.x) {
    int32_t i = base + threadIdx.x;
    int32_t v = i < n ? in[i] : 0;
    int32_t s = v, m = v;
    for (int o = 1; o < 32; o <<= 1) {
      int32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
      m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    }
    if (lane == 31) warp_s[wid] = s;
    if (lane == 0) warp_m[wid] = m;
    __syncthreads();
    if (wid == 0) {
      int nw = blockDim.x >> 5;
      int32_t x = lane < nw ? warp_s[lane] : 0;
      int32_t y = lane < nw ? warp_m[lane] : 0;
      for (int o = 1; o < 32; o <<= 1) {
        int32_t z = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += z;
        y = max(y, __shfl_xor_sync(0xffffffffu, y, o));
      }
      warp_s[lane] = x;
      if (lane == 0) mx = max(mx, y);
    }
    __syncthreads();
    int32_t excl = (wid ? warp_s[wid - 1] : 0) + s - v + carry;
    if (i < n) out[i] = excl;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = excl + v;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    out[n] = carry;
    if (max_out) *max_out = mx;
  }
}

// per entry: kv-page histogram and visible pair count
__global__ void k_page_hist(const octo_entry* __restrict__ entries, int64_t n, const int32_t* __restrict__ tile_rows,
                            int32_t* __restrict__ page_cnt, unsigned long long* __restrict__ pairs) {
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  unsigned long long pr = 0;
  if (i < n) {
    octo_entry e = entries[i];
    atomicAdd(&page_cnt[e.kv_page], 1);
    int32_t rows = tile_rows[e.q_tile];
    if (!(e.flags & 1)) {
      pr = (unsigned long long)(rows - e.q_lo) * (unsigned long long)(e.kv_hi - e.kv_lo);
    } else {
      for (int32_t r = e.q_lo; r < rows; r++) {
        int32_t hi = min((int32_t)e.kv_hi, r + e.diag + 1);
        if (hi > e.kv_lo) pr += (unsigned long long)(hi - e.kv_lo);
      }
    }
  }
  for (int o = 16; o; o >>= 1) pr += __shfl_xor_sync(0xffffffffu, pr, o);
  if ((threadIdx.x & 31) == 0 && pr) atomicAdd(pairs, pr);
}

__global__ void k_csc_scatter(const octo_entry* __restrict__ entries, int64_t n, const int32_t* __restrict__ page_off,
                              int32_t* __restrict__ page_fill, int32_t* __restrict__ csc) {
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  int32_t p = entries[i].kv_page;
  int32_t slot = atomicAdd(&page_fill[p], 1);
  csc[page_off[p] + slot] = (int32_t)i;
}

// one block per touched page: sort its CSC slice ascending (bitonic in shared memory)
// Advances a decode plan by one token per cursor, one warp per cursor: the cursor's
// entries move to their new place; its newest token either widens the entry of its own
// page (kv_hi + 1) or, on a fresh page, adds that page's entry at the end of the list (own
// pages follow everything else in context order); the row moves to the new token.
// adv[2 i] = the token's page, adv[2 i + 1] = 1 if the page is fresh.
__global__ void k_decode_advance(const octo_entry* __restrict__ old_e, const int32_t* __restrict__ old_off,
                                 const int32_t* __restrict__ new_off, const int32_t* __restrict__ adv, int32_t n,
                                 octo_entry* __restrict__ out, int32_t* __restrict__ tile_t0,
                                 int32_t* __restrict__ row_pos) {
  const int32_t i = (int32_t)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= n) return;
  const int32_t a = old_off[i], b = old_off[i + 1], o = new_off[i];
  const int32_t page = adv[2 * i], fresh = adv[2 * i + 1];
  for (int32_t k = lane; k < b - a; k += 32) {
    octo_entry e = old_e[a + k];
    if (!fresh && e.kv_page == (uint32_t)page && e.src == -1) e.kv_hi = (uint16_t)(e.kv_hi + 1);
    out[o + k] = e;
  }
  if (lane == 0) {
    if (fresh) {
      octo_entry e;
      e.q_tile = (uint32_t)i;
      e.kv_page = (uint32_t)page;
      e.kv_lo = 0;
      e.kv_hi = 1;
      e.q_lo = 0;
      e.flags = 0;
      e.diag = 0;
      e.src = -1;
      out[o + (b - a)] = e;
    }
    tile_t0[i] += 1;
    row_pos[i] += 1;
  }
}

// Advance of a decode plan in which no cursor's newest token opens a page: in place, one
// thread per cursor.  The newest token sits on the cursor's last own page, whose entry is
// the last path entry (src -1) of the cursor's list (mounts placed after it in context
// order come later and are skipped); it widens by one slot, and the row moves on.
__global__ void k_decode_widen(octo_entry* __restrict__ entries, const int32_t* __restrict__ tile_off, int32_t n,
                               int32_t* __restrict__ tile_t0, int32_t* __restrict__ row_pos) {
  const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  for (int32_t k = tile_off[i + 1] - 1; k >= tile_off[i]; k--)
    if (entries[k].src == -1) {
      entries[k].kv_hi = (uint16_t)(entries[k].kv_hi + 1);
      break;
    }
  tile_t0[i] += 1;
  row_pos[i] += 1;
}

// number of values of the ascending array a[0, n) below x
__device__ __forceinline__ int32_t count_below(const int32_t* __restrict__ a, int32_t n, int32_t x) {
  int32_t lo = 0, hi = n;
  while (lo < hi) {
    const int32_t mid = (lo + hi) >> 1;
    if (a[mid] < x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// CSC of an advanced decode plan whose fresh pages (ascending, none read before) each get
// one entry: an old position k of page p moves up by the fresh pages below p and its entry
// index by the entries inserted before its cursor; each fresh page lists its new entry.
// Threads [0, n_old) move the old positions, [n_old, n_old + n) place the cursors' new
// entries.  adv[2 i] = cursor i's newest page, adv[2 i + 1] = 1 if it is fresh.
__global__ void k_csc_advance(const int32_t* __restrict__ old_csc, const octo_entry* __restrict__ old_e,
                              int32_t n_old, const int32_t* __restrict__ old_off, const int32_t* __restrict__ new_off,
                              const int32_t* __restrict__ old_page_off, const int32_t* __restrict__ fresh_pages,
                              int32_t m, const int32_t* __restrict__ adv, int32_t n, int32_t* __restrict__ out) {
  const int32_t k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k < n_old) {
    const int32_t e = old_csc[k];
    const octo_entry x = old_e[e];
    const int32_t t = (int32_t)x.q_tile;
    out[k + count_below(fresh_pages, m, (int32_t)x.kv_page)] = e + (new_off[t] - old_off[t]);
  } else if (k < n_old + n) {
    const int32_t i = k - n_old;
    if (adv[2 * i + 1]) {
      const int32_t p = adv[2 * i];
      out[old_page_off[p] + count_below(fresh_pages, m, p)] = new_off[i + 1] - 1;
    }
  }
}

// page_off after adding one entry on each fresh page
__global__ void k_pageoff_advance(const int32_t* __restrict__ old_page_off, int32_t num_pages,
                                  const int32_t* __restrict__ fresh_pages, int32_t m, int32_t* __restrict__ out) {
  const int32_t p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p <= num_pages) out[p] = old_page_off[p] + count_below(fresh_pages, m, p);
}

// ascending merge of the touched pages with the fresh ones
__global__ void k_touched_advance(const int32_t* __restrict__ old_t, int32_t n_old,
                                  const int32_t* __restrict__ fresh_pages, int32_t m, int32_t* __restrict__ out) {
  const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n_old) {
    out[i + count_below(fresh_pages, m, old_t[i])] = old_t[i];
  } else if (i < n_old + m) {
    const int32_t k = i - n_old;
    out[count_below(old_t, n_old, fresh_pages[k]) + k] = fresh_pages[k];
  }
}

// kv_page of the first entry of each split (decode plans)
__global__ void k_split_first_page(const octo_entry* __restrict__ entries, const int32_t* __restrict__ split_e0,
                                   int32_t n, int32_t* __restrict__ out) {
  const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = (int32_t)entries[split_e0[i]].kv_page;
}

__global__ void k_csc_sort(const int32_t* __restrict__ touched, const int32_t* __restrict__ page_off,
                           int32_t* __restrict__ csc, int32_t cap) {
  extern __shared__ int32_t sm[];
  int32_t p = touched[blockIdx.x];
  int32_t lo = page_off[p], n = page_off[p + 1] - lo;
  if (n <= 1) return;
  int32_t m = 1;
  while (m < n) m <<= 1;
  for (int32_t i = threadIdx.x; i < m; i += blockDim.x) sm[i] = i < n ? csc[lo + i] : 0x7fffffff;
  __syncthreads();
  for (int32_t k = 2; k <= m; k <<= 1) {
    for (int32_t j = k >> 1; j > 0; j >>= 1) {
      for (int32_t i = threadIdx.x; i < m; i += blockDim.x) {
        int32_t l = i ^ j;
        if (l > i) {
          bool up = (i & k) == 0;
          int32_t a = sm[i], b = sm[l];
          if ((a > b) == up) {
            sm[i] = b;
            sm[l] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int32_t i = threadIdx.x; i < n; i += blockDim.x) csc[lo + i] = sm[i];
  (void)cap;
}

// touched pages (ascending) by compaction of page_off differences; single block
__global__ void k_touched(const int32_t* __restrict__ page_off, int32_t num_pages, int32_t* __restrict__ touched,
                          int32_t* __restrict__ n_out) {
  __shared__ int32_t warp_s[32];
  __shared__ int32_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int32_t base = 0; base < num_pages; base += blockDim.x) {
    int32_t i = base + threadIdx.x;
    int32_t v = (i < num_pages && page_off[i + 1] > page_off[i]) ? 1 : 0;
    int32_t s = v;
    for (int o = 1; o < 32; o <<= 1) {
      int32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane == 31) warp_s[wid] = s;
    __syncthreads();
    if (wid == 0) {
      int nw = blockDim.x >> 5;
      int32_t x = lane < nw ? warp_s[lane] : 0;
      for (int o = 1; o < 32; o <<= 1) {
        int32_t z = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += z;
      }
      warp_s[lane] = x;
    }
    __syncthreads();
    int32_t excl = (wid ? warp_s[wid - 1] : 0) + s - v + carry;
    if (v) touched[excl] = i;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = excl + v;
    __syncthreads();
  }
  if (threadIdx.x == 0) *n_out = carry;
}

// One block per page pair (pa, pb): the pair's work items.  Every entry of pa's reader
// list gives an item; when the next entry of the tile list is pb's, for the same query
// tile, it joins that item as its second half.  pb's remaining entries follow as items
// of their own, in list order (a block-wide compaction).  Items of one pair are thus in
// a fixed order, and every entry of pa and pb is in exactly one of them.
__device__ __forceinline__ void pair_half(PairItem& it, int h, const octo_entry* e) {
  if (e) {
    it.lo[h] = (int16_t)e->kv_lo;
    it.hi[h] = (int16_t)e->kv_hi;
    it.qlo[h] = (int16_t)e->q_lo;
    if (e->flags & 1) it.causal |= (int16_t)(1 << h);
    it.diag[h] = e->diag;
  } else {
    it.lo[h] = it.hi[h] = it.qlo[h] = 0;
    it.diag[h] = 0;
  }
}

__global__ void k_pair_items(const int32_t* __restrict__ pair_pages, const int32_t* __restrict__ pair_off,
                             const int32_t* __restrict__ page_off, const int32_t* __restrict__ csc,
                             const octo_entry* __restrict__ entries, int32_t n_entries,
                             const int32_t* __restrict__ tile_row0, const int32_t* __restrict__ tile_rows,
                             PairItem* __restrict__ items, int32_t* __restrict__ pair_n) {
  __shared__ int32_t warp_s[32];
  __shared__ int32_t carry;
  const int32_t b = blockIdx.x;
  const int32_t pa = pair_pages[2 * b], pb = pair_pages[2 * b + 1];
  const int32_t base = pair_off[b];
  const int32_t oa = page_off[pa], la = page_off[pa + 1] - oa;
  for (int32_t i = threadIdx.x; i < la; i += blockDim.x) {
    const int32_t e = csc[oa + i];
    const octo_entry E = entries[e];
    PairItem it;
    it.tile = (int32_t)E.q_tile;
    it.row0 = tile_row0[E.q_tile];
    it.rows = (int16_t)tile_rows[E.q_tile];
    it.causal = 0;
    pair_half(it, 0, &E);
    bool joined = false;
    if (pb >= 0 && e + 1 < n_entries) {
      const octo_entry F = entries[e + 1];
      if ((int32_t)F.kv_page == pb && F.q_tile == E.q_tile) {
        pair_half(it, 1, &F);
        joined = true;
      }
    }
    if (!joined) pair_half(it, 1, nullptr);
    items[base + i] = it;
  }
  int32_t n = la;
  if (pb >= 0) {
    const int32_t ob = page_off[pb], lb = page_off[pb + 1] - ob;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int32_t s0 = 0; s0 < lb; s0 += blockDim.x) {
      const int32_t i = s0 + threadIdx.x;
      int32_t e = -1;
      bool keep = false;
      if (i < lb) {
        e = csc[ob + i];
        keep = !(e >= 1 && (int32_t)entries[e - 1].kv_page == pa && entries[e - 1].q_tile == entries[e].q_tile);
      }
      const uint32_t bal = __ballot_sync(0xffffffffu, keep);
      if (lane == 0) warp_s[wid] = __popc(bal);
      __syncthreads();
      int32_t before = carry;
      for (int w2 = 0; w2 < wid; w2++) before += warp_s[w2];
      if (keep) {
        const octo_entry F = entries[e];
        PairItem it;
        it.tile = (int32_t)F.q_tile;
        it.row0 = tile_row0[F.q_tile];
        it.rows = (int16_t)tile_rows[F.q_tile];
        it.causal = 0;
        pair_half(it, 0, nullptr);
        pair_half(it, 1, &F);
        items[base + la + before + __popc(bal & ((1u << lane) - 1))] = it;
      }
      __syncthreads();
      if (threadIdx.x == 0)
        for (int w2 = 0; w2 < nw; w2++) carry += warp_s[w2];
      __syncthreads();
    }
    n = la + carry;
  }
  if (threadIdx.x == 0) pair_n[b] = n;
}

template <typename T>
int dalloc(octo_plan_s* pl, T** ptr, size_t n, cudaStream_t s) {
  void* p = nullptr;
  OCTO_CUDA(cudaMallocAsync(&p, std::max<size_t>(n, 1) * sizeof(T), s));
  pl->allocs.push_back(p);
  *ptr = (T*)p;
  return OCTO_OK;
}

// frees one of the plan's allocations, stream-ordered
void dfree(octo_plan_s* pl, void* p, cudaStream_t s) {
  auto it = std::find(pl->allocs.begin(), pl->allocs.end(), p);
  if (it == pl->allocs.end()) return;
  pl->allocs.erase(it);
  cudaFreeAsync(p, s);
}

}  // namespace

#define OCTO_TRY(x)                 \
  do {                              \
    int _s = (x);                   \
    if (_s != OCTO_OK) {            \
      octo_plan_destroy(pl);        \
      return _s;                    \
    }                               \
  } while (0)

#define OCTO_RET(x)                 \
  do {                              \
    int _s = (x);                   \
    if (_s != OCTO_OK) return _s;   \
  } while (0)

// The parts of a plan that follow from its entries: the CSC view, the pair count and page
// statistics, the launch orders, and the dK/dV page pairs (training plans) or the split-KV
// runs (decode plans, whose host copies are kept for octo_decode_plan_advance).  Ends with
// a stream synchronisation.
int finish_plan(octo_plan_s* pl, cudaStream_t s) {
  octo_pool_s* pool = pl->pool;
  const bool is_decode = pl->info.is_decode != 0;
  const int64_t n_tiles = pl->info.n_tiles;
  const int32_t n_entries = pl->info.n_entries;
  int32_t* d_cnt = pl->d_cnt;
  int32_t* d_scratch = pl->d_scratch;
  OCTO_RET(dalloc(pl, &pl->csc_perm, n_entries, s));
  pl->csc_cap = (size_t)n_entries;
  // ---- CSC ----
  OCTO_RET(cuda_status(cudaMemsetAsync(d_cnt, 0, (size_t)pl->num_pages * 4, s)));
  if (n_entries > 0) {
    k_page_hist<<<(n_entries + 255) / 256, 256, 0, s>>>(pl->entries, n_entries, pl->tile_rows, d_cnt,
                                                        (unsigned long long*)(d_scratch + 4));
    count_launch();
  }
  k_scan<<<1, 1024, 0, s>>>(d_cnt, pl->num_pages, pl->page_off, d_scratch + 2);
  count_launch();
  OCTO_RET(cuda_status(cudaMemsetAsync(d_cnt, 0, (size_t)pl->num_pages * 4, s)));
  if (n_entries > 0) {
    k_csc_scatter<<<(n_entries + 255) / 256, 256, 0, s>>>(pl->entries, n_entries, pl->page_off, d_cnt,
                                                          pl->csc_perm);
    count_launch();
  }
  k_touched<<<1, 1024, 0, s>>>(pl->page_off, pl->num_pages, pl->touched, d_scratch + 3);
  count_launch();
  OCTO_RET(cuda_status(cudaGetLastError()));
  int32_t hs2[6];
  OCTO_RET(cuda_status(cudaMemcpyAsync(hs2, d_scratch, 24, cudaMemcpyDeviceToHost, s)));
  OCTO_RET(cuda_status(cudaStreamSynchronize(s)));
  pl->info.max_page_entries = hs2[2];
  pl->info.n_touched_pages = hs2[3];
  unsigned long long pairs;
  std::memcpy(&pairs, &hs2[4], 8);
  pl->info.pairs = (int64_t)pairs;
  if (hs2[2] > kSortCap) return OCTO_ENOTSUP;
  if (hs2[3] > 0 && hs2[2] > 1) {
    int32_t m = 1;
    while (m < hs2[2]) m <<= 1;
    size_t smem = (size_t)m * 4;
    if (smem > 48 * 1024) OCTO_RET(cuda_status(cudaFuncSetAttribute(k_csc_sort, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)));
    k_csc_sort<<<hs2[3], 512, smem, s>>>(pl->touched, pl->page_off, pl->csc_perm, m);
    count_launch();
  }
  OCTO_RET(cuda_status(cudaGetLastError()));
  // ---- launch orders: tree by tree (concurrent CTAs then read the same tree's rows and
  // pages, which keeps their shared tiles in L2), heaviest tiles / page pairs first within
  // a tree (longest-processing-time first) ----
  {
    std::vector<int32_t> toff(n_tiles + 1), poff((size_t)pl->num_pages + 1);
    OCTO_RET(cuda_status(cudaMemcpyAsync(toff.data(), pl->tile_off, (n_tiles + 1) * 4, cudaMemcpyDeviceToHost, s)));
    OCTO_RET(cuda_status(
        cudaMemcpyAsync(poff.data(), pl->page_off, ((size_t)pl->num_pages + 1) * 4, cudaMemcpyDeviceToHost, s)));
    OCTO_RET(cuda_status(cudaStreamSynchronize(s)));
    if (is_decode) pl->h_toff = toff;
    std::vector<int32_t> tord(n_tiles);
    for (int64_t t = 0; t < n_tiles; t++) tord[t] = (int32_t)t;
    const std::vector<int32_t>& ttree = pl->h_tile_tree;
    std::stable_sort(tord.begin(), tord.end(), [&](int32_t a, int32_t b) {
      if (!ttree.empty() && ttree[a] != ttree[b]) return ttree[a] < ttree[b];
      return toff[a + 1] - toff[a] > toff[b + 1] - toff[b];
    });
    if (is_decode) pl->h_tord = tord;   // re-sorted incrementally by each advance
    const bool any_touched = pl->info.n_touched_pages > 0;
    // dK/dV work units: consecutive own pages of each segment, two at a time, among the
    // touched pages; a touched page without a touched partner runs alone
    if (!is_decode && any_touched) {
      std::vector<int32_t> pp, ptree;   // page pairs, and the tree of each
      std::vector<char> seen((size_t)pl->num_pages, 0);
      auto cnt = [&](int32_t pg) { return pg < 0 ? 0 : poff[pg + 1] - poff[pg]; };
      for (size_t gi = 0; gi < pool->segs.size(); gi++) {
        const Segment& g = pool->segs[gi];
        if (g.freed) continue;
        const int32_t tr = gi < pl->h_seg_tree.size() ? pl->h_seg_tree[gi] : INT32_MAX;
        int32_t pend = -1;
        for (int32_t pg : g.pages) {
          if (pg < 0 || pg >= pl->num_pages || cnt(pg) == 0 || seen[pg]) {
            if (pend >= 0) { pp.push_back(pend); pp.push_back(-1); ptree.push_back(tr); pend = -1; }
            continue;
          }
          seen[pg] = 1;
          if (pend < 0) {
            pend = pg;
          } else {
            pp.push_back(pend);
            pp.push_back(pg);
            ptree.push_back(tr);
            pend = -1;
          }
        }
        if (pend >= 0) { pp.push_back(pend); pp.push_back(-1); ptree.push_back(tr); }
      }
      for (int32_t pg = 0; pg < pl->num_pages; pg++)
        if (cnt(pg) > 0 && !seen[pg]) { pp.push_back(pg); pp.push_back(-1); ptree.push_back(INT32_MAX); }
      const int32_t np = (int32_t)(pp.size() / 2);
      std::vector<int32_t> poff2(np + 1, 0), pord2(np);
      for (int32_t i = 0; i < np; i++) {
        poff2[i + 1] = poff2[i] + cnt(pp[2 * i]) + cnt(pp[2 * i + 1]);
        pord2[i] = i;
      }
      std::stable_sort(pord2.begin(), pord2.end(), [&](int32_t a, int32_t b) {
        if (ptree[a] != ptree[b]) return ptree[a] < ptree[b];
        return poff2[a + 1] - poff2[a] > poff2[b + 1] - poff2[b];
      });
      pl->n_pairs = np;
      OCTO_RET(dalloc(pl, &pl->pair_pages, pp.size(), s));
      OCTO_RET(dalloc(pl, &pl->pair_item_off, poff2.size(), s));
      OCTO_RET(dalloc(pl, &pl->pair_n_items, np, s));
      OCTO_RET(dalloc(pl, &pl->pair_order, np, s));
      OCTO_RET(dalloc(pl, &pl->pair_items, (size_t)n_entries, s));
      OCTO_RET(cuda_status(cudaMemcpyAsync(pl->pair_pages, pp.data(), pp.size() * 4, cudaMemcpyHostToDevice, s)));
      OCTO_RET(cuda_status(
          cudaMemcpyAsync(pl->pair_item_off, poff2.data(), poff2.size() * 4, cudaMemcpyHostToDevice, s)));
      OCTO_RET(cuda_status(cudaMemcpyAsync(pl->pair_order, pord2.data(), np * 4, cudaMemcpyHostToDevice, s)));
      k_pair_items<<<np, 256, 0, s>>>(pl->pair_pages, pl->pair_item_off, pl->page_off, pl->csc_perm, pl->entries,
                                      n_entries, pl->tile_row0, pl->tile_rows, pl->pair_items, pl->pair_n_items);
      count_launch();
      OCTO_RET(cuda_status(cudaGetLastError()));
    }
    OCTO_RET(dalloc(pl, &pl->tile_order, n_tiles, s));
    if (n_tiles > 0)
      OCTO_RET(cuda_status(cudaMemcpyAsync(pl->tile_order, tord.data(), n_tiles * 4, cudaMemcpyHostToDevice, s)));
    // decode plans: split each cursor's entries into runs of kSplitEntries
    std::vector<int32_t> sp_tile, sp_e0, sp_e1, sp_order, cur0(n_tiles + 1, 0);
    if (is_decode) {
      for (int64_t t = 0; t < n_tiles; t++) {
        cur0[t] = (int32_t)sp_tile.size();
        for (int32_t e = toff[t]; e < toff[t + 1]; e += kSplitEntries) {
          sp_tile.push_back((int32_t)t);
          sp_e0.push_back(e);
          sp_e1.push_back(std::min(e + kSplitEntries, toff[t + 1]));
        }
      }
      cur0[n_tiles] = (int32_t)sp_tile.size();
      pl->n_splits = (int32_t)sp_tile.size();
      OCTO_RET(dalloc(pl, &pl->split_tile, sp_tile.size(), s));
      OCTO_RET(dalloc(pl, &pl->split_e0, sp_tile.size(), s));
      OCTO_RET(dalloc(pl, &pl->split_e1, sp_tile.size(), s));
      OCTO_RET(dalloc(pl, &pl->split_order, sp_tile.size(), s));
      OCTO_RET(dalloc(pl, &pl->cur_split0, cur0.size(), s));
      if (!sp_tile.empty()) {
        const int32_t ns = (int32_t)sp_tile.size();
        size_t b = sp_tile.size() * 4;
        OCTO_RET(cuda_status(cudaMemcpyAsync(pl->split_tile, sp_tile.data(), b, cudaMemcpyHostToDevice, s)));
        OCTO_RET(cuda_status(cudaMemcpyAsync(pl->split_e0, sp_e0.data(), b, cudaMemcpyHostToDevice, s)));
        OCTO_RET(cuda_status(cudaMemcpyAsync(pl->split_e1, sp_e1.data(), b, cudaMemcpyHostToDevice, s)));
        // Launch order: by the first page a split reads (then cursor, then split).  A
        // cursor's entries follow its context (prefix run, own run, mounted spans at their
        // points), so cursors sharing a prefix have splits starting on the same page, and
        // a mounted span's pages sit next to its owner's run: such splits start together
        // and their repeated reads are served from L2.  The order array goes to
        // split_order's buffer first as the first-page keys.
        k_split_first_page<<<(ns + 255) / 256, 256, 0, s>>>(pl->entries, pl->split_e0, ns, pl->split_order);
        count_launch();
        OCTO_RET(cuda_status(cudaGetLastError()));
        std::vector<int32_t> first(ns);
        OCTO_RET(cuda_status(cudaMemcpyAsync(first.data(), pl->split_order, b, cudaMemcpyDeviceToHost, s)));
        OCTO_RET(cuda_status(cudaStreamSynchronize(s)));
        sp_order.resize(ns);
        for (int32_t i = 0; i < ns; i++) sp_order[i] = i;
        std::stable_sort(sp_order.begin(), sp_order.end(), [&](int32_t a, int32_t c) { return first[a] < first[c]; });
        OCTO_RET(cuda_status(cudaMemcpyAsync(pl->split_order, sp_order.data(), b, cudaMemcpyHostToDevice, s)));
        pl->h_sp_first = first;
      }
      OCTO_RET(cuda_status(cudaMemcpyAsync(pl->cur_split0, cur0.data(), cur0.size() * 4, cudaMemcpyHostToDevice, s)));
      pl->h_sp_tile = sp_tile;
      pl->h_sp_e0 = sp_e0;
      pl->h_sp_e1 = sp_e1;
      pl->h_sp_order = sp_order;
      pl->h_cur0 = cur0;
    }
    // the host vectors are pageable and go out of scope
    OCTO_RET(cuda_status(cudaStreamSynchronize(s)));
  }
  return OCTO_OK;
}

int compile_plan(octo_pool_s* pool, const int32_t* tile_segs_host, const int32_t* seg_order_host, int32_t n_segs,
                 bool is_decode, int32_t bm, cudaStream_t s, octo_plan_s** out) {
  const int32_t P = pool->desc.page_size;
  const int32_t nseg_all = (int32_t)pool->segs.size();
  // ---- host mirror of the pool metadata ----
  std::vector<DevSeg> hseg(nseg_all);
  std::vector<int32_t> hpages;
  std::vector<DevMount> hmounts;
  for (int32_t i = 0; i < nseg_all; i++) {
    const Segment& g = pool->segs[i];
    DevSeg d;
    d.parent = g.parent;
    d.fork = g.fork;
    d.len = g.len;
    d.page_off = (int32_t)hpages.size();
    d.mount_off = (int32_t)hmounts.size();
    d.mount_cnt = (int32_t)g.mounts.size();
    d.p0 = g.p0;
    d.created_lo = (int32_t)g.created;
    hpages.insert(hpages.end(), g.pages.begin(), g.pages.end());
    for (int32_t mid : g.mounts) {
      const MountRec& m = pool->mounts[mid];
      hmounts.push_back({m.m, (int32_t)m.created, m.producer, m.a, m.b, mid, m.jump, 0});
    }
    hseg[i] = d;
  }
  if (!pool->d_status) {
    OCTO_CUDA(cudaMalloc(&pool->d_status, sizeof(int32_t) * 4));
    OCTO_CUDA(cudaMemset(pool->d_status, 0, sizeof(int32_t) * 4));
  }
  octo_plan_s* pl = new octo_plan_s();
  pl->pool = pool;
  pl->last_stream = s;
  pl->num_pages = pool->desc.num_pages;
  std::memset(&pl->info, 0, sizeof(pl->info));
  pl->info.bm = bm;
  pl->info.page_size = P;
  pl->info.is_decode = is_decode ? 1 : 0;
  int64_t n_rows = 0, n_tiles = 0;
  if (is_decode) {
    n_rows = n_tiles = n_segs;
  } else {
    for (int32_t i = 0; i < n_segs; i++) {
      int32_t L = pool->segs[seg_order_host[i]].len;
      n_rows += L;
      n_tiles += (L + bm - 1) / bm;
    }
  }
  if (n_rows > INT32_MAX / 2 || n_tiles > INT32_MAX / 2) {
    delete pl;
    return OCTO_EINVAL;
  }
  pl->info.n_rows = n_rows;
  pl->info.n_tiles = n_tiles;
  pl->info.n_segments = n_segs;

  DevSeg* d_segs;
  int32_t *d_pages, *d_seg_tile_base, *d_cnt, *d_scratch, *d_status;
  DevMount* d_mounts;
  OCTO_TRY(dalloc(pl, &d_segs, hseg.size(), s));
  OCTO_TRY(dalloc(pl, &d_pages, hpages.size(), s));
  OCTO_TRY(dalloc(pl, &d_mounts, hmounts.size(), s));
  OCTO_TRY(dalloc(pl, &pl->seg_order, n_segs, s));
  OCTO_TRY(dalloc(pl, &pl->seg_row_base, n_segs, s));
  OCTO_TRY(dalloc(pl, &d_seg_tile_base, n_segs + 1, s));
  OCTO_TRY(dalloc(pl, &pl->row_pos, n_rows, s));
  OCTO_TRY(dalloc(pl, &pl->tile_seg, n_tiles, s));
  OCTO_TRY(dalloc(pl, &pl->tile_t0, n_tiles, s));
  OCTO_TRY(dalloc(pl, &pl->tile_rows, n_tiles, s));
  OCTO_TRY(dalloc(pl, &pl->tile_row0, n_tiles, s));
  OCTO_TRY(dalloc(pl, &pl->tile_off, n_tiles + 1, s));
  OCTO_TRY(dalloc(pl, &d_cnt, std::max<int64_t>(n_tiles, pl->num_pages), s));
  OCTO_TRY(dalloc(pl, &d_scratch, 8, s));
  OCTO_TRY(dalloc(pl, &pl->page_off, (size_t)pl->num_pages + 1, s));
  OCTO_TRY(dalloc(pl, &pl->touched, (size_t)pl->num_pages, s));
  pl->poff_cap = (size_t)pl->num_pages + 1;
  pl->touched_cap = (size_t)pl->num_pages;
  d_status = d_scratch;  // [0] status, [1] max tile entries, [2] max page entries, [3] touched, [4..5] pairs
  OCTO_TRY(cuda_status(cudaMemsetAsync(d_scratch, 0, 8 * sizeof(int32_t), s)));
  OCTO_TRY(cuda_status(cudaMemcpyAsync(d_segs, hseg.data(), hseg.size() * sizeof(DevSeg), cudaMemcpyHostToDevice, s)));
  if (!hpages.empty())
    OCTO_TRY(cuda_status(cudaMemcpyAsync(d_pages, hpages.data(), hpages.size() * 4, cudaMemcpyHostToDevice, s)));
  if (!hmounts.empty())
    OCTO_TRY(cuda_status(
        cudaMemcpyAsync(d_mounts, hmounts.data(), hmounts.size() * sizeof(DevMount), cudaMemcpyHostToDevice, s)));
  const int32_t* order_src = is_decode ? tile_segs_host : seg_order_host;
  if (n_segs > 0)
    OCTO_TRY(cuda_status(cudaMemcpyAsync(pl->seg_order, order_src, n_segs * 4, cudaMemcpyHostToDevice, s)));

  // ---- tree of every packed segment and tile (training plans: tree-major launch orders) ----
  if (!is_decode) {
    pl->h_seg_tree.assign(nseg_all, INT32_MAX);
    int32_t rank = -1, prev_root = -1;
    for (int32_t k = 0; k < n_segs; k++) {
      int32_t r = seg_order_host[k];
      while (pool->segs[r].parent >= 0) r = pool->segs[r].parent;
      if (r != prev_root) rank++, prev_root = r;
      pl->h_seg_tree[seg_order_host[k]] = rank;
      const int32_t nt = (pool->segs[seg_order_host[k]].len + bm - 1) / bm;
      pl->h_tile_tree.insert(pl->h_tile_tree.end(), nt, rank);
    }
  }

  // ---- path predecessors of the packed rows (training plans) ----
  std::vector<int32_t> spred, ep, er;  // pageable sources of async copies: kept to the end
  std::vector<int32_t> runs, chunks, lruns, coff, clist;
  if (!is_decode && n_segs > 0) {
    std::vector<int32_t> rbase(n_segs), kpos(nseg_all, -1);
    spred.assign(n_segs, -1);
    int32_t acc = 0;
    for (int32_t k = 0; k < n_segs; k++) {
      rbase[k] = acc;
      kpos[seg_order_host[k]] = k;
      acc += pool->segs[seg_order_host[k]].len;
    }
    std::vector<std::pair<int32_t, int32_t>> ex;
    for (int32_t k = 0; k < n_segs; k++) {
      const Segment& g = pool->segs[seg_order_host[k]];
      if (g.len == 0) continue;
      int32_t par = g.parent, f = g.fork;
      while (par >= 0 && f == 0) {  // a fork at point 0 sees none of the parent's own tokens
        f = pool->segs[par].fork;
        par = pool->segs[par].parent;
      }
      if (par >= 0 && kpos[par] >= 0) {
        spred[k] = rbase[kpos[par]] + f - 1;
        ex.push_back({spred[k], rbase[k]});
      }
    }
    std::sort(ex.begin(), ex.end());
    int32_t run = 0;
    for (size_t i = 0; i < ex.size(); i++) {
      run = (i > 0 && ex[i].first == ex[i - 1].first) ? run + 1 : 1;
      pl->max_succ = std::max(pl->max_succ, run + 1);  // + the next own row
    }
    pl->max_succ = std::max(pl->max_succ, 1);
    ep.resize(ex.size());
    er.resize(ex.size());
    for (size_t i = 0; i < ex.size(); i++) ep[i] = ex[i].first, er[i] = ex[i].second;
    pl->n_succ_extra = (int32_t)ex.size();
    OCTO_TRY(dalloc(pl, &pl->seg_pred, n_segs, s));
    OCTO_TRY(dalloc(pl, &pl->succ_pred, std::max<size_t>(ex.size(), 1), s));
    OCTO_TRY(dalloc(pl, &pl->succ_row, std::max<size_t>(ex.size(), 1), s));
    OCTO_TRY(cuda_status(cudaMemcpyAsync(pl->seg_pred, spred.data(), n_segs * 4, cudaMemcpyHostToDevice, s)));
    if (!ex.empty()) {
      OCTO_TRY(cuda_status(cudaMemcpyAsync(pl->succ_pred, ep.data(), ep.size() * 4, cudaMemcpyHostToDevice, s)));
      OCTO_TRY(cuda_status(cudaMemcpyAsync(pl->succ_row, er.data(), er.size() * 4, cudaMemcpyHostToDevice, s)));
    }
    // runs and chunks of the recurrent layer: cut at every segment start and after every
    // row another segment continues from (a row with several successors)
    std::vector<char> cut((size_t)acc + 1, 0);
    for (int32_t k = 0; k < n_segs; k++) {
      cut[rbase[k]] = 1;
      if (spred[k] >= 0) cut[spred[k] + 1] = 1;
    }
    std::vector<int32_t> end_run((size_t)acc, -1);
    std::vector<int32_t> lvl;
    for (int32_t k = 0; k < n_segs; k++) {
      const int32_t b = rbase[k], e = b + pool->segs[seg_order_host[k]].len;
      for (int32_t r0 = b; r0 < e;) {
        int32_t r1 = r0 + 1;
        while (r1 < e && !cut[r1]) r1++;
        const int32_t pred = (r0 == b) ? spred[k] : r0 - 1;
        const int32_t pr = pred >= 0 ? end_run[pred] : -1;
        const int32_t id = (int32_t)(runs.size() / 4);
        runs.insert(runs.end(), {r0, r1, pr, (int32_t)(chunks.size() / 2)});
        for (int32_t c = r0; c < r1; c += kRecChunk) chunks.insert(chunks.end(), {c, std::min(kRecChunk, r1 - c)});
        lvl.push_back(pr >= 0 ? lvl[pr] + 1 : 0);
        end_run[r1 - 1] = id;
        r0 = r1;
      }
    }
    const int32_t nr = (int32_t)lvl.size();
    pl->n_runs = nr;
    pl->n_chunks = (int32_t)(chunks.size() / 2);
    pl->info.n_rec_runs = nr;
    pl->info.n_rec_chunks = pl->n_chunks;
    pl->n_levels = nr ? *std::max_element(lvl.begin(), lvl.end()) + 1 : 0;
    pl->h_level_off.assign(pl->n_levels + 1, 0);
    for (int32_t l : lvl) pl->h_level_off[l + 1]++;
    for (int32_t l = 0; l < pl->n_levels; l++) pl->h_level_off[l + 1] += pl->h_level_off[l];
    lruns.resize(nr);
    {
      std::vector<int32_t> fill(pl->h_level_off.begin(), pl->h_level_off.end() - (pl->n_levels ? 1 : 0));
      for (int32_t i = 0; i < nr; i++) lruns[fill[lvl[i]]++] = i;
    }
    coff.assign(nr + 1, 0);
    for (int32_t i = 0; i < nr; i++)
      if (runs[4 * i + 2] >= 0) coff[runs[4 * i + 2] + 1]++;
    for (int32_t i = 0; i < nr; i++) coff[i + 1] += coff[i];
    clist.resize(std::max(nr, 1));
    {
      std::vector<int32_t> fill(coff.begin(), coff.end() - 1);
      for (int32_t i = 0; i < nr; i++)
        if (runs[4 * i + 2] >= 0) clist[fill[runs[4 * i + 2]]++] = i;
    }
    OCTO_TRY(dalloc(pl, &pl->run_info, runs.size(), s));
    OCTO_TRY(dalloc(pl, &pl->run_child_off, coff.size(), s));
    OCTO_TRY(dalloc(pl, &pl->run_child, clist.size(), s));
    OCTO_TRY(dalloc(pl, &pl->level_runs, lruns.size(), s));
    OCTO_TRY(dalloc(pl, &pl->chunk_info, chunks.size(), s));
    if (nr > 0) {
      OCTO_TRY(cuda_status(cudaMemcpyAsync(pl->run_info, runs.data(), runs.size() * 4, cudaMemcpyHostToDevice, s)));
      OCTO_TRY(cuda_status(cudaMemcpyAsync(pl->run_child_off, coff.data(), coff.size() * 4, cudaMemcpyHostToDevice, s)));
      OCTO_TRY(cuda_status(cudaMemcpyAsync(pl->run_child, clist.data(), clist.size() * 4, cudaMemcpyHostToDevice, s)));
      OCTO_TRY(cuda_status(cudaMemcpyAsync(pl->level_runs, lruns.data(), lruns.size() * 4, cudaMemcpyHostToDevice, s)));
      OCTO_TRY(cuda_status(cudaMemcpyAsync(pl->chunk_info, chunks.data(), chunks.size() * 4, cudaMemcpyHostToDevice, s)));
    }
  }

  // ---- layout ----
  if (is_decode) {
    if (n_segs > 0) {
      k_decode_tiles<<<(n_segs + 255) / 256, 256, 0, s>>>(d_segs, d_mounts, pl->seg_order, n_segs, pl->tile_seg,
                                                         pl->tile_t0, pl->tile_rows, pl->tile_row0, pl->row_pos,
                                                         pl->seg_row_base);
      count_launch();
    }
  } else {
    k_layout<<<1, 1024, 0, s>>>(d_segs, pl->seg_order, n_segs, bm, pl->seg_row_base, d_seg_tile_base);
    count_launch();
    if (n_segs > 0) {
      k_tiles<<<n_segs, 256, 0, s>>>(d_segs, d_mounts, pl->seg_order, pl->seg_row_base, d_seg_tile_base, bm,
                                     pl->tile_seg, pl->tile_t0, pl->tile_rows, pl->tile_row0, pl->row_pos);
      count_launch();
    }
  }
  WalkArgs w{d_segs, d_pages, d_mounts, P};
  const int wpb = 8;  // warps per block
  int grid_t = (int)((n_tiles + wpb - 1) / wpb);
  if (n_tiles > 0) {
    k_count<<<grid_t, 32 * wpb, 0, s>>>(w, pl->tile_seg, pl->tile_t0, pl->tile_rows, (int32_t)n_tiles, d_cnt,
                                        d_status);
    count_launch();
  }
  k_scan<<<1, 1024, 0, s>>>(d_cnt, (int32_t)n_tiles, pl->tile_off, d_scratch + 1);
  count_launch();
  OCTO_TRY(cuda_status(cudaGetLastError()));
  int32_t hs[2];
  int32_t n_entries = 0;
  OCTO_TRY(cuda_status(cudaMemcpyAsync(&n_entries, pl->tile_off + n_tiles, 4, cudaMemcpyDeviceToHost, s)));
  OCTO_TRY(cuda_status(cudaMemcpyAsync(hs, d_scratch, 8, cudaMemcpyDeviceToHost, s)));
  OCTO_TRY(cuda_status(cudaStreamSynchronize(s)));
  if (hs[0] != OCTO_OK) {
    octo_plan_destroy(pl);
    return hs[0];
  }
  pl->info.n_entries = n_entries;
  pl->info.max_tile_entries = hs[1];
  OCTO_TRY(dalloc(pl, &pl->entries, n_entries, s));
  pl->entries_cap = (size_t)n_entries;
  if (n_tiles > 0) {
    k_fill<<<grid_t, 32 * wpb, 0, s>>>(w, pl->tile_seg, pl->tile_t0, pl->tile_rows, (int32_t)n_tiles, pl->tile_off,
                                       pl->entries, d_status);
    count_launch();
  }
  pl->d_cnt = d_cnt;
  pl->d_scratch = d_scratch;
  if (is_decode) {
    pl->cur_seg.assign(tile_segs_host, tile_segs_host + n_segs);
    std::vector<int32_t> sorted_cur(pl->cur_seg);
    std::sort(sorted_cur.begin(), sorted_cur.end());
    pl->dup_cursors = std::adjacent_find(sorted_cur.begin(), sorted_cur.end()) != sorted_cur.end();
    pl->cur_len.resize(n_segs);
    for (int32_t i = 0; i < n_segs; i++) pl->cur_len[i] = pool->segs[tile_segs_host[i]].len;
  }
  OCTO_TRY(finish_plan(pl, s));
  *out = pl;
  return OCTO_OK;
}

}  // namespace octo

extern "C" {

int octo_pack_tree(octo_pool_t pool, const octo_cursor_t* roots, int32_t n_roots, int32_t bm, void* stream,
                   octo_plan_t* out) {
  octo::NvtxRange nv("octo_pack_tree");
  if (!pool || !out || n_roots < 0 || (n_roots > 0 && !roots) || bm < 1 || bm > 128) return OCTO_EINVAL;
  const int32_t nseg = (int32_t)pool->segs.size();
  std::vector<int32_t> root_of(nseg, -1);
  for (int32_t i = 0; i < nseg; i++) {
    // segments are created after their parents, so the parent's root is known
    const octo::Segment& g = pool->segs[i];
    root_of[i] = g.parent < 0 ? i : root_of[g.parent];
  }
  std::vector<int32_t> order;
  for (int32_t ri = 0; ri < n_roots; ri++) {
    int32_t r = roots[ri];
    if (r < 0 || r >= nseg || pool->segs[r].freed || pool->segs[r].parent != -1) return OCTO_EINVAL;
    for (int32_t k = 0; k < ri; k++)
      if (roots[k] == r) return OCTO_EINVAL;
    for (int32_t i = 0; i < nseg; i++)
      if (root_of[i] == r && !pool->segs[i].freed) order.push_back(i);
  }
  return octo::compile_plan(pool, nullptr, order.data(), (int32_t)order.size(), false, bm, (cudaStream_t)stream, out);
}

int octo_decode_plan(octo_pool_t pool, const octo_cursor_t* cursors, int32_t n, void* stream, octo_plan_t* out) {
  octo::NvtxRange nv("octo_decode_plan");
  if (!pool || !out || n < 0 || (n > 0 && !cursors)) return OCTO_EINVAL;
  for (int32_t i = 0; i < n; i++) {
    int32_t c = cursors[i];
    if (c < 0 || c >= (int32_t)pool->segs.size() || pool->segs[c].freed) return OCTO_EINVAL;
    if (pool->segs[c].len == 0) return OCTO_EINVAL;
  }
  return octo::compile_plan(pool, cursors, nullptr, n, true, 1, (cudaStream_t)stream, out);
}

int octo_decode_plan_advance(octo_plan_t pl, void* stream) {
  using namespace octo;
  NvtxRange nv("octo_decode_plan_advance");
  if (!pl || !pl->info.is_decode) return OCTO_EINVAL;
  octo_pool_s* pool = pl->pool;
  const int32_t n = (int32_t)pl->info.n_tiles, P = pool->desc.page_size;
  cudaStream_t s = (cudaStream_t)stream;
  if ((int32_t)pl->cur_seg.size() != n || (int32_t)pl->h_toff.size() != n + 1 || pl->dup_cursors) return OCTO_ESTATE;
  if (n == 0) return OCTO_OK;
  // every cursor exactly one token longer, and nothing else in its context: no mount at or
  // after the point where the new token sits (a mount at that point becomes visible to it)
  std::vector<int32_t>& stage = pl->h_stage;
  stage.assign(3 * (size_t)n + 1, 0);
  int32_t* adv = stage.data();             // [2 n] newest page, fresh flag
  int32_t* off = stage.data() + 2 * n;     // [n + 1] new tile_off
  int32_t mx = 0;
  std::vector<int32_t> fresh_pages;
  for (int32_t i = 0; i < n; i++) {
    const int32_t c = pl->cur_seg[i], L = pl->cur_len[i];
    if (c < 0 || c >= (int32_t)pool->segs.size()) return OCTO_ESTATE;
    const Segment& g = pool->segs[c];
    if (g.freed || g.len != L + 1 || L / P >= (int32_t)g.pages.size()) return OCTO_ESTATE;
    for (int32_t mid : g.mounts)
      if (pool->mounts[mid].m >= L) return OCTO_ESTATE;
    adv[2 * i] = g.pages[L / P];
    adv[2 * i + 1] = (L % P == 0) ? 1 : 0;
    if (adv[2 * i + 1]) fresh_pages.push_back(adv[2 * i]);
    const int32_t cnt = pl->h_toff[i + 1] - pl->h_toff[i] + adv[2 * i + 1];
    off[i + 1] = off[i] + cnt;
    mx = std::max(mx, cnt);
  }
  // from here on the plan changes; an error leaves it unusable (destroy it).  The plan's
  // arrays are rewritten and freed in order after the work already queued on the stream
  // that last used them.
  if (pl->last_stream != s) {
    if (!pl->order_ev) OCTO_CUDA(cudaEventCreateWithFlags(&pl->order_ev, cudaEventDisableTiming));
    OCTO_CUDA(cudaEventRecord(pl->order_ev, pl->last_stream));
    OCTO_CUDA(cudaStreamWaitEvent(s, pl->order_ev, 0));
  }
  pl->last_stream = s;
  const int32_t m = (int32_t)fresh_pages.size();
  if (m == 0) {
    // no entry moves: the cursors' own-page entries widen in place
    k_decode_widen<<<(n + 255) / 256, 256, 0, s>>>(pl->entries, pl->tile_off, n, pl->tile_t0, pl->row_pos);
    count_launch();
    OCTO_CUDA(cudaGetLastError());
    for (int32_t i = 0; i < n; i++) pl->cur_len[i] += 1;
    pl->info.pairs += n;
    return OCTO_OK;
  }
  std::sort(fresh_pages.begin(), fresh_pages.end());
  // split-KV runs of kSplitEntries entries per cursor: existing runs keep their first
  // entry (entries are only added at the end of a cursor's list); a cursor whose list was
  // a whole number of runs starts a new one on its fresh page
  std::vector<int32_t>&sp_tile = pl->x_sp_tile, &sp_e0 = pl->x_sp_e0, &sp_e1 = pl->x_sp_e1,
                      &sp_first = pl->x_sp_first, &cur0 = pl->x_cur0;
  sp_tile.clear();
  sp_e0.clear();
  sp_e1.clear();
  sp_first.clear();
  cur0.assign(n + 1, 0);
  for (int32_t i = 0; i < n; i++) {
    cur0[i] = (int32_t)sp_tile.size();
    const int32_t old_runs = pl->h_cur0[i + 1] - pl->h_cur0[i];
    for (int32_t e = off[i], j = 0; e < off[i + 1]; e += kSplitEntries, j++) {
      sp_tile.push_back(i);
      sp_e0.push_back(e);
      sp_e1.push_back(std::min(e + kSplitEntries, off[i + 1]));
      sp_first.push_back(j < old_runs ? pl->h_sp_first[pl->h_cur0[i] + j] : adv[2 * i]);
    }
  }
  const int32_t ns = (int32_t)sp_tile.size();
  cur0[n] = ns;
  std::vector<int32_t>& sp_order = pl->x_sp_order;
  if (ns == pl->n_splits) {
    sp_order = pl->h_sp_order;   // same runs, same first pages: same launch order
  } else {
    sp_order.resize(ns);
    for (int32_t i = 0; i < ns; i++) sp_order[i] = i;
    std::stable_sort(sp_order.begin(), sp_order.end(),
                     [&](int32_t a, int32_t c) { return sp_first[a] < sp_first[c]; });
  }
  // tiles by entry count, most first, ties by cursor (the compile's stable sort): the
  // previous order re-sorted by insertion, as only the cursors that opened a page moved
  std::vector<int32_t>& tord = pl->h_tord;
  if ((int32_t)tord.size() != n) {
    tord.resize(n);
    for (int32_t t = 0; t < n; t++) tord[t] = t;
  }
  {
    auto before = [&](int32_t a, int32_t b) {
      const int32_t ca = off[a + 1] - off[a], cb = off[b + 1] - off[b];
      return ca > cb || (ca == cb && a < b);
    };
    for (int32_t i = 1; i < n; i++) {
      const int32_t x = tord[i];
      int32_t k = i;
      for (; k > 0 && before(x, tord[k - 1]); k--) tord[k] = tord[k - 1];
      tord[k] = x;
    }
  }
  // one upload: adv | tile_off | fresh pages | split cursor, first, end, order | first split
  // per cursor | tile order
  const size_t o_fp = 3 * (size_t)n + 1, o_st = o_fp + m, o_e0 = o_st + ns, o_e1 = o_e0 + ns,
               o_so = o_e1 + ns, o_c0 = o_so + ns, o_to = o_c0 + n + 1, total = o_to + n;
  stage.resize(total);
  adv = stage.data();
  off = stage.data() + 2 * n;
  std::copy(fresh_pages.begin(), fresh_pages.end(), stage.begin() + o_fp);
  std::copy(sp_tile.begin(), sp_tile.end(), stage.begin() + o_st);
  std::copy(sp_e0.begin(), sp_e0.end(), stage.begin() + o_e0);
  std::copy(sp_e1.begin(), sp_e1.end(), stage.begin() + o_e1);
  std::copy(sp_order.begin(), sp_order.end(), stage.begin() + o_so);
  std::copy(cur0.begin(), cur0.end(), stage.begin() + o_c0);
  std::copy(tord.begin(), tord.end(), stage.begin() + o_to);
  const int32_t e_old = (int32_t)pl->info.n_entries, e_new = off[n];
  const int32_t t_old = pl->info.n_touched_pages;
  // the arrays this advance writes: the ones the previous such advance replaced, when they
  // are large enough (no allocation then), else new ones with some room to grow
  int32_t *buf = nullptr, *csc = nullptr, *poff = nullptr, *touched = nullptr;
  octo_entry* ent = nullptr;
  size_t buf_cap = 0, ent_cap = 0, csc_cap = 0, poff_cap = 0, touched_cap = 0;
  auto take = [&](auto*& spare, size_t& spare_cap, size_t need, auto*& out, size_t& out_cap) -> int {
    if (spare && spare_cap >= need) {
      out = spare;
      out_cap = spare_cap;
    } else {
      if (spare) dfree(pl, spare, s);
      out_cap = need + need / 8 + 256;
      if (int st = dalloc(pl, &out, out_cap, s)) return st;
    }
    spare = nullptr;
    spare_cap = 0;
    return OCTO_OK;
  };
  int st;
  if ((st = take(pl->sp_buf, pl->sp_buf_cap, total, buf, buf_cap)) ||
      (st = take(pl->sp_entries, pl->sp_entries_cap, (size_t)e_new, ent, ent_cap)) ||
      (st = take(pl->sp_csc, pl->sp_csc_cap, (size_t)e_new, csc, csc_cap)) ||
      (st = take(pl->sp_poff, pl->sp_poff_cap, (size_t)pl->num_pages + 1, poff, poff_cap)) ||
      (st = take(pl->sp_touched, pl->sp_touched_cap, (size_t)t_old + m, touched, touched_cap)))
    return st;
  // pageable source: staged by the runtime before the call returns
  OCTO_CUDA(cudaMemcpyAsync(buf, stage.data(), total * 4, cudaMemcpyHostToDevice, s));
  const int32_t* d_adv = buf;
  int32_t* d_off = buf + 2 * n;
  const int32_t* d_fp = buf + o_fp;
  k_decode_advance<<<(unsigned)(((int64_t)n * 32 + 255) / 256), 256, 0, s>>>(pl->entries, pl->tile_off, d_off, d_adv, n,
                                                                           ent, pl->tile_t0, pl->row_pos);
  k_csc_advance<<<(unsigned)((e_old + n + 255) / 256), 256, 0, s>>>(pl->csc_perm, pl->entries, e_old, pl->tile_off,
                                                                   d_off, pl->page_off, d_fp, m, d_adv, n, csc);
  k_pageoff_advance<<<(unsigned)((pl->num_pages + 1 + 255) / 256), 256, 0, s>>>(pl->page_off, pl->num_pages, d_fp, m,
                                                                               poff);
  k_touched_advance<<<(unsigned)((t_old + m + 255) / 256), 256, 0, s>>>(pl->touched, t_old, d_fp, m, touched);
  count_launch(4);
  OCTO_CUDA(cudaGetLastError());
  // the replaced small arrays of the plan's compile go back in stream order (the ones that
  // lived in the previous advance's buffer are not allocations of their own: dfree skips
  // them); the replaced entries, CSC, page offsets, touched pages and buffer become the
  // next advance's spares, which it writes only after the work queued here
  for (void* p : {(void*)pl->tile_off, (void*)pl->split_tile, (void*)pl->split_e0, (void*)pl->split_e1,
                  (void*)pl->split_order, (void*)pl->cur_split0, (void*)pl->tile_order})
    if (p) dfree(pl, p, s);
  pl->sp_buf = static_cast<int32_t*>(pl->adv_buf);
  pl->sp_buf_cap = pl->buf_cap;
  pl->sp_entries = pl->entries;
  pl->sp_entries_cap = pl->entries_cap;
  pl->sp_csc = pl->csc_perm;
  pl->sp_csc_cap = pl->csc_cap;
  pl->sp_poff = pl->page_off;
  pl->sp_poff_cap = pl->poff_cap;
  pl->sp_touched = pl->touched;
  pl->sp_touched_cap = pl->touched_cap;
  pl->adv_buf = buf;
  pl->buf_cap = buf_cap;
  pl->entries = ent;
  pl->entries_cap = ent_cap;
  pl->csc_perm = csc;
  pl->csc_cap = csc_cap;
  pl->page_off = poff;
  pl->poff_cap = poff_cap;
  pl->touched = touched;
  pl->touched_cap = touched_cap;
  pl->tile_off = d_off;
  pl->split_tile = buf + o_st;
  pl->split_e0 = buf + o_e0;
  pl->split_e1 = buf + o_e1;
  pl->split_order = buf + o_so;
  pl->cur_split0 = buf + o_c0;
  pl->tile_order = buf + o_to;
  pl->n_splits = ns;
  pl->h_toff.assign(off, off + n + 1);
  pl->h_sp_tile.swap(sp_tile);
  pl->h_sp_e0.swap(sp_e0);
  pl->h_sp_e1.swap(sp_e1);
  pl->h_sp_first.swap(sp_first);
  pl->h_sp_order.swap(sp_order);
  pl->h_cur0.swap(cur0);
  for (int32_t i = 0; i < n; i++) pl->cur_len[i] += 1;
  pl->info.n_entries = e_new;
  pl->info.max_tile_entries = mx;
  pl->info.max_page_entries = std::max(pl->info.max_page_entries, 1);
  pl->info.n_touched_pages = t_old + m;
  pl->info.pairs += n;
  return OCTO_OK;
}

int octo_plan_info(octo_plan_t plan, octo_plan_info_t* info) {
  if (!plan || !info) return OCTO_EINVAL;
  *info = plan->info;
  return OCTO_OK;
}

int octo_plan_copy_out(octo_plan_t pl, int32_t* seg_order, int32_t* seg_row_base, int32_t* row_pos, int32_t* tile_seg,
                       int32_t* tile_t0, int32_t* tile_rows, int32_t* tile_off, octo_entry* entries, int32_t* csc_perm,
                       int32_t* page_off) {
  if (!pl) return OCTO_EINVAL;
  const octo_plan_info_t& I = pl->info;
  auto cp = [](void* dst, const void* src, size_t bytes) -> int {
    if (!dst || bytes == 0) return OCTO_OK;
    return octo::cuda_status(cudaMemcpy(dst, src, bytes, cudaMemcpyDeviceToHost));
  };
  int st;
  if ((st = cp(seg_order, pl->seg_order, I.n_segments * 4))) return st;
  if ((st = cp(seg_row_base, pl->seg_row_base, I.n_segments * 4))) return st;
  if ((st = cp(row_pos, pl->row_pos, I.n_rows * 4))) return st;
  if ((st = cp(tile_seg, pl->tile_seg, I.n_tiles * 4))) return st;
  if ((st = cp(tile_t0, pl->tile_t0, I.n_tiles * 4))) return st;
  if ((st = cp(tile_rows, pl->tile_rows, I.n_tiles * 4))) return st;
  if ((st = cp(tile_off, pl->tile_off, (I.n_tiles + 1) * 4))) return st;
  if ((st = cp(entries, pl->entries, I.n_entries * sizeof(octo_entry)))) return st;
  if ((st = cp(csc_perm, pl->csc_perm, I.n_entries * 4))) return st;
  if ((st = cp(page_off, pl->page_off, ((size_t)pl->num_pages + 1) * 4))) return st;
  return OCTO_OK;
}

int octo_plan_destroy(octo_plan_t pl) {
  if (!pl) return OCTO_EINVAL;
  // stream-ordered: the arrays go back to the pool only after the work already enqueued
  // on the plan's last stream has finished with them
  for (void* p : pl->allocs) cudaFreeAsync(p, pl->last_stream);
  if (pl->order_ev) cudaEventDestroy(pl->order_ev);
  delete pl;
  return OCTO_OK;
}

}  // extern "C"
