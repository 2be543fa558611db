// Oracle for packed DAG attention -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, fp64 CPU model of what the Octopus hot path computes.  Only the
// tests, the smoke check and the CPU-baseline leg of the benchmark may load it; the
// library never does.  It shares no code, header, table or helper with the CUDA path.
//
// Sources (Octopus project page, shatianming5.github.io/octopus):
//   * "Architecture & Co-Design", item 02 (Memory): zero-copy KV mount of sibling
//     pages into attention layers, monotonic offset s(c'_B) = max(p_B, e_A + 1),
//     0 new pages.
//   * the five-primitives table: fork shares the parent prefix by reference count
//     (+K), read_thread mounts c_A[s_A:e_A), rewind restores step k and keeps the
//     pruned leaf, done freezes the cursor and pins its pages.
//   * item 03 (Training): one unpadded 1D pass with single-ownership masking; reader
//     gradients reach the producer's KV.
//
// Readings taken where the pages are silent (each is listed in the design notes):
//   * attention is softmax(q k^T * scale) v with scale a parameter (1/sqrt(d)),
//     q head h uses kv head h / (Hq/Hkv); LSE is the natural log of the row sum;
//   * a child (fork or rewind) sees the first f tokens of its parent and the mounts
//     its parent held when the child was created whose point m <= f;
//   * a mount at point m (the reader's length when mounting) is visible to the
//     reader's rows with index >= m; its span [a,b) is in producer-local indices;
//   * e_A is the exclusive end of the span in positions: pos(A, b-1) + 1;
//   * rewind(k) on segment S makes a continuation child at k; S's tail stays.
//
//   * rotary embedding (the "RoPE flip" of unshifted zero-copy KV in the cross-branch
//     sharing table; mounted keys are rotation-free): the half-split rotation, pair
//     (i, i + d/2) turned by pos * base^(-2i/d).  A plain loop below, orc_rope.
//
// Every value here is computed the direct way: each row's context is materialised as
// an explicit list of (token, source), and attention is a dense loop over that list.
// The tile list is derived by brute force from the materialised visibility, not from a
// DAG walk.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <vector>
#include <utility>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

enum { ORC_OK = 0, ORC_EINVAL = 1, ORC_ENOMEM = 2, ORC_ESTATE = 3 };

struct Seg {
  int parent = -1;        // segment this one continues from (-1 for a root)
  int fork = 0;           // tokens of the parent it sees
  long created = 0;       // op sequence number of its creation
  std::vector<int> tok;   // global token ids (append order)
  std::vector<int> pos;   // position id of each own token
  std::vector<int> pages; // physical pages, page i holds own tokens [i*P, (i+1)*P)
  int p_next = 0;         // next position
  bool cursor = true;     // live cursor handle
  bool pinned = false;
  bool frozen = false;    // done: no more appends
  bool dead = false;      // rewound away from: no more appends
  bool freed = false;
};

struct Mount {
  int reader, m, producer, a, b;
  long created;
};

struct Entry {  // rectangle form of one (q-tile, kv-page, source) block
  int q_tile, kv_page, kv_lo, kv_hi, q_lo, flags, diag, src;
};

struct CtxItem {
  int token;   // global token id
  int src;     // -1: the row's own tree path; >= 0: mount id
  int from;    // first own row index of the segment that sees it (0 for inherited)
};

struct Oracle {
  int P, num_pages, Hkv, d;
  std::vector<Seg> segs;
  std::vector<Mount> mounts;
  std::vector<char> used;          // page in use
  std::vector<double> K, V;        // [T, Hkv, d]
  std::vector<int> tok_seg, tok_idx;
  long seq = 0;

  bool valid_seg(int s) const { return s >= 0 && s < (int)segs.size() && !segs[s].freed; }

  // ---- reference counts, recounted from scratch every time ----
  int refcount(int s) const {
    const Seg& g = segs[s];
    if (g.freed) return 0;
    int r = (g.cursor ? 1 : 0) + (g.pinned ? 1 : 0);
    for (const Seg& c : segs)
      if (!c.freed && c.parent == s) r++;
    for (const Mount& mt : mounts)
      if (mt.producer == s && !segs[mt.reader].freed) r++;
    return r;
  }
  // A segment stays allocated while a live cursor or a pin needs it, directly or through
  // the prefix it shares (parent) or a span it mounted (producer).  Reachability is
  // recomputed from scratch by fixpoint iteration.
  void collect() {
    std::vector<char> need(segs.size(), 0);
    for (size_t s = 0; s < segs.size(); s++)
      if (!segs[s].freed && (segs[s].cursor || segs[s].pinned)) need[s] = 1;
    bool grew = true;
    while (grew) {
      grew = false;
      for (size_t s = 0; s < segs.size(); s++) {
        if (!need[s]) continue;
        int par = segs[s].parent;
        if (par >= 0 && !need[par] && !segs[par].freed) { need[par] = 1; grew = true; }
        for (const Mount& mt : mounts)
          if (mt.reader == (int)s && !need[mt.producer] && !segs[mt.producer].freed) {
            need[mt.producer] = 1;
            grew = true;
          }
      }
    }
    for (size_t s = 0; s < segs.size(); s++)
      if (!segs[s].freed && !need[s]) {
        for (int p : segs[s].pages) used[p] = 0;
        segs[s].freed = true;
      }
  }
  int free_count() const {
    int n = 0;
    for (char u : used) n += u ? 0 : 1;
    return n;
  }
  int lowest_free() const {
    for (int p = 0; p < num_pages; p++)
      if (!used[p]) return p;
    return -1;
  }

  // ---- context materialisation ----
  // Own events of segment x: tokens [0, L) and the mounts of x with point m <= mcap
  // created before `before`.  A mount at m goes right before token m (after all
  // tokens when m == L).  `from_own` selects whether `from` is the event index
  // (the segment's own rows) or 0 (inherited by a descendant).
  void own_events(int x, int L, int mcap, long before, bool from_own,
                  std::vector<CtxItem>& out) const {
    std::vector<int> mids;
    for (int i = 0; i < (int)mounts.size(); i++) {
      const Mount& mt = mounts[i];
      if (mt.reader == x && mt.m <= mcap && mt.created < before) mids.push_back(i);
    }
    auto emit_mount = [&](int i) {
      const Mount& mt = mounts[i];
      for (int t = mt.a; t < mt.b; t++)
        out.push_back({segs[mt.producer].tok[t], i, from_own ? mt.m : 0});
    };
    size_t k = 0;  // mids are in creation order, and m never decreases with creation
    for (int idx = 0; idx < L; idx++) {
      while (k < mids.size() && mounts[mids[k]].m <= idx) emit_mount(mids[k++]);
      out.push_back({segs[x].tok[idx], -1, from_own ? idx : 0});
    }
    while (k < mids.size()) emit_mount(mids[k++]);
  }
  void inherited(int s, std::vector<CtxItem>& out) const {
    const Seg& g = segs[s];
    if (g.parent < 0) return;
    inherited(g.parent, out);
    own_events(g.parent, g.fork, g.fork, g.created, false, out);
  }
  // Everything any row of s (up to its current length) can see; row i sees the items
  // with from <= i.
  std::vector<CtxItem> full_ctx(int s) const {
    std::vector<CtxItem> out;
    inherited(s, out);
    int L = (int)segs[s].tok.size();
    own_events(s, L, L - 1, seq + 1, true, out);
    return out;
  }
  // Context a new own row at index m would see (used to validate a mount at point m).
  std::vector<CtxItem> ctx_at(int s, int m) const {
    std::vector<CtxItem> out;
    inherited(s, out);
    own_events(s, m, m, seq + 1, true, out);
    return out;
  }
};

struct Plan {
  const Oracle* o;
  int bm;
  int tile_stride = 1;   // derive the entries of every tile_stride-th tile only
  std::vector<int> seg_order, seg_row_base;    // packed segments and first packed row
  std::vector<int> row_seg, row_idx, row_pos;  // per packed row
  std::vector<int> tile_seg, tile_t0, tile_rows;
  std::vector<int> tile_off;
  std::vector<Entry> entries;
  std::vector<int> csc_perm, page_off;
  long long pairs = 0;
  int err = ORC_OK;
};

// Tile list by brute force: for each q-tile, take the context of its last row in order,
// group it by (physical page, source) in order of first appearance, evaluate the
// visibility of every (row, slot) of each group, and reduce it to the tightest
// rectangle.  Fails if the rectangle formula does not reproduce the visibility exactly.
int derive_tiles(Plan& pl) {
  const Oracle& o = *pl.o;
  const int P = o.P;
  pl.tile_off.push_back(0);
  for (size_t si = 0; si < pl.seg_order.size(); si++) {
    int s = pl.seg_order[si];
    int len = (int)o.segs[s].tok.size();
    std::vector<CtxItem> ctx = o.full_ctx(s);
    for (int t0 = 0; t0 < len; t0 += pl.bm) {
      int rows = std::min(pl.bm, len - t0);
      int t1 = t0 + rows;
      int tile = (int)pl.tile_seg.size();
      pl.tile_seg.push_back(s);
      pl.tile_t0.push_back(t0);
      pl.tile_rows.push_back(rows);
      if (tile % pl.tile_stride != 0) {
        pl.tile_off.push_back((int)pl.entries.size());
        continue;
      }
      // groups in first-appearance order within the last row's context
      std::vector<std::pair<int, int>> keys;  // (page, src)
      std::map<std::pair<int, int>, int> key_index;
      std::vector<std::vector<const CtxItem*>> members;
      for (const CtxItem& c : ctx) {
        if (c.from > t1 - 1) continue;
        int owner = o.tok_seg[c.token], idx = o.tok_idx[c.token];
        int page = o.segs[owner].pages[idx / P];
        auto key = std::make_pair(page, c.src);
        auto it = key_index.find(key);
        if (it == key_index.end()) {
          key_index[key] = (int)keys.size();
          keys.push_back(key);
          members.emplace_back();
          members.back().push_back(&c);
        } else {
          members[it->second].push_back(&c);
        }
      }
      for (size_t gi = 0; gi < keys.size(); gi++) {
        // visibility matrix [rows][P]
        std::vector<char> vis((size_t)rows * P, 0);
        for (const CtxItem* c : members[gi]) {
          int slot = o.tok_idx[c->token] % P;
          for (int r = 0; r < rows; r++)
            if (c->from <= t0 + r) vis[(size_t)r * P + slot] = 1;
        }
        int kv_lo = P, kv_hi = 0, q_lo = rows;
        for (int r = 0; r < rows; r++)
          for (int j = 0; j < P; j++)
            if (vis[(size_t)r * P + j]) {
              kv_lo = std::min(kv_lo, j);
              kv_hi = std::max(kv_hi, j + 1);
              q_lo = std::min(q_lo, r);
            }
        if (q_lo == rows) return ORC_EINVAL;  // an empty group cannot happen
        bool full = true;
        for (int r = q_lo; r < rows && full; r++)
          for (int j = kv_lo; j < kv_hi; j++)
            if (!vis[(size_t)r * P + j]) { full = false; break; }
        int diag = 0, flags = 0;
        if (!full) {
          flags = 1;
          int jmax = -1;
          for (int j = kv_lo; j < kv_hi; j++)
            if (vis[(size_t)q_lo * P + j]) jmax = j;
          diag = jmax - q_lo;
        }
        // the rectangle formula must reproduce the visibility exactly
        for (int r = 0; r < rows; r++)
          for (int j = 0; j < P; j++) {
            bool f = r >= q_lo && j >= kv_lo && j < kv_hi && (!flags || j <= r + diag);
            if (f != (bool)vis[(size_t)r * P + j]) return ORC_EINVAL;
            pl.pairs += f ? 1 : 0;
          }
        pl.entries.push_back({tile, keys[gi].first, kv_lo, kv_hi, q_lo, flags, diag, keys[gi].second});
      }
      pl.tile_off.push_back((int)pl.entries.size());
    }
  }
  // CSC: entries stably ordered by kv page
  pl.csc_perm.resize(pl.entries.size());
  for (size_t i = 0; i < pl.entries.size(); i++) pl.csc_perm[i] = (int)i;
  std::stable_sort(pl.csc_perm.begin(), pl.csc_perm.end(), [&](int a, int b) {
    return pl.entries[a].kv_page < pl.entries[b].kv_page;
  });
  pl.page_off.assign(o.num_pages + 1, 0);
  for (const Entry& e : pl.entries) pl.page_off[e.kv_page + 1]++;
  for (int p = 0; p < o.num_pages; p++) pl.page_off[p + 1] += pl.page_off[p];
  return ORC_OK;
}

// Per-row dense attention over a materialised context, fp64.
struct RowOut {
  std::vector<double> s;  // scores
};

inline double dot(const double* a, const double* b, int d) {
  double acc = 0.0;
  for (int i = 0; i < d; i++) acc += a[i] * b[i];
  return acc;
}

void row_forward(const Oracle& o, const std::vector<int>& toks, const double* q, int g,
                 double scale, std::vector<double>& s, double* out, double* lse) {
  const int d = o.d, Hkv = o.Hkv;
  size_t n = toks.size();
  s.resize(n);
  double mx = -INFINITY;
  for (size_t c = 0; c < n; c++) {
    s[c] = scale * dot(q, &o.K[((size_t)toks[c] * Hkv + g) * d], d);
    mx = std::max(mx, s[c]);
  }
  double sum = 0.0;
  for (size_t c = 0; c < n; c++) sum += std::exp(s[c] - mx);
  double L = mx + std::log(sum);
  for (int i = 0; i < d; i++) out[i] = 0.0;
  for (size_t c = 0; c < n; c++) {
    double p = std::exp(s[c] - L);
    const double* v = &o.V[((size_t)toks[c] * Hkv + g) * d];
    for (int i = 0; i < d; i++) out[i] += p * v[i];
  }
  *lse = L;
}

}  // namespace

extern "C" {

void* orc_new(int page_size, int num_pages, int n_kv_heads, int head_dim) {
  if (page_size <= 0 || num_pages <= 0 || n_kv_heads <= 0 || head_dim <= 0) return nullptr;
  Oracle* o = new Oracle();
  o->P = page_size;
  o->num_pages = num_pages;
  o->Hkv = n_kv_heads;
  o->d = head_dim;
  o->used.assign(num_pages, 0);
  return o;
}

void orc_delete(void* h) { delete static_cast<Oracle*>(h); }

static int new_seg(Oracle* o, int parent, int fork, int p_next) {
  Seg g;
  g.parent = parent;
  g.fork = fork;
  g.created = ++o->seq;
  g.p_next = p_next;
  o->segs.push_back(g);
  return (int)o->segs.size() - 1;
}

static bool writable(const Oracle* o, int c) {
  if (!o->valid_seg(c)) return false;
  const Seg& g = o->segs[c];
  return g.cursor && !g.frozen && !g.dead;
}

int orc_root(void* h, int* out) {
  Oracle* o = static_cast<Oracle*>(h);
  *out = new_seg(o, -1, 0, 0);
  return ORC_OK;
}

// k, v: [n, Hkv, d] or null (zeros)
int orc_append(void* h, int c, int n, const double* k, const double* v, int* pos_out) {
  Oracle* o = static_cast<Oracle*>(h);
  if (c < 0 || c >= (int)o->segs.size() || n < 0) return ORC_EINVAL;
  if (!writable(o, c)) return ORC_ESTATE;
  Seg& g = o->segs[c];
  int len = (int)g.tok.size();
  int have = (int)g.pages.size() * o->P;
  int need = std::max(0, (len + n - have + o->P - 1) / o->P);
  if (need > o->free_count()) return ORC_ENOMEM;
  for (int i = 0; i < need; i++) {
    int p = o->lowest_free();
    o->used[p] = 1;
    g.pages.push_back(p);
  }
  const int row = o->Hkv * o->d;
  for (int i = 0; i < n; i++) {
    int t = (int)o->tok_seg.size();
    o->tok_seg.push_back(c);
    o->tok_idx.push_back((int)g.tok.size());
    g.tok.push_back(t);
    if (pos_out) pos_out[i] = g.p_next;
    g.pos.push_back(g.p_next++);
    for (int j = 0; j < row; j++) {
      o->K.push_back(k ? k[(size_t)i * row + j] : 0.0);
      o->V.push_back(v ? v[(size_t)i * row + j] : 0.0);
    }
  }
  o->seq++;
  return ORC_OK;
}

int orc_fork(void* h, int c, int n, int* out) {
  Oracle* o = static_cast<Oracle*>(h);
  if (c < 0 || c >= (int)o->segs.size() || n < 1) return ORC_EINVAL;
  if (!writable(o, c)) return ORC_ESTATE;
  int f = (int)o->segs[c].tok.size();
  int p = o->segs[c].p_next;
  for (int i = 0; i < n; i++) out[i] = new_seg(o, c, f, p);
  return ORC_OK;
}

int orc_mount(void* h, int r, int a_seg, int a, int b, int* new_pos) {
  Oracle* o = static_cast<Oracle*>(h);
  if (r < 0 || r >= (int)o->segs.size()) return ORC_EINVAL;
  if (!writable(o, r)) return ORC_ESTATE;
  if (!o->valid_seg(a_seg)) return ORC_EINVAL;
  const Seg& A = o->segs[a_seg];
  if (a < 0 || a >= b || b > (int)A.tok.size()) return ORC_EINVAL;
  // no token may become visible twice: the span must not already be in the context
  int m = (int)o->segs[r].tok.size();
  std::vector<CtxItem> ctx = o->ctx_at(r, m);
  for (const CtxItem& c : ctx)
    if (o->tok_seg[c.token] == a_seg && o->tok_idx[c.token] >= a && o->tok_idx[c.token] < b)
      return ORC_EINVAL;
  int e_A = A.pos[b - 1] + 1;
  Seg& R = o->segs[r];
  R.p_next = std::max(R.p_next, e_A + 1);
  o->mounts.push_back({r, m, a_seg, a, b, ++o->seq});
  if (new_pos) *new_pos = R.p_next;
  return ORC_OK;
}

int orc_rewind(void* h, int c, int k, int* out) {
  Oracle* o = static_cast<Oracle*>(h);
  if (c < 0 || c >= (int)o->segs.size()) return ORC_EINVAL;
  if (!writable(o, c)) return ORC_ESTATE;
  int len = (int)o->segs[c].tok.size();
  if (k < 0 || k > len) return ORC_EINVAL;
  int p = k < len ? o->segs[c].pos[k] : o->segs[c].p_next;
  o->segs[c].dead = true;
  o->segs[c].cursor = false;  // the handle moves to the continuation
  *out = new_seg(o, c, k, p);
  return ORC_OK;
}

int orc_done(void* h, int c) {
  Oracle* o = static_cast<Oracle*>(h);
  if (c < 0 || c >= (int)o->segs.size()) return ORC_EINVAL;
  if (!writable(o, c)) return ORC_ESTATE;
  o->segs[c].frozen = true;
  o->segs[c].pinned = true;
  o->seq++;
  return ORC_OK;
}

int orc_release(void* h, int c) {
  Oracle* o = static_cast<Oracle*>(h);
  if (c < 0 || c >= (int)o->segs.size()) return ORC_EINVAL;
  if (!o->valid_seg(c) || !o->segs[c].cursor) return ORC_ESTATE;
  o->segs[c].cursor = false;
  o->seq++;
  o->collect();
  return ORC_OK;
}

int orc_unpin(void* h, int c) {
  Oracle* o = static_cast<Oracle*>(h);
  if (c < 0 || c >= (int)o->segs.size()) return ORC_EINVAL;
  if (!o->valid_seg(c) || !o->segs[c].pinned) return ORC_ESTATE;
  o->segs[c].pinned = false;
  o->seq++;
  o->collect();
  return ORC_OK;
}

// Overwrites the K/V rows of the given tokens (k, v: [n, Hkv, d]); lets a caller that
// appended without values supply only the rows a sampled check reads.
int orc_set_kv(void* h, int n, const int* tokens, const double* k, const double* v) {
  Oracle* o = static_cast<Oracle*>(h);
  const size_t row = (size_t)o->Hkv * o->d;
  for (int i = 0; i < n; i++) {
    if (tokens[i] < 0 || tokens[i] >= (int)o->tok_seg.size()) return ORC_EINVAL;
    for (size_t j = 0; j < row; j++) {
      o->K[(size_t)tokens[i] * row + j] = k[(size_t)i * row + j];
      o->V[(size_t)tokens[i] * row + j] = v[(size_t)i * row + j];
    }
  }
  return ORC_OK;
}

int orc_num_segments(void* h) { return (int)static_cast<Oracle*>(h)->segs.size(); }
int orc_free_pages(void* h) { return static_cast<Oracle*>(h)->free_count(); }
int orc_num_mounts(void* h) { return (int)static_cast<Oracle*>(h)->mounts.size(); }

// info: parent, fork, len, n_pages, refcount, p_next, flags(bit0 cursor, 1 pinned,
// 2 frozen, 3 dead, 4 freed)
int orc_seg_info(void* h, int s, int* info) {
  Oracle* o = static_cast<Oracle*>(h);
  if (s < 0 || s >= (int)o->segs.size()) return ORC_EINVAL;
  const Seg& g = o->segs[s];
  info[0] = g.parent;
  info[1] = g.fork;
  info[2] = (int)g.tok.size();
  info[3] = (int)g.pages.size();
  info[4] = o->refcount(s);
  info[5] = g.p_next;
  info[6] = (g.cursor ? 1 : 0) | (g.pinned ? 2 : 0) | (g.frozen ? 4 : 0) | (g.dead ? 8 : 0) |
            (g.freed ? 16 : 0);
  return ORC_OK;
}
int orc_seg_pos(void* h, int s, int* pos) {
  Oracle* o = static_cast<Oracle*>(h);
  const Seg& g = o->segs[s];
  std::copy(g.pos.begin(), g.pos.end(), pos);
  return ORC_OK;
}
int orc_seg_pages(void* h, int s, int* pages) {
  Oracle* o = static_cast<Oracle*>(h);
  const Seg& g = o->segs[s];
  std::copy(g.pages.begin(), g.pages.end(), pages);
  return ORC_OK;
}
// mount record: reader, m, producer, a, b
int orc_mount_info(void* h, int i, int* info) {
  Oracle* o = static_cast<Oracle*>(h);
  if (i < 0 || i >= (int)o->mounts.size()) return ORC_EINVAL;
  const Mount& m = o->mounts[i];
  info[0] = m.reader; info[1] = m.m; info[2] = m.producer; info[3] = m.a; info[4] = m.b;
  return ORC_OK;
}

// ---- packing ----
void* orc_pack(void* h, const int* roots, int n_roots, int bm, int tile_stride, int* status) {
  Oracle* o = static_cast<Oracle*>(h);
  *status = ORC_OK;
  if (bm <= 0 || n_roots < 0) { *status = ORC_EINVAL; return nullptr; }
  Plan* pl = new Plan();
  pl->o = o;
  pl->bm = bm;
  pl->tile_stride = tile_stride < 1 ? 1 : tile_stride;
  for (int ri = 0; ri < n_roots; ri++) {
    int r = roots[ri];
    if (!o->valid_seg(r) || o->segs[r].parent != -1) { *status = ORC_EINVAL; delete pl; return nullptr; }
    for (int ri2 = 0; ri2 < ri; ri2++)
      if (roots[ri2] == r) { *status = ORC_EINVAL; delete pl; return nullptr; }
    for (int s = 0; s < (int)o->segs.size(); s++) {
      if (o->segs[s].freed) continue;
      int x = s;
      while (o->segs[x].parent >= 0) x = o->segs[x].parent;
      if (x == r) pl->seg_order.push_back(s);
    }
  }
  int row = 0;
  for (int s : pl->seg_order) {
    pl->seg_row_base.push_back(row);
    const Seg& g = o->segs[s];
    for (int i = 0; i < (int)g.tok.size(); i++) {
      pl->row_seg.push_back(s);
      pl->row_idx.push_back(i);
      pl->row_pos.push_back(g.pos[i]);
    }
    row += (int)g.tok.size();
  }
  int st = derive_tiles(*pl);
  if (st != ORC_OK) { *status = st; delete pl; return nullptr; }
  return pl;
}

// Visible (row, key) pairs of the whole plan: the length of every packed row's context.
long long orc_plan_total_pairs(void* p) {
  Plan* pl = static_cast<Plan*>(p);
  long long n = 0;
  for (int s : pl->seg_order) {
    std::vector<CtxItem> ctx = pl->o->full_ctx(s);
    int len = (int)pl->o->segs[s].tok.size();
    std::vector<long long> at(len + 1, 0);
    for (const CtxItem& c : ctx) at[c.from] += 1;
    long long run = 0;
    for (int i = 0; i < len; i++) {
      run += at[i];
      n += run;
    }
  }
  return n;
}

void orc_plan_delete(void* p) { delete static_cast<Plan*>(p); }

// what: 0 rows, 1 tiles, 2 entries, 3 segments, 4 visible pairs
long long orc_plan_size(void* p, int what) {
  Plan* pl = static_cast<Plan*>(p);
  switch (what) {
    case 0: return (long long)pl->row_seg.size();
    case 1: return (long long)pl->tile_seg.size();
    case 2: return (long long)pl->entries.size();
    case 3: return (long long)pl->seg_order.size();
    case 4: return pl->pairs;
  }
  return -1;
}

// entries: [E, 8] ints (q_tile, kv_page, kv_lo, kv_hi, q_lo, flags, diag, src)
void orc_plan_arrays(void* p, int* seg_order, int* seg_row_base, int* row_pos, int* tile_seg,
                     int* tile_t0, int* tile_rows, int* tile_off, int* entries, int* csc_perm,
                     int* page_off) {
  Plan* pl = static_cast<Plan*>(p);
  auto cp = [](const std::vector<int>& v, int* dst) { if (dst) std::copy(v.begin(), v.end(), dst); };
  cp(pl->seg_order, seg_order);
  cp(pl->seg_row_base, seg_row_base);
  cp(pl->row_pos, row_pos);
  cp(pl->tile_seg, tile_seg);
  cp(pl->tile_t0, tile_t0);
  cp(pl->tile_rows, tile_rows);
  cp(pl->tile_off, tile_off);
  cp(pl->csc_perm, csc_perm);
  cp(pl->page_off, page_off);
  if (entries)
    for (size_t i = 0; i < pl->entries.size(); i++) {
      const Entry& e = pl->entries[i];
      int* x = entries + 8 * i;
      x[0] = e.q_tile; x[1] = e.kv_page; x[2] = e.kv_lo; x[3] = e.kv_hi;
      x[4] = e.q_lo; x[5] = e.flags; x[6] = e.diag; x[7] = e.src;
    }
}

// Visible tokens of one packed row, in context order.
static void row_tokens(const Plan& pl, const std::vector<CtxItem>& ctx, int i, std::vector<int>& toks) {
  toks.clear();
  for (const CtxItem& c : ctx)
    if (c.from <= i) toks.push_back(c.token);
}

// Forward over packed rows.  Q, O: [N, Hq, d]; LSE: [Hq, N].  rows: optional subset
// (n_rows >= 0); only those rows of O / LSE are written.
int orc_fwd(void* p, int Hq, const double* Q, double scale, const int* rows, int n_rows,
            double* O, double* LSE, int nthreads) {
  Plan* pl = static_cast<Plan*>(p);
  const Oracle& o = *pl->o;
  if (Hq % o.Hkv) return ORC_EINVAL;
  const int G = Hq / o.Hkv, d = o.d;
  const long long N = (long long)pl->row_seg.size();
  std::vector<int> list;
  if (rows) list.assign(rows, rows + n_rows);
  else for (long long r = 0; r < N; r++) list.push_back((int)r);
  std::map<int, std::vector<CtxItem>> ctxs;
  for (int r : list) {
    int s = pl->row_seg[r];
    if (!ctxs.count(s)) ctxs[s] = o.full_ctx(s);
  }
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 4)
#endif
  for (long long li = 0; li < (long long)list.size(); li++) {
    int r = list[li];
    std::vector<int> toks;
    std::vector<double> s;
    row_tokens(*pl, ctxs.at(pl->row_seg[r]), pl->row_idx[r], toks);
    for (int h = 0; h < Hq; h++) {
      row_forward(o, toks, &Q[((size_t)r * Hq + h) * d], h / G, scale, s,
                  &O[((size_t)r * Hq + h) * d], &LSE[(size_t)h * N + r]);
    }
  }
  return ORC_OK;
}

// Backward.  dQ: [N, Hq, d] for rows with need_dq[r]; dK, dV: [T, Hkv, d] per token id,
// the adjoint of every copied context entry summed back onto its owner token, for
// tokens with need_dkdv[t] (null = all).  With `partial`, only the need_dq rows are
// processed and dK/dV hold their contributions alone (used to time a row sample).  Rows are processed in packed order and the
// sums are taken in that order, one kv head at a time.
int orc_bwd(void* p, int Hq, const double* Q, const double* dO, double scale,
            const unsigned char* need_dq, const unsigned char* need_dkdv,
            double* dQ, double* dK, double* dV, int nthreads, int partial) {
  Plan* pl = static_cast<Plan*>(p);
  const Oracle& o = *pl->o;
  if (Hq % o.Hkv) return ORC_EINVAL;
  const int G = Hq / o.Hkv, d = o.d, Hkv = o.Hkv;
  const long long N = (long long)pl->row_seg.size();
  const size_t T = o.tok_seg.size();
  std::map<int, std::vector<CtxItem>> ctxs;
  for (int s : pl->seg_order) ctxs[s] = o.full_ctx(s);
  // which rows are needed: dq rows, plus every row whose context holds a needed token
  // (a row of segment s sees the context items with from <= its index, so it needs the
  // earliest `from` of a needed token in s's context)
  std::vector<char> need_row(N, 0);
  std::map<int, int> first_need;   // segment -> smallest own-row index that sees a needed token
  if (!partial && need_dkdv != nullptr) {
    for (int s : pl->seg_order) {
      int mf = 0x7fffffff;
      for (const CtxItem& c : ctxs.at(s))
        if (need_dkdv[c.token]) mf = std::min(mf, c.from);
      first_need[s] = mf;
    }
  }
  for (long long r = 0; r < N; r++) {
    if (need_dq == nullptr || need_dq[r]) { need_row[r] = 1; continue; }
    if (partial) continue;   // dK/dV from the dq rows only (a sample of the full sums)
    if (need_dkdv == nullptr) { need_row[r] = 1; continue; }
    if (pl->row_idx[r] >= first_need.at(pl->row_seg[r])) need_row[r] = 1;
  }
  if (dK) std::fill(dK, dK + T * Hkv * d, 0.0);
  if (dV) std::fill(dV, dV + T * Hkv * d, 0.0);
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
  // kv heads are independent: each thread owns whole kv heads, so every dK/dV sum is
  // taken in packed row order whatever the thread count
#ifdef _OPENMP
#pragma omp parallel for schedule(static, 1)
#endif
  for (int g = 0; g < Hkv; g++) {
    std::vector<int> toks;
    std::vector<double> s, o_row(d), dp;
    for (long long r = 0; r < N; r++) {
      if (!need_row[r]) continue;
      row_tokens(*pl, ctxs.at(pl->row_seg[r]), pl->row_idx[r], toks);
      for (int h = g * G; h < (g + 1) * G; h++) {
        const double* q = &Q[((size_t)r * Hq + h) * d];
        const double* dout = &dO[((size_t)r * Hq + h) * d];
        double lse;
        row_forward(o, toks, q, g, scale, s, o_row.data(), &lse);
        double D = dot(dout, o_row.data(), d);
        double* dq = (dQ && (need_dq == nullptr || need_dq[r])) ? &dQ[((size_t)r * Hq + h) * d] : nullptr;
        if (dq) for (int i = 0; i < d; i++) dq[i] = 0.0;
        for (size_t c = 0; c < toks.size(); c++) {
          const double* k = &o.K[((size_t)toks[c] * Hkv + g) * d];
          const double* v = &o.V[((size_t)toks[c] * Hkv + g) * d];
          double pc = std::exp(s[c] - lse);
          double dpc = dot(dout, v, d);
          double ds = pc * (dpc - D);
          if (dq) for (int i = 0; i < d; i++) dq[i] += scale * ds * k[i];
          if (need_dkdv == nullptr || need_dkdv[toks[c]]) {
            double* dk = &dK[((size_t)toks[c] * Hkv + g) * d];
            double* dv = &dV[((size_t)toks[c] * Hkv + g) * d];
            for (int i = 0; i < d; i++) {
              dk[i] += scale * ds * q[i];
              dv[i] += pc * dout[i];
            }
          }
        }
      }
    }
  }
  return ORC_OK;
}

// Decode: one query per cursor against the context of the cursor's last token.
// q, out: [n, Hq, d]; lse: [n, Hq].
int orc_decode(void* h, const int* cursors, int n, int Hq, const double* q, double scale,
               double* out, double* lse) {
  Oracle* o = static_cast<Oracle*>(h);
  if (Hq % o->Hkv) return ORC_EINVAL;
  const int G = Hq / o->Hkv, d = o->d;
  for (int i = 0; i < n; i++) {
    int c = cursors[i];
    if (!o->valid_seg(c) || o->segs[c].tok.empty()) return ORC_EINVAL;
    std::vector<CtxItem> ctx = o->full_ctx(c);
    int last = (int)o->segs[c].tok.size() - 1;
    std::vector<int> toks;
    for (const CtxItem& x : ctx)
      if (x.from <= last) toks.push_back(x.token);
    std::vector<double> s;
    for (int hh = 0; hh < Hq; hh++)
      row_forward(*o, toks, &q[((size_t)i * Hq + hh) * d], hh / G, scale, s,
                  &out[((size_t)i * Hq + hh) * d], &lse[(size_t)i * Hq + hh]);
  }
  return ORC_OK;
}

// Context of one packed row as (token, src) pairs; returns its length (writes up to cap).
int orc_row_context(void* p, int r, int* tokens, int* srcs, int cap) {
  Plan* pl = static_cast<Plan*>(p);
  const Oracle& o = *pl->o;
  std::vector<CtxItem> ctx = o.full_ctx(pl->row_seg[r]);
  int n = 0;
  for (const CtxItem& c : ctx)
    if (c.from <= pl->row_idx[r]) {
      if (n < cap) { tokens[n] = c.token; srcs[n] = c.src; }
      n++;
    }
  return n;
}

// token id -> (segment, index)
void orc_token_owner(void* h, int* seg, int* idx) {
  Oracle* o = static_cast<Oracle*>(h);
  std::copy(o->tok_seg.begin(), o->tok_seg.end(), seg);
  std::copy(o->tok_idx.begin(), o->tok_idx.end(), idx);
}
int orc_num_tokens(void* h) { return (int)static_cast<Oracle*>(h)->tok_seg.size(); }

// Rotary embedding of x [n][H][d] (fp64, in place): row t at position pos[t]; for each
// head and i < d/2 the pair (x_i, x_{i+d/2}) is multiplied by the 2x2 rotation through
// theta = pos * base^(-2i/d) (inverse != 0: through -theta).
int orc_rope(double* x, int n, int H, int d, const int* pos, double base, int inverse) {
  if (d < 2 || d % 2 != 0 || base <= 0) return 1;
  const int half = d / 2;
  for (int t = 0; t < n; t++)
    for (int h = 0; h < H; h++)
      for (int i = 0; i < half; i++) {
        const double theta = (double)pos[t] * std::pow(base, -2.0 * i / d) * (inverse ? -1.0 : 1.0);
        const double c = std::cos(theta), s = std::sin(theta);
        double* row = x + ((size_t)t * H + h) * d;
        const double a = row[i], b = row[i + half];
        row[i] = c * a - s * b;
        row[i + half] = s * a + c * b;
      }
  return 0;
}

}  // extern "C"
