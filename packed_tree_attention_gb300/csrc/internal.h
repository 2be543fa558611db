// Internal structures shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include <set>
#include <vector>

#include "../../include/octopus.h"

namespace octo {

// ---- host metadata of one segment (a maximal run of tokens owned by one branch) ----
struct Segment {
  int32_t parent = -1;
  int32_t fork = 0;          // parent tokens it sees
  int64_t created = 0;       // op sequence number
  int32_t len = 0;
  int32_t p0 = 0;            // position of its first token (before own mounts at m = 0)
  int32_t p_next = 0;
  int32_t refcount = 1;
  bool cursor = true, pinned = false, frozen = false, dead = false, freed = false;
  std::vector<int32_t> pages;
  std::vector<int32_t> pos;
  std::vector<int32_t> mounts;  // ids of the mounts this segment reads, creation order
};

struct MountRec {
  int32_t reader, m, producer, a, b;
  int32_t jump;     // position jump the mount applied: new p - old p (>= 0)
  int64_t created;
};

// Device-side mirror of the pool metadata used by the compiler kernels.
struct DevSeg {
  int32_t parent, fork, len, page_off;   // page_off: first own page in dev pages[]
  int32_t mount_off, mount_cnt;          // own mounts in dev mounts[]
  int32_t p0;
  int32_t created_lo;                    // creation sequence (fits 31 bits per pool)
};
struct DevMount {
  int32_t m, created, producer, a, b, id, jump, pad;
};

// One work item of the dK/dV kernel: a query tile against a pair of pages (keys 0-63 from
// the first page, 64-127 from the second), with each half's visibility rectangle copied
// from its tile-list entry (lo = hi = 0: no entry for that half).  32 bytes.
struct PairItem {
  int32_t tile, row0;     // query tile, its first packed row
  int16_t lo[2], hi[2];   // visible slots [lo, hi) of each page
  int16_t qlo[2];         // first visible tile row
  int16_t rows;           // rows in the tile
  int16_t causal;         // bit h: half h is causal
  int32_t diag[2];        // causal: row r sees slot j iff j <= r + diag
};

}  // namespace octo

struct octo_pool_s {
  octo_pool_desc desc;
  std::vector<octo::Segment> segs;
  std::vector<octo::MountRec> mounts;
  std::set<int32_t> free_pages;
  int64_t seq = 0;
  int32_t* d_status = nullptr;   // device status word (bounded waits), shared by plans
};

struct octo_plan_s {
  octo_pool_s* pool;
  octo_plan_info_t info;
  int32_t num_pages;
  // device arrays (owned)
  int32_t* seg_order = nullptr;      // [n_segments]
  int32_t* seg_row_base = nullptr;   // [n_segments]
  int32_t* row_pos = nullptr;        // [n_rows]
  int32_t* tile_seg = nullptr;       // [n_tiles] segment id
  int32_t* tile_t0 = nullptr;        // [n_tiles] first own row index of the segment
  int32_t* tile_rows = nullptr;      // [n_tiles]
  int32_t* tile_row0 = nullptr;      // [n_tiles] first packed row
  int32_t* tile_off = nullptr;       // [n_tiles+1]
  octo_entry* entries = nullptr;     // [n_entries]
  int32_t* csc_perm = nullptr;       // [n_entries]
  int32_t* page_off = nullptr;       // [num_pages+1]
  int32_t* touched = nullptr;        // [n_touched_pages] pages with >= 1 entry, ascending
  int32_t* tile_order = nullptr;     // [n_tiles] tiles by descending entry count (scheduling)
  // dK/dV work units: pairs of consecutive own pages of a segment (second -1: one page)
  int32_t n_pairs = 0;
  int32_t* pair_pages = nullptr;     // [2 n_pairs]
  int32_t* pair_item_off = nullptr;  // [n_pairs+1] item slice of each pair (upper bound)
  int32_t* pair_n_items = nullptr;   // [n_pairs] items actually written
  int32_t* pair_order = nullptr;     // [n_pairs] launch order, heaviest first
  octo::PairItem* pair_items = nullptr;  // [n_entries]
  // path predecessors of the packed rows (per-token log-probability): row r's successors
  // are r + 1 inside its segment plus the first rows of the segments continuing from r
  int32_t* seg_pred = nullptr;       // [n_segments] row before the packed segment's first row, -1 none
  int32_t n_succ_extra = 0;
  int32_t* succ_pred = nullptr;      // [n_succ_extra] predecessor row, ascending
  int32_t* succ_row = nullptr;       // [n_succ_extra] first row of the continuing segment
  int32_t max_succ = 0;              // most successors of one row
  // tree-packed recurrent layer: the packed rows cut into runs -- a new run at every
  // segment start and after every row that other segments continue from -- so a run
  // starts from the state after one row (its predecessor run's last row, or nothing) and
  // no row inside a run feeds another run.  Runs are cut into chunks of kRecChunk rows.
  int32_t n_runs = 0, n_chunks = 0, n_levels = 0;
  int32_t* run_info = nullptr;       // [n_runs][4] first row, end row, predecessor run (-1 none), first chunk
  int32_t* run_child_off = nullptr;  // [n_runs + 1] runs continuing from each run's last row
  int32_t* run_child = nullptr;      // [n_runs] (ascending run ids per run)
  int32_t* level_runs = nullptr;     // [n_runs] run ids by level (a run's level = its predecessor's + 1)
  int32_t* chunk_info = nullptr;     // [n_chunks][2] first row, rows
  std::vector<int32_t> h_level_off;  // [n_levels + 1] level slices of level_runs
  // pack plans: the tree (rank of its root among the packed roots) of every pool segment
  // (INT32_MAX if not packed) and of every tile, for tree-major launch orders
  std::vector<int32_t> h_seg_tree, h_tile_tree;
  // decode plans: runs of up to kSplitEntries entries of one cursor (split-KV)
  int32_t n_splits = 0;
  int32_t* split_tile = nullptr;     // [n_splits] cursor (tile) of the split
  int32_t* split_e0 = nullptr;       // [n_splits] first entry
  int32_t* split_e1 = nullptr;       // [n_splits] one past the last entry
  int32_t* split_order = nullptr;    // [n_splits] launch order: first page read, then cursor, then split
  int32_t* cur_split0 = nullptr;     // [n_tiles+1] first split of each cursor
  std::vector<void*> allocs;
  int32_t* d_cnt = nullptr;          // [max(n_tiles, num_pages)] compile scratch
  int32_t* d_scratch = nullptr;      // [8] compile scratch (status, maxima, counts, pairs)
  // decode plans: the cursors, their lengths when the plan was built or last advanced, and
  // host copies of tile_off and of the split-KV tables (split cursor, first / end entry,
  // kv page of the first entry, launch order, first split per cursor), kept so that an
  // advance by one token per cursor updates them without reading the device
  std::vector<int32_t> cur_seg, cur_len, h_toff;
  std::vector<int32_t> h_sp_tile, h_sp_e0, h_sp_e1, h_sp_first, h_sp_order, h_cur0;
  // the advance's host-side counterparts: last time's split arrays (their storage is
  // reused) and the decode plan's tile order, kept to re-sort it incrementally
  std::vector<int32_t> x_sp_tile, x_sp_e0, x_sp_e1, x_sp_first, x_sp_order, x_cur0, h_tord;
  bool dup_cursors = false;          // a cursor listed twice (advance then refuses)
  std::vector<int32_t> h_stage;      // staging of the small arrays an advance uploads
  void* adv_buf = nullptr;           // device copy of the last advance's small arrays
  // An advance that opens pages writes the entries, CSC, page offsets, touched pages and
  // its small arrays into spare arrays and swaps them in; the arrays it replaced are the
  // next such advance's spares (capacities in elements).
  octo_entry* sp_entries = nullptr;
  int32_t *sp_csc = nullptr, *sp_poff = nullptr, *sp_touched = nullptr, *sp_buf = nullptr;
  size_t sp_entries_cap = 0, sp_csc_cap = 0, sp_poff_cap = 0, sp_touched_cap = 0, sp_buf_cap = 0;
  size_t entries_cap = 0, csc_cap = 0, poff_cap = 0, touched_cap = 0, buf_cap = 0;   // current arrays
  cudaEvent_t order_ev = nullptr;    // orders an advance after work on another stream
  cudaStream_t last_stream = nullptr;  // stream of the last call that used the plan
};

namespace octo {

extern thread_local int g_last_cuda_error;
void count_launch(int n = 1);
// Raises a kernel's dynamic shared-memory limit to `bytes` on the current device, once per
// (kernel, device, size): the attribute is per device, and one process may drive several.
int set_smem_limit(const void* func, int bytes);

inline int cuda_status(cudaError_t e) {
  if (e != cudaSuccess) {
    g_last_cuda_error = (int)e;
    return OCTO_ECUDA;
  }
  return OCTO_OK;
}

#define OCTO_CUDA(call)                                   \
  do {                                                    \
    int _st = ::octo::cuda_status(call);                  \
    if (_st != OCTO_OK) return _st;                       \
  } while (0)

// kernels launched by the host pool code
int launch_zero_pages(const octo_pool_desc& d, const int32_t* d_pages, int32_t n, cudaStream_t s);
int launch_append_rows(const octo_pool_desc& d, const int32_t* d_dst_rows, int32_t n, const void* k,
                       const void* v, cudaStream_t s);
// rotary embedding (rope.cu): K rotated at each appended token's position while copied
int rope_validate(int32_t head_dim, float base);
int launch_append_rope(const octo_pool_desc& d, const int32_t* d_dst_rows, const int32_t* d_pos, int32_t n,
                       const void* k, const void* v, float base, cudaStream_t s);

// plan compilation (compile.cu)
int compile_plan(octo_pool_s* pool, const int32_t* tile_segs_host, const int32_t* seg_order, int32_t n_segs,
                 bool is_decode, int32_t bm, cudaStream_t s, octo_plan_s** out);

constexpr int32_t kSplitEntries = 32;
constexpr int32_t kRecChunk = 64;   // rows per chunk of the tree-packed recurrent layer

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// An NVTX range over the scope (seen by nsys / ncu range filters; a no-op without a tool).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace octo
