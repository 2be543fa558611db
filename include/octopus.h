/* octopus.h -- C ABI of liboctopus: packed DAG attention over a paged, refcounted KV pool.
 *
 * The operations follow the Octopus project page (shatianming5.github.io/octopus):
 *   - "Architecture & Co-Design", item 01 (Runtime): server-resident radix cursors;
 *   - item 02 (Memory): zero-copy KV mount of a sibling span into attention layers at the
 *     monotonic position offset s(c'_B) = max(p_B, e_A + 1), allocating 0 new KV pages;
 *   - item 03 (Training): one unpadded 1D packed forward/backward pass with
 *     single-ownership masking, reader gradients routed into the producer's KV;
 *   - the five-primitives table (fork, read_thread, rewind, wait, done).
 *
 * Conventions
 *   - Every call returns an int status (OCTO_OK = 0).  Out-parameters are written only on
 *     success.  No C++ exception crosses this boundary.
 *   - Handles are opaque.  A pool and its plans are not thread-safe: one host thread at a
 *     time per pool.
 *   - Device memory for tensors (K/V pools, Q, O, LSE, dO, dQ, dK, dV, workspaces) is
 *     allocated and owned by the caller and passed as raw device pointers.  The library
 *     owns the host metadata of a pool and the device metadata arrays of a plan.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Kernels are enqueued asynchronously on it.  octo_pack_tree and octo_decode_plan
 *     synchronise the stream once (to size the tile list); the attention calls never do.
 *   - Cursor ids are segment ids: the n-th segment created by octo_root / octo_fork /
 *     octo_rewind in a pool has id n.
 *   - Sizes: a pool holds at most 2^31-1 tokens per plan; page_size <= 128; head_dim is
 *     64 or 128; n_q_heads a multiple of n_kv_heads.
 */
#ifndef OCTOPUS_H
#define OCTOPUS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---- */
enum {
  OCTO_OK = 0,
  OCTO_EINVAL = 1,   /* bad argument, out-of-range span, or a mount that would show a token twice */
  OCTO_ENOMEM = 2,   /* the pool has no free page for an append (nothing is changed) */
  OCTO_ESTATE = 3,   /* cursor is done, rewound away from, released, or freed */
  OCTO_ECUDA = 4,    /* a CUDA call failed; see octo_last_cuda_error() */
  OCTO_ETIMEOUT = 5, /* a bounded device wait expired; the kernel returned early */
  OCTO_ENOTSUP = 6,  /* shape or dtype the library has no kernel for */
  OCTO_ESCRATCH = 7  /* request needs more than the built-in scratch of octo_decode_noalloc */
};

enum { OCTO_DTYPE_F32 = 0, OCTO_DTYPE_BF16 = 1 };

typedef struct octo_pool_s* octo_pool_t;
typedef struct octo_plan_s* octo_plan_t;
typedef int32_t octo_cursor_t;

/* Pool description.  k_pool / v_pool: device arrays [num_pages][n_kv_heads][page_size]
 * [head_dim] of `dtype`, owned by the caller, alive as long as the pool.  octo_append
 * writes appended K/V rows into them; the attention calls read whatever pool arrays they
 * are given, which must have this layout (so one pool's page tables can serve the K/V of
 * several layers). */
typedef struct {
  int32_t num_pages;
  int32_t page_size;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t dtype;
  void* k_pool;
  void* v_pool;
} octo_pool_desc;

/* One block of the block-sparse schedule: query tile q_tile against the slots of
 * physical page kv_page that one source (src = -1: the tile's own tree path; src >= 0:
 * the mount with that id) makes visible.  Tile row r (0-based) sees page slot j iff
 *     r >= q_lo  &&  kv_lo <= j < kv_hi  &&  (!(flags & 1) || j <= r + diag).
 * 24 bytes, naturally aligned. */
typedef struct {
  uint32_t q_tile;
  uint32_t kv_page;
  uint16_t kv_lo;
  uint16_t kv_hi;
  uint16_t q_lo;
  uint16_t flags;
  int32_t diag;
  int32_t src;
} octo_entry;

/* Segment record returned by octo_seg_query.  flags: bit0 live cursor, bit1 pinned
 * (done), bit2 frozen (done), bit3 rewound away from, bit4 freed. */
typedef struct {
  int32_t parent;   /* segment it continues from, -1 for a root */
  int32_t fork;     /* tokens of the parent it sees */
  int32_t len;      /* own tokens */
  int32_t n_pages;  /* own pages */
  int32_t refcount; /* live cursor + live children + mounts reading it + pin */
  int32_t p_next;   /* position the next appended token gets */
  int32_t flags;
} octo_seg_info;

typedef struct {
  int64_t n_rows;      /* packed query rows (decode plan: one per cursor) */
  int64_t n_tiles;
  int64_t n_entries;
  int64_t n_segments;  /* packed segments */
  int64_t pairs;       /* visible (row, key) pairs: the useful work of one head */
  int32_t bm;          /* rows per q-tile */
  int32_t page_size;
  int32_t max_tile_entries;
  int32_t max_page_entries;
  int32_t n_touched_pages; /* pages some entry reads */
  int32_t is_decode;
  int32_t n_rec_runs;      /* pack plans: runs of the recurrent layer (rows with one path predecessor chain) */
  int32_t n_rec_chunks;    /* pack plans: their chunks of up to 64 rows */
} octo_plan_info_t;

/* ---- pool (host metadata; primitives table of the project page) ---- */

/* Creates a pool.  All pages start free.  EINVAL on a bad description.  No device
 * memory is touched until the first plan is compiled. */
int octo_pool_create(const octo_pool_desc* desc, octo_pool_t* out);
/* Destroys the pool (waits for the device first).  Its plans must be destroyed before. */
int octo_pool_destroy(octo_pool_t pool);

/* New root segment with a live cursor; positions start at 0. */
int octo_root(octo_pool_t pool, octo_cursor_t* out);

/* Appends n tokens to the cursor's segment.  Pages are taken lowest-free-id first as the
 * segment needs them; a segment's tokens fill its own pages in order.  pos_out (host,
 * n entries, may be NULL) receives each token's position: the cursor's next position,
 * which then advances by one.  k, v: device [n][n_kv_heads][head_dim] of the pool dtype,
 * copied into the pool arrays on `stream`; both NULL = no rows copied.  Every page newly
 * given to the segment is first zeroed in the pool's own arrays (when the pool has them):
 * the attention kernels read whole pages and mask the slots a row does not see, so those
 * slots must hold finite values.  Pool arrays passed directly to the attention calls must
 * keep the same property (zero-initialise them).
 * ENOMEM if the free pages do not suffice (nothing changes), ESTATE if the cursor is
 * frozen, rewound away from or released. */
int octo_append(octo_pool_t pool, octo_cursor_t cur, int32_t n, const void* k, const void* v,
                void* stream, int32_t* pos_out);

/* One token appended to each of n distinct cursors (a decode step's new tokens): the same
 * pages, positions and zeroing as n octo_append calls of one token, in one call and two
 * kernels.  k, v: device [n][n_kv_heads][head_dim] of the pool dtype, row i for cursors[i];
 * both NULL = layout only.  rope_base > 0: the K rows are rotated at the positions their
 * tokens receive, as octo_append_rope does; 0 = copied as given.  pos_out (host, n entries,
 * may be NULL) receives the positions.  All or nothing: EINVAL (a cursor listed twice or
 * out of range, a bad rope_base), ESTATE (a cursor frozen, rewound away from or
 * released) and ENOMEM (fewer free pages than the cursors that open one) leave the pool
 * unchanged.  Queued on `stream` without waiting for the device. */
int octo_append_step(octo_pool_t pool, const octo_cursor_t* cursors, int32_t n, const void* k,
                     const void* v, float rope_base, void* stream, int32_t* pos_out);

/* fork: n children that each see the parent's current tokens and the mounts the parent
 * holds now (O(1): no page is allocated or copied; the parent's refcount grows by n).
 * Each child starts on a fresh page and at the parent's next position.  out: n ids. */
int octo_fork(octo_pool_t pool, octo_cursor_t parent, int32_t n, octo_cursor_t* out);

/* read_thread: mounts the producer's own tokens [a, b) into the reader's attention
 * context from the reader's next token on (point m = reader's current length); later
 * children of the reader inherit it.  No page is allocated.  The reader's next position
 * becomes max(p_B, e_A + 1) with p_B its next position before the mount and
 * e_A = pos(producer, b-1) + 1.  new_pos (may be NULL) receives it.  EINVAL if
 * 0 <= a < b <= len(producer) fails or if any token of the span is already in the
 * reader's context (its own path, or an earlier mount it sees). */
int octo_mount(octo_pool_t pool, octo_cursor_t reader, octo_cursor_t producer, int32_t a,
               int32_t b, int32_t* new_pos);

/* rewind: a continuation segment that sees the first k tokens of `cur` (and the mounts
 * with point <= k); its next position is that of token k.  The cursor moves to the
 * continuation (returned in out); the old segment keeps its tail as a dead-end leaf
 * (still packed and trained) until released with its continuation. */
int octo_rewind(octo_pool_t pool, octo_cursor_t cur, int32_t k, octo_cursor_t* out);

/* done: freezes the segment (no more appends, forks or mounts into it) and pins its
 * pages (+1 refcount) so that they stay readable by mounts after the cursor is
 * released.  octo_unpin drops the pin. */
int octo_done(octo_pool_t pool, octo_cursor_t cur);
int octo_unpin(octo_pool_t pool, octo_cursor_t cur);

/* Drops the cursor's reference.  A segment whose refcount reaches 0 is freed: its pages
 * return to the pool and its references on its parent and on the producers it mounted
 * are dropped in turn. */
int octo_release(octo_pool_t pool, octo_cursor_t cur);

/* Pool state in one call: the primitives table's refcounts ("+K refs" on fork, the pin of
 * done) and page ownership.  Inputs: seg_capacity, and the optional host arrays refcount
 * and n_pages ([seg_capacity] entries, indexed by segment id; EINVAL if seg_capacity is
 * below the number of segments while either is given) and page_owner ([num_pages]: the
 * segment owning each page, -1 for a free page).  Outputs: the counts. */
typedef struct {
  int32_t n_segments;    /* out: segments created so far (freed ones included) */
  int32_t free_pages;    /* out */
  int32_t n_mounts;      /* out: mounts made so far */
  int32_t num_pages;     /* out */
  int32_t seg_capacity;  /* in */
  int32_t* refcount;     /* in/out, may be NULL: live cursor + live children + mounts reading it + pin (0 when freed) */
  int32_t* n_pages;      /* in/out, may be NULL: pages the segment owns */
  int32_t* page_owner;   /* in/out, may be NULL */
} octo_pool_state;
int octo_pool_query(octo_pool_t pool, octo_pool_state* state);

/* The counts of octo_pool_query alone. */
int octo_pool_info(octo_pool_t pool, int32_t* n_segments, int32_t* free_pages,
                   int32_t* n_mounts);
/* One segment: its record, and the optional host outputs pos (len entries: each token's
 * position) and pages (n_pages entries: its own pages in token order). */
int octo_seg_query(octo_pool_t pool, octo_cursor_t seg, octo_seg_info* info, int32_t* pos,
                   int32_t* pages);

/* ---- plans (item 03: compile the tree and its mount edges into one packed pass) ---- */

/* Packs every live segment descending from the given roots, in (root order, segment id)
 * order, unpadded: row_base = exclusive scan of the segment lengths.  Each segment's
 * rows are cut into q-tiles of bm rows (the last one ragged); the GPU compiler emits, per
 * tile, one entry per (page, source) block of visible keys, in the order those keys
 * first appear in the context of the tile's last row, then a kv-page-major view (CSC)
 * for the backward pass.  Synchronises `stream` once.  1 <= bm <= 128 (multiples of 16
 * for the tensor-core kernels: bm = 128 is what they run). */
int octo_pack_tree(octo_pool_t pool, const octo_cursor_t* roots, int32_t n_roots, int32_t bm,
                   void* stream, octo_plan_t* out);

/* Decode plan: one row per cursor -- the cursor's last token -- against its whole
 * context (prefix pages, own pages, mounted spans).  Same entry format, one tile per
 * cursor.  Synchronises `stream` once. */
int octo_decode_plan(octo_pool_t pool, const octo_cursor_t* cursors, int32_t n, void* stream,
                     octo_plan_t* out);

/* Moves a decode plan on by one token per cursor, after each of its cursors had exactly
 * one token appended (octo_append / octo_append_rope) since the plan was built or last
 * advanced: the result equals octo_decode_plan on the same cursors, array for array and
 * bit for bit (octopus project page, "Architecture & Co-Design" item 01: a turn extends
 * a cursor over the same shared pages, so the view changes only by the new token; the
 * pages quote 128K prompt assembly in 1.44 ms).  Per cursor, the newest token either
 * widens the entry of its own last page or, when it opens a page, adds that page's entry
 * at the end of the cursor's list.  When no cursor opens a page this is one kernel that
 * updates the plan in place; otherwise the entries, the CSC view, page offsets and touched
 * pages are rebuilt by device kernels from the old ones, and the split-KV runs and launch
 * orders from host copies kept with the plan; the arrays replaced are kept with the plan
 * and written by the next such advance, which allocates only when they are too small.
 * It never waits for the device; the work is
 * queued on `stream`, ordered after the work queued on the stream that last used the plan.
 * OCTO_ESTATE, with the plan unchanged, when a cursor is not exactly one token longer, was
 * freed, has a mount at or after the point of its new token (its context then grows by
 * more than that token), or is listed twice in the plan: build a fresh plan instead.
 * Segments whose pages the plan reads must not be released in between.  On any other
 * error the plan must be destroyed.  The plan can have more split-KV runs afterwards:
 * query octo_decode_workspace_size again. */
int octo_decode_plan_advance(octo_plan_t plan, void* stream);

int octo_plan_info(octo_plan_t plan, octo_plan_info_t* info);

/* Copies the plan to host buffers (each may be NULL); synchronous.  Sizes: seg_order,
 * seg_row_base [n_segments]; row_pos [n_rows]; tile_seg, tile_t0, tile_rows [n_tiles];
 * tile_off [n_tiles+1]; entries, csc_perm [n_entries]; page_off [num_pages+1]. */
int octo_plan_copy_out(octo_plan_t plan, int32_t* seg_order, int32_t* seg_row_base,
                       int32_t* row_pos, int32_t* tile_seg, int32_t* tile_t0,
                       int32_t* tile_rows, int32_t* tile_off, octo_entry* entries,
                       int32_t* csc_perm, int32_t* page_off);
/* Frees the plan's device arrays in stream order on the stream of the last call that
 * used the plan, so it may be called while that work is still running; work using the
 * plan on any other stream must have completed. */
int octo_plan_destroy(octo_plan_t plan);

/* ---- rotary position embedding at the packed positions ----
 * Octopus project page, "Architecture & Co-Design" item 02 and the cross-branch sharing
 * table: mounted sibling keys are read rotation-free (as stored) under the monotonic
 * offset s = max(p_B, e_A + 1); only the reader's positions jump.  Without the jump a
 * longer sibling's keys would sit at or after the reader's queries ("RoPE flip").  So keys
 * are rotated once, when appended, at the position the pool gives each token, and queries
 * at the position of their packed row.  Rotation, half-split form: for a head vector x of
 * dimension d at position p and i < d/2, (x_i, x_{i+d/2}) turns by the angle
 * p * base^(-2i/d), formed and reduced modulo 2 pi in double precision.  head_dim must be
 * even and at most 128; base > 0 and finite (EINVAL otherwise). */

/* octo_append with each K row rotated at the position its token receives (V copied as
 * is); same pages, positions, zeroing and errors as octo_append. */
int octo_append_rope(octo_pool_t pool, octo_cursor_t cur, int32_t n, const void* k, const void* v,
                     float base, void* stream, int32_t* pos_out);

/* Rotates in place x [n_rows][n_heads][head_dim] (dtype OCTO_DTYPE_BF16 or
 * OCTO_DTYPE_F32, device) in the plan's packed row order, each row at its position: a
 * pack plan's rows, or a decode plan's one row per cursor (its newest token).  inverse = 0
 * before attention (queries); inverse = 1 turns back, mapping the gradient with respect
 * to the rotated rows (octo_attn_bwd's dq) to the gradient with respect to the rows as
 * given.  Async on stream. */
int octo_rope_rows(octo_plan_t plan, int32_t n_heads, void* x, int32_t dtype, float base,
                   int32_t inverse, void* stream);

/* Turns key gradients from octo_attn_bwd (fp32, pool-shaped [num_pages][n_kv_heads]
 * [page_size][head_dim]) back through the append rotation: every slot of every page the
 * plan reads, at its token's position, with the inverse rotation; slots holding no token
 * and pages the plan does not read are left as they are.  dv needs nothing (V is not
 * rotated).  Uploads a host-built table of slot positions and waits for the stream before
 * returning. */
int octo_rope_pool_grad(octo_plan_t plan, float* dk_pool, float base, void* stream);

/* ---- per-token log-probability and loss over the packed rows ----
 * Octopus project page, "Architecture & Co-Design" item 03 (1D packed DAG-GRPO): every
 * branch trains in one packed pass and single-ownership masking counts a shared prefix
 * once; the five-primitives table, row done, has an untrainable close reminder (mask
 * m = 0).  Each packed row t is one owned token, with id ids[t] and weight w[t] (the
 * caller's m * advantage; NULL weight = 1).  Its term uses the logits row of pred(t), the
 * row of the token before it on its path: t - 1 inside a segment; for a segment's first
 * row the parent's row at the fork point minus one (through forks at point 0); none for a
 * root's first token, whose logp is 0 and which adds nothing.  Mounted spans change no
 * predecessor.  With lse(r) = log sum_v exp(x[r][v]):
 *     logp[t] = x[pred t][ids t] - lse(pred t),   loss = - sum_t w[t] logp[t],
 *     dlogits[r][v] = grad_scale * (W_r softmax(x[r])_v - sum over t with pred t = r and
 *                     ids t = v of w[t]),  W_r = sum over t with pred t = r of w[t]. */

/* Workspace (bytes) for octo_token_logprob over n_rows rows. */
int octo_token_logprob_workspace_size(int32_t n_rows, size_t* bytes);

/* Rows [row0, row0 + n_rows) of a pack plan (not a decode plan): logits [n_rows][ld]
 * (dtype OCTO_DTYPE_BF16 or OCTO_DTYPE_F32, device, 16-byte aligned, ld * element size a
 * multiple of 16, ld >= vocab), row row0 + i at logits + i * ld.  ids, weight, logp:
 * device arrays over ALL rows of the plan (a row's successor can lie past the chunk).
 * Writes logp[t] for every t whose predecessor is in the chunk, and 0 for the chunk's path
 * starts; row_lse [n_rows] (natural log, optional); dlogits (optional, same dtype, layout
 * and alignment as logits; may be logits itself: the gradient then overwrites the logits);
 * loss (optional, one device float: - sum of w[t] logp[t] over the chunk's rows' successors,
 * summed in a fixed order).  ws: device workspace of the size above.  Ids outside
 * [0, vocab) give NaN logp, no gradient term, and OCTO_EINVAL at the next octo_sync.
 * OCTO_ENOTSUP if a row of the plan has more than 64 successors.  Async on stream. */
int octo_token_logprob(octo_plan_t plan, int32_t row0, int32_t n_rows, const void* logits, int32_t dtype,
                       int64_t ld, int32_t vocab, const int32_t* ids, const float* weight, float* logp,
                       float* row_lse, void* dlogits, float grad_scale, float* loss, void* ws, size_t ws_bytes,
                       void* stream);

/* ---- tree-packed recurrent layer (gated delta rule), device, async on stream ----
 * ia.com.br summary, associative versus working memory: the hybrid model pairs attention
 * with linear-recurrent layers (Gated DeltaNet / Mamba-2) whose state is the branch's
 * working memory.  Octopus project page, five-primitives table: fork clones the recurrent
 * checkpoint at the fork point, rewind restores the exact state of step k, and
 * read_thread's mounted span is skipped by the recurrent layers; "Architecture &
 * Co-Design" item 03: the packed pass carries the recurrent boundary checkpoints.
 * Per head, state S [head_dim x head_dim] (rows: value dimension):
 *     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t,
 * S_{t-1} the state after the row before t on its path (the previous own row; for a
 * segment's first row the parent's row at the fork or rewind point minus one, through
 * forks at point 0), S = 0 before a path's first row; mounts change nothing.  The gate
 * activations, feature maps and normalisation are the caller's: q, k, v, alpha, beta
 * arrive as they enter the recurrence.  Computed in chunks of 64 rows along runs of the
 * pack plan, fp32 on the CUDA cores. */

/* Workspace bytes of octo_recurrent_fwd / bwd for this pack plan (0 on bad arguments). */
size_t octo_recurrent_workspace_size(octo_plan_t plan, int32_t n_heads, int32_t head_dim);

/* Forward over a pack plan's rows: q, k, v, o fp32 [n_rows][n_heads][head_dim]; alpha, beta
 * fp32 [n_rows][n_heads], alpha in (0, 1] (its log is taken), beta any finite value.
 * head_dim 64 or 128 (EINVAL otherwise, and for a decode plan).  ws: device workspace of
 * octo_recurrent_workspace_size bytes; the forward leaves in it the chunk states the
 * backward reads, so pass the same ws, unchanged, to octo_recurrent_bwd.  Deterministic. */
int octo_recurrent_fwd(octo_plan_t plan, int32_t n_heads, int32_t head_dim, const float* q,
                       const float* k, const float* v, const float* alpha, const float* beta,
                       float* o, void* ws, size_t ws_bytes, void* stream);

/* Backward of octo_recurrent_fwd for the same inputs and workspace: with dout the gradient
 * of the loss with respect to o, writes dq, dk, dv [n_rows][n_heads][head_dim] and dalpha,
 * dbeta [n_rows][n_heads] (fp32).  A row with several successors (a fork or rewind point)
 * receives the sum of their state gradients, taken in a fixed order. */
int octo_recurrent_bwd(octo_plan_t plan, int32_t n_heads, int32_t head_dim, const float* q,
                       const float* k, const float* v, const float* alpha, const float* beta,
                       const float* dout, float* dq, float* dk, float* dv, float* dalpha,
                       float* dbeta, void* ws, size_t ws_bytes, void* stream);

/* ---- packed DAG attention (device, async on stream) ----
 * Octopus project page, "Architecture & Co-Design" item 03 (Training): one unpadded 1D
 * packed forward/backward pass over the branched trees and their live mount edges, with
 * single-ownership masking (every token stored and owned once; each query row sees its
 * tree-ancestor path and the spans mounted on it), the reader's gradients routed directly
 * into the producer's KV; the ia.com.br summary calls it a block-sparse attention pass.
 * The schedule is the plan's entry list; attention itself is softmax(scale q k^T) v. */

/* Forward over a packed plan.  For query head h the kv head is h / (n_q_heads /
 * n_kv_heads).  q, o: [n_rows][n_q_heads][head_dim] of the pool dtype; lse: fp32
 * [n_q_heads][n_rows], natural log of the softmax denominator of the scaled scores.
 * k_pool / v_pool NULL = the pool's own arrays.  scale multiplies q.k (1/sqrt(d) is
 * the usual choice). */
int octo_attn_fwd(octo_plan_t plan, int32_t n_q_heads, const void* q, const void* k_pool,
                  const void* v_pool, void* o, float* lse, float scale, void* stream);

/* Workspace bytes octo_attn_bwd needs for this plan and head count. */
size_t octo_attn_bwd_workspace_size(octo_plan_t plan, int32_t n_q_heads);

/* Backward of octo_attn_fwd given o, lse and dout (same layouts as the forward).
 * dq: fp32 [n_rows][n_q_heads][head_dim].  dk_pool, dv_pool: fp32, pool-shaped
 * [num_pages][n_kv_heads][page_size][head_dim]; every page some entry of the plan reads
 * is overwritten with the sum, over every reader row and the query heads of its group,
 * of that key's gradient (slots no row sees get 0); other pages are not touched.  The
 * sums are taken in a fixed order without atomics, so results are deterministic. */
int octo_attn_bwd(octo_plan_t plan, int32_t n_q_heads, const void* q, const void* k_pool,
                  const void* v_pool, const void* o, const float* lse, const void* dout,
                  float* dq, float* dk_pool, float* dv_pool, float scale, void* ws,
                  size_t ws_bytes, void* stream);

/* ---- paged decode over cursors ----
 * Octopus project page, "Architecture & Co-Design" item 01 (Runtime): cursors stay resident
 * on the serving side over shared KV pages, and each turn extends a cursor; item 02 and
 * the primitives table, row read_thread: a reader's attention also sees its mounted
 * sibling spans, read in place.  Decoding one token per cursor is the last row of a packed
 * pass over that cursor's context.  The decode takes a plan (octo_decode_plan) so that the
 * context walk is done once and the plan moved on by one token per step
 * (octo_decode_plan_advance) while the kernel streams the pages; octo_decode_cursors does
 * all of it in one call. */

/* Workspace bytes octo_decode needs for this plan and head count (split-KV partials). */
size_t octo_decode_workspace_size(octo_plan_t plan, int32_t n_q_heads);

/* Paged decode over a decode plan: for cursor i and query head h, out[i][h] =
 * softmax(scale * q[i][h] . K_ctx) V_ctx over the cursor's context (its last token
 * included), kv head h / (n_q_heads / n_kv_heads).  q, out: [n][n_q_heads][head_dim] of
 * the pool dtype (device); lse: fp32 [n][n_q_heads] natural log (may be NULL).  ws: device
 * workspace of octo_decode_workspace_size bytes (EINVAL if smaller).  k_pool / v_pool NULL
 * = the pool's arrays.  Async on stream; the split partials are combined in a fixed
 * order, so results are deterministic. */
int octo_decode(octo_plan_t plan, int32_t n_q_heads, const void* q, const void* k_pool,
                const void* v_pool, void* out, float* lse, float scale, void* ws,
                size_t ws_bytes, void* stream);

/* The decode straight from cursors: octo_decode_plan, octo_decode, octo_plan_destroy in one
 * call (arguments as there).  ws may be NULL: the library then takes the workspace from
 * the stream-ordered allocator (cudaMallocAsync on `stream`) and returns it after the
 * decode.  Synchronises the stream once (the plan compile).  A caller decoding the same
 * cursors step after step keeps a plan and advances it instead. */
int octo_decode_cursors(octo_pool_t pool, const octo_cursor_t* cursors, int32_t n,
                        int32_t n_q_heads, const void* q, const void* k_pool, const void* v_pool,
                        void* out, float* lse, float scale, void* ws, size_t ws_bytes,
                        void* stream);

/* Allocation-free variant of octo_decode, for callers that must not allocate device
 * memory: engines whose device memory is all handed out by their own allocator at
 * start-up, or code running where a cudaMalloc (or a torch allocation) is not allowed.
 * Such callers still pass q, out and lse, but cannot provide octo_decode's workspace.
 * The pages have no counterpart for this entry point; it is a deployment convenience.
 *
 * The split partials live in a file-scope device array of OCTO_NOALLOC_SCRATCH_BYTES
 * bytes (32 MiB) that every GPU which loads the library holds until the process exits.
 * A call needs octo_decode_workspace_size(plan, n_q_heads) bytes of it; larger requests
 * return OCTO_ESCRATCH and launch nothing.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current, once per CUDA
 * context (again after the context is destroyed and made anew, e.g. by cudaDeviceReset);
 * make that first call before any stream capture.  The call itself allocates nothing.  Every call
 * shares the one array and each call overwrites the part it reads before reading it, so
 * nothing needs clearing between calls -- but calls that overlap on the GPU (on different
 * streams, or on different host threads) race on it and must be serialised by the
 * caller.  Arguments, layouts and results are those of octo_decode; bf16 pools with
 * head_dim 128 and page size 64 only (OCTO_ENOTSUP otherwise). */
#define OCTO_NOALLOC_SCRATCH_BYTES (32u << 20)
int octo_decode_noalloc(octo_plan_t plan, int32_t n_q_heads, const void* q, const void* k_pool,
                        const void* v_pool, void* out, float* lse, float scale, void* stream);

/* ---- diagnostics ---- */
const char* octo_strerror(int status);
int octo_last_cuda_error(void);   /* last cudaError_t seen by the library */
/* Waits for the stream, then returns the device status word of the pool's plans
 * (OCTO_ETIMEOUT if a bounded wait expired) and clears it. */
int octo_sync(octo_plan_t plan, void* stream);
/* Self-test of the failure path of the kernels' bounded waits (the pages have no
 * counterpart): one CTA waits, through the same bounded mbarrier wait the tensor-core and
 * decode kernels use, on a barrier phase that nothing completes, gives up after max_polls
 * polls (1 .. 2^27), records OCTO_ETIMEOUT in the status word of the plan's pool and
 * returns.  No copy or MMA is in flight and nothing else is written, so the context stays
 * usable: the next octo_sync on the plan returns OCTO_ETIMEOUT (and clears it), and later
 * calls run normally.  Async on stream. */
int octo_wait_selftest(octo_plan_t plan, uint32_t max_polls, void* stream);
/* Which kernel family octo_attn_fwd / bwd / decode will use for this plan:
 * 0 = CUDA-core (SIMT) kernels, 1 = tcgen05 tensor-core kernels (the backward takes them
 * only with a nonzero scale), 2 = split-KV decode kernels.  which: 0 fwd, 1 bwd,
 * 2 decode. */
int octo_kernel_path(octo_plan_t plan, int32_t n_q_heads, int32_t which);
/* Number of kernels the library has enqueued in this process so far (all pools, all
 * streams).  The difference across a region counts the region's launches. */
int64_t octo_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* OCTOPUS_H */
