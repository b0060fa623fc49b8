/*
 * dendrite.h -- C ABI of a copy-on-write, tree-structured paged KV cache with
 * tree-aware decode attention, for NVIDIA GB300 (sm_103a).
 *
 * The method (Dendrite article, ainews.cool "Dendrite: O(1) KV cache forking",
 * section 技术深度解析; dendrite demo.tape, section "The problem"):
 *   - KV rows live in fixed-size blocks; each branch has a block table.
 *   - A fork at token t shares every block of positions 0..t-1 with the
 *     parent (table copy + refcount increment, no KV copied); the child then
 *     owns only the leaf blocks it appends.
 *   - An append into a partially filled tail block that is still shared
 *     (refcount > 1) first copies that block (copy-on-write).
 *   - Decode attention walks the tree: keys/values of the shared ancestor path
 *     and of the branch's own leaf path.  Shared-prefix blocks are streamed
 *     from HBM once for all descendant queries (short shared ranges in trees
 *     of short nodes may instead be re-read by the ranges that follow them:
 *     pool option fold_segments); partial (max, sum, acc) triples are merged
 *     with a log-sum-exp step.
 *
 * Conventions (all calls):
 *   - Every call returns an int: DENDRITE_OK (0) or a negative error code.
 *   - Host-checkable errors (bad argument, bad handle, capacity, dtype) are
 *     returned immediately and the call changes nothing.
 *   - Device work is stream-ordered on the caller's stream (a cudaStream_t
 *     passed as void*; NULL = the legacy default stream).  Calls return before
 *     the GPU work finishes.
 *   - Errors found on the device (an exhausted block pool, a wait that timed
 *     out) are sticky: the offending call's device effects are not applied,
 *     every later kernel of the pool becomes a no-op, and the error is
 *     returned by dendrite_sync() and by every call after the host has seen
 *     it.  A pool in this state can only be inspected and destroyed.
 *   - A pool is not thread-safe; calls on different streams must be ordered
 *     by the caller.
 *
 * Ownership:
 *   - The pool owns the KV block storage, refcounts, free stack, block tables
 *     and its scratch (cudaMalloc'd at create time, plus a grow-only
 *     attention workspace).
 *   - The caller owns Q, K, V and out (device pointers).  They must stay valid
 *     until the stream work of the call has completed.  The library keeps no
 *     caller pointer after a call returns.
 *   - Host arrays (branch lists, counts) are read during the call only.
 *   - Branch handles (int32) are owned by the caller until dendrite_free.
 */
#ifndef DENDRITE_H
#define DENDRITE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------- error codes */
#define DENDRITE_OK           0
#define DENDRITE_EINVAL      -1  /* bad argument (size, layout, duplicate branch, ...) */
#define DENDRITE_ENOMEM      -2  /* block pool exhausted (found on the device; sticky) */
#define DENDRITE_EBADHANDLE  -3  /* handle not live */
#define DENDRITE_ELIMIT      -4  /* capacity exceeded: branches, table row, plan size, scratch */
#define DENDRITE_EDTYPE      -5  /* unsupported dtype / head_dim / block_size combination */
#define DENDRITE_ECUDA       -6  /* a CUDA runtime call failed */
#define DENDRITE_ETIMEOUT    -7  /* a bounded device wait gave up (sticky) */
#define DENDRITE_ECORRUPT    -8  /* device metadata inconsistent (refcount underflow; sticky) */

/* ------------------------------------------------------------------ dtypes */
#define DENDRITE_FP32  0   /* fp32 K/V/Q/out; attention in fp32 FMA (no TF32)          */
#define DENDRITE_BF16  1   /* bf16 K/V/Q/out; attention on tensor cores, fp32 accumulate */
#define DENDRITE_TURBO 2   /* compressed blocks (dendrite_pool_create_turbo): bf16 K/V/Q/out
                            * in the calls, TurboQuant records in the pool               */

typedef struct dendrite_pool dendrite_pool;

/* Optional pool settings; pass NULL for defaults. */
typedef struct dendrite_pool_opts {
    int32_t max_branches;          /* live handles at once (default 4096)                 */
    int32_t max_blocks_per_branch; /* block-table row length (default 4096 = 64K tokens)  */
    int32_t tc_min_rows;           /* bf16 attention: sharing segments read by more than  *
                                    * this many query rows per KV head run on the tcgen05 *
                                    * (tensor memory) kernel, the others on the mma.sync  *
                                    * kernel.  0 = default (64); -1 = never.               */
    int32_t n_layers;              /* model layers held (0 = 1): every layer has its own  *
                                    * K and V pools; block ids, tables, refcounts and the *
                                    * free stack are shared by all layers.                */
    int32_t fold_segments;         /* attention planning: a short sharing segment whose   *
                                    * rows continue into several longer ones is read      *
                                    * again by each of them instead of producing partial  *
                                    * rows of its own, when an estimate of the kernels'   *
                                    * time says that is cheaper.  0 = default (fold when  *
                                    * the estimate drops); k > 0 = fold when it drops     *
                                    * below k percent; -1 = never.                        */
    int32_t device_planning;       /* bf16 attention plans: expand the sharing segments   *
                                    * into work units and split them over CTAs on the GPU *
                                    * (a kernel between the plan upload and the partial   *
                                    * kernels) rather than on the host.  0 = default      *
                                    * (plans of at least 2048 units averaging fewer than  *
                                    * 32 tiles per unit, whose host expansion rivals the  *
                                    * kernels' work), 1 = always, -1 = never.  The result *
                                    * is the same plan either way.                        */
    int32_t tc_sms;                /* bf16 attention calls with work for both partial     *
                                    * kernels: SMs given to the tcgen05 kernel (one CTA   *
                                    * each) while the mma.sync kernel's CTAs take the     *
                                    * others, so the two run side by side.  0 = default   *
                                    * (an estimate of both kernels' time picks the split, *
                                    * or none: then each SM goes to the mma.sync kernel   *
                                    * when its tcgen05 CTA finishes); k > 0 = k SMs (no   *
                                    * split from the SM count up); -1 = never split.      */
    int32_t pack_segments;         /* bf16 attention planning: a sharing segment takes    *
                                    * the tiles of the segments that follow it, when none *
                                    * of those has followers of its own, as extra tiles   *
                                    * read by their own rows only (one unit instead of    *
                                    * several; dendrite_plan_segments_packed), when an    *
                                    * estimate of the kernels' time drops.  0 = default;  *
                                    * k > 0 = when it drops below k percent; -1 = never.  */
    int32_t reserved[1];           /* must be zero                                         */
} dendrite_pool_opts;

/*
 * Create a block pool.
 *   num_blocks  > 0: number of KV blocks.
 *   block_size  tokens per block; 16 (the attention kernels' tile height).
 *   n_kv_heads  KV heads per token (1..64).
 *   head_dim    bf16: 128.  fp32: a multiple of 32, at most 256.
 *   dtype       DENDRITE_FP32 or DENDRITE_BF16.
 * Device layout: K and V pools are [n_layers][num_blocks][n_kv_heads][block_size][head_dim]
 * (one (block, head) tile is contiguous); refcount int32[num_blocks]; the free
 * stack int32[num_blocks] starts as [num_blocks-1, ..., 0] so block 0 is handed
 * out first; block tables int32[max_branches][max_blocks_per_branch] (-1 = empty).
 * Synchronous.  Uses the current CUDA device.
 */
int dendrite_pool_create(int64_t num_blocks, int32_t block_size, int32_t n_kv_heads,
                         int32_t head_dim, int32_t dtype, const dendrite_pool_opts* opts,
                         dendrite_pool** out);

/*
 * A pool whose blocks hold compressed rows (dendrite demo.tape, section
 * "TurboQuant": "TurboQuant KV compression (PolarQuant + QJL)"; the pages
 * name the methods and give a 3.05x ratio at head_dim 128, not the
 * algorithm, so the steps follow the published PolarQuant, QJL and
 * TurboQuant methods):
 *   - every K and V row r (head_dim 128) is rotated, x = H (s * r) / sqrt(128),
 *     H the Walsh-Hadamard matrix and s = rot_signs (host float[128], each
 *     +1 or -1);
 *   - the recursive polar transform of x is stored as its norm (fp32), 64
 *     level-1 angle codes of 4 bits (16 equal bins of [0, 2 pi)) and 63 codes
 *     of 3 bits for the angles of levels 2..7 (8 equal bins of
 *     [pi/4 - w, pi/4 + w], w = min(pi/4, 1.6 / sqrt(k - 1)) for halves of
 *     k = 2^(level - 1) coordinates);
 *   - a key row also stores sign(S e) (128 bits) and |e| (fp32) for its
 *     residual e = x - x_hat, S = qjl_matrix (host float[128][128], row-major,
 *     normally i.i.d. N(0, 1)), and attention scores it as
 *     <q', x_hat> + sqrt(pi/2)/128 |e| <S q', sign(S e)> with q' the rotated
 *     query.
 * Records: a value row is 64 bytes (norm; 32 bytes of 4-bit codes, code i in
 * byte 4 + i/2, low nibble for even i; 24 bytes holding the 3-bit codes of
 * levels 2..7 in level order, code i at bit 3 i of a little-endian stream;
 * 4 zero bytes); a key row is 96 bytes (the value layout, then the 128 sign
 * bits, bit j in byte 64 + j/8 at bit j % 8, then |e|, then 12 zero bytes).
 * K + V take 160 bytes per token and head instead of 512 in bf16 (3.2x).
 * The encoder takes its bin and sign decisions in fp32, one rounded operation
 * at a time in a fixed order, so records depend only on the input bits.
 * K and V of dendrite_append_kv / _append_layer, and Q and out of the
 * attention calls, are bf16; dendrite_read_block returns the raw records
 * ([n_kv_heads][block_size][96] and [...][64] bytes).  head_dim must be 128;
 * other arguments and errors as dendrite_pool_create (dtype DENDRITE_TURBO).
 */
int dendrite_pool_create_turbo(int64_t num_blocks, int32_t block_size, int32_t n_kv_heads, int32_t head_dim,
                               const float* rot_signs, const float* qjl_matrix, const dendrite_pool_opts* opts,
                               dendrite_pool** out);

/* Synchronises the device, then releases everything the pool owns. */
int dendrite_pool_destroy(dendrite_pool* pool);

/* New empty root branch (length 0).  Host only: no device work. */
int dendrite_branch_new(dendrite_pool* pool, int32_t* out_branch);

/*
 * Fork: n_children new branches that share every block of `parent`
 * (Dendrite article, section 技术深度解析: a fork at t keeps positions 0..t-1
 * shared and gives each branch an empty leaf for positions >= t).
 * On the device: each child's table row is a copy of the parent's
 * ceil(len/block_size) entries and each of those blocks gains n_children
 * references.  No KV is copied.  The parent stays live and unchanged.
 * out_children: host int32[n_children], written before the call returns.
 */
int dendrite_fork(dendrite_pool* pool, int32_t parent, int32_t n_children,
                  int32_t* out_children, void* stream);

/*
 * Batched fork: parent i gets n_children[i] children, written in order to
 * out_children (host int32[sum n_children]).  One kernel launch for the whole
 * batch.  A parent may appear more than once.
 */
int dendrite_fork_batch(dendrite_pool* pool, const int32_t* parents, const int32_t* n_children,
                        int32_t n_parents, int32_t* out_children, void* stream);

/*
 * Append n_new tokens to every branch in `branches` (host int32[n_branches],
 * no duplicates).  K, V: device, [n_branches][n_new][n_kv_heads][head_dim] in
 * the pool dtype, contiguous.
 * Copy-on-write (dendrite demo.tape, section "The problem"): a branch whose
 * tail block is partially filled copies the tail's valid slots into a fresh
 * block first iff the tail's refcount is above 1 at its turn; the branches of
 * one call are served as if one after the other in argument order.  New blocks
 * come off the free stack in argument order, copy first, then in position
 * order.  All-or-nothing: if the pool has too few free blocks the call
 * applies nothing and the pool reports DENDRITE_ENOMEM (sticky).
 * n_new == 0 is a no-op.
 * A pool of n_layers > 1 takes every layer at once: K, V are
 * [n_layers][n_branches][n_new][n_kv_heads][head_dim]; the copy-on-write and
 * allocation decisions are made once and applied to every layer.
 * DENDRITE_EINVAL while a split append (below) is pending.
 */
int dendrite_append_kv(dendrite_pool* pool, const int32_t* branches, int32_t n_branches,
                       int32_t n_new, const void* K, const void* V, void* stream);

/*
 * Split append for a decode step through a multi-layer model, where layer l's
 * K and V only exist once layer l has run.  No counterpart on the pages: it
 * is dendrite_append_kv cut at its one natural seam (the block decisions are
 * the same for every layer; only the rows differ).
 *   dendrite_append_begin: the copy-on-write decisions, block allocation,
 *     table and refcount updates and the new lengths, for all layers at once
 *     (same rules, order and all-or-nothing behaviour as dendrite_append_kv).
 *     No rows are written yet.
 *   dendrite_append_layer: writes layer `layer`'s rows of the pending append
 *     (K, V: [n_branches][n_new][n_kv_heads][head_dim] as in dendrite_append_kv)
 *     and that layer's copy-on-write slot copies.  Each layer exactly once, in
 *     any order; the append stops being pending when every layer is written.
 * While an append is pending: dendrite_append_kv, dendrite_append_begin,
 * dendrite_free and dendrite_truncate return DENDRITE_EINVAL, and attention
 * on a layer whose rows are not written yet returns DENDRITE_EINVAL.
 * Forks are allowed (a child shares the pending rows like any other).
 */
int dendrite_append_begin(dendrite_pool* pool, const int32_t* branches, int32_t n_branches,
                          int32_t n_new, void* stream);
int dendrite_append_layer(dendrite_pool* pool, int32_t layer, const void* K, const void* V, void* stream);

/*
 * Tree decode attention (Dendrite article, section 技术深度解析: attention
 * gathers keys and values from the shared ancestor path and the branch's own
 * leaf path).
 *   Q:   device, [n_branches][q_len][n_q_heads][head_dim], pool dtype.
 *   out: device, same shape and dtype (written).
 *   n_q_heads: a multiple of n_kv_heads; query head h reads KV head h / (n_q_heads / n_kv_heads).
 *   q_len >= 1: the queries are the branch's last q_len positions; query j sees
 *        positions <= len - q_len + j.  Every branch needs len >= q_len.
 * out = softmax(q K^T / sqrt(head_dim)) V per query row.  Blocks shared by
 * several queried branches are streamed once for all of them (split-KV
 * partials, then a log-sum-exp merge); a short shared range may instead be
 * read again by each longer range that follows it (pool option
 * fold_segments).  The plan built from the branch tree is cached until the
 * tree changes; after appends alone, where no queried branch reached a new
 * block, only its members' lengths are refreshed, and where some did, the
 * cached sharing segments are lengthened instead of found again when each of
 * those branches reads its last segment alone.  `branches` may not hold
 * duplicates.
 * DENDRITE_ELIMIT if a shared range would be read by 2^24 or more query rows
 * per KV head, or the plan outgrows 32-bit indices.
 * Reads layer 0 of a multi-layer pool.
 * Stream order: the call's work is ordered on `stream`.  When a bf16 call
 * has segments on both partial kernels (the tcgen05 one for segments read by
 * more than 64 rows per KV head, the mma.sync one for the rest), the
 * mma.sync kernel runs on a stream the pool owns, forked from `stream` and
 * joined back into it with events before the merge, so it overlaps the
 * tcgen05 kernel; work queued on `stream` after the call still sees the
 * output.
 */
int dendrite_tree_attn_decode(dendrite_pool* pool, const void* Q, int32_t n_q_heads, int32_t q_len,
                              const int32_t* branches, int32_t n_branches, void* out, void* stream);

/*
 * The same attention over layer `layer` (0 <= layer < n_layers) of a
 * multi-layer pool.  The plan depends only on the tree and the queried
 * branches, so the calls of one decode step for layers 0..n_layers-1 build it
 * once and reuse it.  DENDRITE_EINVAL if a pending split append has not
 * written this layer's rows yet.
 */
int dendrite_tree_attn_decode_layer(dendrite_pool* pool, int32_t layer, const void* Q, int32_t n_q_heads,
                                    int32_t q_len, const int32_t* branches, int32_t n_branches, void* out,
                                    void* stream);

/*
 * Free branches (host int32[n_branches], no duplicates): every block of each
 * table loses one reference; blocks that reach zero are pushed on the free
 * stack in descending id order (so one call that frees everything restores
 * the initial stack).  Handles become invalid at once.
 */
int dendrite_free(dendrite_pool* pool, const int32_t* branches, int32_t n_branches, void* stream);

/*
 * Rollback: branch i keeps only its first new_lens[i] tokens (host int32
 * arrays; 0 <= new_lens[i] <= current length; no duplicate branches).  This is
 * the reject step of speculative decoding (DSpark blog, section 第二层:
 * predict, verify in parallel, accept or roll back).  Table entries past
 * ceil(new_len / block_size) each drop one reference; blocks that reach zero
 * are pushed on the free stack in descending id order, as for free.  A kept
 * tail block that is now partially valid and still shared is copied on the
 * next append.  Branches forked from this one earlier keep everything they
 * share with it.  Accepting one draft path and discarding its siblings is a
 * truncate of the winner plus a free of the others.
 */
int dendrite_truncate(dendrite_pool* pool, const int32_t* branches, const int32_t* new_lens,
                      int32_t n_branches, void* stream);

/* Wait for the pool's work on `stream`, then return its sticky device status. */
int dendrite_sync(dendrite_pool* pool, void* stream);

/* ------------------------------------------------------------ inspection
 * Synchronous helpers for tests and tools (they synchronise `stream`).     */

/* Current length (tokens) of a live branch (host mirror; no device work). */
int dendrite_branch_len(dendrite_pool* pool, int32_t branch, int32_t* out_len);

/* Copy the first ceil(len/block_size) table entries of `branch` to host
 * int32 out[cap]; *n_out receives the count. */
int dendrite_read_table(dendrite_pool* pool, int32_t branch, int32_t* out, int32_t cap,
                        int32_t* n_out, void* stream);

/* Copy refcount[0..num_blocks) to host int32 out[num_blocks]. */
int dendrite_read_refcounts(dendrite_pool* pool, int32_t* out, void* stream);

/* Copy the live part of the free stack (bottom to top) to host int32
 * out[num_blocks]; *top_out receives its size. */
int dendrite_read_free_stack(dendrite_pool* pool, int32_t* out, int32_t* top_out, void* stream);

/* Copy one block's K and V ([n_kv_heads][block_size][head_dim], pool dtype;
 * the records for DENDRITE_TURBO pools) to host buffers k_out / v_out
 * (layer 0; dendrite_read_block_layer for any). */
int dendrite_read_block(dendrite_pool* pool, int32_t block, void* k_out, void* v_out, void* stream);
int dendrite_read_block_layer(dendrite_pool* pool, int32_t layer, int32_t block, void* k_out, void* v_out,
                              void* stream);

/*
 * Test hook for the device-side failure handling (no counterpart on the
 * pages): launches one thread that waits on an mbarrier nothing arrives at,
 * through the bounded wait every attention kernel uses (about 2 s of
 * %globaltimer).  When it gives up the pool records DENDRITE_ETIMEOUT, which
 * dendrite_sync then returns and every later call of the pool reports (the
 * pool is poisoned).  The device and the CUDA context stay usable.
 */
int dendrite_selftest_bounded_wait(dendrite_pool* pool, void* stream);

/* Number of layers the pool holds. */
int dendrite_pool_layers(dendrite_pool* pool, int32_t* n_layers);

/* Pool geometry: num_blocks, block_size, n_kv_heads, head_dim, dtype. */
int dendrite_pool_info(dendrite_pool* pool, int64_t* num_blocks, int32_t* block_size,
                       int32_t* n_kv_heads, int32_t* head_dim, int32_t* dtype);

/* ------------------------------------------------------------ profiling
 * With enable = 1, each call records CUDA events around each of its kernels
 * on the caller's stream; with enable = 2, only around whole attention calls
 * (ms[6]), so that a call's kernels keep overlapping one another as they do
 * unprofiled; 0 turns profiling off (other values: DENDRITE_EINVAL).
 * dendrite_last_timings() synchronises on them and
 * returns the device milliseconds of the most recent call of each kind:
 *   ms[0] fork, ms[1] append metadata, ms[2] append copy/scatter,
 *   ms[3] attention partial kernels, ms[4] log-sum-exp merge kernel,
 *   ms[5] free (or truncate), ms[6] whole attention call (plan upload and
 *   expansion when the call builds a plan, partial kernels, merge),
 *   ms[7] the tcgen05 partial kernel alone (part of ms[3]),
 *   ms[8] the mma.sync partial kernel alone when it ran beside the tcgen05
 *   kernel (events on the pool's side stream; ms[3] then spans both).
 * Entries with no recorded call are set to -1.                                */
#define DENDRITE_N_TIMINGS 9
int dendrite_set_profiling(dendrite_pool* pool, int32_t enable);
int dendrite_last_timings(dendrite_pool* pool, float* ms, int32_t n);

/* Attention plan statistics of the most recent dendrite_tree_attn_decode call. */
typedef struct dendrite_plan_stats {
    int32_t n_segments;     /* shared + private block ranges planned               */
    int32_t n_units;        /* (segment, kv head, row group) work units            */
    int32_t n_ctas;         /* CTAs of the partial kernel                           */
    int32_t n_partials;     /* partial triples written                              */
    int64_t tiles;          /* (block, kv head) tiles streamed by the partial kernel */
    int64_t unique_tiles;   /* distinct (block, kv head) tiles among them            */
    double  plan_us;        /* host time spent building or refreshing the plan      *
                             * (0 if it was reused as it was)                        */
    int32_t n_tc_units;     /* units among n_units run on the tcgen05 kernel        */
    int32_t n_tc_ctas;      /* CTAs of the tcgen05 kernel (not counted in n_ctas)   */
    int32_t refreshed;      /* 1: the cached plan only had its members' lengths     *
                             * refreshed (only appends since it was built, and no   *
                             * queried branch reached a new block); 2: only appends *
                             * since it was built and the branches that reached new *
                             * blocks each read their last segment (or, packed,     *
                             * their last extra tile) alone, so the cached segments *
                             * were lengthened and only the units, CTA partition    *
                             * and paths rebuilt; 0: built anew                     */
    int32_t reserved;
} dendrite_plan_stats;
int dendrite_last_plan_stats(dendrite_pool* pool, dendrite_plan_stats* out);

/* ------------------------------------------------------------ planner
 * The sharing planner as a pure host function (no pool, no GPU), used by the
 * attention call and exposed for tests.
 * Tree: node i has parent[i] (-1 for a root) and fork_len[i] (the parent's
 * length when i was forked; 0 for a root); len[i] is its current length.
 * For the queried nodes it returns the segments: maximal ranges of logical
 * blocks that a fixed set of queried branches reads from the same physical
 * blocks.  Only blocks that were full at every fork on the way are shared; a
 * partial block at a fork point counts as the child's own.
 * segs[k] = {rep, block_start, block_count, member_offset, n_members}:
 * members[member_offset .. +n_members) are indices into `queried`, and rep is
 * a member whose table holds the segment.  Segment order: by owner node in
 * first-visit order, then by block_start.
 * Returns DENDRITE_ELIMIT if seg_cap or member_cap is too small (the needed
 * sizes are still written to *n_segs / *n_members).
 */
typedef struct dendrite_segment {
    int32_t rep;
    int32_t block_start;
    int32_t block_count;
    int32_t member_offset;
    int32_t n_members;
} dendrite_segment;

int dendrite_plan_segments(int32_t n_nodes, const int32_t* parent, const int32_t* fork_len,
                           const int32_t* len, int32_t block_size,
                           const int32_t* queried, int32_t n_queried,
                           dendrite_segment* segs, int32_t seg_cap, int32_t* n_segs,
                           int32_t* members, int32_t member_cap, int32_t* n_members);

/*
 * The segments the bf16 attention call actually reads: those of
 * dendrite_plan_segments after folding (pool option fold_segments).  A
 * segment s is folded when the segments that follow it in its members' block
 * order (each holding a subset of s's members) are estimated to read s's
 * blocks again with their own rows faster than s's own row groups cost: every
 * following segment is then extended down to s's first block, and the members
 * whose blocks end in s keep a segment over s's range.  The result still has
 * each queried branch read each of its logical blocks exactly once, and every
 * position of a segment is the same physical block for all its members; it is
 * no longer maximal.
 *   rows_per_member  query rows per KV head of one member (q_len x GQA group), > 0.
 *   tc_min_rows      as the pool option (0 = default, -1 = no tcgen05 class).
 *   fold_pct         as the pool option fold_segments (0 = default, -1 = never).
 * Other arguments, results and errors as dendrite_plan_segments; segments keep
 * their order, a folded segment's place going to the segment of the members
 * that end in it, if any.
 */
int dendrite_plan_segments_folded(int32_t n_nodes, const int32_t* parent, const int32_t* fork_len,
                                  const int32_t* len, int32_t block_size,
                                  const int32_t* queried, int32_t n_queried,
                                  int32_t rows_per_member, int32_t tc_min_rows, int32_t fold_pct,
                                  dendrite_segment* segs, int32_t seg_cap, int32_t* n_segs,
                                  int32_t* members, int32_t member_cap, int32_t* n_members);

/*
 * The segments of the bf16 attention call with packing (pool option
 * pack_segments) before folding.  A segment whose following segments (those
 * that continue its members' block order) have no followers of their own can
 * take their tiles as extra tiles: extra tile {rep, block, member_mask} is
 * logical block `block` of node `rep`'s table, read only by the segment's
 * members whose bit is set (bit k: members[member_offset + k]); the followers
 * then disappear.  It packs when an estimate of one unit over all the tiles
 * (every tile multiplied with all the segment's rows) beats the separate
 * units; only segments of at most 32 members and one row group per kv head
 * (64 rows on the mma.sync kernel, 256 on the tcgen05 kernel) pack.  Folding
 * then runs as in dendrite_plan_segments_folded: a packed segment is never
 * folded, and a folded segment before it extends its shared range (the
 * blocks all its members read) downwards.  Every queried branch still reads
 * each of its logical blocks exactly once, through the shared range or
 * through the extra tiles of exactly one segment.
 *   pack_pct  0 = default (pack when the estimate drops), k > 0 = when it drops
 *             below k percent, -1 = never.
 *   extra_off [seg_cap + 1]: segment k's extra tiles are extras[extra_off[k] ..
 *             extra_off[k + 1]) (may be NULL).
 * Returns DENDRITE_ELIMIT if a capacity is too small (the needed counts are
 * still written).
 */
typedef struct dendrite_extra_tile {
    int32_t rep;
    int32_t block;
    uint32_t member_mask;
    int32_t reserved;
} dendrite_extra_tile;

int dendrite_plan_segments_packed(int32_t n_nodes, const int32_t* parent, const int32_t* fork_len,
                                  const int32_t* len, int32_t block_size,
                                  const int32_t* queried, int32_t n_queried,
                                  int32_t rows_per_member, int32_t tc_min_rows, int32_t fold_pct,
                                  int32_t pack_pct, dendrite_segment* segs, int32_t seg_cap, int32_t* n_segs,
                                  int32_t* members, int32_t member_cap, int32_t* n_members,
                                  int32_t* extra_off, dendrite_extra_tile* extras, int32_t extra_cap,
                                  int32_t* n_extras);

/* ------------------------------------------------- allocation-free variant
 * No counterpart on the pages: this entry point exists for callers that must
 * not have the library allocate device memory during decoding -- a serving
 * process whose device memory already belongs to its own caching allocator,
 * a latency-critical loop that cannot absorb the device synchronisation that
 * cudaMalloc / cudaFree may trigger, or a deployment that fixes each
 * library's memory at load time.
 *
 * Same arguments, layouts, results and errors as dendrite_tree_attn_decode,
 * but its scratch (the uploaded plan and the partial (max, sum, acc) rows)
 * lives in one file-scope device array of DENDRITE_NOALLOC_SCRATCH_BYTES
 * (16 MiB) that every GPU loading the library holds until the process exits.
 * The call itself calls no cudaMalloc, cudaFree, cudaMallocHost or other
 * allocating CUDA or torch routine; its host-side planning reuses per-thread
 * host buffers.  It does not use or grow the pool's attention workspace, and
 * it neither reads nor updates the pool's plan cache: every call builds its
 * plan anew, and dendrite_last_plan_stats keeps describing the last
 * dendrite_tree_attn_decode call.
 *   - The plan goes up with a cudaMemcpyAsync from one process-wide pageable
 *     host buffer, under a lock held while the plan is packed and copied, so
 *     threads that drive different pools do not mix their plans.  Such a
 *     copy first waits for the work queued earlier on `stream`: the call
 *     blocks the host until then.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) once for that device; make that first call before
 *     any stream capture.
 *   - The call cannot be captured into a CUDA graph (a captured copy from
 *     the pageable buffer would read it only when the graph runs): while
 *     `stream` is capturing it returns DENDRITE_EINVAL and enqueues nothing.
 *   - A call whose plan plus partial rows exceed the array returns
 *     DENDRITE_ELIMIT and launches nothing (roughly: more than ~30,000 partial
 *     rows of head_dim 128).
 *   - Pools of compressed blocks (DENDRITE_TURBO) return DENDRITE_EDTYPE.
 *   - Nothing in the array needs to start at zero: each call writes the plan
 *     and every partial row before reading them.
 *   - All calls share the one device array per device and it keeps the last
 *     call's contents: calls whose GPU work overlaps on one device (other
 *     streams, other pools on the same device, other threads) race on it and
 *     must be ordered by the caller.  Calls on different devices do not
 *     share device scratch.
 */
#define DENDRITE_NOALLOC_SCRATCH_BYTES (16u << 20)
int dendrite_tree_attn_decode_noalloc(dendrite_pool* pool, const void* Q, int32_t n_q_heads, int32_t q_len,
                                      const int32_t* branches, int32_t n_branches, void* out, void* stream);

/* Library version string. */
const char* dendrite_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DENDRITE_H */
