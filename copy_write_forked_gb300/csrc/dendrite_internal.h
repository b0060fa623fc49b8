// Internal declarations of the dendrite library (host + device).
// Not part of the public ABI; see include/dendrite.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <chrono>
#include <deque>
#include <string>
#include <utility>
#include <vector>

#include "dendrite.h"

namespace dendrite {

// ------------------------------------------------------------------ limits
constexpr int kBlockSize = 16;        // tokens per block (= attention tile height)
constexpr int kMaxUnitRowsBf16 = 64;  // rows per mma.sync attention unit (4 row tiles of 16)
constexpr int kMaxUnitRowsF32 = 16;
constexpr int kMaxUnitRowsTurbo = 64;  // rows per compressed-pool unit (4 warps x 16 rows)
constexpr int kMaxUnitRowsTc = 256;   // rows per tcgen05 attention unit (2 row tiles of 128)
constexpr int kTcMinRowsDefault = 64; // segments with more rows per kv head use the tcgen05 kernel
constexpr int32_t kFoldPctDefault = 100;  // fold a segment when that is estimated cheaper
constexpr int32_t kPackPctDefault = 100;  // pack a segment's followers into it when that is estimated cheaper
constexpr int kAppendMetaThreads = 1024;
constexpr int kFreeCollectThreads = 1024;

// Device-resident pool metadata words.
struct DevMeta {
    int32_t top;        // free stack size
    int32_t status;     // sticky error code (0 = ok)
    int32_t rel_lo;     // smallest block id released by the current free call
    int32_t rel_hi;     // largest block id released by the current free call
    int32_t rel_count;  // blocks released by the current free call
    int32_t rel_done;   // CTAs of the current free call that finished releasing
    int32_t pad[2];
};

// One sharing segment: blocks [blk_start, blk_start + n_blk) of the table row
// `table_row`, read by the queried branches listed in members[mem_off ..).
// Its units are unit_base + kv_head * ngroups + row_group.
struct AttnSeg {
    int32_t table_row;
    int32_t blk_start;
    int32_t n_blk;
    int32_t mem_off;
    int32_t n_mem;
    int32_t unit_base;
    int32_t ngroups;
    int32_t group_rows; // rows per row group (kMaxUnitRowsTc for tensor-core segments)
};

// A queried branch as a segment member: its index in the query list and length.
struct AttnMember {
    int32_t qi;
    int32_t len;
};

// One attention work unit: a (segment, kv head, row group).  Its rows are
// segment rows [row_lo, row_lo + n_rows); segment row sr belongs to member
// sr / (q_len * G), query token (sr % (q_len * G)) / G and head group g = sr % G.
// The segment's table row, block range and first member are repeated here so
// the partial kernels need no second lookup; a row's Q/out row and visibility
// limit follow from its member (unit_row).
struct AttnUnit {
    int32_t seg;
    int32_t kv_head;
    int32_t row_lo;
    int32_t n_rows;     // 1..max rows per unit
    int32_t rt;         // row tiles: of 16 rows (1, 2 or 4), of 128 rows in tc units (1 or 2)
    int32_t tile_off;   // index of the unit's first tile within its class's tile list
    int32_t cfirst;     // CTA (of its class's kernel) holding the unit's first tile
    int32_t nchunks;    // CTAs its tiles are split over (all non-empty)
    int32_t prow_base;  // first partial row; chunk k uses rows prow_base + k * n_rows ..
    int32_t table_row;  // branch handle whose table row holds the segment's block ids
    int32_t blk_start;  // first logical block of the segment
    int32_t n_blk;      // blocks (tiles) of the segment
    int32_t mem_off;    // the segment's first entry in the member list
    int32_t n_shared;   // tiles [0, n_shared) are blocks blk_start + i of table_row, read by all rows;
    int32_t x_off;      // tiles from n_shared on are the plan's extra tiles x_off + (i - n_shared)
    int32_t pad;
};
static_assert(sizeof(AttnUnit) == 64, "AttnUnit layout");

// An extra tile of a packed unit: logical block `blk` of branch handle
// `table_row`'s table, read by the unit's rows whose member (index within the
// segment's member list) has its bit set in `mask`.
struct AttnXTile {
    int32_t blk;
    uint32_t mask;
    int32_t table_row;
    int32_t pad;
};

// One query row of a unit (computed by unit_row).
struct AttnRow {
    int32_t q_row;   // row of Q/out viewed as [rows][head_dim]
    int32_t limit;   // visible positions: the row sees positions < limit
    int32_t member;  // index of the row's member within its segment's member list
};

// Device view of an uploaded attention plan.
struct AttnPlanDev {
    const AttnSeg* segs;
    const AttnMember* members;
    const AttnUnit* units;
    // Units [0, n_tc_units) run on the tcgen05 kernel, the rest on the
    // mma.sync (or fp32) kernel; each class has its own tile numbering and
    // its own CTA partition.
    const int32_t* cta_begin;      // [n_ctas + 1] strictly increasing tile boundaries
    const int32_t* cta_unit;       // [n_ctas] unit holding cta_begin[c]
    const int32_t* tc_cta_begin;   // [n_tc_ctas + 1], same for the tc class
    const int32_t* tc_cta_unit;    // [n_tc_ctas]
    const int32_t* path_off;       // [n_queried + 1] into path
    const AttnXTile* xtiles;       // extra tiles of packed units
    const int32_t* path;           // per path entry: (first unit of the segment, row groups per kv head,
                                   //  first segment row of the member, rows per row group)
    const int32_t* counts;         // plans expanded on the device: [0] CTAs of the mma.sync class,
                                   // [1] CTAs of the tc class, [2], [3] partial rows (low, high 32 bits);
                                   // CTAs at or past a class's count exit at once.  Null otherwise.
    int32_t n_units;
    int32_t n_ctas;
    int32_t n_tc_units;
    int32_t n_tc_ctas;
    int32_t n_queried;
    int32_t q_len;
    int32_t n_q_heads;
    int32_t group;                 // G = n_q_heads / n_kv
    float rcp_rows_per_member;     // 1 / (q_len G)
    float rcp_group;               // 1 / G
    int32_t packed;                // some unit reads extra tiles (the mma.sync kernel then needs its tile info)
};

// ------------------------------------------------------- host bookkeeping
struct Branch {
    int32_t live = 0;
    int32_t len = 0;
    int32_t node = -1;
};

struct Node {
    int32_t parent = -1;
    int32_t fork_len = 0;
    int32_t len = 0;
    int32_t handle = -1;
    int32_t refs = 0;   // (live handle ? 1 : 0) + number of child nodes
    int32_t first_child = -1, next_sib = -1, prev_sib = -1;   // the child nodes, as a list
};

// Pinned host -> device staging ring for per-call argument arrays.
class Staging {
public:
    int init(size_t cap);
    void destroy();
    // Reserve `bytes` (256-aligned); returns host and device pointers.
    int reserve(size_t bytes, char** h, char** d);
    // Copy the reserved region to the device on `stream`.
    int upload(cudaStream_t stream, char* h, size_t bytes);
    // Mark every region reserved since the last release as reusable once
    // the work queued on `stream` so far has completed.
    int release(cudaStream_t stream);

private:
    int grow(size_t need);
    int wait_overlap(size_t off, size_t n);
    char* h_ = nullptr;
    char* d_ = nullptr;
    size_t cap_ = 0;
    size_t head_ = 0;
    size_t pending_begin_ = 0, pending_end_ = 0;
    bool pending_ = false;
    bool pending_wrapped_ = false;
    struct Region { size_t off, end; cudaEvent_t ev; };
    std::deque<Region> inflight_;
    std::vector<cudaEvent_t> spare_;
};

enum TimingKind { T_FORK = 0, T_APPEND_META, T_APPEND_COPY, T_ATTN_PARTIAL, T_ATTN_MERGE, T_FREE,
                  T_ATTN_TOTAL, T_ATTN_TC, T_ATTN_MMA_SIDE, T_COUNT };

// 128-byte opaque CUtensorMap storage.
struct alignas(64) TensorMapBlob {
    unsigned char bytes[128];
};

// A split append (dendrite_append_begin) whose rows are not all written yet.
struct PendingAppend {
    bool active = false;
    std::vector<int32_t> branches;
    std::vector<int32_t> lens;        // lengths before the append
    int32_t n_new = 0;
    int64_t touched = 0;              // (branch, block) pairs the rows land in
    std::vector<uint8_t> layer_done;
    int32_t n_done = 0;
};

// A sharing segment found by the planner (planner.cpp).  A packed segment
// (pack_segments) also holds the tiles of the segments that followed it:
// extra tiles [x_off, x_off + n_x) of the planner's extra-tile list, each
// read by a subset of the members only.
struct Segment {
    int32_t rep_node;
    int32_t block_start;
    int32_t block_count;
    int32_t member_offset;
    int32_t n_members;
    int32_t owner;      // node whose blocks these are (a node's segments are consecutive, ascending)
    int32_t x_off = 0;
    int32_t n_x = 0;
};

// One extra tile of a packed segment: logical block `blk` of node `rep`'s
// table row, read by the segment's members whose bit is set in `mask`
// (bit k: the segment's k-th member).
struct ExtraTile {
    int32_t rep_node;
    int32_t blk;
    uint32_t mask;
};
constexpr int kMaxPackMembers = 32;
constexpr int kMaxTcExtraTiles = 64;   // extra tiles of a packed segment on the tcgen05 kernel

struct PlanCache {
    bool valid = false;
    bool device = false;             // units and CTA split expanded on the device
    int32_t n_segplan = 0;           // segments of the device expansion's list
    size_t upload_bytes = 0;         // host-written prefix of the packed plan
    size_t sec_off[16] = {};         // section offsets of the packed plan
    uint64_t version = 0, shape_version = 0;
    int32_t q_len = 0, n_q_heads = 0;
    std::vector<int32_t> branches;
    std::vector<int32_t> n_blocks;   // each queried branch's block count when the plan was built
    AttnPlanDev dev{};
    size_t n_partial_rows = 0;
    int buf = 0;                     // plan buffer pair holding the plan
    size_t bytes = 0;                // packed plan size
    size_t members_off = 0;          // byte offset of the member list in the packed plan
    int32_t n_members = 0;
    dendrite_plan_stats stats{};
    // The plan's segments (after folding) and, per queried branch, the index
    // of its last segment when that segment is read by that branch alone and
    // ends at its last block (-1 otherwise): appends that take such branches
    // into new blocks only lengthen those segments.
    std::vector<Segment> segs;
    std::vector<int32_t> seg_members;
    std::vector<ExtraTile> seg_xt;
    std::vector<int32_t> last_seg;
    // per queried branch: the extra tile (index in seg_xt) holding its last
    // block when that tile is read by it alone, else -1; appends that take
    // such branches into new blocks add extra tiles after it
    std::vector<int32_t> last_xt;
    int64_t unique_tiles = 0;
};

}  // namespace dendrite

struct dendrite_pool {
    // geometry
    int64_t num_blocks = 0;
    int32_t block_size = 0, n_kv = 0, head_dim = 0, dtype = 0, elt = 0;
    int32_t max_branches = 0, bpb = 0;
    int device = 0;
    int sm_count = 0;
    int attn_ctas_per_sm = 1;
    int32_t tc_min_rows = dendrite::kTcMinRowsDefault;   // < 0: tensor-core attention kernel off
    int32_t tc_sms = 0;   // SMs of the tcgen05 kernel beside the mma.sync one (0: estimated, -1: no split)
    int32_t fold_pct = dendrite::kFoldPctDefault;        // < 0: segments are never folded
    int32_t pack_pct = dendrite::kPackPctDefault;        // < 0: segments are never packed
    int32_t device_planning = 0;                         // 0 auto, 1 always, -1 never (bf16 plans)

    // device state
    void* d_k = nullptr;
    void* d_v = nullptr;
    int32_t* d_refcount = nullptr;
    int32_t* d_stack = nullptr;
    int32_t* d_table = nullptr;
    dendrite::DevMeta* d_meta = nullptr;
    int32_t* d_holders = nullptr;    // [num_blocks] holders of a shared tail within one append
    int32_t* d_last = nullptr;       // [num_blocks] last holder index within one append
    int32_t* d_released = nullptr;   // bitmap of the blocks a free released (word k: ids 32 k ..)
    int32_t* d_call_i32 = nullptr;   // [4 * max_branches] per-call scratch (offsets, cow sources)

    // layers: layer l's K pool starts at d_k + l * layer_bytes, its V pool at
    // d_v + l * layer_bytes_v (the same except for compressed pools)
    int32_t n_layers = 1;
    size_t layer_bytes = 0, layer_bytes_v = 0;
    // compressed pools (DENDRITE_TURBO): rotation signs [128] and QJL matrix
    // [128][128] on the device; rotated queries and projections of a call
    float* d_tq_signs = nullptr;
    float* d_tq_S = nullptr;
    float* d_tq_qs = nullptr;
    size_t tq_qs_rows = 0;

    // tensor maps of every layer's K and V pool for the bf16 attention
    // kernels (opaque 128-byte blobs)
    std::vector<dendrite::TensorMapBlob> tmap_k, tmap_v;
    bool tmaps_ok = false;
    bool tc_ready = false;           // tcgen05 attention kernel configured for this device

    // attention workspace (grow-only)
    char* d_plan[2] = {nullptr, nullptr};      // device copies, used alternately by plan builds
    size_t plan_cap = 0;                       // capacity of each
    char* h_plan[2] = {nullptr, nullptr};      // pinned, used alternately by plan builds
    size_t h_plan_cap = 0;                     // capacity of each
    cudaEvent_t plan_copied[2] = {nullptr, nullptr};
    // the mma.sync partial kernel runs beside the tcgen05 one on this stream
    // (forked from and joined back into the caller's stream)
    cudaStream_t side = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
    int plan_buf = 0;                          // buffer the next plan build packs into
    float* d_partial = nullptr;      // partial rows: [rows][head_dim] acc then [rows][2] (m, l)
    size_t partial_rows_cap = 0;
    dendrite::PlanCache plan;

    // host mirror
    std::vector<dendrite::Branch> br;
    std::vector<int32_t> free_handles;
    std::vector<dendrite::Node> nodes;
    std::vector<int32_t> free_nodes;
    uint64_t version = 1;          // any change to the tree or its lengths
    uint64_t shape_version = 1;    // any change but appends (forks, frees, truncations, new branches)
    int32_t poisoned = 0;

    dendrite::Staging staging;
    dendrite::PendingAppend pending;

    // profiling
    int profiling = 0;   // 0 off, 1 every kernel, 2 whole attention calls only
    cudaEvent_t ev[dendrite::T_COUNT][2] = {};
    bool ev_recorded[dendrite::T_COUNT] = {};
};

namespace dendrite {

// -------------------------------------------------------------- helpers
int cuda_err(cudaError_t e);     // maps a CUDA error to DENDRITE_ECUDA (and clears it)

// Programmatic dependent launch: the kernel may be scheduled while the
// previous kernel on the stream drains; it waits (griddepcontrol.wait) before
// touching anything that kernel produced.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
void prof_begin(dendrite_pool* p, TimingKind k, cudaStream_t s);
void prof_end(dendrite_pool* p, TimingKind k, cudaStream_t s);
int check_live(const dendrite_pool* p, int32_t h);

// Planner (planner.cpp): segments over the node forest (struct Segment above).
void plan_segments(int32_t n_nodes, const int32_t* parent, const int32_t* fork_len,
                   const int32_t* len, int32_t block_size, const int32_t* queried, int32_t n_queried,
                   std::vector<Segment>& segs, std::vector<int32_t>& members);
// How the attention plan will split a segment's rows, for the folding estimate:
// more than tc_rows rows per kv head (tc_rows < 0: never) go to the tcgen05
// kernel in groups of 256, the others to the small-row kernel in groups of
// small_rows.  fold_pct: fold when the estimate after folding is below this
// percentage of the estimate before.
struct FoldParams {
    int32_t rows_per_member;
    int32_t tc_rows;
    int32_t small_rows;
    int32_t fold_pct;
};
void fold_segments(const FoldParams& fp, int32_t n_nodes, const int32_t* parent, const int32_t* fork_len,
                   const int32_t* len, int32_t block_size, const int32_t* queried, int32_t n_queried,
                   std::vector<Segment>& segs, std::vector<int32_t>& members,
                   const std::vector<int32_t>* prev_in = nullptr);
// Packing: a segment whose following segments have none of their own takes
// their tiles as extra tiles (each read by that follower's members only) when
// the estimate of one unit per row group over all the tiles beats the
// separate units by pack_pct percent (< 0: never); the followers disappear.
// Runs before folding; only segments of at most kMaxPackMembers members and
// one row group per kv head pack.  prev_out (optional) receives each kept
// segment's predecessor in its members' block order, which folding can take
// as prev_in instead of finding it again.
void pack_segments(const FoldParams& fp, int32_t pack_pct, int32_t n_nodes, const int32_t* parent,
                   const int32_t* fork_len, int32_t block_size, std::vector<Segment>& segs,
                   std::vector<int32_t>& members, std::vector<ExtraTile>& xt,
                   std::vector<int32_t>* prev_out = nullptr);

// Attention (attn.cu)
int attn_setup(dendrite_pool* p);      // tensor maps, occupancy
void attn_teardown(dendrite_pool* p);

}  // namespace dendrite

#define DENDRITE_TRY(x)                   \
    do {                                  \
        int _rc = (x);                    \
        if (_rc != DENDRITE_OK) return _rc; \
    } while (0)

#define DENDRITE_CUDA(x)                                  \
    do {                                                  \
        cudaError_t _e = (x);                             \
        if (_e != cudaSuccess) return dendrite::cuda_err(_e); \
    } while (0)
