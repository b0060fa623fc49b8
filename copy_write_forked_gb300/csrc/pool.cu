// Block pool, fork, copy-on-write append and free.
//
// Method: Dendrite article (ainews.cool, "Dendrite: O(1) KV cache forking",
// section 技术深度解析) and dendrite demo.tape (section "The problem":
// copy-on-write block table).  A fork copies block-table entries and raises
// refcounts; it never copies KV.  An append copies a partially filled tail
// block only when it is still shared (refcount > 1).  Freed blocks go back to
// a free stack.
//
// Device state (all owned by the pool):
//   K, V pools   [num_blocks][n_kv][block_size][head_dim]
//   refcount     int32[num_blocks]
//   free stack   int32[num_blocks], size in DevMeta::top; pop = stack[--top]
//   tables       int32[max_branches][bpb], -1 = empty
//   DevMeta      top, sticky status, scratch words of the free call
//
// Determinism: block ids handed out by one append follow argument order
// (copy of the tail first, then new blocks in position order), and the blocks
// released by one free are pushed in descending id order, so tables, refcounts
// and the free stack are bit-for-bit reproducible.
#include <algorithm>
#include <climits>
#include <cstdio>
#include <cstring>
#include <unordered_set>

#include "dendrite_internal.h"
#include "turbo.h"

using namespace dendrite;

// =================================================================== kernels
namespace {

__device__ __forceinline__ void set_status(DevMeta* m, int32_t code) {
    atomicCAS(&m->status, 0, code);
}

// Programmatic dependent launch: every kernel here first waits for the
// previous kernel in the stream (pdl_wait), then lets the next one launch its
// prologue (it still waits for this whole grid before reading anything).
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Per-call argument arrays: small ones travel as kernel parameters (no copy
// on the stream), large ones are staged in device memory.  Kernel parameters
// may fill up to 32,764 bytes; the largest tier keeps the argument words at
// 16 KiB (a fork batch of 1,024 pairs, the tiled free of 1,024 branches),
// for kernels whose lanes read the same argument word (a lane reading its
// own word of kernel parameters is served one lane at a time).
constexpr int kParamCapLarge = 4096;
template <int CAP>
struct ParamArgs {
    int32_t v[CAP];
    __device__ __forceinline__ int32_t operator[](int64_t i) const { return v[i]; }
    const int32_t* dev_ptr() const { return nullptr; }
};
struct GlobalArgs {
    const int32_t* p;
    __device__ __forceinline__ int32_t operator[](int64_t i) const { return p[i]; }
    const int32_t* dev_ptr() const { return p; }
};

__global__ void k_init(int32_t* stack, int32_t* refcount, int32_t* holders, int32_t* last,
                       int32_t* released, int64_t n, int32_t* table, int64_t n_table, DevMeta* meta) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        stack[i] = (int32_t)(n - 1 - i);
        refcount[i] = 0;
        holders[i] = 0;
        last[i] = -1;
        released[i] = 0;
    }
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_table; i += stride) table[i] = -1;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        meta->top = (int32_t)n;
        meta->status = 0;
        meta->rel_lo = INT_MAX;
        meta->rel_hi = -1;
        meta->rel_count = 0;
        meta->rel_done = 0;
    }
}

// ---------------------------------------------------------------- fork
// One warp per (parent, child) pair: the child's table row becomes a copy of
// the parent's first nb entries.  The pair flagged with add > 0 also raises
// the refcount of each of those blocks by `add` (the parent's child count),
// so each parent's blocks see exactly one atomic add per fork call.
template <int CAP>
struct ForkParams {
    int32_t n_pairs;
    int32_t child[CAP];
    int32_t parent[CAP];
    int32_t nb[CAP];
    int32_t add[CAP];
};

__device__ __forceinline__ void fork_pair(int32_t* __restrict__ table, int32_t* __restrict__ refcount,
                                          int32_t bpb, int32_t child, int32_t parent, int32_t nb,
                                          int32_t add, int lane, int32_t n_blocks, DevMeta* meta,
                                          int32_t first = 0) {
    // the parent's row is not written by this launch (children are new handles),
    // so its entries are read through the read-only path, 8 per lane at once;
    // entries [first, nb)
    const int32_t* src = table + (int64_t)parent * bpb;
    int32_t* dst = table + (int64_t)child * bpb;
    constexpr int U = 8;
    for (int32_t base = first; base < nb; base += 32 * U) {
        int32_t v[U];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const int32_t k = base + i * 32 + lane;
            v[i] = k < nb ? __ldg(src + k) : -1;
        }
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const int32_t k = base + i * 32 + lane;
            if (k >= nb) continue;
            dst[k] = v[i];
            if ((uint32_t)v[i] >= (uint32_t)n_blocks) {
                set_status(meta, DENDRITE_ECORRUPT);
                continue;
            }
            if (add) atomicAdd(refcount + v[i], add);
        }
    }
}

// One warp per (pair, kForkChunk entries of its row): a fork of a long row
// takes as long as one of a short row.
constexpr int32_t kForkChunk = 256;
template <int CAP>
__global__ void k_fork_param(const __grid_constant__ ForkParams<CAP> a, int32_t* table,
                             int32_t* refcount, int32_t bpb, int32_t n_blocks, DevMeta* meta) {
    pdl_wait();
    if (meta->status) return;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (warp >= a.n_pairs) return;
    const int32_t first = (int32_t)blockIdx.y * kForkChunk;
    const int32_t nb = min(a.nb[warp], first + kForkChunk);
    if (first >= nb) return;
    fork_pair(table, refcount, bpb, a.child[warp], a.parent[warp], nb, a.add[warp], threadIdx.x & 31, n_blocks, meta,
              first);
}

// Same for batches too large for kernel parameters: the four arrays
// (child, parent, nb, add) are read from device memory.
// blockIdx.y: a chunk of kForkChunk entries, so a large batch of long rows
// keeps enough warps in flight (one warp per pair and chunk).
__global__ void k_fork_global(const int32_t* __restrict__ args, int32_t n_pairs, int32_t* table,
                              int32_t* refcount, int32_t bpb, int32_t n_blocks, DevMeta* meta) {
    pdl_wait();
    if (meta->status) return;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (warp >= n_pairs) return;
    const int32_t first = (int32_t)blockIdx.y * kForkChunk;
    const int32_t nb = min(args[2 * n_pairs + warp], first + kForkChunk);
    if (first >= nb) return;
    fork_pair(table, refcount, bpb, args[warp], args[n_pairs + warp], nb, args[3 * n_pairs + warp],
              threadIdx.x & 31, n_blocks, meta, first);
}

// ------------------------------------------------------------ block scan
template <int NT>
__device__ __forceinline__ int32_t block_exclusive_scan(int32_t v, int32_t* warp_sums, int32_t* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int32_t s = lane < NT / 32 ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < NT / 32) warp_sums[lane] = s;   // inclusive warp prefix
        if (lane == NT / 32 - 1) *total = s;
    }
    __syncthreads();
    const int32_t res = x - v + (wid ? warp_sums[wid - 1] : 0);
    __syncthreads();
    return res;
}

// ------------------------------------------------------- append, phase 1
// One CTA.  Decides, for every branch of the call in argument order, whether
// its partially filled tail must be copied, reserves its blocks from the free
// stack with one exclusive scan, checks capacity (all-or-nothing) and writes
// the table/refcount updates.
//
// Copy-on-write decision as if the branches were served one after the other:
// a branch copies iff the tail's refcount is above 1 at its turn.  Earlier
// holders of the same tail in this call all copy (each leaves one reference),
// so with r = refcount[tail] and k holders in the call, holder number j
// (0-based, argument order) copies iff r - j > 1.  Since r >= k, only the last
// holder can write in place, and only when r == k.
//
// The kernel is a chain of dependent memory round trips, so it keeps them
// few: with at most one branch per thread the tail id, the decision and the
// stack offset stay in registers, and the table rows are written by one warp
// per branch with its lanes over the new blocks (one stack read per lane
// rather than one per block in turn).
template <typename A>
__global__ void __launch_bounds__(kAppendMetaThreads)
k_append_meta(const __grid_constant__ A args, int32_t n, int32_t n_new, int32_t bs, int32_t bpb,
              int32_t n_blocks, int32_t* table, int32_t* refcount, const int32_t* stack, int32_t* holders,
              int32_t* last, int32_t* call, DevMeta* meta) {
    constexpr int NT = kAppendMetaThreads, NW = NT / 32;
    __shared__ int32_t warp_sums[NW];
    __shared__ int32_t chunk_total;
    __shared__ int32_t status0, top0, bad;
    __shared__ int32_t s_off[NT], s_src[NT];
    // args: branch[n], len[n]
    int32_t* offs = call;              // [n] first stack offset of each branch (n > NT only)
    int32_t* cow_src = call + n;       // [n] copied tail (-1 = none), read by the copy kernel
    const int32_t t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const bool one = n <= NT;          // branch t of thread t: per-branch values in registers
    pdl_wait();
    if (t == 0) {
        status0 = meta->status;
        top0 = meta->top;
        bad = 0;
    }
    // with one branch per thread, its tail id is loaded with the status word
    int32_t my_tail = -1;
    if (one && t < n && args[n + t] % bs) my_tail = table[(int64_t)args[t] * bpb + args[n + t] / bs];
    __syncthreads();
    if (status0) return;
    // holders of each shared tail within the call; a tail id that is not a
    // block id poisons the pool instead of being dereferenced
    for (int32_t i = t; i < n; i += NT) {
        const int32_t L = args[n + i];
        if (L % bs) {
            const int32_t tail = one ? my_tail : table[(int64_t)args[i] * bpb + L / bs];
            if ((uint32_t)tail >= (uint32_t)n_blocks) {
                bad = 1;
            } else {
                atomicAdd(holders + tail, 1);
                atomicMax(last + tail, i);
            }
        }
    }
    __syncthreads();
    if (bad) {
        if (t == 0) set_status(meta, DENDRITE_ECORRUPT);
        return;
    }
    // decisions and one exclusive scan of the blocks each branch takes
    int32_t carry = 0, my_off = 0, my_src = -1;
    for (int32_t base = 0; base < n; base += NT) {
        const int32_t i = base + t;
        int32_t demand = 0, src = -1;
        if (i < n) {
            const int32_t L = args[n + i];
            if (L % bs) {
                const int32_t tail = one ? my_tail : table[(int64_t)args[i] * bpb + L / bs];
                const bool cow = !(__ldcg(refcount + tail) == __ldcg(holders + tail) && __ldcg(last + tail) == i);
                src = cow ? tail : -1;
            }
            demand = (src >= 0) + (L + n_new + bs - 1) / bs - (L + bs - 1) / bs;
            cow_src[i] = src;
        }
        const int32_t ex = block_exclusive_scan<NT>(demand, warp_sums, &chunk_total);
        if (i < n) {
            if (one) {
                my_off = ex;
                my_src = src;
            } else {
                offs[i] = carry + ex;
            }
        }
        carry += chunk_total;
        __syncthreads();
    }
    const bool fits = carry <= top0;
    // small appends with one branch per thread (decode steps: one token, at
    // most a copied tail and one new block each): every thread writes its own
    // branch's entries, so the whole call is one round of stack reads instead
    // of one per branch of a warp
    int32_t my_demand = 0;
    if (one && t < n) {
        const int32_t L = args[n + t];
        my_demand = (my_src >= 0) + (L + n_new + bs - 1) / bs - (L + bs - 1) / bs;
    }
    const bool per_thread = one && !__syncthreads_or(my_demand > 4);
    if (fits && per_thread) {
        if (t < n) {
            const int32_t b = args[t], L = args[n + t];
            int32_t o = my_off;
            int32_t* row = table + (int64_t)b * bpb;
            if (my_src >= 0) {
                const int32_t blk = stack[top0 - 1 - o];
                atomicSub(refcount + my_src, 1);
                refcount[blk] = 1;
                row[L / bs] = blk;
                ++o;
            }
            const int32_t nb0 = (L + bs - 1) / bs, nb1 = (L + n_new + bs - 1) / bs;
            for (int32_t j = nb0; j < nb1; ++j) {
                const int32_t blk = stack[top0 - 1 - (o + j - nb0)];
                refcount[blk] = 1;
                row[j] = blk;
            }
        }
    } else if (fits) {
        for (int32_t base = 0; base < n; base += NT) {
            const int32_t i = base + t;
            if (i < n) {
                s_off[t] = one ? my_off : __ldcg(offs + i);
                s_src[t] = one ? my_src : __ldcg(cow_src + i);
            }
            __syncthreads();
            const int32_t cnt = min(NT, n - base);
            for (int32_t k = warp; k < cnt; k += NW) {
                const int32_t b = args[base + k], L = args[n + base + k];
                int32_t o = s_off[k];
                const int32_t src = s_src[k];
                int32_t* row = table + (int64_t)b * bpb;
                if (src >= 0) {
                    if (lane == 0) {
                        const int32_t blk = stack[top0 - 1 - o];
                        atomicSub(refcount + src, 1);
                        refcount[blk] = 1;
                        row[L / bs] = blk;
                    }
                    ++o;
                }
                const int32_t nb0 = (L + bs - 1) / bs, nb1 = (L + n_new + bs - 1) / bs;
                for (int32_t j = nb0 + lane; j < nb1; j += 32) {
                    const int32_t blk = stack[top0 - 1 - (o + j - nb0)];
                    refcount[blk] = 1;
                    row[j] = blk;
                }
            }
            __syncthreads();
        }
    }
    // reset the holder scratch for the next call (the original tail id: a
    // copied tail's is in cow_src, an in-place tail is still in the table)
    for (int32_t i = t; i < n; i += NT) {
        const int32_t L = args[n + i];
        if (L % bs) {
            int32_t tail = my_tail;
            if (!one) {
                const int32_t src = __ldcg(cow_src + i);
                tail = src >= 0 ? src : table[(int64_t)args[i] * bpb + L / bs];
            }
            holders[tail] = 0;
            last[tail] = -1;
        }
    }
    if (t == 0) {
        if (fits) meta->top = top0 - carry;
        else set_status(meta, DENDRITE_ENOMEM);
    }
}

// ------------------------------------------------------- append, phase 2
// One CTA at a time per (branch, touched block, kv head) tile: copies the
// valid slots of a copied-on-write tail (if any) and scatters the new rows
// into their slots with 16-byte vector moves.  tile_pre[i] is the exclusive prefix of
// touched blocks per branch (host computed; depends only on lengths).
// blockIdx.y selects the layer: the input rows of layer y start y * in_layer
// 16-byte words after Kin / Vin, its pool y * pool_layer words after Kp / Vp.
template <typename A>
__global__ void __launch_bounds__(128, 16) k_append_copy(const __grid_constant__ A args, int32_t n, int32_t n_new, int32_t bs, int32_t bpb, int32_t n_kv,
                              int32_t row_vec, int32_t n_blocks, const int32_t* __restrict__ table,
                              const int32_t* __restrict__ call, const uint4* __restrict__ Kin0,
                              const uint4* __restrict__ Vin0, uint4* __restrict__ Kp0, uint4* __restrict__ Vp0,
                              int64_t in_layer, int64_t pool_layer, const DevMeta* meta, int64_t n_tiles,
                              int32_t uniform) {
    pdl_wait();
    // one tile per CTA up to 64 CTAs per SM (the scheduler starts the next
    // tile's CTA as one finishes), beyond that the grid strides over the tiles
    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const uint4* __restrict__ Kin = Kin0 + blockIdx.y * in_layer;
    const uint4* __restrict__ Vin = Vin0 + blockIdx.y * in_layer;
    uint4* __restrict__ Kp = Kp0 + blockIdx.y * pool_layer;
    uint4* __restrict__ Vp = Vp0 + blockIdx.y * pool_layer;
    // args: branch[n], len[n], tile prefix[n]
    const int32_t* cow_src = call + n;
    const int32_t h = (int32_t)(tile % n_kv);
    const int32_t t = (int32_t)(tile / n_kv);   // touched-block index over the call
    // branch i with tile_pre[i] <= t < tile_pre[i+1]: a division when every
    // branch touches `uniform` blocks (decode steps: one each), else a search
    int32_t i, t0;
    if (uniform > 0) {
        i = t / uniform;
        t0 = i * uniform;
    } else {
        int32_t lo = 0, hi = n - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (args[2 * n + mid] <= t) lo = mid; else hi = mid - 1;
        }
        i = lo;
        t0 = args[2 * n + i];
    }
    const int32_t L = args[n + i];
    const int32_t lblk = L / bs + (t - t0);
    const int32_t s0 = lblk == L / bs ? L % bs : 0;
    const int32_t s1 = min(bs, L + n_new - lblk * bs);
    const int64_t tile_vec = (int64_t)bs * row_vec;
    const int32_t total = s1 * row_vec;   // slots [0, s1) of the destination tile
    // Slots s >= s0 take the new rows (token lblk*bs + s - L of branch i),
    // slots s < s0 of a copied-on-write tail its source's rows.  The first
    // batch of new rows is loaded together with the status word, the
    // destination block id and the copy-on-write source, none of which its
    // addresses depend on; each thread issues its loads before its stores so
    // the moves of a tile are in flight together.
    constexpr int U = 2;   // 2 x 128 threads cover a bf16 tile of head_dim 128 (256 slots)
    uint4 kv[U], vv[U];
    int32_t idx[U];
    auto gather = [&](int32_t e0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int32_t e = e0 + u * (int32_t)blockDim.x;
            idx[u] = e < total ? e : -1;
            if (e >= total) continue;
            const int32_t s = e / row_vec, v = e % row_vec;
            if (s >= s0) {
                const int64_t tok = (int64_t)lblk * bs + s - L;
                const int64_t src = (((int64_t)i * n_new + tok) * n_kv + h) * row_vec + v;
                kv[u] = __ldg(Kin + src);
                vv[u] = __ldg(Vin + src);
            }
        }
    };
    const int32_t status = meta->status;
    const int32_t dst = table[(int64_t)args[i] * bpb + lblk];
    const int32_t csrc = lblk == L / bs ? cow_src[i] : -1;
    gather(threadIdx.x);
    if (status) return;
    if ((uint32_t)dst >= (uint32_t)n_blocks || csrc >= n_blocks) {
        if (threadIdx.x == 0) atomicCAS(const_cast<int32_t*>(&meta->status), 0, DENDRITE_ECORRUPT);
        return;
    }
    uint4* kd = Kp + ((int64_t)dst * n_kv + h) * tile_vec;
    uint4* vd = Vp + ((int64_t)dst * n_kv + h) * tile_vec;
    const bool cow = csrc >= 0;
    const uint4* ks = cow ? Kp + ((int64_t)csrc * n_kv + h) * tile_vec : nullptr;
    const uint4* vs = cow ? Vp + ((int64_t)csrc * n_kv + h) * tile_vec : nullptr;
    for (int32_t e0 = threadIdx.x; e0 < total; e0 += U * blockDim.x) {
        if (e0 != (int32_t)threadIdx.x) gather(e0);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (idx[u] < 0 || idx[u] / row_vec >= s0) continue;
            if (!cow) {            // an in-place tail keeps its rows
                idx[u] = -1;
                continue;
            }
            kv[u] = ks[idx[u]];
            vv[u] = vs[idx[u]];
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (idx[u] < 0) continue;
            kd[idx[u]] = kv[u];
            vd[idx[u]] = vv[u];
        }
    }
    }
}

// ------------------------------------------------------- free / truncate
// The end of a free kernel.  free_fold: thread (rel, blk) released block blk
// if rel; one lane per warp folds the warp's released ids into the call's
// range (any number of times per thread).  free_finish: the last CTA to
// finish pushes the released blocks onto the free stack in descending id
// order (a block scan over [rel_lo, rel_hi] from the top down).
__device__ __forceinline__ void free_fold(bool rel, int32_t blk, DevMeta* meta) {
    const unsigned m = __ballot_sync(0xffffffffu, rel);
    if (m) {
        const int32_t wlo = __reduce_min_sync(0xffffffffu, rel ? blk : INT_MAX);
        const int32_t whi = __reduce_max_sync(0xffffffffu, rel ? blk : -1);
        if ((threadIdx.x & 31) == 0) {
            atomicMin(&meta->rel_lo, wlo);
            atomicMax(&meta->rel_hi, whi);
            atomicAdd(&meta->rel_count, __popc(m));
        }
    }
}

__device__ __forceinline__ void free_finish(int32_t* released, int32_t* stack, DevMeta* meta, int32_t n_blocks) {
    __shared__ int32_t warp_sums[kFreeCollectThreads / 32];
    __shared__ int32_t chunk_total;
    __shared__ int32_t st, is_last, lo, hi, top0, cnt;
    const int32_t n_ctas = (int32_t)(gridDim.x * gridDim.y);
    __syncthreads();
    if (threadIdx.x == 0) {
        // a single CTA is its own last one: the barrier above already ordered
        // its threads' updates.  Otherwise one acquire-release increment both
        // publishes this CTA's updates (ordered before it by the barrier) and,
        // in the last CTA, makes every other CTA's updates visible.
        if (n_ctas == 1) {
            is_last = 1;
        } else {
            int32_t prev;
            asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(prev) : "l"(&meta->rel_done) : "memory");
            is_last = prev == n_ctas - 1;
        }
        if (is_last) {
            volatile DevMeta* vm = meta;
            lo = vm->rel_lo;
            hi = vm->rel_hi;
            cnt = vm->rel_count;
            top0 = vm->top;
            st = vm->status;
        }
    }
    __syncthreads();
    if (!is_last) return;
    if (!st && cnt > 0) {
        // the released bits of [lo, hi] (word g holds ids 32 g .. 32 g + 31),
        // from the top word down: thread t of a pass takes one word, and a
        // block scan of the words' counts places its released ids, highest
        // first.  Bits outside [lo, hi] are zero.
        uint32_t* bits = reinterpret_cast<uint32_t*>(released);
        int32_t carry = 0;
        const int32_t g_hi = hi >> 5, g_lo = lo >> 5;
        for (int32_t g0 = g_hi; g0 >= g_lo; g0 -= (int32_t)blockDim.x) {
            const int32_t g = g0 - (int32_t)threadIdx.x;
            const uint32_t mask = g >= g_lo ? __ldcg(bits + g) : 0u;   // bit k: id 32 g + k
            const int32_t ex = block_exclusive_scan<kFreeCollectThreads>(__popc(mask), warp_sums, &chunk_total);
            int32_t o = top0 + carry + ex;
            for (uint32_t m = mask; m; m &= ~(1u << (31 - __clz(m)))) {   // highest id first
                const int32_t j = (g << 5) + (31 - __clz(m));
                stack[o++] = j;
            }
            if (mask) bits[g] = 0;
            carry += chunk_total;
            __syncthreads();
        }
        if (threadIdx.x == 0) meta->top = top0 + carry;
    }
    if (threadIdx.x == 0) {
        meta->rel_lo = INT_MAX;
        meta->rel_hi = -1;
        meta->rel_count = 0;
        meta->rel_done = 0;
    }
}

// One thread per released table entry (branch i releases its entries
// [start_i, start_i + count_i)) drops one reference and clears the entry; an
// entry whose refcount reaches zero marks its block released.  The last CTA
// to finish then pushes the released blocks onto the free stack in
// descending id order (a block scan over [rel_lo, rel_hi] from the top down).
template <typename A>
__global__ void __launch_bounds__(kFreeCollectThreads)
k_free(const __grid_constant__ A args, int32_t n, int32_t total, int32_t bpb, int32_t n_blocks, int32_t* table,
       int32_t* refcount, int32_t* released, int32_t* stack, DevMeta* meta) {
    pdl_wait();
    // args: branch[n], entry prefix[n], first released entry[n]
    const int32_t e = blockIdx.x * blockDim.x + threadIdx.x;
    int32_t* slot = nullptr;
    int32_t blk = -1;
    if (e < total) {
        int32_t l = 0, h = n - 1;
        while (l < h) {
            const int32_t mid = (l + h + 1) >> 1;
            if (args[n + mid] <= e) l = mid; else h = mid - 1;
        }
        slot = table + (int64_t)args[l] * bpb + args[2 * n + l] + (e - args[n + l]);
        blk = *slot;   // loaded together with the status word; nothing is written before it is checked
    }
    // one decision per CTA, from one status load (a status set by another
    // CTA meanwhile may be seen by some CTAs only)
    if (__syncthreads_or(threadIdx.x == 0 && *reinterpret_cast<volatile const int32_t*>(&meta->status) != 0))
        return;
    bool rel = false;
    if (slot) {
        *slot = -1;
        if ((uint32_t)blk >= (uint32_t)n_blocks) {
            set_status(meta, DENDRITE_ECORRUPT);
        } else {
            const int32_t old = atomicSub(refcount + blk, 1);
            if (old == 1) {
                atomicOr(reinterpret_cast<uint32_t*>(released) + (blk >> 5), 1u << (blk & 31));
                rel = true;
            } else if (old < 1) {
                set_status(meta, DENDRITE_ECORRUPT);
            }
        }
    }
    free_fold(rel, blk, meta);
    free_finish(released, stack, meta, n_blocks);
}

// Frees of many branches whose rows share blocks (siblings of one prompt): a
// CTA takes 32 branches x kFreeTileEntries of their entries.  Warp w reads and
// clears branch w's entries (coalesced, four per lane); transposed through
// shared memory, warp w then takes entries w, w + 32, ... of the 32
// branches, and lanes holding the same block drop their references with one
// atomic.  args as for k_free; blockIdx.y: entry chunk.
constexpr int kFreeTileEntries = 128;
template <typename A>
__global__ void __launch_bounds__(kFreeCollectThreads)
k_free_tiles(const __grid_constant__ A args, int32_t n, int32_t total, int32_t bpb, int32_t n_blocks,
             int32_t* table, int32_t* refcount, int32_t* released, int32_t* stack, DevMeta* meta) {
    static_assert(kFreeCollectThreads == 1024, "one warp per branch row of a 32-branch tile");
    constexpr int PER = kFreeTileEntries / 32;
    __shared__ int32_t tile[32][kFreeTileEntries + 1];
    pdl_wait();
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t i = blockIdx.x * 32 + w;
    const int32_t pos0 = blockIdx.y * kFreeTileEntries + lane;
    int32_t* row = nullptr;
    int32_t count = 0;
    if (i < n) {
        const int32_t c0 = args[n + i], c1 = i + 1 < n ? args[n + i + 1] : total;
        count = c1 - c0;
        row = table + (int64_t)args[i] * bpb + args[2 * n + i];
    }
    int32_t blk[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) blk[k] = (row && pos0 + 32 * k < count) ? row[pos0 + 32 * k] : -1;
    if (__syncthreads_or(threadIdx.x == 0 && *reinterpret_cast<volatile const int32_t*>(&meta->status) != 0))
        return;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        if (row && pos0 + 32 * k < count) {
            row[pos0 + 32 * k] = -1;
            if ((uint32_t)blk[k] >= (uint32_t)n_blocks) {
                set_status(meta, DENDRITE_ECORRUPT);
                blk[k] = -1;
            }
        }
        tile[w][lane + 32 * k] = blk[k];
    }
    __syncthreads();
    // all PER reference drops are issued before any result is looked at
    int32_t bb[PER], cc[PER], old[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        bb[k] = tile[lane][w + 32 * k];
        const unsigned grp = __match_any_sync(0xffffffffu, bb[k]);
        cc[k] = (bb[k] >= 0 && lane == __ffs(grp) - 1) ? __popc(grp) : 0;
        old[k] = cc[k] ? atomicSub(refcount + bb[k], cc[k]) : 0;
    }
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        bool rel = false;
        if (cc[k]) {
            if (old[k] == cc[k]) {
                atomicOr(reinterpret_cast<uint32_t*>(released) + (bb[k] >> 5), 1u << (bb[k] & 31));
                rel = true;
            } else if (old[k] < cc[k]) {
                set_status(meta, DENDRITE_ECORRUPT);
            }
        }
        free_fold(rel, bb[k], meta);
    }
    free_finish(released, stack, meta, n_blocks);
}

}  // namespace

// ============================================================ host helpers
namespace dendrite {

int cuda_err(cudaError_t e) {
    (void)e;
    cudaGetLastError();
    return DENDRITE_ECUDA;
}

// Level 2 records only whole attention calls: events between a call's
// kernels would end the overlap of each kernel's start with the previous
// one's tail (programmatic dependent launch) and time a slower call.
static bool prof_on(const dendrite_pool* p, TimingKind k) {
    return p->profiling == 1 || (p->profiling == 2 && k == T_ATTN_TOTAL);
}
void prof_begin(dendrite_pool* p, TimingKind k, cudaStream_t s) {
    if (prof_on(p, k)) cudaEventRecord(p->ev[k][0], s);
}
void prof_end(dendrite_pool* p, TimingKind k, cudaStream_t s) {
    if (prof_on(p, k)) {
        cudaEventRecord(p->ev[k][1], s);
        p->ev_recorded[k] = true;
    }
}

int check_live(const dendrite_pool* p, int32_t h) {
    if (h < 0 || h >= p->max_branches || !p->br[h].live) return DENDRITE_EBADHANDLE;
    return DENDRITE_OK;
}

// ----------------------------------------------------------------- staging
int Staging::init(size_t cap) {
    cap_ = cap;
    if (cudaMallocHost(&h_, cap) != cudaSuccess) return cuda_err(cudaErrorMemoryAllocation);
    if (cudaMalloc(&d_, cap) != cudaSuccess) return cuda_err(cudaErrorMemoryAllocation);
    return DENDRITE_OK;
}

void Staging::destroy() {
    for (auto& r : inflight_) cudaEventDestroy(r.ev);
    for (auto e : spare_) cudaEventDestroy(e);
    inflight_.clear();
    spare_.clear();
    if (h_) cudaFreeHost(h_);
    if (d_) cudaFree(d_);
    h_ = d_ = nullptr;
}

int Staging::wait_overlap(size_t off, size_t n) {
    while (!inflight_.empty()) {
        const Region& r = inflight_.front();
        const bool overlap = r.off < off + n && off < r.end;
        if (!overlap) {
            // regions are handed out in ring order; stop at the first one that
            // does not overlap unless it lies behind the new range
            bool later = false;
            for (const Region& q : inflight_)
                if (q.off < off + n && off < q.end) later = true;
            if (!later) break;
        }
        DENDRITE_CUDA(cudaEventSynchronize(r.ev));
        spare_.push_back(r.ev);
        inflight_.pop_front();
    }
    return DENDRITE_OK;
}

int Staging::grow(size_t need) {
    // wait for everything in flight, then reallocate
    for (auto& r : inflight_) {
        cudaEventSynchronize(r.ev);
        spare_.push_back(r.ev);
    }
    inflight_.clear();
    size_t cap = cap_;
    while (cap < need) cap *= 2;
    cudaFreeHost(h_);
    cudaFree(d_);
    h_ = d_ = nullptr;
    cap_ = 0;
    head_ = 0;
    pending_ = false;
    return init(cap);
}

int Staging::reserve(size_t bytes, char** h, char** d) {
    bytes = (bytes + 255) & ~size_t(255);
    if (bytes == 0) bytes = 256;
    if (bytes > cap_ / 2) {
        if (pending_) return DENDRITE_EINVAL;   // one oversized region per call only
        DENDRITE_TRY(grow(bytes * 2));
    }
    size_t off = head_;
    if (off + bytes > cap_) {
        off = 0;
        if (pending_) pending_wrapped_ = true;
    }
    DENDRITE_TRY(wait_overlap(off, bytes));
    if (!pending_) {
        pending_ = true;
        pending_wrapped_ = false;
        pending_begin_ = off;
    }
    pending_end_ = off + bytes;
    head_ = off + bytes;
    *h = h_ + off;
    *d = d_ + off;
    return DENDRITE_OK;
}

int Staging::upload(cudaStream_t stream, char* h, size_t bytes) {
    DENDRITE_CUDA(cudaMemcpyAsync(d_ + (h - h_), h, bytes, cudaMemcpyHostToDevice, stream));
    return DENDRITE_OK;
}

int Staging::release(cudaStream_t stream) {
    if (!pending_) return DENDRITE_OK;
    cudaEvent_t ev;
    if (!spare_.empty()) {
        ev = spare_.back();
        spare_.pop_back();
    } else {
        DENDRITE_CUDA(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    }
    DENDRITE_CUDA(cudaEventRecord(ev, stream));
    if (pending_wrapped_) {
        inflight_.push_back({pending_begin_, cap_, ev});
        cudaEvent_t ev2;
        DENDRITE_CUDA(cudaEventCreateWithFlags(&ev2, cudaEventDisableTiming));
        DENDRITE_CUDA(cudaEventRecord(ev2, stream));
        inflight_.push_back({0, pending_end_, ev2});
    } else {
        inflight_.push_back({pending_begin_, pending_end_, ev});
    }
    pending_ = false;
    return DENDRITE_OK;
}

}  // namespace dendrite

// ================================================================ host API
namespace {

// A node's child nodes form a doubly linked list (first_child, next_sib,
// prev_sib), so that a node left with one child can hand its place to it.
void link_child(dendrite_pool* p, int32_t parent, int32_t id) {
    Node& n = p->nodes[id];
    n.parent = parent;
    n.prev_sib = -1;
    n.next_sib = -1;
    if (parent < 0) return;
    Node& par = p->nodes[parent];
    n.next_sib = par.first_child;
    if (par.first_child >= 0) p->nodes[par.first_child].prev_sib = id;
    par.first_child = id;
}

void unlink_child(dendrite_pool* p, int32_t id) {
    Node& n = p->nodes[id];
    if (n.parent < 0) return;
    if (n.prev_sib >= 0) p->nodes[n.prev_sib].next_sib = n.next_sib;
    else p->nodes[n.parent].first_child = n.next_sib;
    if (n.next_sib >= 0) p->nodes[n.next_sib].prev_sib = n.prev_sib;
    n.prev_sib = n.next_sib = -1;
}

int32_t new_node(dendrite_pool* p, int32_t parent, int32_t fork_len, int32_t handle) {
    int32_t id;
    if (!p->free_nodes.empty()) {
        id = p->free_nodes.back();
        p->free_nodes.pop_back();
    } else {
        id = (int32_t)p->nodes.size();
        p->nodes.emplace_back();
    }
    Node& n = p->nodes[id];
    n = Node();
    n.fork_len = fork_len;
    n.len = fork_len;
    n.handle = handle;
    n.refs = 1;
    link_child(p, parent, id);
    if (parent >= 0) p->nodes[parent].refs++;
    return id;
}

// Drops one reference of node id: its handle or one of its child nodes.  A
// node with no references left is freed (and drops its reference on its
// parent).  A node left with no handle and one child node is spliced out:
// the child takes its place under its parent and its fork position, so the
// child's own range starts where the node's did.  That changes no branch's
// blocks and which branches share them (the node's own blocks were read by
// the child's subtree alone), and it keeps the chain from a branch to its
// root as short as the tree's real forks, however many times its leaves
// were forked and freed (a decode loop that forks every leaf at every step
// would otherwise add a node per branch per step).
void drop_node_ref(dendrite_pool* p, int32_t id) {
    while (id >= 0) {
        Node& n = p->nodes[id];
        if (--n.refs > 0) {
            if (n.refs == 1 && n.handle < 0 && n.first_child >= 0) {
                const int32_t c = n.first_child, up = n.parent, fl = n.fork_len;
                unlink_child(p, c);
                unlink_child(p, id);
                // (a child cut below the node's own start, by a truncation,
                // already starts earlier and keeps its position)
                p->nodes[c].fork_len = std::min(p->nodes[c].fork_len, fl);
                link_child(p, up, c);
                p->nodes[id] = Node();
                p->free_nodes.push_back(id);
            }
            return;
        }
        const int32_t up = n.parent;
        unlink_child(p, id);
        n = Node();
        p->free_nodes.push_back(id);
        id = up;
    }
}

int32_t alloc_handle(dendrite_pool* p) {
    const int32_t h = p->free_handles.back();
    p->free_handles.pop_back();
    return h;
}

int prelude(dendrite_pool* p) {
    if (!p) return DENDRITE_EINVAL;
    if (p->poisoned) return p->poisoned;
    DENDRITE_CUDA(cudaSetDevice(p->device));
    return DENDRITE_OK;
}

int check_unique_live(dendrite_pool* p, const int32_t* b, int32_t n) {
    for (int32_t i = 0; i < n; ++i) DENDRITE_TRY(check_live(p, b[i]));
    if (n > 1) {
        std::vector<int32_t> s(b, b + n);
        std::sort(s.begin(), s.end());
        if (std::adjacent_find(s.begin(), s.end()) != s.end()) return DENDRITE_EINVAL;
    }
    return DENDRITE_OK;
}

template <int CAP>
int launch_fork_param(dendrite_pool* p, const std::vector<int32_t>& child, const std::vector<int32_t>& par,
                      const std::vector<int32_t>& nb, const std::vector<int32_t>& add, cudaStream_t s) {
    ForkParams<CAP> a;
    a.n_pairs = (int32_t)child.size();
    for (size_t i = 0; i < child.size(); ++i) {
        a.child[i] = child[i];
        a.parent[i] = par[i];
        a.nb[i] = nb[i];
        a.add[i] = add[i];
    }
    const int threads = 128;
    const int blocks = (int)((child.size() * 32 + threads - 1) / threads);
    const int32_t max_nb = child.empty() ? 0 : *std::max_element(nb.begin(), nb.end());
    const unsigned chunks = (unsigned)std::max<int32_t>(1, (max_nb + kForkChunk - 1) / kForkChunk);
    DENDRITE_CUDA(launch_pdl(k_fork_param<CAP>, dim3(blocks, chunks), dim3(threads), 0, s, a, p->d_table,
                             p->d_refcount, p->bpb, (int32_t)p->num_blocks, p->d_meta));
    return DENDRITE_OK;
}

}  // namespace

namespace {

// Host checks of an append: live, distinct branches and table capacity.
// touched: the (branch, block) pairs the new rows land in.
int append_check(dendrite_pool* p, const int32_t* branches, int32_t n, int32_t n_new, int64_t* touched) {
    DENDRITE_TRY(check_unique_live(p, branches, n));
    const int32_t bs = p->block_size;
    int64_t t = 0;
    for (int32_t i = 0; i < n; ++i) {
        const int64_t L = p->br[branches[i]].len;
        if (L + n_new > INT32_MAX / 2) return DENDRITE_ELIMIT;
        if ((L + n_new + bs - 1) / bs > p->bpb) return DENDRITE_ELIMIT;
        t += (L + n_new - 1) / bs - L / bs + 1;
    }
    if (t * p->n_kv > INT32_MAX) return DENDRITE_ELIMIT;
    *touched = t;
    return DENDRITE_OK;
}

// Launches the metadata kernel (meta) and/or the copy kernel (copy) of an
// append whose branches had lengths lens[] before it.  The copy writes layers
// [layer0, layer0 + n_layers_in) from K/V (layer y's rows in_layer 16-byte
// words after layer y - 1's).
int append_launch(dendrite_pool* p, const int32_t* branches, const int32_t* lens, int32_t n, int32_t n_new,
                  int64_t touched, bool copy, const void* K, const void* V, int32_t layer0, int32_t n_layers_in,
                  int64_t in_layer, cudaStream_t s, bool meta = true) {
    const int32_t bs = p->block_size;
    // args: branch[n], len[n], tile prefix[n]
    constexpr int CAP = 768;
    const int32_t row_vec = p->head_dim * p->elt / 16;
    const int64_t n_tiles = touched * p->n_kv;
    const unsigned grid = (unsigned)std::min<int64_t>(n_tiles, (int64_t)p->sm_count * 64);
    const int64_t pool_layer = (int64_t)(p->layer_bytes / 16);
    // blocks each branch touches, when the same for all (else 0)
    int32_t uniform = -1;
    for (int32_t i = 0; i < n && uniform != 0; ++i) {
        const int32_t k = (lens[i] + n_new - 1) / bs - lens[i] / bs + 1;
        uniform = uniform < 0 ? k : (uniform == k ? k : 0);
    }
    uniform = std::max(uniform, 0);
    auto fill = [&](int32_t* a) {
        int32_t acc = 0;
        for (int32_t i = 0; i < n; ++i) {
            const int32_t L = lens[i];
            a[i] = branches[i];
            a[n + i] = L;
            a[2 * n + i] = acc;
            acc += (L + n_new - 1) / bs - L / bs + 1;
        }
    };
    auto launch = [&](auto args) -> int {
        if (meta) {
            prof_begin(p, T_APPEND_META, s);
            DENDRITE_CUDA(launch_pdl(k_append_meta<decltype(args)>, dim3(1), dim3(kAppendMetaThreads), 0, s, args,
                                     n, n_new, bs, p->bpb, (int32_t)p->num_blocks, p->d_table, p->d_refcount,
                                     p->d_stack, p->d_holders, p->d_last, p->d_call_i32, p->d_meta));
            prof_end(p, T_APPEND_META, s);
        }
        if (copy && p->dtype == DENDRITE_TURBO) {
            prof_begin(p, T_APPEND_COPY, s);
            TurboAppend t{};
            t.args = args.dev_ptr();
            t.n = n;
            t.n_new = n_new;
            t.bs = bs;
            t.bpb = p->bpb;
            t.n_kv = p->n_kv;
            t.n_blocks = (int32_t)p->num_blocks;
            t.table = p->d_table;
            t.call = p->d_call_i32;
            t.K = static_cast<const __nv_bfloat16*>(K);
            t.V = static_cast<const __nv_bfloat16*>(V);
            t.kp = static_cast<unsigned char*>(p->d_k) + (size_t)layer0 * p->layer_bytes;
            t.vp = static_cast<unsigned char*>(p->d_v) + (size_t)layer0 * p->layer_bytes_v;
            t.in_layer = in_layer * 8;   // 16-byte words -> bf16 elements
            t.kp_layer = (int64_t)p->layer_bytes;
            t.vp_layer = (int64_t)p->layer_bytes_v;
            t.signs = p->d_tq_signs;
            t.S = p->d_tq_S;
            t.meta = p->d_meta;
            t.n_tiles = n_tiles;
            t.n_layers_in = n_layers_in;
            t.sm_count = p->sm_count;
            DENDRITE_TRY(launch_append_turbo(t, s));
            prof_end(p, T_APPEND_COPY, s);
        } else if (copy) {
            prof_begin(p, T_APPEND_COPY, s);
            uint4* kp = reinterpret_cast<uint4*>(static_cast<char*>(p->d_k) + (size_t)layer0 * p->layer_bytes);
            uint4* vp = reinterpret_cast<uint4*>(static_cast<char*>(p->d_v) + (size_t)layer0 * p->layer_bytes);
            DENDRITE_CUDA(launch_pdl(k_append_copy<decltype(args)>, dim3(grid, (unsigned)n_layers_in), dim3(128), 0,
                                     s, args, n, n_new, bs, p->bpb, p->n_kv, row_vec, (int32_t)p->num_blocks,
                                     (const int32_t*)p->d_table, (const int32_t*)p->d_call_i32, (const uint4*)K,
                                     (const uint4*)V, kp, vp, in_layer, pool_layer, (const DevMeta*)p->d_meta, n_tiles,
                                     uniform));
            prof_end(p, T_APPEND_COPY, s);
        }
        return DENDRITE_OK;
    };
    // compressed pools encode from device-resident arguments
    // (k_append_meta reads the arguments of a different branch in every
    // lane: from kernel parameters such reads are serialised, so larger
    // calls keep them in device memory)
    if (3 * n <= CAP && !(copy && p->dtype == DENDRITE_TURBO)) {
        ParamArgs<CAP> a;
        fill(a.v);
        return launch(a);
    }
    char *h, *d;
    const size_t bytes = (size_t)n * 12;
    DENDRITE_TRY(p->staging.reserve(bytes, &h, &d));
    fill((int32_t*)h);
    DENDRITE_TRY(p->staging.upload(s, h, bytes));
    DENDRITE_TRY(launch(GlobalArgs{(const int32_t*)d}));
    return p->staging.release(s);
}

void append_commit_lengths(dendrite_pool* p, const int32_t* branches, int32_t n, int32_t n_new) {
    for (int32_t i = 0; i < n; ++i) {
        Branch& b = p->br[branches[i]];
        b.len += n_new;
        p->nodes[b.node].len = b.len;
    }
    p->version++;
}

}  // namespace

extern "C" {

const char* dendrite_version(void) { return "dendrite-gb300 0.1.0 (sm_103a)"; }

}  // extern "C"

namespace {

int pool_create(int64_t num_blocks, int32_t block_size, int32_t n_kv_heads, int32_t head_dim, int32_t dtype,
                const float* tq_signs, const float* tq_S, const dendrite_pool_opts* opts, dendrite_pool** out) {
    if (!out) return DENDRITE_EINVAL;
    *out = nullptr;
    if (num_blocks <= 0 || num_blocks >= INT32_MAX || n_kv_heads < 1 || n_kv_heads > 64) return DENDRITE_EINVAL;
    if (block_size != kBlockSize) return DENDRITE_EDTYPE;
    if (dtype == DENDRITE_TURBO) {
        if (head_dim != kTurboDim) return DENDRITE_EDTYPE;
        if (!tq_signs || !tq_S) return DENDRITE_EINVAL;
        for (int i = 0; i < kTurboDim; ++i)
            if (tq_signs[i] != 1.f && tq_signs[i] != -1.f) return DENDRITE_EINVAL;
    } else if (dtype == DENDRITE_BF16) {
        if (head_dim != 128) return DENDRITE_EDTYPE;
    } else if (dtype == DENDRITE_FP32) {
        if (head_dim <= 0 || head_dim > 256 || head_dim % 32) return DENDRITE_EDTYPE;
    } else {
        return DENDRITE_EDTYPE;
    }
    int32_t max_branches = 4096, bpb = 4096;
    if (opts) {
        for (int32_t r : opts->reserved)
            if (r) return DENDRITE_EINVAL;
        if (opts->max_branches) max_branches = opts->max_branches;
        if (opts->max_blocks_per_branch) bpb = opts->max_blocks_per_branch;
        if (opts->tc_min_rows < -1 || opts->fold_segments < -1) return DENDRITE_EINVAL;
        if (opts->device_planning < -1 || opts->device_planning > 1) return DENDRITE_EINVAL;
        if (opts->n_layers < 0 || opts->n_layers > 1024) return DENDRITE_EINVAL;
        if (opts->tc_sms < -1 || opts->pack_segments < -1) return DENDRITE_EINVAL;
    }
    if (max_branches < 1 || bpb < 1 || (int64_t)max_branches * bpb > (int64_t)1 << 34) return DENDRITE_EINVAL;

    dendrite_pool* p = new dendrite_pool();
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->n_kv = n_kv_heads;
    p->head_dim = head_dim;
    p->dtype = dtype;
    p->elt = dtype == DENDRITE_FP32 ? 4 : 2;   // compressed pools take bf16 rows
    p->max_branches = max_branches;
    p->bpb = bpb;
    if (opts && opts->tc_min_rows) p->tc_min_rows = opts->tc_min_rows;
    if (opts) p->tc_sms = opts->tc_sms;
    if (opts && opts->pack_segments) p->pack_pct = opts->pack_segments;
    if (opts && opts->n_layers) p->n_layers = opts->n_layers;
    if (opts && opts->fold_segments) p->fold_pct = opts->fold_segments;
    if (opts) p->device_planning = opts->device_planning;
    int rc = DENDRITE_OK;
    auto fail = [&](int code) {
        dendrite_pool_destroy(p);
        return code;
    };
    if (cudaGetDevice(&p->device) != cudaSuccess) return fail(cuda_err(cudaErrorNoDevice));
    cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, p->device);
    const size_t slots = (size_t)num_blocks * n_kv_heads * block_size;
    if (dtype == DENDRITE_TURBO) {
        p->layer_bytes = slots * kTurboKeyBytes;
        p->layer_bytes_v = slots * kTurboValueBytes;
    } else {
        p->layer_bytes = p->layer_bytes_v = slots * head_dim * p->elt;
    }
    const size_t k_bytes = p->layer_bytes * p->n_layers, v_bytes = p->layer_bytes_v * p->n_layers;
    if (cudaMalloc(&p->d_k, k_bytes) != cudaSuccess || cudaMalloc(&p->d_v, v_bytes) != cudaSuccess)
        return fail(cuda_err(cudaErrorMemoryAllocation));
    // Slots past a branch's length are read by the attention tiles and given
    // weight zero; they must hold finite values (0 x NaN is NaN; a zero record
    // decodes to a zero row).  Zero them once here; afterwards they only ever
    // hold appended rows.
    if (cudaMemset(p->d_k, 0, k_bytes) != cudaSuccess || cudaMemset(p->d_v, 0, v_bytes) != cudaSuccess)
        return fail(cuda_err(cudaErrorUnknown));
    if (dtype == DENDRITE_TURBO) {
        if (cudaMalloc(&p->d_tq_signs, kTurboDim * sizeof(float)) != cudaSuccess ||
            cudaMalloc(&p->d_tq_S, (size_t)kTurboQjlBits * kTurboDim * sizeof(float)) != cudaSuccess)
            return fail(cuda_err(cudaErrorMemoryAllocation));
        if (cudaMemcpy(p->d_tq_signs, tq_signs, kTurboDim * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess ||
            cudaMemcpy(p->d_tq_S, tq_S, (size_t)kTurboQjlBits * kTurboDim * sizeof(float),
                       cudaMemcpyHostToDevice) != cudaSuccess)
            return fail(cuda_err(cudaErrorUnknown));
        if ((rc = turbo_setup_tables()) != DENDRITE_OK) return fail(rc);
    }
    const size_t nb4 = (size_t)num_blocks * 4;
    if (cudaMalloc(&p->d_refcount, nb4) != cudaSuccess || cudaMalloc(&p->d_stack, nb4) != cudaSuccess ||
        cudaMalloc(&p->d_holders, nb4) != cudaSuccess || cudaMalloc(&p->d_last, nb4) != cudaSuccess ||
        cudaMalloc(&p->d_released, nb4) != cudaSuccess ||
        cudaMalloc(&p->d_table, (size_t)max_branches * bpb * 4) != cudaSuccess ||
        cudaMalloc(&p->d_call_i32, (size_t)max_branches * 4 * 4) != cudaSuccess ||
        cudaMalloc(&p->d_meta, sizeof(DevMeta)) != cudaSuccess)
        return fail(cuda_err(cudaErrorMemoryAllocation));
    if ((rc = p->staging.init(4u << 20)) != DENDRITE_OK) return fail(rc);
    for (int k = 0; k < T_COUNT; ++k)
        if (cudaEventCreate(&p->ev[k][0]) != cudaSuccess || cudaEventCreate(&p->ev[k][1]) != cudaSuccess)
            return fail(cuda_err(cudaErrorUnknown));
    // the side stream (the mma.sync partial kernel beside the tcgen05 one) at
    // the lowest priority: the tcgen05 kernel's CTAs take the SMs first and
    // the mma.sync CTAs fill what they leave
    int lo_prio = 0, hi_prio = 0;
    if (cudaEventCreateWithFlags(&p->plan_copied[0], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->plan_copied[1], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_join, cudaEventDisableTiming) != cudaSuccess ||
        cudaDeviceGetStreamPriorityRange(&lo_prio, &hi_prio) != cudaSuccess ||
        cudaStreamCreateWithPriority(&p->side, cudaStreamNonBlocking, lo_prio) != cudaSuccess)
        return fail(cuda_err(cudaErrorUnknown));
    k_init<<<std::max(1, std::min(4 * p->sm_count, (int)((num_blocks + 255) / 256))), 256>>>(
        p->d_stack, p->d_refcount, p->d_holders, p->d_last, p->d_released, num_blocks, p->d_table,
        (int64_t)max_branches * bpb, p->d_meta);
    if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
        return fail(cuda_err(cudaErrorUnknown));
    if ((rc = attn_setup(p)) != DENDRITE_OK) return fail(rc);
    p->br.assign(max_branches, Branch());
    p->free_handles.reserve(max_branches);
    for (int32_t h = max_branches - 1; h >= 0; --h) p->free_handles.push_back(h);
    *out = p;
    return DENDRITE_OK;
}

}  // namespace

extern "C" {

int dendrite_pool_create(int64_t num_blocks, int32_t block_size, int32_t n_kv_heads, int32_t head_dim,
                         int32_t dtype, const dendrite_pool_opts* opts, dendrite_pool** out) {
    if (dtype == DENDRITE_TURBO) return DENDRITE_EINVAL;   // needs its codec: dendrite_pool_create_turbo
    return pool_create(num_blocks, block_size, n_kv_heads, head_dim, dtype, nullptr, nullptr, opts, out);
}

int dendrite_pool_create_turbo(int64_t num_blocks, int32_t block_size, int32_t n_kv_heads, int32_t head_dim,
                               const float* rot_signs, const float* qjl_matrix, const dendrite_pool_opts* opts,
                               dendrite_pool** out) {
    return pool_create(num_blocks, block_size, n_kv_heads, head_dim, DENDRITE_TURBO, rot_signs, qjl_matrix, opts,
                       out);
}

int dendrite_pool_destroy(dendrite_pool* p) {
    if (!p) return DENDRITE_EINVAL;
    cudaSetDevice(p->device);
    cudaDeviceSynchronize();
    attn_teardown(p);
    p->staging.destroy();
    void* bufs[] = {p->d_k, p->d_v, p->d_refcount, p->d_stack, p->d_holders, p->d_last,
                    p->d_released, p->d_table, p->d_call_i32, p->d_meta, p->d_tq_signs, p->d_tq_S};
    for (void* b : bufs)
        if (b) cudaFree(b);
    for (int k = 0; k < T_COUNT; ++k)
        for (int j = 0; j < 2; ++j)
            if (p->ev[k][j]) cudaEventDestroy(p->ev[k][j]);
    for (cudaEvent_t e : p->plan_copied)
        if (e) cudaEventDestroy(e);
    if (p->ev_fork) cudaEventDestroy(p->ev_fork);
    if (p->ev_join) cudaEventDestroy(p->ev_join);
    if (p->side) cudaStreamDestroy(p->side);
    cudaGetLastError();
    delete p;
    return DENDRITE_OK;
}

int dendrite_branch_new(dendrite_pool* p, int32_t* out) {
    DENDRITE_TRY(prelude(p));
    if (!out) return DENDRITE_EINVAL;
    if (p->free_handles.empty()) return DENDRITE_ELIMIT;
    const int32_t h = alloc_handle(p);
    p->br[h].live = 1;
    p->br[h].len = 0;
    p->br[h].node = new_node(p, -1, 0, h);
    p->version++;
    p->shape_version++;   // the tree's shape changed, not only lengths
    *out = h;
    return DENDRITE_OK;
}

int dendrite_fork_batch(dendrite_pool* p, const int32_t* parents, const int32_t* n_children, int32_t n_parents,
                        int32_t* out_children, void* stream) {
    DENDRITE_TRY(prelude(p));
    if (n_parents < 0 || (n_parents > 0 && (!parents || !n_children || !out_children))) return DENDRITE_EINVAL;
    int64_t total = 0;
    for (int32_t i = 0; i < n_parents; ++i) {
        DENDRITE_TRY(check_live(p, parents[i]));
        if (n_children[i] <= 0) return DENDRITE_EINVAL;
        total += n_children[i];
    }
    if (total > (int64_t)p->free_handles.size()) return DENDRITE_ELIMIT;
    if (total == 0) return DENDRITE_OK;
    cudaStream_t s = (cudaStream_t)stream;
    std::vector<int32_t> child, par, nb, add;
    child.reserve(total);
    par.reserve(total);
    nb.reserve(total);
    add.reserve(total);
    int64_t k = 0;
    for (int32_t i = 0; i < n_parents; ++i) {
        const int32_t pa = parents[i];
        const int32_t L = p->br[pa].len;
        const int32_t nblk = (L + p->block_size - 1) / p->block_size;
        for (int32_t c = 0; c < n_children[i]; ++c) {
            const int32_t h = alloc_handle(p);
            p->br[h].live = 1;
            p->br[h].len = L;
            p->br[h].node = new_node(p, p->br[pa].node, L, h);
            out_children[k++] = h;
            child.push_back(h);
            par.push_back(pa);
            nb.push_back(nblk);
            add.push_back(c == 0 ? n_children[i] : 0);
        }
    }
    p->version++;
    p->shape_version++;   // the tree's shape changed, not only lengths
    prof_begin(p, T_FORK, s);
    int rc;
    const size_t n = child.size();
    if (n <= 4) rc = launch_fork_param<4>(p, child, par, nb, add, s);
    else if (n <= 32) rc = launch_fork_param<32>(p, child, par, nb, add, s);
    else if (n <= 256) rc = launch_fork_param<256>(p, child, par, nb, add, s);
    else if (n <= kParamCapLarge / 4) rc = launch_fork_param<kParamCapLarge / 4>(p, child, par, nb, add, s);
    else {
        char *h, *d;
        DENDRITE_TRY(p->staging.reserve(n * 16, &h, &d));
        int32_t* a = (int32_t*)h;
        std::memcpy(a, child.data(), n * 4);
        std::memcpy(a + n, par.data(), n * 4);
        std::memcpy(a + 2 * n, nb.data(), n * 4);
        std::memcpy(a + 3 * n, add.data(), n * 4);
        DENDRITE_TRY(p->staging.upload(s, h, n * 16));
        const int threads = 128;
        const int blocks = (int)((n * 32 + threads - 1) / threads);
        const int32_t max_nb = *std::max_element(nb.begin(), nb.end());
        const unsigned chunks = (unsigned)std::max<int32_t>(1, (max_nb + kForkChunk - 1) / kForkChunk);
        rc = launch_pdl(k_fork_global, dim3(blocks, chunks), dim3(threads), 0, s, (const int32_t*)d, (int32_t)n,
                        p->d_table, p->d_refcount, p->bpb, (int32_t)p->num_blocks, p->d_meta) == cudaSuccess
                 ? DENDRITE_OK : DENDRITE_ECUDA;
        DENDRITE_TRY(p->staging.release(s));
    }
    prof_end(p, T_FORK, s);
    return rc;
}

int dendrite_fork(dendrite_pool* p, int32_t parent, int32_t n_children, int32_t* out_children, void* stream) {
    return dendrite_fork_batch(p, &parent, &n_children, 1, out_children, stream);
}

int dendrite_append_kv(dendrite_pool* p, const int32_t* branches, int32_t n, int32_t n_new, const void* K,
                       const void* V, void* stream) {
    DENDRITE_TRY(prelude(p));
    if (p->pending.active) return DENDRITE_EINVAL;
    if (n < 0 || n_new < 0 || (n > 0 && !branches)) return DENDRITE_EINVAL;
    if (n == 0 || n_new == 0) return DENDRITE_OK;
    if (!K || !V) return DENDRITE_EINVAL;
    if (((uintptr_t)K | (uintptr_t)V) & 15) return DENDRITE_EINVAL;
    int64_t touched = 0;
    DENDRITE_TRY(append_check(p, branches, n, n_new, &touched));
    cudaStream_t s = (cudaStream_t)stream;
    std::vector<int32_t> lens(n);
    for (int32_t i = 0; i < n; ++i) lens[i] = p->br[branches[i]].len;
    const int64_t in_layer = (int64_t)n * n_new * p->n_kv * p->head_dim * p->elt / 16;
    DENDRITE_TRY(append_launch(p, branches, lens.data(), n, n_new, touched, true, K, V, 0, p->n_layers, in_layer, s));
    append_commit_lengths(p, branches, n, n_new);
    return DENDRITE_OK;
}

int dendrite_append_begin(dendrite_pool* p, const int32_t* branches, int32_t n, int32_t n_new, void* stream) {
    DENDRITE_TRY(prelude(p));
    if (p->pending.active) return DENDRITE_EINVAL;
    if (n < 0 || n_new < 0 || (n > 0 && !branches)) return DENDRITE_EINVAL;
    if (n == 0 || n_new == 0) return DENDRITE_OK;
    int64_t touched = 0;
    DENDRITE_TRY(append_check(p, branches, n, n_new, &touched));
    cudaStream_t s = (cudaStream_t)stream;
    PendingAppend& pa = p->pending;
    pa.branches.assign(branches, branches + n);
    pa.lens.resize(n);
    for (int32_t i = 0; i < n; ++i) pa.lens[i] = p->br[branches[i]].len;
    DENDRITE_TRY(append_launch(p, branches, pa.lens.data(), n, n_new, touched, false, nullptr, nullptr, 0, 0, 0, s));
    pa.n_new = n_new;
    pa.touched = touched;
    pa.layer_done.assign(p->n_layers, 0);
    pa.n_done = 0;
    pa.active = true;
    append_commit_lengths(p, branches, n, n_new);
    return DENDRITE_OK;
}

int dendrite_append_layer(dendrite_pool* p, int32_t layer, const void* K, const void* V, void* stream) {
    DENDRITE_TRY(prelude(p));
    PendingAppend& pa = p->pending;
    if (!pa.active || layer < 0 || layer >= p->n_layers || pa.layer_done[layer]) return DENDRITE_EINVAL;
    if (!K || !V || (((uintptr_t)K | (uintptr_t)V) & 15)) return DENDRITE_EINVAL;
    cudaStream_t s = (cudaStream_t)stream;
    const int32_t n = (int32_t)pa.branches.size();
    DENDRITE_TRY(append_launch(p, pa.branches.data(), pa.lens.data(), n, pa.n_new, pa.touched, true, K, V, layer, 1,
                               0, s, /*meta=*/false));
    pa.layer_done[layer] = 1;
    if (++pa.n_done == p->n_layers) pa.active = false;
    return DENDRITE_OK;
}

int dendrite_pool_layers(dendrite_pool* p, int32_t* n_layers) {
    if (!p || !n_layers) return DENDRITE_EINVAL;
    *n_layers = p->n_layers;
    return DENDRITE_OK;
}

}  // extern "C"

namespace {

// Releases table entries [start_i, end_i) of each branch on the device.
int release_entries(dendrite_pool* p, const int32_t* branches, const int32_t* start, const int32_t* end,
                    int32_t n, cudaStream_t s) {
    int64_t total = 0;
    int32_t max_count = 0;
    for (int32_t i = 0; i < n; ++i) {
        total += end[i] - start[i];
        max_count = std::max(max_count, end[i] - start[i]);
    }
    if (total > INT32_MAX / 2) return DENDRITE_ELIMIT;
    if (total == 0) return DENDRITE_OK;
    // many branches: 32-branch tiles (one atomic per block shared within a tile)
    const bool tiles = n >= 32 && (max_count + kFreeTileEntries - 1) / kFreeTileEntries <= 65535;
    auto fill = [&](int32_t* a) {
        int32_t acc = 0;
        for (int32_t i = 0; i < n; ++i) {
            a[i] = branches[i];
            a[n + i] = acc;
            a[2 * n + i] = start[i];
            acc += end[i] - start[i];
        }
    };
    const unsigned grid = (unsigned)((total + kFreeCollectThreads - 1) / kFreeCollectThreads);
    auto launch = [&](auto args) -> int {
        if (tiles) {
            DENDRITE_CUDA(launch_pdl(k_free_tiles<decltype(args)>,
                                     dim3((unsigned)((n + 31) / 32),
                                          (unsigned)((max_count + kFreeTileEntries - 1) / kFreeTileEntries)),
                                     dim3(kFreeCollectThreads), 0, s, args, n, (int32_t)total, p->bpb,
                                     (int32_t)p->num_blocks, p->d_table, p->d_refcount, p->d_released, p->d_stack,
                                     p->d_meta));
            return DENDRITE_OK;
        }
        DENDRITE_CUDA(launch_pdl(k_free<decltype(args)>, dim3(grid), dim3(kFreeCollectThreads), 0, s, args, n,
                                 (int32_t)total, p->bpb, (int32_t)p->num_blocks, p->d_table, p->d_refcount,
                                 p->d_released, p->d_stack, p->d_meta));
        return DENDRITE_OK;
    };
    constexpr int CAP = 1536;
    if (3 * n <= CAP) {
        ParamArgs<CAP> a;
        fill(a.v);
        return launch(a);
    }
    if (tiles && 3 * n <= kParamCapLarge) {   // the tiled kernel reads one branch's arguments per warp
        ParamArgs<kParamCapLarge> a;
        fill(a.v);
        return launch(a);
    }
    char *h, *d;
    const size_t bytes = (size_t)n * 12;
    DENDRITE_TRY(p->staging.reserve(bytes, &h, &d));
    fill((int32_t*)h);
    DENDRITE_TRY(p->staging.upload(s, h, bytes));
    DENDRITE_TRY(launch(GlobalArgs{(const int32_t*)d}));
    return p->staging.release(s);
}

}  // namespace

extern "C" {

int dendrite_free(dendrite_pool* p, const int32_t* branches, int32_t n, void* stream) {
    DENDRITE_TRY(prelude(p));
    if (p->pending.active) return DENDRITE_EINVAL;
    if (n < 0 || (n > 0 && !branches)) return DENDRITE_EINVAL;
    if (n == 0) return DENDRITE_OK;
    DENDRITE_TRY(check_unique_live(p, branches, n));
    cudaStream_t s = (cudaStream_t)stream;
    const int32_t bs = p->block_size;
    static thread_local std::vector<int32_t> start, end;
    start.assign(n, 0);
    end.resize(n);
    for (int32_t i = 0; i < n; ++i) end[i] = (p->br[branches[i]].len + bs - 1) / bs;
    prof_begin(p, T_FREE, s);
    DENDRITE_TRY(release_entries(p, branches, start.data(), end.data(), n, s));
    prof_end(p, T_FREE, s);
    for (int32_t i = 0; i < n; ++i) {
        Branch& b = p->br[branches[i]];
        const int32_t node = b.node;
        p->nodes[node].handle = -1;
        b = Branch();
        p->free_handles.push_back(branches[i]);
        drop_node_ref(p, node);
    }
    p->version++;
    p->shape_version++;   // the tree's shape changed, not only lengths
    return DENDRITE_OK;
}

int dendrite_truncate(dendrite_pool* p, const int32_t* branches, const int32_t* new_lens, int32_t n,
                      void* stream) {
    DENDRITE_TRY(prelude(p));
    if (p->pending.active) return DENDRITE_EINVAL;
    if (n < 0 || (n > 0 && (!branches || !new_lens))) return DENDRITE_EINVAL;
    if (n == 0) return DENDRITE_OK;
    DENDRITE_TRY(check_unique_live(p, branches, n));
    for (int32_t i = 0; i < n; ++i)
        if (new_lens[i] < 0 || new_lens[i] > p->br[branches[i]].len) return DENDRITE_EINVAL;
    cudaStream_t s = (cudaStream_t)stream;
    const int32_t bs = p->block_size;
    static thread_local std::vector<int32_t> start, end;
    start.resize(n);
    end.resize(n);
    for (int32_t i = 0; i < n; ++i) {
        start[i] = (new_lens[i] + bs - 1) / bs;
        end[i] = (p->br[branches[i]].len + bs - 1) / bs;
    }
    prof_begin(p, T_FREE, s);
    DENDRITE_TRY(release_entries(p, branches, start.data(), end.data(), n, s));
    prof_end(p, T_FREE, s);
    // the branch continues as a new node cut from its old one at new_len, so
    // children forked from the old node keep the blocks they share with it
    for (int32_t i = 0; i < n; ++i) {
        Branch& b = p->br[branches[i]];
        if (new_lens[i] == b.len) continue;
        const int32_t old = b.node;
        b.node = new_node(p, old, new_lens[i], branches[i]);
        b.len = new_lens[i];
        p->nodes[old].handle = -1;
        drop_node_ref(p, old);
    }
    p->version++;
    p->shape_version++;   // the tree's shape changed, not only lengths
    return DENDRITE_OK;
}

int dendrite_sync(dendrite_pool* p, void* stream) {
    if (!p) return DENDRITE_EINVAL;
    DENDRITE_CUDA(cudaSetDevice(p->device));
    DENDRITE_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
    int32_t st = 0;
    DENDRITE_CUDA(cudaMemcpy(&st, &p->d_meta->status, 4, cudaMemcpyDeviceToHost));
    if (st && !p->poisoned) p->poisoned = st;
    return p->poisoned;
}

int dendrite_branch_len(dendrite_pool* p, int32_t branch, int32_t* out_len) {
    if (!p || !out_len) return DENDRITE_EINVAL;
    DENDRITE_TRY(check_live(p, branch));
    *out_len = p->br[branch].len;
    return DENDRITE_OK;
}

int dendrite_read_table(dendrite_pool* p, int32_t branch, int32_t* out, int32_t cap, int32_t* n_out,
                        void* stream) {
    if (!p || !n_out) return DENDRITE_EINVAL;
    DENDRITE_TRY(check_live(p, branch));
    DENDRITE_CUDA(cudaSetDevice(p->device));
    const int32_t nb = (p->br[branch].len + p->block_size - 1) / p->block_size;
    *n_out = nb;
    if (nb > cap) return DENDRITE_ELIMIT;
    if (nb == 0) return DENDRITE_OK;
    if (!out) return DENDRITE_EINVAL;
    DENDRITE_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
    DENDRITE_CUDA(cudaMemcpy(out, p->d_table + (int64_t)branch * p->bpb, (size_t)nb * 4, cudaMemcpyDeviceToHost));
    return DENDRITE_OK;
}

int dendrite_read_refcounts(dendrite_pool* p, int32_t* out, void* stream) {
    if (!p || !out) return DENDRITE_EINVAL;
    DENDRITE_CUDA(cudaSetDevice(p->device));
    DENDRITE_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
    DENDRITE_CUDA(cudaMemcpy(out, p->d_refcount, (size_t)p->num_blocks * 4, cudaMemcpyDeviceToHost));
    return DENDRITE_OK;
}

int dendrite_read_free_stack(dendrite_pool* p, int32_t* out, int32_t* top_out, void* stream) {
    if (!p || !out || !top_out) return DENDRITE_EINVAL;
    DENDRITE_CUDA(cudaSetDevice(p->device));
    DENDRITE_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
    DevMeta m;
    DENDRITE_CUDA(cudaMemcpy(&m, p->d_meta, sizeof(m), cudaMemcpyDeviceToHost));
    *top_out = m.top;
    if (m.top < 0 || m.top > p->num_blocks) return DENDRITE_ECORRUPT;
    if (m.top) DENDRITE_CUDA(cudaMemcpy(out, p->d_stack, (size_t)m.top * 4, cudaMemcpyDeviceToHost));
    return DENDRITE_OK;
}

int dendrite_read_block_layer(dendrite_pool* p, int32_t layer, int32_t block, void* k_out, void* v_out,
                              void* stream) {
    if (!p || !k_out || !v_out || block < 0 || block >= p->num_blocks) return DENDRITE_EINVAL;
    if (layer < 0 || layer >= p->n_layers) return DENDRITE_EINVAL;
    DENDRITE_CUDA(cudaSetDevice(p->device));
    DENDRITE_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
    const size_t kb = p->layer_bytes / p->num_blocks, vb = p->layer_bytes_v / p->num_blocks;   // per block
    DENDRITE_CUDA(cudaMemcpy(k_out, (char*)p->d_k + (size_t)layer * p->layer_bytes + kb * block, kb,
                             cudaMemcpyDeviceToHost));
    DENDRITE_CUDA(cudaMemcpy(v_out, (char*)p->d_v + (size_t)layer * p->layer_bytes_v + vb * block, vb,
                             cudaMemcpyDeviceToHost));
    return DENDRITE_OK;
}

int dendrite_read_block(dendrite_pool* p, int32_t block, void* k_out, void* v_out, void* stream) {
    return dendrite_read_block_layer(p, 0, block, k_out, v_out, stream);
}

int dendrite_pool_info(dendrite_pool* p, int64_t* num_blocks, int32_t* block_size, int32_t* n_kv_heads,
                       int32_t* head_dim, int32_t* dtype) {
    if (!p) return DENDRITE_EINVAL;
    if (num_blocks) *num_blocks = p->num_blocks;
    if (block_size) *block_size = p->block_size;
    if (n_kv_heads) *n_kv_heads = p->n_kv;
    if (head_dim) *head_dim = p->head_dim;
    if (dtype) *dtype = p->dtype;
    return DENDRITE_OK;
}

int dendrite_set_profiling(dendrite_pool* p, int32_t enable) {
    if (!p) return DENDRITE_EINVAL;
    if (enable < 0 || enable > 2) return DENDRITE_EINVAL;
    p->profiling = enable;
    for (int k = 0; k < T_COUNT; ++k) p->ev_recorded[k] = false;
    return DENDRITE_OK;
}

int dendrite_last_timings(dendrite_pool* p, float* ms, int32_t n) {
    if (!p || !ms || n < 0) return DENDRITE_EINVAL;
    DENDRITE_CUDA(cudaSetDevice(p->device));
    for (int32_t k = 0; k < n; ++k) {
        ms[k] = -1.f;
        if (k < T_COUNT && p->ev_recorded[k]) {
            DENDRITE_CUDA(cudaEventSynchronize(p->ev[k][1]));
            float t = 0;
            DENDRITE_CUDA(cudaEventElapsedTime(&t, p->ev[k][0], p->ev[k][1]));
            ms[k] = t;
        }
    }
    return DENDRITE_OK;
}

}  // extern "C"
