// Tree-aware split-KV decode attention over the copy-on-write block pool.
//
// Method (Dendrite article, ainews.cool, section 技术深度解析): attention walks
// the cache tree and gathers keys and values from the shared ancestor path and
// from the branch's own leaf path; the shared prefix is stored once.  Here the
// tree is cut into segments (block ranges read by a fixed set of queried
// branches, see planner.cpp).  Every segment is streamed from HBM once for all
// of its query rows (branches x q_len x GQA group), producing partial
// (max, sum, acc) triples per row; a log-sum-exp merge combines the partials
// of each output row:
//     M = max_i m_i,  L = sum_i l_i 2^(m_i - M),  out = sum_i acc_i 2^(m_i - M) / L
// (scores are kept in base-2 units: s * log2(e) / sqrt(head_dim)).
//
// Work decomposition: a unit is (segment, kv head, group of <= 64 rows); its
// tiles are (block, kv head) pairs of 16 tokens x head_dim.  All tiles of all
// units form one list that is split evenly (by tiles x row tiles) over a
// persistent grid; a CTA that crosses a unit boundary writes one partial per
// unit it touched.
//
// bf16 kernel (head_dim 128): 4 consumer warps + 1 producer warp.  The
// producer streams K and V tiles with TMA (cp.async.bulk.tensor, 128-byte
// swizzle) into a 3-stage mbarrier ring; a stage holds up to 4 tiles of one
// unit.  Each consumer warp owns one 16-row query tile and one tile position
// within the stage: for units with 1, 2 or 4 row tiles a stage carries 4, 2 or
// 1 tiles.  S = Q K^T and O += P V run on tensor cores (mma.sync m16n8k16,
// bf16 in, fp32 accumulate) with an online softmax in registers.  Warps that
// worked on the same rows combine their states through shared memory at the
// end of a unit.
//
// Every mbarrier wait is bounded (about 2 s of %globaltimer): on expiry the
// kernel records DENDRITE_ETIMEOUT in the pool status, skips the rest of its
// work (keeping the same barrier sequence) and waits, again bounded, for its
// own copies still in flight before it exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <climits>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "attn_common.cuh"
#include "turbo.h"

using namespace dendrite;

namespace {

constexpr int NSTAGE = 3;
constexpr int SLOT_BYTES = 4 * HALF_BYTES;       // K (2 halves) + V (2 halves) of one tile
constexpr int STAGE_BYTES = 4 * SLOT_BYTES;
constexpr int NCONS = 4;
constexpr int THREADS = (NCONS + 1) * 32;
constexpr int ML_BYTES = NCONS * 16 * 2 * 4;
constexpr int INFO_BYTES = NSTAGE * 4 * 16;  // per stage and tile: logical block, 64-bit row mask
// plans with packed units also hold the tile info (INFO_BYTES more): kept
// out of the others, which stay within the smaller shared-memory carveout
constexpr size_t SMEM_BF16 = 1024 + (size_t)NSTAGE * STAGE_BYTES + 2 * NSTAGE * 8 + ML_BYTES;
constexpr size_t SMEM_BF16_PACKED = SMEM_BF16 + INFO_BYTES;


// ------------------------------------------------ log-sum-exp merge of one row
// One warp merges output row o (branch qi, query token j, query head h*G + g)
// of head_dim 128: the row's partials are the chunks of one unit per segment
// on the branch's path; lanes enumerate them (lane e takes path entry e, a
// warp scan turns chunk counts into partial indices), load every (m, l) at
// once, and reduce
//     M = max m_i,  L = sum l_i 2^(m_i - M),  out = sum acc_i 2^(m_i - M) / L
// with lane l owning columns 4 l .. 4 l + 3 (one 16-byte load per partial
// row), eight acc rows in flight.  Partial rows are read through L2 only.
// Nothing is stored when the pool's status word is set.
// Waits (once per thread) for the partial kernel before the first read of its
// partial rows or of the status word: the plan lookups before it (path, units,
// chunk enumeration) overlap the partial kernel's tail.  Every kernel that
// wrote the plan completed before the partial kernel passed its own wait,
// which comes before it lets the merge launch.
__device__ __forceinline__ void wait_partials(bool& waited) {
    if (!waited) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        waited = true;
    }
}

template <typename T>
__device__ __forceinline__ void merge_row_wide(const AttnArgs& a, int32_t o, int lane) {
    const AttnPlanDev& pl = a.plan;
    bool waited = false;
    const int G = pl.group;
    const int32_t qi = o / (pl.q_len * pl.n_q_heads);
    const int32_t rem = o - qi * pl.q_len * pl.n_q_heads;
    const int32_t j = rem / pl.n_q_heads, hq = rem - j * pl.n_q_heads;
    const int32_t h = hq / G, g = hq - h * G;
    const int32_t pbeg = pl.path_off[qi], pend = pl.path_off[qi + 1];
    float M = -INFINITY, L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int32_t e0 = pbeg; e0 < pend; e0 += 32) {
        // lane e: one path entry -> its unit's chunks for this row
        const int32_t e = e0 + lane;
        int32_t nch = 0, base = 0, stride = 0;
        if (e < pend) {
            // unit_base, ngroups, first segment row, rows per group
            const int4 pe = __ldg(reinterpret_cast<const int4*>(pl.path) + e);
            const int32_t sr = pe.z + j * G + g;
            const int32_t grp = sr / pe.w;
            const AttnUnit U = pl.units[pe.x + h * pe.y + grp];
            nch = U.nchunks;
            base = U.prow_base + (sr - grp * pe.w);
            stride = U.n_rows;
        }
        int32_t incl = nch;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        const int32_t total = __shfl_sync(0xffffffffu, incl, 31);
        const int32_t excl = incl - nch;
        for (int32_t p0 = 0; p0 < total; p0 += 32) {
            // lane p: partial p of this batch -> its partial row
            const int32_t pidx = p0 + lane;
            int32_t ent = 0;
            const int n_ent = min(32, pend - e0);   // lanes past it hold no chunks
            for (int k = 0; k < n_ent; ++k) ent += (__shfl_sync(0xffffffffu, incl, k) <= pidx) ? 1 : 0;
            ent = min(ent, 31);
            const int32_t eb = __shfl_sync(0xffffffffu, base, ent);
            const int32_t es = __shfl_sync(0xffffffffu, stride, ent);
            const int32_t ex = __shfl_sync(0xffffffffu, excl, ent);
            const bool valid = pidx < total;
            const int32_t prow = valid ? eb + (pidx - ex) * es : 0;
            const int nb = min(32, total - p0);
            wait_partials(waited);
            // the first eight acc rows go out with the (m, l) loads
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int32_t pr = __shfl_sync(0xffffffffu, prow, min(u, nb - 1));
                v[u] = u < nb ? __ldcg(reinterpret_cast<const float4*>(a.part_acc + (int64_t)pr * D) + lane)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float2 ml = valid ? __ldcg(a.part_ml + prow) : make_float2(-INFINITY, 0.f);
            // running max over this batch
            float mb = ml.x;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
            const float Mn = fmaxf(M, mb);
            const float Mu = Mn == -INFINITY ? 0.f : Mn;
            const float sc = exp2f(M - Mu);   // rescale of the running state
            const float w = ml.x == -INFINITY ? 0.f : exp2f(ml.x - Mu);
            float lw = w * ml.y;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, off);
            L = L * sc + lw;
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[k] *= sc;
            M = Mn;
            for (int q = 0; q < nb; q += 8) {
                float wq[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int src = min(q + u, nb - 1);
                    const float ww = __shfl_sync(0xffffffffu, w, src);
                    wq[u] = q + u < nb ? ww : 0.f;
                    if (q > 0) {
                        const int32_t pr = __shfl_sync(0xffffffffu, prow, src);
                        v[u] = q + u < nb
                                   ? __ldcg(reinterpret_cast<const float4*>(a.part_acc + (int64_t)pr * D) + lane)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    acc[0] = fmaf(v[u].x, wq[u], acc[0]);
                    acc[1] = fmaf(v[u].y, wq[u], acc[1]);
                    acc[2] = fmaf(v[u].z, wq[u], acc[2]);
                    acc[3] = fmaf(v[u].w, wq[u], acc[3]);
                }
            }
        }
    }
    wait_partials(waited);
    if (*reinterpret_cast<volatile const int32_t*>(&a.meta->status)) return;
    const float inv = 1.f / L;
    float y[4] = {acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv};
    if (a.tq_signs) {
        // compressed pools: the partials live in the rotated space; rotate
        // the merged row back, out = s * (H y) / sqrt(128)
        tq_fwht(y, lane);
        const float4 sg = __ldg(reinterpret_cast<const float4*>(a.tq_signs) + lane);
        const float c = 0.0883883476483184405501055452631f;
        y[0] = y[0] * c * sg.x;
        y[1] = y[1] * c * sg.y;
        y[2] = y[2] * c * sg.z;
        y[3] = y[3] * c * sg.w;
    }
    T* dst = static_cast<T*>(a.out) + (int64_t)o * D + 4 * lane;
    if constexpr (sizeof(T) == 2) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(y[0], y[1]);
        __nv_bfloat162 hi = __floats2bfloat162_rn(y[2], y[3]);
        *reinterpret_cast<uint2*>(dst) = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    } else {
        *reinterpret_cast<float4*>(dst) = make_float4(y[0], y[1], y[2], y[3]);
    }
}

// ------------------------------------------------ consumer side of one chunk
// The P = 4 / rt consumer warps of a row tile split head_dim: warp w owns row
// tile r = w / P and columns [(w % P) NCOL, (w % P + 1) NCOL), NCOL = 128 / P,
// and runs every tile of every stage.  Each of those warps computes the row
// tile's scores and softmax in full (identical bits in all of them), and its
// own slice of P V, so at the chunk's end every warp stores its slice of the
// partial rows directly: no exchange between warps, and fewer accumulator
// registers (128 / P columns per row).
struct ConsumerCtx {
    const AttnArgs* a;
    uint32_t base, bar_full, bar_empty;
    volatile int* abortp;
    const int4* info;   // [NSTAGE][4]: each tile's logical block and row mask, written by the producer
    int warp, lane, c;
};

template <int P, bool PACKED>
__device__ __forceinline__ void consume_chunk(const ConsumerCtx& x, const AttnUnit& U, int32_t t, int32_t cend,
                                              int32_t& stage) {
    constexpr int NCOL = D / P, NT = NCOL / 8;   // columns and 8-column n-tiles of this warp
    const AttnArgs& a = *x.a;
    const AttnPlanDev& pl = a.plan;
    const int warp = x.warp, lane = x.lane;
    const int r = warp / P, col0 = (warp % P) * NCOL;
    const float NEG_INF = -INFINITY;
    const __nv_bfloat16* Q = static_cast<const __nv_bfloat16*>(a.Q);
    // query fragments of rows r*16 + lane/4 (+8), and their visibility limits
    uint32_t qa[8][4];
    int32_t lim0 = 0, lim1 = 0;
    {
        const int row0 = r * 16 + (lane >> 2), row1 = row0 + 8;
        const bool v0 = row0 < U.n_rows, v1 = row1 < U.n_rows;
        const AttnRow R0 = v0 ? unit_row(pl, U, row0) : AttnRow{0, 0};
        const AttnRow R1 = v1 ? unit_row(pl, U, row1) : AttnRow{0, 0};
        lim0 = R0.limit;
        lim1 = R1.limit;
        const uint32_t* q0 = reinterpret_cast<const uint32_t*>(Q + (int64_t)R0.q_row * D);
        const uint32_t* q1 = reinterpret_cast<const uint32_t*>(Q + (int64_t)R1.q_row * D);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int w = ks * 8 + (lane & 3);   // 32-bit word index of column ks*16 + 2*(lane&3)
            qa[ks][0] = v0 ? q0[w] : 0u;
            qa[ks][1] = v1 ? q1[w] : 0u;
            qa[ks][2] = v0 ? q0[w + 4] : 0u;
            qa[ks][3] = v1 ? q1[w + 4] : 0u;
        }
    }
    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;

    for (int32_t st = t; st < cend; st += 4, ++stage) {
        const int slot = stage % NSTAGE;
        const uint32_t ph = (uint32_t)(stage / NSTAGE) & 1u;
        const int ntiles = min(4, cend - st);
        const bool last = st + 4 >= cend;
        bool ok = !*x.abortp;
        if (ok) {
            ok = mbar_wait(x.bar_full + 8 * slot, ph, x.abortp);
            if (!ok) {
                *x.abortp = 1;
                atomicCAS(&a.meta->status, 0, DENDRITE_ETIMEOUT);
            }
        }
        ok = __all_sync(0xffffffffu, ok) && !*x.abortp;
        for (int ti = 0; ok && ti < ntiles; ++ti) {
            const uint32_t kt = x.base + slot * STAGE_BYTES + ti * SLOT_BYTES;
            const uint32_t vt = kt + 2 * HALF_BYTES;
            // S = Q K^T (16 rows x 16 tokens)
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            {
                const int mi = lane >> 3;
                const int tok = (mi >> 1) * 8 + (lane & 7);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kt + swz(tok, ks * 16 + (mi & 1) * 8), b0, b1, b2, b3);
                    mma16816(sc[0], qa[ks], b0, b1);
                    mma16816(sc[1], qa[ks], b2, b3);
                }
            }
            // scale, mask by per-row visibility (the row's limit; in a
            // packed unit also the tile's rows), online softmax
            int32_t pos0, vl0 = lim0, vl1 = lim1;
            if (PACKED) {
                const int4 inf = x.info[slot * 4 + ti];
                pos0 = inf.x * BS + (lane & 3) * 2;
                const uint64_t rmask = (uint64_t)(uint32_t)inf.y | (uint64_t)(uint32_t)inf.z << 32;
                const int row0 = r * 16 + (lane >> 2);
                vl0 = (rmask >> row0) & 1u ? lim0 : INT_MIN;
                vl1 = (rmask >> (row0 + 8)) & 1u ? lim1 : INT_MIN;
            } else {
                pos0 = (U.blk_start + (st - U.tile_off) + ti) * BS + (lane & 3) * 2;
            }
            float mx0 = NEG_INF, mx1 = NEG_INF;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int32_t pos = pos0 + nt * 8 + e;
                    sc[nt][e] = pos < vl0 ? sc[nt][e] * a.scale_log2 : NEG_INF;
                    sc[nt][2 + e] = pos < vl1 ? sc[nt][2 + e] * a.scale_log2 : NEG_INF;
                    mx0 = fmaxf(mx0, sc[nt][e]);
                    mx1 = fmaxf(mx1, sc[nt][2 + e]);
                }
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
            const float u0s = n0 == NEG_INF ? 0.f : n0, u1s = n1 == NEG_INF ? 0.f : n1;
            const float al0 = exp2f(m0 - u0s), al1 = exp2f(m1 - u1s);
            m0 = n0;
            m1 = n1;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    sc[nt][e] = exp2f(sc[nt][e] - u0s);
                    sc[nt][2 + e] = exp2f(sc[nt][2 + e] - u1s);
                }
            }
            // P goes to the tensor cores in bf16; the row sums use the same
            // rounded weights so numerator and denominator stay consistent
            uint32_t pa[4];
            pa[0] = pack_bf16(sc[0][0], sc[0][1]);
            pa[1] = pack_bf16(sc[0][2], sc[0][3]);
            pa[2] = pack_bf16(sc[1][0], sc[1][1]);
            pa[3] = pack_bf16(sc[1][2], sc[1][3]);
            const float ps0 = bf16_pair_sum(pa[0]) + bf16_pair_sum(pa[2]);
            const float ps1 = bf16_pair_sum(pa[1]) + bf16_pair_sum(pa[3]);
            l0 = l0 * al0 + ps0;
            l1 = l1 * al1 + ps1;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                o[n][0] *= al0;
                o[n][1] *= al0;
                o[n][2] *= al1;
                o[n][3] *= al1;
            }
            // O[:, col0 : col0 + NCOL] += P V[:, col0 : col0 + NCOL]
            {
                const int mi = lane >> 3;
                const int tok = (mi & 1) * 8 + (lane & 7);
#pragma unroll
                for (int np = 0; np < NT / 2; ++np) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(vt + swz(tok, col0 + np * 16 + (mi >> 1) * 8), b0, b1, b2, b3);
                    mma16816(o[2 * np], pa, b0, b1);
                    mma16816(o[2 * np + 1], pa, b2, b3);
                }
            }
        }

        if (last) {
            // ---------------------------------------- end of this unit's chunk
            l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
            l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
            const int32_t prow0 = U.prow_base + (x.c - U.cfirst) * U.n_rows;
            if (ok) {
                const int row0 = r * 16 + (lane >> 2), row1 = row0 + 8;
                if (row0 < U.n_rows) {
                    float* dst = a.part_acc + (int64_t)(prow0 + row0) * D + col0 + (lane & 3) * 2;
#pragma unroll
                    for (int n = 0; n < NT; ++n) *reinterpret_cast<float2*>(dst + n * 8) = make_float2(o[n][0], o[n][1]);
                    if (col0 == 0 && (lane & 3) == 0) a.part_ml[prow0 + row0] = make_float2(m0, l0);
                }
                if (row1 < U.n_rows) {
                    float* dst = a.part_acc + (int64_t)(prow0 + row1) * D + col0 + (lane & 3) * 2;
#pragma unroll
                    for (int n = 0; n < NT; ++n) *reinterpret_cast<float2*>(dst + n * 8) = make_float2(o[n][2], o[n][3]);
                    if (col0 == 0 && (lane & 3) == 0) a.part_ml[prow0 + row1] = make_float2(m1, l1);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(x.bar_empty + 8 * slot);
    }
}

// ============================================================ bf16 kernel
// PACKED: the plan has packed units; the producer then writes every tile's
// logical block and row mask into shared memory and the consumers mask by
// them (plans without packed units run without that step or its memory).
template <bool PACKED>
__global__ void __launch_bounds__(THREADS, 2)
k_attn_partial_bf16(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const AttnArgs a) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ int abort_flag;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* sm = smem_raw + (base - raw);
    const uint32_t bar_full = base + NSTAGE * STAGE_BYTES;
    const uint32_t bar_empty = bar_full + NSTAGE * 8;
    float* ml = reinterpret_cast<float*>(sm + NSTAGE * STAGE_BYTES + 2 * NSTAGE * 8);
    int4* info = reinterpret_cast<int4*>(sm + NSTAGE * STAGE_BYTES + 2 * NSTAGE * 8 + ML_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, NCONS);
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");   // inputs of the previous kernel are ready
    pdl_trigger();
    // this CTA's share of the plan is loaded together with the status word
    const AttnPlanDev& pl = a.plan;
    const int c = blockIdx.x;
    if (pl.counts && c >= pl.counts[0]) return;   // past the split expanded on the device
    const int32_t t_begin = pl.cta_begin[c], t_end = pl.cta_begin[c + 1];
    const int32_t u0 = pl.cta_unit[c];
    if (threadIdx.x == 0) {
        abort_flag = a.meta->status != 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (abort_flag) return;
    volatile int* abortp = &abort_flag;

    if (warp == NCONS) {
        // ------------------------------------------------------ producer
        // Each stage is up to 4 consecutive tiles (blocks x one kv head) of
        // one unit; lane i reads tile i's block id (for a packed unit's extra
        // tile through its entry in the plan, which also gives the tile's
        // logical block and member mask), writes the tile's logical block
        // and the mask of the unit's rows that see it for the consumers, and
        // after the stage's arrival issues its four TMA boxes (K and V, two
        // 64-column halves each).
        uint32_t issued = 0, parity_bits = 0;
        int32_t stage = 0;
        int32_t t = t_begin, u = u0;
        while (t < t_end) {
            const AttnUnit U = pl.units[u];
            const int32_t uend = U.tile_off + U.n_blk;
            if (t >= uend) { ++u; continue; }
            const int32_t cend = min(t_end, uend);
            const int32_t* trow = a.table + (int64_t)U.table_row * a.bpb + U.blk_start - U.tile_off;
            // packed: the entry of this lane's extra tile in the next stage,
            // loaded one stage ahead (the block id load still depends on it)
            AttnXTile pre{0, 0u, 0, 0};
            auto prefetch = [&](int32_t tt) {
                const int32_t ti = tt - U.tile_off;
                if (PACKED && lane < 4 && tt < cend && ti >= U.n_shared) pre = pl.xtiles[U.x_off + ti - U.n_shared];
            };
            prefetch(t + lane);
            for (int32_t st = t; st < cend; st += 4, ++stage) {
                const int slot = stage % NSTAGE;
                const uint32_t ph = (uint32_t)(stage / NSTAGE) & 1u;
                const int ntiles = min(4, cend - st);
                bool ok = true;
                if (lane == 0 && !*abortp) {
                    ok = mbar_wait(bar_empty + 8 * slot, ph ^ 1u, abortp);
                    if (!ok) {
                        *abortp = 1;
                        atomicCAS(&a.meta->status, 0, DENDRITE_ETIMEOUT);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) && !*abortp;
                if (!ok) continue;
                int32_t blk = 0;
                if (!PACKED) {
                    if (lane == 0) mbar_expect_tx(bar_full + 8 * slot, (uint32_t)(ntiles * SLOT_BYTES));
                    __syncwarp();
                    if (lane < ntiles) blk = trow[st + lane];
                } else if (lane < ntiles) {
                    const int32_t ti = st + lane - U.tile_off;
                    int4 inf;
                    if (ti < U.n_shared) {
                        blk = trow[st + lane];
                        inf = make_int4(U.blk_start + ti, -1, -1, 0);
                    } else {
                        // packed units hold one row group: row k belongs to member k / (q_len G)
                        const AttnXTile e = pre;
                        blk = a.table[(int64_t)e.table_row * a.bpb + e.blk];
                        const int32_t RM = pl.q_len * pl.group;
                        const uint64_t one = RM >= 64 ? ~0ull : (1ull << RM) - 1ull;
                        uint64_t rm = 0;
                        for (uint32_t mm = e.mask; mm; mm &= mm - 1u) {
                            const int32_t m = __ffs(mm) - 1;
                            if (m * RM < 64) rm |= one << (m * RM);
                        }
                        inf = make_int4(e.blk, (int32_t)(uint32_t)rm, (int32_t)(uint32_t)(rm >> 32), 0);
                    }
                    info[slot * 4 + lane] = inf;
                }
                if (PACKED) {
                    __syncwarp();   // the tile info is written before the stage's arrival releases it
                    if (lane == 0) mbar_expect_tx(bar_full + 8 * slot, (uint32_t)(ntiles * SLOT_BYTES));
                    __syncwarp();
                }
                if (lane < ntiles) {
                    if ((uint32_t)blk >= (uint32_t)a.n_blocks) {   // broken table: poison, read zeros
                        atomicCAS(&a.meta->status, 0, DENDRITE_ECORRUPT);
                        blk = -1;
                    }
                    const int32_t row0 = (blk * a.n_kv + U.kv_head) * BS;
                    const uint32_t dst = base + slot * STAGE_BYTES + lane * SLOT_BYTES;
                    const uint32_t fb = bar_full + 8 * slot;
                    tma_load_3d(dst, &tmK, 0, 0, row0, fb);
                    tma_load_3d(dst + HALF_BYTES, &tmK, 0, 1, row0, fb);
                    tma_load_3d(dst + 2 * HALF_BYTES, &tmV, 0, 0, row0, fb);
                    tma_load_3d(dst + 3 * HALF_BYTES, &tmV, 0, 1, row0, fb);
                }
                issued |= 1u << slot;
                parity_bits = (parity_bits & ~(1u << slot)) | (ph << slot);
                prefetch(st + 4 + lane);
            }
            t = cend;
            ++u;
        }
        // after a timeout, wait (bounded) for this CTA's copies still in flight
        if (lane == 0 && *abortp) {
            for (int s = 0; s < NSTAGE; ++s) {
                if (!(issued >> s & 1u)) continue;
                const uint32_t fb = bar_full + 8 * s, ph = parity_bits >> s & 1u;
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(fb, ph) && globaltimer() - t0 < WAIT_LIMIT_NS) {
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    // Units of up to 16 rows (one row tile): warp w takes tiles w, w + 4, ...
    // of each stage and the four warps combine their states at the chunk's
    // end.  Units of 32 or 64 rows: consume_chunk (the warps of a row tile
    // split head_dim instead).  Splitting head_dim for 16-row units too made
    // every warp compute each tile's scores, which the beam step could not
    // afford (34.7 -> 40.8 us); for 32 rows it wins (spec-verify leaves).
    const float NEG_INF = -INFINITY;
    const __nv_bfloat16* Q = static_cast<const __nv_bfloat16*>(a.Q);
    int32_t stage = 0;
    int32_t t = t_begin, u = u0;
    const ConsumerCtx ctx{&a, base, bar_full, bar_empty, abortp, info, warp, lane, c};
    while (t < t_end) {
        const AttnUnit U = pl.units[u];
        const int32_t uend = U.tile_off + U.n_blk;
        if (t >= uend) { ++u; continue; }
        const int32_t cend = min(t_end, uend);
        if (U.rt != 1) {
            // 32 or 64 rows: the warps of a row tile split head_dim (no exchange)
            if (U.rt == 2) consume_chunk<2, PACKED>(ctx, U, t, cend, stage);
            else consume_chunk<1, PACKED>(ctx, U, t, cend, stage);
            t = cend;
            ++u;
            continue;
        }
        // up to 16 rows: the four warps split each stage's tiles and combine
        // their states at the chunk's end
        constexpr int P = 4;
        const int r = 0, pidx = warp;

        // query fragments of rows r*16 + lane/4 (+8), and their visibility limits
        uint32_t qa[8][4];
        int32_t lim0 = 0, lim1 = 0;
        {
            const int row0 = r * 16 + (lane >> 2), row1 = row0 + 8;
            const bool v0 = row0 < U.n_rows, v1 = row1 < U.n_rows;
            const AttnRow R0 = v0 ? unit_row(pl, U, row0) : AttnRow{0, 0};
            const AttnRow R1 = v1 ? unit_row(pl, U, row1) : AttnRow{0, 0};
            lim0 = R0.limit;
            lim1 = R1.limit;
            const uint32_t* q0 = reinterpret_cast<const uint32_t*>(Q + (int64_t)R0.q_row * D);
            const uint32_t* q1 = reinterpret_cast<const uint32_t*>(Q + (int64_t)R1.q_row * D);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int w = ks * 8 + (lane & 3);   // 32-bit word index of column ks*16 + 2*(lane&3)
                qa[ks][0] = v0 ? q0[w] : 0u;
                qa[ks][1] = v1 ? q1[w] : 0u;
                qa[ks][2] = v0 ? q0[w + 4] : 0u;
                qa[ks][3] = v1 ? q1[w + 4] : 0u;
            }
        }
        float o[16][4];
#pragma unroll
        for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;

        for (int32_t st = t; st < cend; st += 4, ++stage) {
            const int slot = stage % NSTAGE;
            const uint32_t ph = (uint32_t)(stage / NSTAGE) & 1u;
            const int ntiles = min(4, cend - st);
            const bool last = st + 4 >= cend;
            bool ok = !*abortp;
            if (ok) {
                ok = mbar_wait(bar_full + 8 * slot, ph, abortp);
                if (!ok) {
                    *abortp = 1;
                    atomicCAS(&a.meta->status, 0, DENDRITE_ETIMEOUT);
                }
            }
            ok = __all_sync(0xffffffffu, ok) && !*abortp;
            for (int ti = pidx; ok && ti < ntiles; ti += P) {
                const uint32_t kt = base + slot * STAGE_BYTES + ti * SLOT_BYTES;
                const uint32_t vt = kt + 2 * HALF_BYTES;
                // S = Q K^T (16 rows x 16 tokens)
                float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                {
                    const int mi = lane >> 3;
                    const int tok = (mi >> 1) * 8 + (lane & 7);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(kt + swz(tok, ks * 16 + (mi & 1) * 8), b0, b1, b2, b3);
                        mma16816(s[0], qa[ks], b0, b1);
                        mma16816(s[1], qa[ks], b2, b3);
                    }
                }
                // scale, mask by per-row visibility (the row's limit; in a
                // packed unit also the tile's rows), online softmax
                int32_t pos0, vl0 = lim0, vl1 = lim1;
                if (PACKED) {
                    const int4 inf = info[slot * 4 + ti];
                    pos0 = inf.x * BS + (lane & 3) * 2;
                    vl0 = ((uint32_t)inf.y >> (lane >> 2)) & 1u ? lim0 : INT_MIN;
                    vl1 = ((uint32_t)inf.y >> ((lane >> 2) + 8)) & 1u ? lim1 : INT_MIN;
                } else {
                    pos0 = (U.blk_start + (st - U.tile_off) + ti) * BS + (lane & 3) * 2;
                }
                float mx0 = NEG_INF, mx1 = NEG_INF;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int32_t pos = pos0 + nt * 8 + e;
                        s[nt][e] = pos < vl0 ? s[nt][e] * a.scale_log2 : NEG_INF;
                        s[nt][2 + e] = pos < vl1 ? s[nt][2 + e] * a.scale_log2 : NEG_INF;
                        mx0 = fmaxf(mx0, s[nt][e]);
                        mx1 = fmaxf(mx1, s[nt][2 + e]);
                    }
                }
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
                const float u0s = n0 == NEG_INF ? 0.f : n0, u1s = n1 == NEG_INF ? 0.f : n1;
                const float al0 = exp2f(m0 - u0s), al1 = exp2f(m1 - u1s);
                m0 = n0;
                m1 = n1;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        s[nt][e] = exp2f(s[nt][e] - u0s);
                        s[nt][2 + e] = exp2f(s[nt][2 + e] - u1s);
                    }
                }
                // P goes to the tensor cores in bf16; the row sums use the same
                // rounded weights so numerator and denominator stay consistent
                uint32_t pa[4];
                pa[0] = pack_bf16(s[0][0], s[0][1]);
                pa[1] = pack_bf16(s[0][2], s[0][3]);
                pa[2] = pack_bf16(s[1][0], s[1][1]);
                pa[3] = pack_bf16(s[1][2], s[1][3]);
                const float ps0 = bf16_pair_sum(pa[0]) + bf16_pair_sum(pa[2]);
                const float ps1 = bf16_pair_sum(pa[1]) + bf16_pair_sum(pa[3]);
                l0 = l0 * al0 + ps0;
                l1 = l1 * al1 + ps1;
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    o[n][0] *= al0;
                    o[n][1] *= al0;
                    o[n][2] *= al1;
                    o[n][3] *= al1;
                }
                // O += P V
                {
                    const int mi = lane >> 3;
                    const int tok = (mi & 1) * 8 + (lane & 7);
#pragma unroll
                    for (int np = 0; np < 8; ++np) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(vt + swz(tok, np * 16 + (mi >> 1) * 8), b0, b1, b2, b3);
                        mma16816(o[2 * np], pa, b0, b1);
                        mma16816(o[2 * np + 1], pa, b2, b3);
                    }
                }
            }

            if (last) {
                // ---------------------------------------- end of this unit's chunk
                l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
                l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
                l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
                l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
                const int32_t prow0 = U.prow_base + (c - U.cfirst) * U.n_rows;
                // combine the P warps of each row tile through this stage's buffer
                consumer_sync();   // every warp is done reading the stage's K/V
                float* ob = reinterpret_cast<float*>(sm + slot * STAGE_BYTES) + warp * 16 * D;
                {
                    const int ra = lane >> 2, rb = ra + 8;
#pragma unroll
                    for (int n = 0; n < 16; ++n) {
                        const int col = n * 8 + (lane & 3) * 2;
                        *reinterpret_cast<float2*>(ob + ra * D + (col ^ ((ra & 7) << 3))) =
                            make_float2(o[n][0], o[n][1]);
                        *reinterpret_cast<float2*>(ob + rb * D + (col ^ ((rb & 7) << 3))) =
                            make_float2(o[n][2], o[n][3]);
                    }
                    if ((lane & 3) == 0) {
                        ml[(warp * 16 + ra) * 2] = m0;
                        ml[(warp * 16 + ra) * 2 + 1] = l0;
                        ml[(warp * 16 + rb) * 2] = m1;
                        ml[(warp * 16 + rb) * 2 + 1] = l1;
                    }
                }
                consumer_sync();
                if (ok) {
                    const float* obase = reinterpret_cast<const float*>(sm + slot * STAGE_BYTES);
                    const int items = 16 * (D / 4);   // one row tile
                    for (int idx = threadIdx.x; idx < items; idx += NCONS * 32) {
                        const int rr = idx / (16 * (D / 4));
                        const int row = (idx / (D / 4)) % 16;
                        const int d = (idx % (D / 4)) * 4;
                        const int grow = rr * 16 + row;
                        if (grow >= U.n_rows) continue;
                        float M = NEG_INF;
                        for (int p2 = 0; p2 < P; ++p2) M = fmaxf(M, ml[((rr * P + p2) * 16 + row) * 2]);
                        const float Mu = M == NEG_INF ? 0.f : M;
                        float L = 0.f;
                        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                        for (int p2 = 0; p2 < P; ++p2) {
                            const int w2 = rr * P + p2;
                            const float wgt = exp2f(ml[(w2 * 16 + row) * 2] - Mu);
                            L += ml[(w2 * 16 + row) * 2 + 1] * wgt;
                            const float4 v = *reinterpret_cast<const float4*>(
                                obase + (w2 * 16 + row) * D + (d ^ ((row & 7) << 3)));
                            acc.x += v.x * wgt;
                            acc.y += v.y * wgt;
                            acc.z += v.z * wgt;
                            acc.w += v.w * wgt;
                        }
                        *reinterpret_cast<float4*>(a.part_acc + (int64_t)(prow0 + grow) * D + d) = acc;
                        if (d == 0) a.part_ml[prow0 + grow] = make_float2(M, L);
                    }
                }
                fence_async_smem();
                consumer_sync();   // buffer free again before it is handed back to TMA
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
        }
        t = cend;
        ++u;
    }
}

// ============================================================ fp32 kernel
// CUDA-core path for fp32 pools (FFMA only, no TF32).  One warp per query
// row (up to 4 rows per warp), one 16-token tile at a time in shared memory.
__global__ void __launch_bounds__(128) k_attn_partial_f32(const AttnArgs a) {
    extern __shared__ float fsm[];
    const int d = a.head_dim, nj = d / 32;
    float* Ks = fsm;
    float* Vs = fsm + BS * d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ int st0;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    pdl_trigger();
    if (threadIdx.x == 0) st0 = a.meta->status;
    __syncthreads();
    if (st0) return;
    const AttnPlanDev& pl = a.plan;
    const int c = blockIdx.x;
    int32_t t = pl.cta_begin[c];
    const int32_t t_end = pl.cta_begin[c + 1];
    int32_t u = pl.cta_unit[c];
    const float* Q = static_cast<const float*>(a.Q);
    while (t < t_end) {
        const AttnUnit U = pl.units[u];
        const int32_t uend = U.tile_off + U.n_blk;
        if (t >= uend) { ++u; continue; }
        const int32_t cend = min(t_end, uend);
        float q[4][8], acc[4][8], m[4], l[4];
        int32_t lim[4];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            const int row = warp + 4 * rr;
            const bool v = row < U.n_rows;
            const AttnRow R = v ? unit_row(pl, U, row) : AttnRow{0, 0};
            lim[rr] = R.limit;
            m[rr] = -INFINITY;
            l[rr] = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                q[rr][j] = (v && j < nj) ? Q[(int64_t)R.q_row * d + lane + 32 * j] : 0.f;
                acc[rr][j] = 0.f;
            }
        }
        for (int32_t tt = t; tt < cend; ++tt) {
            const int32_t lb = U.blk_start + (tt - U.tile_off);
            int32_t blk = a.table[(int64_t)U.table_row * a.bpb + lb];
            if ((uint32_t)blk >= (uint32_t)a.n_blocks) {
                if (threadIdx.x == 0) atomicCAS(&a.meta->status, 0, DENDRITE_ECORRUPT);
                blk = 0;   // read a valid block; the pool is poisoned anyway
            }
            const float* kg = a.pool_k + ((int64_t)blk * a.n_kv + U.kv_head) * BS * d;
            const float* vg = a.pool_v + ((int64_t)blk * a.n_kv + U.kv_head) * BS * d;
            __syncthreads();
            for (int e = threadIdx.x; e < BS * d; e += blockDim.x) {
                Ks[e] = kg[e];
                Vs[e] = vg[e];
            }
            __syncthreads();
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                if (warp + 4 * rr >= U.n_rows) continue;
                for (int tok = 0; tok < BS; ++tok) {
                    if (lb * BS + tok >= lim[rr]) break;
                    float dot = 0.f;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (j < nj) dot = fmaf(q[rr][j], Ks[tok * d + lane + 32 * j], dot);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
                    const float sc = dot * a.scale_log2;
                    const float mn = fmaxf(m[rr], sc);
                    const float al = exp2f(m[rr] - mn);
                    const float p = exp2f(sc - mn);
                    l[rr] = l[rr] * al + p;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (j < nj) acc[rr][j] = fmaf(p, Vs[tok * d + lane + 32 * j], acc[rr][j] * al);
                    m[rr] = mn;
                }
            }
        }
        const int32_t prow0 = U.prow_base + (c - U.cfirst) * U.n_rows;
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            const int row = warp + 4 * rr;
            if (row >= U.n_rows) continue;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < nj) a.part_acc[(int64_t)(prow0 + row) * d + lane + 32 * j] = acc[rr][j];
            if (lane == 0) a.part_ml[prow0 + row] = make_float2(m[rr], l[rr]);
        }
        t = cend;
        ++u;
    }
}

// ============================================================ LSE merge
// One warp per output row (branch qi, query token j, query head h*G + g).
// The row's partials are the chunks of one unit per segment on the branch's
// path; lanes enumerate them (lane e takes path entry e, a warp scan turns
// chunk counts into partial indices), load every (m, l) at once, and reduce
//     M = max m_i,  L = sum l_i 2^(m_i - M),  out = sum acc_i 2^(m_i - M) / L
// with the acc rows fetched four partials at a time.  Partial rows are read
// through L2 only (they were written by the previous kernel).
// WIDE (head_dim 128): lane l owns columns 4 l .. 4 l + 3, so a partial row is
// one 16-byte load per lane and eight partials are in flight per warp; the
// launch bound leaves it 128 registers (at 64 it spilled, and the beam step
// took 2 us longer).
template <typename T, bool WIDE>
__global__ void __launch_bounds__(256, WIDE ? 2 : 1) k_attn_merge(const AttnArgs a) {
    pdl_trigger();
    const AttnPlanDev& pl = a.plan;
    const int lane = threadIdx.x & 31;
    const int32_t o = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int32_t n_out = pl.n_queried * pl.q_len * pl.n_q_heads;
    if (o >= n_out) return;
    if constexpr (WIDE) {
        merge_row_wide<T>(a, o, lane);
        return;
    }
    bool waited = false;
    const int G = pl.group;
    const int32_t qi = o / (pl.q_len * pl.n_q_heads);
    const int32_t rem = o - qi * pl.q_len * pl.n_q_heads;
    const int32_t j = rem / pl.n_q_heads, hq = rem - j * pl.n_q_heads;
    const int32_t h = hq / G, g = hq - h * G;
    const int d = a.head_dim, nj = d / 32;
    const int32_t pbeg = pl.path_off[qi], pend = pl.path_off[qi + 1];
    float M = -INFINITY, L = 0.f, acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.f;
    for (int32_t e0 = pbeg; e0 < pend; e0 += 32) {
        // lane e: one path entry -> its unit's chunks for this row
        const int32_t e = e0 + lane;
        int32_t nch = 0, base = 0, stride = 0;
        if (e < pend) {
            // unit_base, ngroups, first segment row, rows per group
            const int4 pe = __ldg(reinterpret_cast<const int4*>(pl.path) + e);
            const int32_t sr = pe.z + j * G + g;
            const int32_t grp = sr / pe.w;
            const AttnUnit U = pl.units[pe.x + h * pe.y + grp];
            nch = U.nchunks;
            base = U.prow_base + (sr - grp * pe.w);
            stride = U.n_rows;
        }
        int32_t incl = nch;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        const int32_t total = __shfl_sync(0xffffffffu, incl, 31);
        const int32_t excl = incl - nch;
        for (int32_t p0 = 0; p0 < total; p0 += 32) {
            // lane p: partial p of this batch -> its partial row
            const int32_t pidx = p0 + lane;
            int32_t ent = 0;
            const int n_ent = min(32, pend - e0);   // lanes past it hold no chunks
            for (int k = 0; k < n_ent; ++k) ent += (__shfl_sync(0xffffffffu, incl, k) <= pidx) ? 1 : 0;
            ent = min(ent, 31);
            const int32_t eb = __shfl_sync(0xffffffffu, base, ent);
            const int32_t es = __shfl_sync(0xffffffffu, stride, ent);
            const int32_t ex = __shfl_sync(0xffffffffu, excl, ent);
            const bool valid = pidx < total;
            const int32_t prow = valid ? eb + (pidx - ex) * es : 0;
            const int nb = min(32, total - p0);
            wait_partials(waited);
            // the first eight acc rows go out with the (m, l) loads
            float4 v[8];
            if constexpr (WIDE) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int32_t pr = __shfl_sync(0xffffffffu, prow, min(u, nb - 1));
                    v[u] = u < nb ? __ldcg(reinterpret_cast<const float4*>(a.part_acc + (int64_t)pr * D) + lane)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            float2 ml = valid ? __ldcg(a.part_ml + prow) : make_float2(-INFINITY, 0.f);
            // running max over this batch
            float mb = ml.x;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
            const float Mn = fmaxf(M, mb);
            const float Mu = Mn == -INFINITY ? 0.f : Mn;
            const float sc = exp2f(M - Mu);   // rescale of the running state
            const float w = ml.x == -INFINITY ? 0.f : exp2f(ml.x - Mu);
            float lw = w * ml.y;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, off);
            L = L * sc + lw;
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] *= sc;
            M = Mn;
            if constexpr (WIDE) {
                for (int q = 0; q < nb; q += 8) {
                    float wq[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int src = min(q + u, nb - 1);
                        const float ww = __shfl_sync(0xffffffffu, w, src);
                        wq[u] = q + u < nb ? ww : 0.f;
                        if (q > 0) {
                            const int32_t pr = __shfl_sync(0xffffffffu, prow, src);
                            v[u] = q + u < nb
                                       ? __ldcg(reinterpret_cast<const float4*>(a.part_acc + (int64_t)pr * D) + lane)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        acc[0] = fmaf(v[u].x, wq[u], acc[0]);
                        acc[1] = fmaf(v[u].y, wq[u], acc[1]);
                        acc[2] = fmaf(v[u].z, wq[u], acc[2]);
                        acc[3] = fmaf(v[u].w, wq[u], acc[3]);
                    }
                }
            } else {
                for (int q = 0; q < nb; q += 4) {
                    float wq[4];
                    float v[4][8];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int src = min(q + u, nb - 1);
                        const int32_t pr = __shfl_sync(0xffffffffu, prow, src);
                        wq[u] = (q + u < nb) ? __shfl_sync(0xffffffffu, w, src) : 0.f;
                        const float* row = a.part_acc + (int64_t)pr * d;
#pragma unroll
                        for (int k = 0; k < 8; ++k) v[u][k] = k < nj ? __ldcg(row + lane + 32 * k) : 0.f;
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int k = 0; k < 8; ++k) acc[k] = fmaf(v[u][k], wq[u], acc[k]);
                }
            }
        }
    }
    wait_partials(waited);
    if (*reinterpret_cast<volatile const int32_t*>(&a.meta->status)) return;
    const float inv = 1.f / L;
    if constexpr (WIDE) {
        T* dst = static_cast<T*>(a.out) + (int64_t)o * D + 4 * lane;
        if constexpr (sizeof(T) == 2) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
            *reinterpret_cast<uint2*>(dst) =
                make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
        } else {
            *reinterpret_cast<float4*>(dst) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
        }
        return;
    }
    T* dst = static_cast<T*>(a.out) + (int64_t)o * d;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        if (k < nj) {
            if constexpr (sizeof(T) == 2) dst[lane + 32 * k] = __float2bfloat16_rn(acc[k] * inv);
            else dst[lane + 32 * k] = acc[k] * inv;
        }
}

// Grouped merge (head_dim 128): one warp per (branch qi, query token j, KV
// head h) and NG = min(G, 4) consecutive query heads g0 .. g0 + NG - 1 of its
// GQA group.  Those heads are NG consecutive rows of every unit the branch
// reads, so they share the unit lookups and the chunk enumeration: the
// partial of row g0 + i is always the one of row g0 plus i.  The plan keeps
// such a run of rows inside one row group when G <= 4 divides 16 or G is a
// multiple of 4 (row groups hold 16, 64 or 256 rows); other group sizes use
// the per-row kernel above.  Lane l owns columns 4 l .. 4 l + 3.  The kernel
// is a chain of dependent loads, so it runs three CTAs per SM (80 registers;
// with four heads one partial's loads in flight at a time, a 28-byte spill):
// stress merge 29 -> 24 us, MCTS call 271 -> 264 us against two CTAs per SM.
template <typename T, int NG>
__global__ void __launch_bounds__(256, 3) k_attn_merge_grouped(const AttnArgs a) {
    pdl_trigger();
    const AttnPlanDev& pl = a.plan;
    const int lane = threadIdx.x & 31;
    const int G = pl.group, gchunks = G / NG, n_kv = pl.n_q_heads / G;
    const int32_t w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int32_t n_w = pl.n_queried * pl.q_len * n_kv * gchunks;
    if (w >= n_w) return;
    int32_t x = w;
    const int gc = x % gchunks;
    x /= gchunks;
    const int h = x % n_kv;
    x /= n_kv;
    const int j = x % pl.q_len;
    const int32_t qi = x / pl.q_len;
    const int g0 = gc * NG;
    bool waited = false;
    const int32_t pbeg = pl.path_off[qi], pend = pl.path_off[qi + 1];
    float M[NG], L[NG];
    float4 acc[NG];
#pragma unroll
    for (int i = 0; i < NG; ++i) {
        M[i] = -INFINITY;
        L[i] = 0.f;
        acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int32_t e0 = pbeg; e0 < pend; e0 += 32) {
        // lane e: one path entry -> its unit's chunks for row g0
        const int32_t e = e0 + lane;
        int32_t nch = 0, base = 0, stride = 0;
        if (e < pend) {
            const int4 pe = __ldg(reinterpret_cast<const int4*>(pl.path) + e);
            const int32_t sr = pe.z + j * G + g0;
            const int32_t grp = sr / pe.w;
            const AttnUnit U = pl.units[pe.x + h * pe.y + grp];
            nch = U.nchunks;
            base = U.prow_base + (sr - grp * pe.w);
            stride = U.n_rows;
        }
        int32_t incl = nch;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        const int32_t total = __shfl_sync(0xffffffffu, incl, 31);
        const int32_t excl = incl - nch;
        const int n_ent = min(32, pend - e0);   // lanes past it hold no chunks
        for (int32_t p0 = 0; p0 < total; p0 += 32) {
            // lane p: partial p of this batch -> its partial row for g0
            const int32_t pidx = p0 + lane;
            int32_t ent = 0;
            for (int k = 0; k < n_ent; ++k) ent += (__shfl_sync(0xffffffffu, incl, k) <= pidx) ? 1 : 0;
            ent = min(ent, 31);
            const int32_t eb = __shfl_sync(0xffffffffu, base, ent);
            const int32_t es = __shfl_sync(0xffffffffu, stride, ent);
            const int32_t ex = __shfl_sync(0xffffffffu, excl, ent);
            const bool valid = pidx < total;
            const int32_t prow = valid ? eb + (pidx - ex) * es : 0;
            const int nb = min(32, total - p0);
            wait_partials(waited);
            float2 ml[NG];
#pragma unroll
            for (int i = 0; i < NG; ++i) ml[i] = valid ? __ldcg(a.part_ml + prow + i) : make_float2(-INFINITY, 0.f);
            float wt[NG];
#pragma unroll
            for (int i = 0; i < NG; ++i) {
                float mb = ml[i].x;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
                const float Mn = fmaxf(M[i], mb);
                const float Mu = Mn == -INFINITY ? 0.f : Mn;
                const float sc = exp2f(M[i] - Mu);   // rescale of the running state
                wt[i] = ml[i].x == -INFINITY ? 0.f : exp2f(ml[i].x - Mu);
                float lw = wt[i] * ml[i].y;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, off);
                L[i] = L[i] * sc + lw;
                acc[i].x *= sc;
                acc[i].y *= sc;
                acc[i].z *= sc;
                acc[i].w *= sc;
                M[i] = Mn;
            }
            // acc rows, eight (partial, head) pairs in flight
            constexpr int PER = NG >= 4 ? 1 : 8 / NG;   // partials per batch of loads (register budget)
            for (int q = 0; q < nb; q += PER) {
                float4 v[PER][NG];
                float wq[PER][NG];
#pragma unroll
                for (int u = 0; u < PER; ++u) {
                    const int src = min(q + u, nb - 1);
                    const int32_t pr = __shfl_sync(0xffffffffu, prow, src);
#pragma unroll
                    for (int i = 0; i < NG; ++i) {
                        const float ww = __shfl_sync(0xffffffffu, wt[i], src);
                        wq[u][i] = q + u < nb ? ww : 0.f;
                        v[u][i] = q + u < nb
                                      ? __ldcg(reinterpret_cast<const float4*>(a.part_acc + (int64_t)(pr + i) * D) + lane)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
#pragma unroll
                for (int u = 0; u < PER; ++u)
#pragma unroll
                    for (int i = 0; i < NG; ++i) {
                        acc[i].x = fmaf(v[u][i].x, wq[u][i], acc[i].x);
                        acc[i].y = fmaf(v[u][i].y, wq[u][i], acc[i].y);
                        acc[i].z = fmaf(v[u][i].z, wq[u][i], acc[i].z);
                        acc[i].w = fmaf(v[u][i].w, wq[u][i], acc[i].w);
                    }
            }
        }
    }
    wait_partials(waited);
    if (*reinterpret_cast<volatile const int32_t*>(&a.meta->status)) return;
#pragma unroll
    for (int i = 0; i < NG; ++i) {
        const float inv = 1.f / L[i];
        const int64_t o = ((int64_t)qi * pl.q_len + j) * pl.n_q_heads + h * G + g0 + i;
        T* dst = static_cast<T*>(a.out) + o * D + 4 * lane;
        if constexpr (sizeof(T) == 2) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc[i].x * inv, acc[i].y * inv);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc[i].z * inv, acc[i].w * inv);
            *reinterpret_cast<uint2*>(dst) =
                make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
        } else {
            *reinterpret_cast<float4*>(dst) = make_float4(acc[i].x * inv, acc[i].y * inv, acc[i].z * inv, acc[i].w * inv);
        }
    }
}

// ============================================================ host planning
// A segment as the unit expansion reads it (host or device): its units are
// unit_base + kv head * ngroups + row group, its tiles (class numbering)
// tile_base + that local unit index * n_blk, and the weight of the class's
// units before it wbase.  Row groups 0 .. ngroups - 2 hold group_rows rows,
// the last one rows_last.
struct SegPlan {
    int64_t wbase;                 // the three search keys first: one 16-byte load
    int32_t tile_base, unit_base;
    int32_t ngroups, group_rows, rows_last, n_blk;
    int32_t rt_full, rt_last, table_row, blk_start;
    int32_t mem_off;
    int32_t row_base;         // rows of all units before this segment's (tensor-core class first)
    int32_t w_full, w_last;   // weight of one unit of a full row group / of the last one
    int32_t n_shared, x_off;  // packed segments: tiles of the table row, first extra tile
    int32_t pad[2];
};
static_assert(sizeof(SegPlan) == 80, "SegPlan layout");

// A class of units (0: tcgen05, 1: mma.sync / fp32) for the CTA split.
struct PlanClass {
    int64_t weight;             // total weight of its units
    int32_t tiles;              // its tiles
    int32_t c0;                 // CTAs the split aims at (cuts are made at c0 - 1 targets)
    int32_t u_lo, u_hi;         // its units
    int32_t s_lo, s_hi;         // its segments in the SegPlan list
    int32_t unit_start, row_shift;   // the class's unit-start weight terms
};
struct PlanHeader {
    PlanClass cls[2];
    int32_t n_units, n_segs, n_rows, pad;   // n_rows: rows of all units (one chunk each)
};


// ====================================================== device plan expansion
// Expands a plan's segment list (SegPlan, class-relative offsets) into its
// work units and splits each class's tiles over CTAs on the device, writing
// exactly what the host expansion writes (build_units, partition_class):
//   - for c = 1 .. c0 - 1, the weight target ceil(weight c / c0) falls in one
//     unit, which starts at weight w after start weight us and has tiles of
//     weight tw; the cut candidate is its first tile plus
//     min(n_blk, max(0, ceil((target - w - us) / tw))).  Candidates do not
//     decrease with c, so the host's rule (keep a candidate above the last
//     kept cut and below the class's tiles) keeps exactly the candidates
//     that exceed their predecessor (0 for the first) and lie below the
//     tiles; a scan over those flags places them;
//   - each CTA's first unit, each unit's first CTA and number of chunks;
//   - each unit's first partial row.  Over the units before u, a unit holds
//     one chunk of its rows plus one more per CTA boundary inside it, so
//     prow_base(u) = (rows of the units before u) + (rows of the unit each
//     interior boundary before u falls in); the first term is the segment's
//     row base plus the rows before u in its segment, the second a prefix
//     over the (at most kMaxExpandCtas) boundaries of each class.
// Every CTA computes the splits (a few binary searches per thread) and then
// expands its own kExpandUnits units, so no step needs a grid-wide scan.  The
// searches run over the segments' keys (weight, first tile, first unit),
// which each CTA first copies to shared memory: kMaxExpandSegs segments at
// most (the host checks).
// It reads the segment list and header from the device copy the upload
// wrote, after waiting for that upload.  (Reading them from the pinned host
// buffer before the wait, to run alongside the append's copy, measured
// slower on the stress plan: the dependent host reads cost more than the
// overlap won.)
constexpr int kMaxExpandCtas = 1024;
constexpr int kMaxExpandSegs = 8192;
constexpr int kExpandThreads = 256;
constexpr int kExpandUnits = 256;   // units per expansion CTA

struct ExpandArgs {
    const SegPlan* sp;
    const PlanHeader* hdr;
    AttnUnit* units;
    int32_t* begin;      // mma.sync class CTA split [c0 + 1]
    int32_t* cunit;      // [c0]
    int32_t* tc_begin;
    int32_t* tc_cunit;
    int32_t* counts;     // [4]: CTAs of each class, partial rows (low, high)
    int32_t nkv;
};

// The segment of class [s_lo, s_hi) whose key range holds x: the last one
// with key(s) <= x (key nondecreasing in s).
template <typename F>
__device__ __forceinline__ int32_t seg_search(int32_t s_lo, int32_t s_hi, F key, int64_t x) {
    int32_t lo = s_lo, hi = s_hi - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (key(mid) <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Exclusive scan of one int per thread over the CTA (kExpandThreads threads);
// returns the thread's prefix and leaves the total in *total.
__device__ __forceinline__ int32_t expand_scan(int32_t v, int32_t* warp_tot, int32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += y;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    int32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kExpandThreads / 32; ++w) {
        const int32_t t = warp_tot[w];
        before += w < warp ? t : 0;
        all += t;
    }
    __syncthreads();   // warp_tot is reused by the next scan
    *total = all;
    return before + inc - v;
}

__global__ void __launch_bounds__(kExpandThreads) k_plan_expand(const ExpandArgs x) {
    constexpr int PER = kMaxExpandCtas / kExpandThreads;   // candidates per thread
    __shared__ int32_t s_cand[kMaxExpandCtas];
    __shared__ int32_t s_begin[2][kMaxExpandCtas + 1];
    __shared__ int32_t s_pre[2][kMaxExpandCtas + 1];   // rows of the interior boundaries 1..i
    __shared__ int32_t s_nc[2];
    __shared__ int32_t s_warp[kExpandThreads / 32];
    extern __shared__ int64_t s_keys[];                 // wbase[n_segs], then tile_base, unit_base
    asm volatile("griddepcontrol.wait;" ::: "memory");
    pdl_trigger();
    const int tid = threadIdx.x;
    const PlanHeader hdr = *x.hdr;
    const SegPlan* sp = x.sp;
    const int32_t nkv = x.nkv;
    const int32_t n_segs = hdr.n_segs;
    int64_t* s_wb = s_keys;
    int32_t* s_tb = reinterpret_cast<int32_t*>(s_keys + n_segs);
    int32_t* s_ub = s_tb + n_segs;
    for (int32_t i = tid; i < n_segs; i += kExpandThreads) {
        const int4 k = *reinterpret_cast<const int4*>(sp + i);
        s_wb[i] = (int64_t)(((uint64_t)(uint32_t)k.y << 32) | (uint32_t)k.x);
        s_tb[i] = k.z;
        s_ub[i] = k.w;
    }
    __syncthreads();
    // ------------------------------------------------------------ CTA splits
    for (int cls = 0; cls < 2; ++cls) {
        const PlanClass pc = hdr.cls[cls];
        for (int32_t c = 1 + tid; c < pc.c0; c += kExpandThreads) {
            const int64_t target = (pc.weight * c + pc.c0 - 1) / pc.c0;
            int32_t cut = pc.tiles;   // no unit holds the target: never kept
            if (target < pc.weight) {
                const int32_t si = seg_search(pc.s_lo, pc.s_hi, [&](int32_t k) { return s_wb[k]; }, target);
                const SegPlan g = sp[si];
                const int64_t w_head = (int64_t)(g.ngroups - 1) * g.w_full + g.w_last;
                const int64_t r = target - g.wbase;
                const int32_t h = (int32_t)min(r / w_head, (int64_t)(nkv - 1));
                const int64_t r2 = r - h * w_head;
                const int32_t grp = r2 < (int64_t)(g.ngroups - 1) * g.w_full ? (int32_t)(r2 / g.w_full) : g.ngroups - 1;
                const int64_t w = g.wbase + h * w_head + (int64_t)grp * g.w_full;
                const bool last = grp == g.ngroups - 1;
                const int32_t rows = last ? g.rows_last : g.group_rows;
                const int64_t us = pc.unit_start + (pc.row_shift >= 0 ? (rows >> pc.row_shift) : 0);
                const int64_t tw = 1 + (last ? g.rt_last : g.rt_full);
                const int64_t k = max((int64_t)0, (target - w - us + tw - 1) / tw);
                cut = g.tile_base + (h * g.ngroups + grp) * g.n_blk + (int32_t)min(k, (int64_t)g.n_blk);
            }
            s_cand[c] = cut;
        }
        __syncthreads();
        // keep flags of this thread's run of candidates c = 1 + PER tid ...
        int32_t keep = 0;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int32_t c = 1 + PER * tid + i;
            if (c < pc.c0) {
                const int32_t cut = s_cand[c], prev = c > 1 ? s_cand[c - 1] : 0;
                keep |= (cut > prev && cut < pc.tiles) << i;
            }
        }
        int32_t n_kept = 0;
        int32_t pos = 1 + expand_scan(__popc(keep), s_warp, &n_kept);
#pragma unroll
        for (int i = 0; i < PER; ++i)
            if (keep >> i & 1) s_begin[cls][pos++] = s_cand[1 + PER * tid + i];
        if (tid == 0) {
            s_begin[cls][0] = 0;
            s_begin[cls][n_kept + 1] = pc.tiles;
            s_nc[cls] = pc.c0 > 0 ? n_kept + 1 : 0;
        }
        __syncthreads();
        // rows of the unit each interior boundary falls in (0 at a unit start)
        const int32_t C = s_nc[cls];
        int32_t run = 0;
        int32_t rows_at[PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int32_t b_i = 1 + PER * tid + i;   // boundary index 1 .. C - 1
            rows_at[i] = 0;
            if (b_i < C) {
                const int32_t b = s_begin[cls][b_i];
                const int32_t si = seg_search(pc.s_lo, pc.s_hi, [&](int32_t k) { return (int64_t)s_tb[k]; }, b);
                const SegPlan g = sp[si];
                const int32_t k = (b - g.tile_base) / g.n_blk;
                const bool interior = b - g.tile_base != k * g.n_blk;
                const bool last = k % g.ngroups == g.ngroups - 1;
                rows_at[i] = interior ? (last ? g.rows_last : g.group_rows) : 0;
            }
            run += rows_at[i];
        }
        int32_t tot = 0;
        int32_t acc = expand_scan(run, s_warp, &tot);
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int32_t b_i = 1 + PER * tid + i;
            acc += rows_at[i];
            if (b_i < C) s_pre[cls][b_i] = acc;
        }
        if (tid == 0) {
            s_pre[cls][0] = 0;
            s_pre[cls][kMaxExpandCtas] = tot;   // all interior boundaries of the class
        }
        __syncthreads();
    }
    // ----------------------------------------- CTA arrays and counts (CTA 0)
    if (blockIdx.x == 0) {
        for (int cls = 0; cls < 2; ++cls) {
            const PlanClass pc = hdr.cls[cls];
            const int32_t C = s_nc[cls];
            int32_t* bg = cls == 0 ? x.tc_begin : x.begin;
            int32_t* cu = cls == 0 ? x.tc_cunit : x.cunit;
            for (int32_t c = tid; c <= C && C > 0; c += kExpandThreads) bg[c] = s_begin[cls][c];
            if (C == 0 && tid == 0) bg[0] = 0;   // an empty class still has begin[0]
            for (int32_t c = tid; c < C; c += kExpandThreads) {
                const int32_t b = s_begin[cls][c];
                const int32_t si = seg_search(pc.s_lo, pc.s_hi, [&](int32_t k) { return (int64_t)s_tb[k]; }, b);
                const SegPlan g = sp[si];
                cu[c] = g.unit_base + (b - g.tile_base) / g.n_blk;
            }
        }
        if (tid == 0) {
            const int64_t rows = (int64_t)hdr.n_rows + s_pre[0][kMaxExpandCtas] + s_pre[1][kMaxExpandCtas];
            x.counts[0] = s_nc[1];
            x.counts[1] = s_nc[0];
            x.counts[2] = (int32_t)(rows & 0xffffffff);
            x.counts[3] = (int32_t)(rows >> 32);
        }
    }
    // ------------------------------------------------------ this CTA's units
    const int32_t u = blockIdx.x * kExpandUnits + tid;
    if (u < hdr.n_units) {
        const int cls = u < hdr.cls[0].u_hi ? 0 : 1;
        const PlanClass& pc = hdr.cls[cls];
        const int32_t si = seg_search(pc.s_lo, pc.s_hi, [&](int32_t k) { return (int64_t)s_ub[k]; }, u);
        const SegPlan g = sp[si];
        const int32_t k = u - g.unit_base;
        const int32_t h = k / g.ngroups, grp = k - h * g.ngroups;
        const bool last = grp == g.ngroups - 1;
        AttnUnit U;
        U.seg = si;
        U.kv_head = h;
        U.row_lo = grp * g.group_rows;
        U.n_rows = last ? g.rows_last : g.group_rows;
        U.rt = last ? g.rt_last : g.rt_full;
        U.tile_off = g.tile_base + k * g.n_blk;
        // first CTA: begin[c] <= tile_off < begin[c + 1]; last CTA likewise for the last tile
        const int32_t C = s_nc[cls];
        auto cta_of = [&](int32_t t) {
            int32_t lo = 0, hi = C - 1;
            while (lo < hi) {
                const int32_t mid = (lo + hi + 1) >> 1;
                if (s_begin[cls][mid] <= t) lo = mid; else hi = mid - 1;
            }
            return lo;
        };
        U.cfirst = cta_of(U.tile_off);
        U.nchunks = cta_of(U.tile_off + g.n_blk - 1) - U.cfirst + 1;
        const int32_t rows_per_head = (g.ngroups - 1) * g.group_rows + g.rows_last;
        U.prow_base = g.row_base + h * rows_per_head + grp * g.group_rows + s_pre[cls][U.cfirst] +
                      (cls == 1 ? s_pre[0][kMaxExpandCtas] : 0);
        U.table_row = g.table_row;
        U.blk_start = g.blk_start;
        U.n_blk = g.n_blk;
        U.mem_off = g.mem_off;
        U.n_shared = g.n_shared;
        U.x_off = g.x_off;
        U.pad = 0;
        x.units[u] = U;
    }
}

// ============================================================ plan upload
// Copies the plan from the pool's pinned host buffer (device-accessible) to
// one of its two device copies.  A kernel rather than cudaMemcpyAsync: the
// copy engines may be busy with the caller's own host-to-device traffic on
// other streams, and a few KB of plan should not queue behind it.
// Launched as a programmatic dependent, it copies while the previous kernel
// (usually the append's copy kernel) is still running: it reads only the
// pinned buffer and writes only the device copy that the plan before the
// previous one used.  The kernels of that older call are complete by the
// time the previous kernel lets dependents launch: every kernel of the
// library does so only after its own griddepcontrol.wait, except this upload
// and the merge, which does so at its start but is itself launched only
// after the partial kernel passed its wait, so that every kernel before the
// merge's own call is complete.  It then waits for the previous kernel like
// any other, so the attention kernels after it see that kernel's results.
__global__ void __launch_bounds__(256) k_plan_upload(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                     int64_t n16) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
    pdl_trigger();
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ============================================================ host planning
struct HostPlan {
    std::vector<AttnSeg> segs;
    std::vector<AttnMember> members;
    std::vector<AttnUnit> units;
    std::vector<int32_t> cta_begin, cta_unit, tc_cta_begin, tc_cta_unit, path_off, path;
    std::vector<int64_t> cuts;
    int64_t tiles = 0, unique_tiles = 0;
    int32_t n_tc_units = 0;
    size_t partial_rows = 0;
    std::vector<int32_t> parent, fork_len, len, queried, seg_members, cursor;
    std::vector<Segment> psegs;
    std::vector<ExtraTile> pxt;      // the planner's extra tiles of packed segments
    std::vector<AttnXTile> xtiles;   // the same for the kernels (branch handles)
    std::vector<SegPlan> segplan;
    PlanHeader hdr{};
    bool device = false;       // units and CTA split left to the device
    bool small_packed = false; // a packed segment in the mma.sync class
    void clear() {   // keeps capacity: plans are rebuilt whenever the tree changes; the unit and
                     // member arrays keep their size too (build_plan resizes and fills them in place)
        segs.clear(); cta_begin.clear(); cta_unit.clear(); segplan.clear(); device = false; small_packed = false;
        pxt.clear(); xtiles.clear();
        tc_cta_begin.clear(); tc_cta_unit.clear(); path_off.clear(); path.clear(); cuts.clear();
        tiles = unique_tiles = 0;
        n_tc_units = 0;
        partial_rows = 0;
    }
};

size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// Partition weights, fitted to per-CTA timelines on GB300.  mma.sync class: a
// tile of a unit with rt row tiles of 16 costs about (1 + rt) units (HBM time
// plus mma time: 0.25 us for rt = 1 vs 0.61 us for rt = 4 per CTA), and every
// chunk boundary (partial store, combine, next unit's Q) about as much as 5
// one-row-tile tiles plus an eighth of a tile per row (its query load,
// combine and partial store grow with the rows).  Per-CTA end times of the
// beam call put a 4-row unit's start at about 1.8 us against 0.32 us per
// tile; on the packed MCTS plan these weights take the call from 237 to
// 215 us against (8, 4 rows per tile) before, with beam, spec-verify and
// stress unchanged.  tcgen05 class (one CTA per SM): a tile
// costs about (1 + rt) with rt row tiles of 128; a chunk boundary drains the
// MMA pipeline and stores up to 256 partial rows of 520 bytes.
struct ClassWeights {
    int64_t unit_start;
    int32_t row_shift;         // a unit start also weighs n_rows >> row_shift (-1: no row term)
    int64_t min_per_cta;       // smallest total weight worth a CTA of its own
};
constexpr ClassWeights kSmallWeights{10, 2, 8};
constexpr ClassWeights kTcWeights{24, -1, 32};
inline int64_t tile_weight(int rt) { return 1 + rt; }
inline int64_t start_weight(const ClassWeights& cw, int32_t n_rows) {
    return cw.unit_start + (cw.row_shift >= 0 ? (n_rows >> cw.row_shift) : 0);
}

// Stream-K split of one class's tile list (units [u_lo, u_hi), tiles
// [0, T)) into at most max_ctas CTAs of about equal weight (tile_weight per
// tile plus start_weight per unit start).  Cuts are made strictly increasing so
// that no CTA is empty.  Fills begin[C + 1], cunit[C] and each unit's cfirst
// and nchunks.
void partition_class(HostPlan& hp, int32_t u_lo, int32_t u_hi, int64_t T, int64_t weight, int max_ctas,
                     const ClassWeights& cw_, std::vector<int32_t>& begin, std::vector<int32_t>& cunit) {
    begin.clear();
    cunit.clear();
    if (u_lo == u_hi) {
        begin.push_back(0);
        return;
    }
    const int C0 = (int)std::max<int64_t>(
        1, std::min<int64_t>(max_ctas, (weight + cw_.min_per_cta - 1) / cw_.min_per_cta));
    hp.cuts.clear();
    hp.cuts.push_back(0);
    {
        // the weight at which cut c falls; one division per cut, not per unit
        int c = 1;
        int64_t target = C0 > 1 ? (weight + C0 - 1) / C0 : INT64_MAX;
        int64_t cw = 0;
        for (int32_t ui = u_lo; ui < u_hi; ++ui) {
            const AttnUnit& U = hp.units[ui];
            const int64_t nb = U.n_blk;
            const int64_t tw = tile_weight(U.rt);
            const int64_t us = start_weight(cw_, U.n_rows);
            const int64_t uw = us + nb * tw;
            while (c < C0 && target < cw + uw) {
                const int64_t k = std::max<int64_t>(0, (target - cw - us + tw - 1) / tw);
                const int64_t cut = U.tile_off + std::min<int64_t>(k, nb);
                if (cut > hp.cuts.back() && cut < T) hp.cuts.push_back(cut);
                ++c;
                target = c < C0 ? (weight * c + C0 - 1) / C0 : INT64_MAX;
            }
            cw += uw;
        }
    }
    hp.cuts.push_back(T);
    const int C = (int)hp.cuts.size() - 1;
    begin.resize(C + 1);
    for (int i = 0; i <= C; ++i) begin[i] = (int32_t)hp.cuts[i];
    cunit.resize(C);
    {
        int32_t u = u_lo;
        for (int c = 0; c < C; ++c) {
            while (u + 1 < u_hi && hp.units[u].tile_off + hp.units[u].n_blk <= begin[c]) ++u;
            cunit[c] = u;
        }
    }
    int c = 0;
    for (int32_t ui = u_lo; ui < u_hi; ++ui) {
        AttnUnit& U = hp.units[ui];
        const int32_t last = U.tile_off + U.n_blk - 1;
        while (begin[c + 1] <= U.tile_off) ++c;
        int cl = c;
        while (begin[cl + 1] <= last) ++cl;
        U.cfirst = c;
        U.nchunks = cl - c + 1;
    }
}

int build_units(dendrite_pool* p, const int32_t* branches, int32_t n, int32_t q_len, int32_t nq, int max_ctas,
                int max_tc_ctas, HostPlan& hp, bool allow_device);
int unit_rows_small(const dendrite_pool* p);

// max_ctas: CTAs of the mma.sync/fp32 kernel; max_tc_ctas: of the tcgen05
// kernel (0 when it is not used).  The segments (after folding) are left in
// hp.psegs / hp.seg_members.
int build_plan(dendrite_pool* p, const int32_t* branches, int32_t n, int32_t q_len, int32_t nq, int max_ctas,
               int max_tc_ctas, HostPlan& hp, bool allow_device) {
    const int32_t G = nq / p->n_kv, nkv = p->n_kv;
    const int32_t RM = q_len * G;
    const bool bf16 = p->dtype == DENDRITE_BF16;
    const int small_rows = unit_rows_small(p);
    const bool tc_on = bf16 && max_tc_ctas > 0 && p->tc_min_rows >= 0;
    const int32_t n_nodes = (int32_t)p->nodes.size();
    hp.parent.resize(n_nodes);
    hp.fork_len.resize(n_nodes);
    hp.len.resize(n_nodes);
    hp.queried.resize(n);
    for (int32_t i = 0; i < n_nodes; ++i) {
        hp.parent[i] = p->nodes[i].parent;
        hp.fork_len[i] = p->nodes[i].fork_len;
        hp.len[i] = p->nodes[i].len;
    }
    for (int32_t i = 0; i < n; ++i) hp.queried[i] = p->br[branches[i]].node;
    plan_segments(n_nodes, hp.parent.data(), hp.fork_len.data(), hp.len.data(), p->block_size, hp.queried.data(), n,
                  hp.psegs, hp.seg_members);
    // distinct tiles: the sharing segments before folding read each (block,
    // kv head) pair once
    for (const Segment& sg : hp.psegs) hp.unique_tiles += (int64_t)sg.block_count * nkv;
    static thread_local std::vector<int32_t> prev;
    prev.clear();
    if (bf16 && p->pack_pct >= 0)
        pack_segments(FoldParams{RM, tc_on ? p->tc_min_rows : -1, small_rows, p->fold_pct}, p->pack_pct, n_nodes,
                      hp.parent.data(), hp.fork_len.data(), p->block_size, hp.psegs, hp.seg_members, hp.pxt, &prev);
    if (p->fold_pct >= 0)
        fold_segments(FoldParams{RM, tc_on ? p->tc_min_rows : -1, small_rows, p->fold_pct}, n_nodes,
                      hp.parent.data(), hp.fork_len.data(), hp.len.data(), p->block_size, hp.queried.data(), n,
                      hp.psegs, hp.seg_members, &prev);
    return build_units(p, branches, n, q_len, nq, max_ctas, max_tc_ctas, hp, allow_device);
}

// Number of CTAs a class's split aims at: one per min_per_cta of weight, at
// most max_ctas, at least one.
int32_t class_ctas(int64_t weight, int max_ctas, const ClassWeights& cw) {
    return (int32_t)std::max<int64_t>(1, std::min<int64_t>(max_ctas, (weight + cw.min_per_cta - 1) / cw.min_per_cta));
}

// Rows per unit of the mma.sync (bf16: 4 row tiles of 16) or compressed
// (64: the CTA decodes each tile once for its four warps' row tiles) partial
// kernels, and of the fp32 kernel (16).
int unit_rows_small(const dendrite_pool* p) {
    return p->dtype == DENDRITE_BF16 ? kMaxUnitRowsBf16 : p->dtype == DENDRITE_TURBO ? kMaxUnitRowsTurbo
                                                                                    : kMaxUnitRowsF32;
}

// bf16 plans of at least this many units, with fewer tiles per unit than
// this on average, are expanded on the device by default
constexpr int32_t kDevicePlanMinUnits = 2048;
constexpr int32_t kDevicePlanMaxTilesPerUnit = 32;

// The plan's units, CTA partitions, partial rows and paths from the segments
// in hp.psegs / hp.seg_members (hp.tiles and the arrays are rebuilt;
// hp.unique_tiles is left as it is).  With allow_device and the pool's
// device_planning setting, a bf16 plan leaves the units and CTA split to
// k_plan_expand (hp.device): the host then fills the segment list (SegPlan)
// that kernel reads, and space for what it writes.
// SMs for the tcgen05 kernel when both partial classes have work (0: all SMs,
// the mma.sync kernel's CTAs taking each SM as its tcgen05 CTA finishes).
// The two kernels' CTAs never share an SM (shared memory), so without a split
// their times add up, although the tcgen05 class is bound by its tensor and
// softmax work once its units hold 256 rows, below the HBM rate, and the
// mma.sync class by HBM on leaves of a few rows.  Given n SMs the tcgen05
// kernel takes about A / n (A: its SM time) and reads its bytes at B_tc n / A,
// and the mma.sync kernel, on the other SMs, streams its bytes through the
// bandwidth left over, at most a per-SM rate; both end at the HBM floor when
// n = A * bandwidth / (B_tc + B_s).  The split is taken when its estimate
// beats the kernels one after the other by 7 %.  Weights are the partition's
// (tile_weight per tile plus the unit starts); the ns per weight are fitted
// to the kernels on GB300 (tcgen05: 255 ns per 16-token tile of a 256-row
// unit per SM; mma.sync: 60 ns per 4-row tile per CTA, two CTAs per SM).
int split_tc_sms(const dendrite_pool* p, int64_t w_tc, int64_t w_small, int64_t tiles_tc, int64_t tiles_small) {
    const int sms = p->sm_count;
    if (p->tc_sms < 0 || sms < 2) return 0;
    if (p->tc_sms > 0) return p->tc_sms < sms ? p->tc_sms : 0;
    constexpr double kTcNsPerWeight = 85.0, kSmallNsPerWeight = 30.0;   // SM ns
    constexpr double kHbmBytesPerNs = 6700.0;                           // measured copy bandwidth
    constexpr double kSmallBytesPerNsPerSm = 70.0;                      // one SM's two mma.sync CTAs
    const double tile_bytes = 2.0 * p->block_size * p->head_dim * 2;   // K and V of one kv head, bf16
    const double A = (double)w_tc * kTcNsPerWeight, S = (double)w_small * kSmallNsPerWeight;
    const double Bt = (double)tiles_tc * tile_bytes, Bs = (double)tiles_small * tile_bytes;
    const double serial = std::max(A / sms, Bt / kHbmBytesPerNs) + std::max(S / sms, Bs / kHbmBytesPerNs);
    const double floor_ns = (Bt + Bs) / kHbmBytesPerNs;
    double best = serial;
    int best_n = 0;
    for (int n = 1; n < sms; ++n) {
        const int m = sms - n;
        const double t = std::max(std::max(A / n, S / m), std::max(floor_ns, Bs / (m * kSmallBytesPerNsPerSm)));
        if (t < best) {
            best = t;
            best_n = n;
        }
    }
    return best < 0.93 * serial ? best_n : 0;
}

int build_units(dendrite_pool* p, const int32_t* branches, int32_t n, int32_t q_len, int32_t nq, int max_ctas,
                int max_tc_ctas, HostPlan& hp, bool allow_device) {
    const int32_t G = nq / p->n_kv, nkv = p->n_kv;
    const int32_t RM = q_len * G;
    const bool bf16 = p->dtype == DENDRITE_BF16;
    const int small_rows = unit_rows_small(p);
    const bool tc_on = bf16 && max_tc_ctas > 0 && p->tc_min_rows >= 0;
    // Segments, their members and their units (kv head major, then row
    // group), tensor-core segments first: pass 0 takes the segments read by
    // more than tc_min_rows rows per kv head, pass 1 the rest.
    size_t n_units_total = 0, n_members_total = 0, n_tiles_total = 0;
    for (const Segment& sg : hp.psegs) {
        if ((int64_t)sg.n_members * RM >= (int64_t)1 << 24) return DENDRITE_ELIMIT;   // rows as exact fp32
        const int32_t rows_per_head = sg.n_members * RM;
        const int32_t group_rows = (tc_on && rows_per_head > p->tc_min_rows) ? kMaxUnitRowsTc : small_rows;
        const size_t units = (size_t)nkv * ((rows_per_head + group_rows - 1) / group_rows);
        if (sg.n_x && units != (size_t)nkv) return DENDRITE_EINVAL;   // packed: one row group per kv head
        if (sg.n_x > kMaxTcExtraTiles && group_rows == kMaxUnitRowsTc) return DENDRITE_ELIMIT;
        n_units_total += units;
        n_tiles_total += units * (size_t)(sg.block_count + sg.n_x);
        n_members_total += sg.n_members;
    }
    if (n_units_total >= (size_t)INT32_MAX / 2) return DENDRITE_ELIMIT;
    // By default only plans whose host expansion rivals the kernels' work go
    // to the device: many units (the expansion's cost) of few tiles each (the
    // kernels' work).  Elsewhere the host expansion hides behind the device's
    // work, while the expansion kernel would sit between the upload and the
    // partial kernels.
    hp.device = allow_device && bf16 && max_ctas <= kMaxExpandCtas && max_tc_ctas <= kMaxExpandCtas &&
                hp.psegs.size() <= (size_t)kMaxExpandSegs &&
                (p->device_planning > 0 ||
                 (p->device_planning == 0 && n_units_total >= (size_t)kDevicePlanMinUnits &&
                  n_tiles_total < (size_t)kDevicePlanMaxTilesPerUnit * n_units_total));
    hp.units.resize(n_units_total);
    hp.members.resize(n_members_total);
    hp.segs.reserve(hp.psegs.size());
    hp.segplan.reserve(hp.psegs.size());
    AttnMember* mp = hp.members.data();
    int32_t n_mem = 0, n_unit = 0;
    int64_t n_rows = 0;
    for (int pass = 0; pass < 2; ++pass) {
        PlanClass& pc = hp.hdr.cls[pass];
        const ClassWeights& cwt = pass == 0 ? kTcWeights : kSmallWeights;
        pc = PlanClass{};
        pc.u_lo = n_unit;
        pc.s_lo = (int32_t)hp.segplan.size();
        pc.unit_start = (int32_t)cwt.unit_start;
        pc.row_shift = cwt.row_shift;
        int64_t tile_off = 0, weight = 0;
        for (const Segment& sg : hp.psegs) {
            const int32_t rows_per_head = sg.n_members * RM;
            const bool tc = tc_on && rows_per_head > p->tc_min_rows;
            if (tc != (pass == 0)) continue;
            const int32_t group_rows = tc ? kMaxUnitRowsTc : small_rows;
            AttnSeg S;
            S.table_row = p->nodes[sg.rep_node].handle;
            S.blk_start = sg.block_start;
            S.n_blk = sg.block_count + sg.n_x;
            S.mem_off = n_mem;
            S.n_mem = sg.n_members;
            S.unit_base = n_unit;
            S.ngroups = (rows_per_head + group_rows - 1) / group_rows;
            S.group_rows = group_rows;
            for (int32_t k = 0; k < sg.n_members; ++k) {
                const int32_t qi = hp.seg_members[sg.member_offset + k];
                mp[n_mem++] = AttnMember{qi, p->br[branches[qi]].len};
            }
            auto rt_of = [&](int32_t rows) { return tc ? (rows + 127) / 128 : rows <= 16 ? 1 : rows <= 32 ? 2 : 4; };
            SegPlan sp;
            sp.unit_base = S.unit_base;
            sp.ngroups = S.ngroups;
            sp.group_rows = group_rows;
            sp.rows_last = rows_per_head - (S.ngroups - 1) * group_rows;
            sp.n_blk = S.n_blk;
            sp.tile_base = (int32_t)tile_off;
            sp.rt_full = rt_of(group_rows);
            sp.rt_last = rt_of(sp.rows_last);
            sp.table_row = S.table_row;
            sp.blk_start = S.blk_start;
            sp.mem_off = S.mem_off;
            sp.n_shared = sg.block_count;
            sp.x_off = (int32_t)hp.xtiles.size();
            sp.pad[0] = sp.pad[1] = 0;
            if (pass == 1 && sg.n_x) hp.small_packed = true;
            for (int32_t k = 0; k < sg.n_x; ++k) {
                const ExtraTile& e = hp.pxt[sg.x_off + k];
                hp.xtiles.push_back(AttnXTile{e.blk, e.mask, p->nodes[e.rep_node].handle, 0});
            }
            sp.row_base = (int32_t)n_rows;
            sp.wbase = weight;
            sp.w_full = (int32_t)(start_weight(cwt, group_rows) + (int64_t)S.n_blk * tile_weight(sp.rt_full));
            sp.w_last = (int32_t)(start_weight(cwt, sp.rows_last) + (int64_t)S.n_blk * tile_weight(sp.rt_last));
            hp.segplan.push_back(sp);
            const int64_t units = (int64_t)nkv * S.ngroups;
            n_unit += (int32_t)units;
            n_rows += (int64_t)nkv * rows_per_head;
            tile_off += units * S.n_blk;
            weight += (int64_t)nkv * ((int64_t)(S.ngroups - 1) * sp.w_full + sp.w_last);
            hp.segs.push_back(S);
        }
        if (tile_off >= INT32_MAX / 2) return DENDRITE_ELIMIT;
        pc.u_hi = n_unit;
        pc.s_hi = (int32_t)hp.segplan.size();
        pc.tiles = (int32_t)tile_off;
        pc.weight = weight;
        if (pass == 0) hp.n_tc_units = n_unit;
    }
    {
        PlanClass& ct = hp.hdr.cls[0];
        PlanClass& cs = hp.hdr.cls[1];
        if (ct.u_hi > ct.u_lo && cs.u_hi > cs.u_lo) {
            const int n = split_tc_sms(p, ct.weight, cs.weight, ct.tiles, cs.tiles);
            if (n > 0) {
                max_tc_ctas = std::min(max_tc_ctas, n);
                max_ctas = std::min(max_ctas, (p->sm_count - n) * p->attn_ctas_per_sm);
            }
        }
        ct.c0 = ct.u_hi > ct.u_lo ? class_ctas(ct.weight, max_tc_ctas, kTcWeights) : 0;
        cs.c0 = cs.u_hi > cs.u_lo ? class_ctas(cs.weight, max_ctas, kSmallWeights) : 0;
    }
    if (n_rows >= INT32_MAX / 2) return DENDRITE_ELIMIT;
    hp.hdr.n_units = n_unit;
    hp.hdr.n_segs = (int32_t)hp.segplan.size();
    hp.hdr.n_rows = (int32_t)n_rows;
    hp.tiles = (int64_t)hp.hdr.cls[0].tiles + hp.hdr.cls[1].tiles;
    if (hp.device) {
        // space for what k_plan_expand writes; the partial rows bounded by one
        // extra chunk of a unit's rows per CTA boundary
        hp.cta_begin.assign((size_t)std::max(hp.hdr.cls[1].c0, 1) + 1, 0);
        hp.cta_unit.assign((size_t)std::max(hp.hdr.cls[1].c0, 1), 0);
        hp.tc_cta_begin.assign((size_t)hp.hdr.cls[0].c0 + 1, 0);
        hp.tc_cta_unit.assign((size_t)hp.hdr.cls[0].c0, 0);
        hp.partial_rows = (size_t)n_rows + (size_t)std::max(hp.hdr.cls[1].c0 - 1, 0) * small_rows +
                          (size_t)std::max(hp.hdr.cls[0].c0 - 1, 0) * kMaxUnitRowsTc;
    } else {
        for (size_t si = 0; si < hp.segplan.size(); ++si) {
            const SegPlan& sp = hp.segplan[si];
            const int32_t rows_per_head = (sp.ngroups - 1) * sp.group_rows + sp.rows_last;
            for (int32_t h = 0; h < nkv; ++h) {
                for (int32_t grp = 0; grp < sp.ngroups; ++grp) {
                    const int32_t k = h * sp.ngroups + grp;
                    AttnUnit& U = hp.units[sp.unit_base + k];
                    U.seg = (int32_t)si;
                    U.kv_head = h;
                    U.row_lo = grp * sp.group_rows;
                    U.n_rows = std::min(sp.group_rows, rows_per_head - U.row_lo);
                    U.rt = grp + 1 < sp.ngroups ? sp.rt_full : sp.rt_last;
                    U.tile_off = sp.tile_base + k * sp.n_blk;
                    U.cfirst = U.nchunks = U.prow_base = 0;
                    U.table_row = sp.table_row;
                    U.blk_start = sp.blk_start;
                    U.n_blk = sp.n_blk;
                    U.mem_off = sp.mem_off;
                    U.n_shared = sp.n_shared;
                    U.x_off = sp.x_off;
                    U.pad = 0;
                }
            }
        }
        partition_class(hp, 0, hp.n_tc_units, hp.hdr.cls[0].tiles, hp.hdr.cls[0].weight, max_tc_ctas, kTcWeights,
                        hp.tc_cta_begin, hp.tc_cta_unit);
        partition_class(hp, hp.n_tc_units, (int32_t)hp.units.size(), hp.hdr.cls[1].tiles, hp.hdr.cls[1].weight,
                        max_ctas, kSmallWeights, hp.cta_begin, hp.cta_unit);
        // partial rows per unit
        size_t prow = 0;
        for (AttnUnit& U : hp.units) {
            U.prow_base = (int32_t)prow;
            prow += (size_t)U.nchunks * U.n_rows;
        }
        if (prow >= (size_t)INT32_MAX) return DENDRITE_ELIMIT;
        hp.partial_rows = prow;
    }
    if (hp.partial_rows >= (size_t)INT32_MAX) return DENDRITE_ELIMIT;
    // path of every queried branch: one entry per segment it reads
    hp.path_off.assign(n + 1, 0);
    for (const AttnSeg& S : hp.segs)
        for (int32_t k = 0; k < S.n_mem; ++k) hp.path_off[hp.members[S.mem_off + k].qi + 1]++;
    for (int32_t i = 0; i < n; ++i) hp.path_off[i + 1] += hp.path_off[i];
    hp.path.resize(4 * (size_t)hp.path_off[n]);
    hp.cursor.assign(hp.path_off.begin(), hp.path_off.end() - 1);
    for (int32_t si = 0; si < (int32_t)hp.segs.size(); ++si) {
        const AttnSeg& S = hp.segs[si];
        for (int32_t k = 0; k < S.n_mem; ++k) {
            const int32_t e = hp.cursor[hp.members[S.mem_off + k].qi]++;
            hp.path[4 * e] = S.unit_base;
            hp.path[4 * e + 1] = S.ngroups;
            hp.path[4 * e + 2] = k * RM;
            hp.path[4 * e + 3] = S.group_rows;
        }
    }
    for (int32_t i = 0; i < n; ++i)
        if (hp.path_off[i + 1] == hp.path_off[i]) return DENDRITE_EINVAL;   // a branch with no visible key
    return DENDRITE_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

int encode_pool_map(dendrite_pool* p, void* base, unsigned char* out) {
    auto enc = get_encode();
    if (!enc) return DENDRITE_ECUDA;
    CUtensorMap m;
    // [rows = blocks * kv heads * 16][2 halves][64 columns] of bf16, one box = 16 rows x 64 columns
    cuuint64_t dims[3] = {64, 2, (cuuint64_t)p->num_blocks * p->n_kv * BS};
    cuuint64_t strides[2] = {128, 256};
    cuuint32_t box[3] = {64, 1, BS};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return DENDRITE_ECUDA;
    static_assert(sizeof(CUtensorMap) == 128, "tensor map size");
    std::memcpy(out, &m, sizeof(m));
    return DENDRITE_OK;
}

// Byte layout of an uploaded plan: the sections of HostPlan one after the
// other, each 16-byte aligned.  off[k] is the start of section k,
// off[kPlanSections] the total size.  The sections the host always writes
// come first (segments, members, paths, the segment list and header of the
// device expansion); from kPlanDeviceSection on, the units, CTA splits and
// counts, which k_plan_expand writes when the plan is expanded on the device
// (only the prefix before them is then uploaded).
enum PlanSection {
    SEC_SEGS, SEC_MEMBERS, SEC_PATH_OFF, SEC_PATH, SEC_SEGPLAN, SEC_HEADER, SEC_XTILES,
    SEC_UNITS, SEC_CTA_BEGIN, SEC_CTA_UNIT, SEC_TC_BEGIN, SEC_TC_UNIT, SEC_COUNTS, kPlanSections
};
constexpr int kPlanDeviceSection = SEC_UNITS;
size_t plan_layout(const HostPlan& hp, size_t (&off)[kPlanSections + 1]) {
    const size_t sz[kPlanSections] = {
        hp.segs.size() * sizeof(AttnSeg),     hp.members.size() * sizeof(AttnMember),
        hp.path_off.size() * 4,               hp.path.size() * 4,
        hp.device ? hp.segplan.size() * sizeof(SegPlan) : 0,
        hp.device ? sizeof(PlanHeader) : 0,
        hp.xtiles.size() * sizeof(AttnXTile),
        hp.units.size() * sizeof(AttnUnit),   hp.cta_begin.size() * 4,
        hp.cta_unit.size() * 4,               hp.tc_cta_begin.size() * 4,
        hp.tc_cta_unit.size() * 4,            hp.device ? 4 * sizeof(int32_t) : 0};
    size_t b = 0;
    for (int k = 0; k < kPlanSections; ++k) {
        off[k] = b;
        b = align16(b + sz[k]);
    }
    off[kPlanSections] = b;
    return b;
}

// Bytes of the packed plan the host writes and uploads.
size_t plan_upload_bytes(const HostPlan& hp, const size_t (&off)[kPlanSections + 1]) {
    return hp.device ? off[kPlanDeviceSection] : off[kPlanSections];
}

void plan_pack(const HostPlan& hp, const size_t (&off)[kPlanSections + 1], char* h) {
    auto put = [&](int k, const void* src, size_t bytes) {
        if (bytes) std::memcpy(h + off[k], src, bytes);
    };
    put(SEC_SEGS, hp.segs.data(), hp.segs.size() * sizeof(AttnSeg));
    put(SEC_MEMBERS, hp.members.data(), hp.members.size() * sizeof(AttnMember));
    put(SEC_PATH_OFF, hp.path_off.data(), hp.path_off.size() * 4);
    put(SEC_PATH, hp.path.data(), hp.path.size() * 4);
    put(SEC_XTILES, hp.xtiles.data(), hp.xtiles.size() * sizeof(AttnXTile));
    if (hp.device) {
        put(SEC_SEGPLAN, hp.segplan.data(), hp.segplan.size() * sizeof(SegPlan));
        put(SEC_HEADER, &hp.hdr, sizeof(PlanHeader));
        return;
    }
    put(SEC_UNITS, hp.units.data(), hp.units.size() * sizeof(AttnUnit));
    put(SEC_CTA_BEGIN, hp.cta_begin.data(), hp.cta_begin.size() * 4);
    put(SEC_CTA_UNIT, hp.cta_unit.data(), hp.cta_unit.size() * 4);
    put(SEC_TC_BEGIN, hp.tc_cta_begin.data(), hp.tc_cta_begin.size() * 4);
    put(SEC_TC_UNIT, hp.tc_cta_unit.data(), hp.tc_cta_unit.size() * 4);
}

AttnPlanDev plan_view(const HostPlan& hp, const size_t (&off)[kPlanSections + 1], const char* d, int32_t n,
                      int32_t q_len, int32_t nq, int32_t group) {
    AttnPlanDev v{};
    v.segs = reinterpret_cast<const AttnSeg*>(d + off[SEC_SEGS]);
    v.members = reinterpret_cast<const AttnMember*>(d + off[SEC_MEMBERS]);
    v.path_off = reinterpret_cast<const int32_t*>(d + off[SEC_PATH_OFF]);
    v.path = reinterpret_cast<const int32_t*>(d + off[SEC_PATH]);
    v.xtiles = reinterpret_cast<const AttnXTile*>(d + off[SEC_XTILES]);
    v.units = reinterpret_cast<const AttnUnit*>(d + off[SEC_UNITS]);
    v.cta_begin = reinterpret_cast<const int32_t*>(d + off[SEC_CTA_BEGIN]);
    v.cta_unit = reinterpret_cast<const int32_t*>(d + off[SEC_CTA_UNIT]);
    v.tc_cta_begin = reinterpret_cast<const int32_t*>(d + off[SEC_TC_BEGIN]);
    v.tc_cta_unit = reinterpret_cast<const int32_t*>(d + off[SEC_TC_UNIT]);
    v.counts = hp.device ? reinterpret_cast<const int32_t*>(d + off[SEC_COUNTS]) : nullptr;
    v.packed = hp.small_packed ? 1 : 0;
    v.n_units = (int32_t)hp.units.size();
    v.n_ctas = (int32_t)hp.cta_unit.size();
    v.n_tc_units = hp.n_tc_units;
    v.n_tc_ctas = (int32_t)hp.tc_cta_unit.size();
    v.n_queried = n;
    v.q_len = q_len;
    v.n_q_heads = nq;
    v.group = group;
    v.rcp_rows_per_member = 1.0f / (float)(q_len * group);
    v.rcp_group = 1.0f / (float)group;
    return v;
}

// The same plan view over another copy of the plan bytes.
AttnPlanDev plan_rebase(AttnPlanDev v, const char* from, const char* to) {
    auto mv = [&](auto*& ptr) {
        using P = std::remove_reference_t<decltype(ptr)>;
        ptr = reinterpret_cast<P>(to + (reinterpret_cast<const char*>(ptr) - from));
    };
    mv(v.segs);
    mv(v.members);
    mv(v.units);
    mv(v.cta_begin);
    mv(v.cta_unit);
    mv(v.tc_cta_begin);
    mv(v.tc_cta_unit);
    mv(v.path_off);
    mv(v.path);
    mv(v.xtiles);
    if (v.counts) mv(v.counts);
    return v;
}

// Launches k_plan_expand over the plan copy at d (section offsets off), after
// the upload that wrote its host sections.
int launch_plan_expand(dendrite_pool* p, char* d, const size_t* off, int32_t n_units, int32_t n_segs,
                       cudaStream_t s) {
    ExpandArgs x{};
    x.sp = reinterpret_cast<const SegPlan*>(d + off[SEC_SEGPLAN]);
    x.hdr = reinterpret_cast<const PlanHeader*>(d + off[SEC_HEADER]);
    x.units = reinterpret_cast<AttnUnit*>(d + off[SEC_UNITS]);
    x.begin = reinterpret_cast<int32_t*>(d + off[SEC_CTA_BEGIN]);
    x.cunit = reinterpret_cast<int32_t*>(d + off[SEC_CTA_UNIT]);
    x.tc_begin = reinterpret_cast<int32_t*>(d + off[SEC_TC_BEGIN]);
    x.tc_cunit = reinterpret_cast<int32_t*>(d + off[SEC_TC_UNIT]);
    x.counts = reinterpret_cast<int32_t*>(d + off[SEC_COUNTS]);
    x.nkv = p->n_kv;
    DENDRITE_CUDA(launch_pdl(k_plan_expand, dim3((unsigned)std::max(1, (n_units + kExpandUnits - 1) / kExpandUnits)),
                             dim3(kExpandThreads), (size_t)n_segs * 16, s, x));
    return DENDRITE_OK;
}

// CTAs the tensor-core kernel may use on this pool (0: not used).
int tc_ctas(const dendrite_pool* p) {
    return (p->dtype == DENDRITE_BF16 && p->tc_ready && p->tc_min_rows >= 0) ? p->sm_count : 0;
}

// The partial kernels of one attention call (tensor-core class, then the
// mma.sync or fp32 class), then the merge.  The mma.sync, fp32 and merge
// kernels are launched with programmatic stream serialisation: their
// prologues overlap the previous kernel's tail, and they wait for its results
// (griddepcontrol.wait) before reading anything.
int launch_attention(dendrite_pool* p, int32_t layer, const AttnArgs& a, cudaStream_t s) {
    const bool bf16 = p->dtype == DENDRITE_BF16;
    prof_begin(p, T_ATTN_PARTIAL, s);
    CUtensorMap mk{}, mv{};
    if (bf16) {
        std::memcpy(&mk, p->tmap_k[layer].bytes, sizeof(mk));
        std::memcpy(&mv, p->tmap_v[layer].bytes, sizeof(mv));
    }
    // Both partial classes: the tcgen05 and the mma.sync kernel write
    // disjoint partial rows and read only the plan and the pool, so the
    // mma.sync kernel runs on the pool's side stream (lowest priority) beside
    // the tcgen05 one, and the caller's stream waits for it before the merge.
    // Their CTAs never share an SM: with an SM split in the plan each
    // kernel's CTAs fit on their own SMs at once and the two run side by
    // side; without one the mma.sync CTAs take the SMs the tcgen05 CTAs
    // leave as they finish.
    const bool beside = bf16 && a.plan.n_tc_ctas > 0 && a.plan.n_ctas > 0 && p->side;
    if (beside) DENDRITE_CUDA(cudaEventRecord(p->ev_fork, s));
    // the tcgen05 kernel is submitted first, so that its CTAs are placed
    // before the side stream's
    if (a.plan.n_tc_ctas > 0) {
        prof_begin(p, T_ATTN_TC, s);
        DENDRITE_TRY(launch_attn_tc(mk, mv, a, a.plan.n_tc_ctas, s));
        prof_end(p, T_ATTN_TC, s);
    } else {
        p->ev_recorded[T_ATTN_TC] = false;   // this call ran no tensor-core kernel
    }
    if (beside) {
        DENDRITE_CUDA(cudaStreamWaitEvent(p->side, p->ev_fork, 0));
        prof_begin(p, T_ATTN_MMA_SIDE, p->side);
        if (a.plan.packed)
            k_attn_partial_bf16<true><<<dim3(a.plan.n_ctas), dim3(THREADS), SMEM_BF16_PACKED, p->side>>>(mk, mv, a);
        else
            k_attn_partial_bf16<false><<<dim3(a.plan.n_ctas), dim3(THREADS), SMEM_BF16, p->side>>>(mk, mv, a);
        DENDRITE_CUDA(cudaGetLastError());
        prof_end(p, T_ATTN_MMA_SIDE, p->side);
        DENDRITE_CUDA(cudaEventRecord(p->ev_join, p->side));
        DENDRITE_CUDA(cudaStreamWaitEvent(s, p->ev_join, 0));
    } else {
        p->ev_recorded[T_ATTN_MMA_SIDE] = false;
    }
    const int32_t n_out_rows = a.plan.n_queried * a.plan.q_len * a.plan.n_q_heads;
    if (beside) {
        // launched above
    } else if (p->dtype == DENDRITE_TURBO) {
        DENDRITE_TRY(launch_turbo_partials(a, a.Q, n_out_rows, p->d_tq_signs, p->d_tq_S, p->d_tq_qs, s));
    } else if (a.plan.n_ctas > 0) {
        if (bf16) {
            if (a.plan.packed)
                DENDRITE_CUDA(launch_pdl(k_attn_partial_bf16<true>, dim3(a.plan.n_ctas), dim3(THREADS),
                                         SMEM_BF16_PACKED, s, mk, mv, a));
            else
                DENDRITE_CUDA(launch_pdl(k_attn_partial_bf16<false>, dim3(a.plan.n_ctas), dim3(THREADS), SMEM_BF16,
                                         s, mk, mv, a));
        } else {
            DENDRITE_CUDA(launch_pdl(k_attn_partial_f32, dim3(a.plan.n_ctas), dim3(128),
                                     2 * BS * p->head_dim * sizeof(float), s, a));
        }
    }
    prof_end(p, T_ATTN_PARTIAL, s);
    prof_begin(p, T_ATTN_MERGE, s);
    {
        // after a join from the side stream the merge is an ordinary launch:
        // its dependence is on an event, not on the previous kernel alone
        auto mlaunch = [&](auto kernel, unsigned g) -> cudaError_t {
            if (!beside) return launch_pdl(kernel, dim3(g), dim3(256), 0, s, a);
            kernel<<<dim3(g), dim3(256), 0, s>>>(a);
            return cudaGetLastError();
        };
        const int32_t n_out = a.plan.n_queried * a.plan.q_len * a.plan.n_q_heads;
        const unsigned grid = (unsigned)((n_out + 7) / 8);
        const int G = a.plan.group;
        const int ng = G >= 4 ? (G % 4 == 0 ? 4 : 0) : (G == 1 || G == 2 ? G : 0);   // rows per grouped warp
        // the grouped merge shares lookups among a group's heads but runs a
        // quarter of the warps; a small merge (beam: 1,024 rows) keeps one
        // row per warp, where the warps' latency chains overlap better
        if (p->dtype == DENDRITE_TURBO) {
            // rows of compressed pools are rotated back by the per-row merge
            DENDRITE_CUDA(mlaunch(k_attn_merge<__nv_bfloat16, true>, grid));
        } else if (p->head_dim == D && ng > 0 && (int64_t)n_out / ng >= (int64_t)16 * p->sm_count) {
            const unsigned ggrid = (unsigned)((n_out / ng + 7) / 8);
            if (bf16) {
                if (ng == 4) DENDRITE_CUDA(mlaunch(k_attn_merge_grouped<__nv_bfloat16, 4>, ggrid));
                else if (ng == 2) DENDRITE_CUDA(mlaunch(k_attn_merge_grouped<__nv_bfloat16, 2>, ggrid));
                else DENDRITE_CUDA(mlaunch(k_attn_merge_grouped<__nv_bfloat16, 1>, ggrid));
            } else {
                if (ng == 4) DENDRITE_CUDA(mlaunch(k_attn_merge_grouped<float, 4>, ggrid));
                else if (ng == 2) DENDRITE_CUDA(mlaunch(k_attn_merge_grouped<float, 2>, ggrid));
                else DENDRITE_CUDA(mlaunch(k_attn_merge_grouped<float, 1>, ggrid));
            }
        } else if (bf16) DENDRITE_CUDA(mlaunch(k_attn_merge<__nv_bfloat16, true>, grid));
        else if (p->head_dim == D) DENDRITE_CUDA(mlaunch(k_attn_merge<float, true>, grid));
        else DENDRITE_CUDA(mlaunch(k_attn_merge<float, false>, grid));
    }
    prof_end(p, T_ATTN_MERGE, s);
    prof_end(p, T_ATTN_TOTAL, s);
    DENDRITE_CUDA(cudaGetLastError());
    return DENDRITE_OK;
}

AttnArgs attn_args(const dendrite_pool* p, int32_t layer, const void* Q, void* out) {
    AttnArgs a{};
    a.Q = Q;
    a.out = out;
    a.table = p->d_table;
    a.pool_k = reinterpret_cast<const float*>(static_cast<const char*>(p->d_k) + (size_t)layer * p->layer_bytes);
    a.pool_v = reinterpret_cast<const float*>(static_cast<const char*>(p->d_v) + (size_t)layer * p->layer_bytes_v);
    a.tq_signs = p->dtype == DENDRITE_TURBO ? p->d_tq_signs : nullptr;
    a.meta = p->d_meta;
    a.bpb = p->bpb;
    a.n_kv = p->n_kv;
    a.head_dim = p->head_dim;
    a.n_blocks = (int32_t)p->num_blocks;
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)p->head_dim));
    return a;
}

int ensure_capacity(dendrite_pool* p, size_t plan_bytes, size_t partial_rows) {
    if (plan_bytes > p->plan_cap) {
        size_t cap = std::max<size_t>(plan_bytes * 2, 1 << 20);
        DENDRITE_CUDA(cudaDeviceSynchronize());
        for (char*& d : p->d_plan) {
            if (d) cudaFree(d);
            d = nullptr;
        }
        p->plan_cap = 0;
        for (char*& d : p->d_plan) DENDRITE_CUDA(cudaMalloc(&d, cap));
        p->plan_cap = cap;
        p->plan.valid = false;
    }
    if (plan_bytes > p->h_plan_cap) {
        size_t cap = std::max<size_t>(plan_bytes * 2, 1 << 20);
        for (int i = 0; i < 2; ++i) {
            DENDRITE_CUDA(cudaEventSynchronize(p->plan_copied[i]));
            if (p->h_plan[i]) cudaFreeHost(p->h_plan[i]);
            p->h_plan[i] = nullptr;
        }
        p->h_plan_cap = 0;
        for (int i = 0; i < 2; ++i) DENDRITE_CUDA(cudaMallocHost(&p->h_plan[i], cap));
        p->h_plan_cap = cap;
    }
    if (partial_rows > p->partial_rows_cap) {
        size_t cap = std::max<size_t>(partial_rows * 3 / 2, 4096);
        DENDRITE_CUDA(cudaDeviceSynchronize());
        if (p->d_partial) cudaFree(p->d_partial);
        p->d_partial = nullptr;
        p->partial_rows_cap = 0;
        DENDRITE_CUDA(cudaMalloc(&p->d_partial, cap * (p->head_dim + 2) * sizeof(float)));
        p->partial_rows_cap = cap;
    }
    return DENDRITE_OK;
}

}  // namespace

namespace dendrite {

int attn_setup(dendrite_pool* p) {
    if (p->dtype == DENDRITE_BF16) {
        p->tmap_k.resize(p->n_layers);
        p->tmap_v.resize(p->n_layers);
        for (int32_t l = 0; l < p->n_layers; ++l) {
            const size_t off = (size_t)l * p->layer_bytes;
            DENDRITE_TRY(encode_pool_map(p, static_cast<char*>(p->d_k) + off, p->tmap_k[l].bytes));
            DENDRITE_TRY(encode_pool_map(p, static_cast<char*>(p->d_v) + off, p->tmap_v[l].bytes));
        }
        p->tmaps_ok = true;
        DENDRITE_CUDA(cudaFuncSetAttribute(k_attn_partial_bf16<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)SMEM_BF16));
        DENDRITE_CUDA(cudaFuncSetAttribute(k_attn_partial_bf16<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)SMEM_BF16_PACKED));
        int occ = 0, occ_packed = 0;
        DENDRITE_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_attn_partial_bf16<false>, THREADS, SMEM_BF16));
        DENDRITE_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_packed, k_attn_partial_bf16<true>, THREADS,
                                                                    SMEM_BF16_PACKED));
        p->attn_ctas_per_sm = std::max(1, std::min(occ, occ_packed));
        p->tc_ready = attn_tc_setup() == DENDRITE_OK;
        DENDRITE_CUDA(cudaFuncSetAttribute(k_plan_expand, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kMaxExpandSegs * 16));
    } else if (p->dtype == DENDRITE_TURBO) {
        p->attn_ctas_per_sm = turbo_ctas_per_sm();
    } else {
        const size_t sm = 2 * BS * p->head_dim * sizeof(float);
        int occ = 0;
        DENDRITE_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_attn_partial_f32, 128, sm));
        p->attn_ctas_per_sm = std::max(1, occ);
    }
    return DENDRITE_OK;
}

void attn_teardown(dendrite_pool* p) {
    for (char*& d : p->d_plan) {
        if (d) cudaFree(d);
        d = nullptr;
    }
    for (char*& h : p->h_plan) {
        if (h) cudaFreeHost(h);
        h = nullptr;
    }
    if (p->d_partial) cudaFree(p->d_partial);
    p->d_partial = nullptr;
    if (p->d_tq_qs) cudaFree(p->d_tq_qs);
    p->d_tq_qs = nullptr;
}

}  // namespace dendrite

extern "C" int dendrite_tree_attn_decode(dendrite_pool* p, const void* Q, int32_t n_q_heads, int32_t q_len,
                                         const int32_t* branches, int32_t n, void* out, void* stream) {
    return dendrite_tree_attn_decode_layer(p, 0, Q, n_q_heads, q_len, branches, n, out, stream);
}

extern "C" int dendrite_tree_attn_decode_layer(dendrite_pool* p, int32_t layer, const void* Q, int32_t n_q_heads,
                                               int32_t q_len, const int32_t* branches, int32_t n, void* out,
                                               void* stream) {
    if (!p) return DENDRITE_EINVAL;
    if (p->poisoned) return p->poisoned;
    if (layer < 0 || layer >= p->n_layers) return DENDRITE_EINVAL;
    if (p->pending.active && !p->pending.layer_done[layer]) return DENDRITE_EINVAL;
    DENDRITE_CUDA(cudaSetDevice(p->device));
    if (!Q || !out || !branches || n <= 0 || q_len <= 0 || n_q_heads <= 0) return DENDRITE_EINVAL;
    if (n_q_heads % p->n_kv) return DENDRITE_EINVAL;
    if (((uintptr_t)Q | (uintptr_t)out) & 15) return DENDRITE_EINVAL;
    if ((int64_t)n * q_len * n_q_heads >= INT32_MAX / 2) return DENDRITE_ELIMIT;
    for (int32_t i = 0; i < n; ++i) {
        DENDRITE_TRY(check_live(p, branches[i]));
        if (p->br[branches[i]].len < q_len) return DENDRITE_EINVAL;
    }
    {
        std::vector<int32_t> s(branches, branches + n);
        std::sort(s.begin(), s.end());
        if (std::adjacent_find(s.begin(), s.end()) != s.end()) return DENDRITE_EINVAL;
    }
    cudaStream_t s = (cudaStream_t)stream;
    // the whole call's device work, plan upload and expansion included (its
    // events start after the host has built the plan)
    bool began = false;
    const int max_ctas = p->sm_count * p->attn_ctas_per_sm;
    PlanCache& pc = p->plan;
    const bool same_query = pc.valid && pc.q_len == q_len && pc.n_q_heads == n_q_heads &&
                            (int32_t)pc.branches.size() == n && std::equal(branches, branches + n, pc.branches.begin());
    const bool hit = same_query && pc.version == p->version;
    // Only appends since the plan was built, and no queried branch reached a
    // new block: the segments, units and partition are unchanged, and only
    // the members' lengths (their rows' visibility limits) need refreshing.
    // Appends alone, and some queried branches reached new blocks: when each
    // of those branches' last segment is its own (read by it alone, ending at
    // its last block), the segments stay as they are but for those segments'
    // lengths, and only the units, partition and paths are rebuilt.
    const bool appends_only = !hit && same_query && pc.shape_version == p->shape_version;
    bool refresh = appends_only, grow = appends_only;
    for (int32_t i = 0; appends_only && i < n; ++i) {
        const int32_t nb = (p->br[branches[i]].len + p->block_size - 1) / p->block_size;
        if (nb == pc.n_blocks[i]) continue;
        refresh = false;
        if (nb < pc.n_blocks[i] || (pc.last_seg[i] < 0 && pc.last_xt[i] < 0)) grow = false;
    }
    grow = grow && !refresh;
    if (refresh) {
        const auto t0 = std::chrono::steady_clock::now();
        const int ib = p->plan_buf;
        p->plan_buf ^= 1;
        DENDRITE_CUDA(cudaEventSynchronize(p->plan_copied[ib]));
        if (ib != pc.buf) std::memcpy(p->h_plan[ib], p->h_plan[pc.buf], pc.upload_bytes);
        AttnMember* m = reinterpret_cast<AttnMember*>(p->h_plan[ib] + pc.members_off);
        for (int32_t e = 0; e < pc.n_members; ++e) m[e].len = p->br[branches[m[e].qi]].len;
        {
            const int64_t n16 = (int64_t)(pc.upload_bytes / 16);
            const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(64, (n16 + 255) / 256));
            prof_begin(p, T_ATTN_TOTAL, s);
            began = true;
            DENDRITE_CUDA(launch_pdl(k_plan_upload, dim3(grid), dim3(256), 0, s,
                                     reinterpret_cast<const uint4*>(p->h_plan[ib]),
                                     reinterpret_cast<uint4*>(p->d_plan[ib]), n16));
        }
        DENDRITE_CUDA(cudaEventRecord(p->plan_copied[ib], s));
        // the other device copy holds an older plan's units: expand again
        if (pc.device)
            DENDRITE_TRY(launch_plan_expand(p, p->d_plan[ib], pc.sec_off, pc.dev.n_units, pc.n_segplan, s));
        pc.dev = plan_rebase(pc.dev, p->d_plan[pc.buf], p->d_plan[ib]);
        pc.buf = ib;
        pc.version = p->version;
        pc.stats.refreshed = 1;
        pc.stats.plan_us = std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now() - t0).count();
    } else if (!hit) {
        const auto t0 = std::chrono::steady_clock::now();
        static thread_local HostPlan hp;
        hp.clear();
        if (grow) {
            hp.psegs = pc.segs;
            hp.seg_members = pc.seg_members;
            hp.unique_tiles = pc.unique_tiles;
            // extra tiles to add: d more blocks after tile last_xt[i], the
            // insertions in increasing position
            static thread_local std::vector<std::pair<int32_t, int32_t>> ins;
            ins.clear();
            for (int32_t i = 0; i < n; ++i) {
                const int32_t d = (p->br[branches[i]].len + p->block_size - 1) / p->block_size - pc.n_blocks[i];
                if (!d) continue;
                if (pc.last_seg[i] >= 0) hp.psegs[pc.last_seg[i]].block_count += d;
                else ins.emplace_back(pc.last_xt[i], d);
                hp.unique_tiles += (int64_t)d * p->n_kv;
            }
            if (ins.empty()) {
                hp.pxt = pc.seg_xt;
            } else {
                std::sort(ins.begin(), ins.end());
                hp.pxt.clear();
                size_t k = 0;
                for (int32_t x = 0; x < (int32_t)pc.seg_xt.size(); ++x) {
                    const ExtraTile e = pc.seg_xt[x];
                    hp.pxt.push_back(e);
                    for (; k < ins.size() && ins[k].first == x; ++k)
                        for (int32_t j = 1; j <= ins[k].second; ++j) hp.pxt.push_back(ExtraTile{e.rep_node, e.blk + j, e.mask});
                }
                // each packed segment's extra range moves by the tiles added before and inside it
                k = 0;
                int32_t added = 0;
                for (Segment& sg : hp.psegs) {   // extra ranges are in segment order
                    if (!sg.n_x) continue;
                    const int32_t end = sg.x_off + sg.n_x;
                    int32_t inside = 0;
                    for (; k < ins.size() && ins[k].first < end; ++k) inside += ins[k].second;
                    sg.x_off += added;
                    sg.n_x += inside;
                    added += inside;
                }
            }
            // a packed segment of the tcgen05 class holds at most
            // kMaxTcExtraTiles extra tiles (the kernel stages them in shared
            // memory): one grown past that is planned anew
            const int32_t rpm = q_len * (n_q_heads / p->n_kv);
            const bool tc_on = p->dtype == DENDRITE_BF16 && tc_ctas(p) > 0;
            for (const Segment& sg : hp.psegs)
                if (tc_on && sg.n_x > kMaxTcExtraTiles && (int64_t)sg.n_members * rpm > p->tc_min_rows) grow = false;
            if (!grow) hp.clear();
        }
        if (grow) {
            DENDRITE_TRY(build_units(p, branches, n, q_len, n_q_heads, max_ctas, tc_ctas(p), hp, true));
        } else {
            DENDRITE_TRY(build_plan(p, branches, n, q_len, n_q_heads, max_ctas, tc_ctas(p), hp, true));
        }
        size_t off[kPlanSections + 1];
        const size_t b = plan_layout(hp, off);
        DENDRITE_TRY(ensure_capacity(p, b, hp.partial_rows));
        // two pinned buffers in turn: this build only waits for the upload
        // of the build before the previous one
        const int ib = p->plan_buf;
        p->plan_buf ^= 1;
        DENDRITE_CUDA(cudaEventSynchronize(p->plan_copied[ib]));
        plan_pack(hp, off, p->h_plan[ib]);
        const size_t up_bytes = plan_upload_bytes(hp, off);
        {
            const int64_t n16 = (int64_t)(up_bytes / 16);
            const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(64, (n16 + 255) / 256));
            prof_begin(p, T_ATTN_TOTAL, s);
            began = true;
            DENDRITE_CUDA(launch_pdl(k_plan_upload, dim3(grid), dim3(256), 0, s,
                                     reinterpret_cast<const uint4*>(p->h_plan[ib]),
                                     reinterpret_cast<uint4*>(p->d_plan[ib]), n16));
        }
        DENDRITE_CUDA(cudaEventRecord(p->plan_copied[ib], s));
        if (hp.device) DENDRITE_TRY(launch_plan_expand(p, p->d_plan[ib], off, hp.hdr.n_units, hp.hdr.n_segs, s));
        pc.dev = plan_view(hp, off, p->d_plan[ib], n, q_len, n_q_heads, n_q_heads / p->n_kv);
        pc.n_partial_rows = hp.partial_rows;
        pc.valid = true;
        pc.device = hp.device;
        pc.n_segplan = hp.hdr.n_segs;
        pc.upload_bytes = up_bytes;
        for (int k = 0; k <= kPlanSections; ++k) pc.sec_off[k] = off[k];
        pc.version = p->version;
        pc.shape_version = p->shape_version;
        pc.buf = ib;
        pc.bytes = off[kPlanSections];
        pc.members_off = off[SEC_MEMBERS];
        pc.n_members = (int32_t)hp.members.size();
        pc.n_blocks.resize(n);
        for (int32_t i = 0; i < n; ++i) pc.n_blocks[i] = (p->br[branches[i]].len + p->block_size - 1) / p->block_size;
        pc.segs = hp.psegs;
        pc.seg_members = hp.seg_members;
        pc.seg_xt = hp.pxt;
        pc.unique_tiles = hp.unique_tiles;
        if (!grow) {   // grown segments still end at their branch's last block
            pc.last_seg.assign(n, -1);
            for (int32_t si = 0; si < (int32_t)hp.psegs.size(); ++si) {
                const Segment& sg = hp.psegs[si];
                if (sg.n_members != 1 || sg.n_x) continue;
                const int32_t m = hp.seg_members[sg.member_offset];
                if (sg.block_start + sg.block_count == pc.n_blocks[m]) pc.last_seg[m] = si;
            }
        }
        pc.last_xt.assign(n, -1);   // extra tiles move when a grow inserts some
        for (const Segment& sg : hp.psegs) {
            for (int32_t x = sg.x_off; x < sg.x_off + sg.n_x; ++x) {
                const ExtraTile& e = hp.pxt[x];
                if (e.mask & (e.mask - 1u)) continue;   // read by several members
                const int32_t m = hp.seg_members[sg.member_offset + __builtin_ctz(e.mask)];
                if (e.blk == pc.n_blocks[m] - 1) pc.last_xt[m] = x;
            }
        }
        pc.q_len = q_len;
        pc.n_q_heads = n_q_heads;
        pc.branches.assign(branches, branches + n);
        pc.stats.n_segments = (int32_t)hp.segs.size();
        pc.stats.n_units = (int32_t)hp.units.size();
        pc.stats.n_ctas = pc.dev.n_ctas;
        pc.stats.n_partials = (int32_t)hp.partial_rows;
        pc.stats.tiles = hp.tiles;
        pc.stats.unique_tiles = hp.unique_tiles;
        pc.stats.n_tc_units = hp.n_tc_units;
        pc.stats.n_tc_ctas = pc.dev.n_tc_ctas;
        pc.stats.refreshed = grow ? 2 : 0;
        pc.stats.plan_us = std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now() - t0).count();
    } else {
        pc.stats.refreshed = 0;
        pc.stats.plan_us = 0.0;
    }
    if (p->dtype == DENDRITE_TURBO) {   // rotated queries and their QJL projections
        const size_t rows = (size_t)n * q_len * n_q_heads;
        if (rows > p->tq_qs_rows) {
            const size_t cap = std::max<size_t>(rows * 3 / 2, 4096);
            DENDRITE_CUDA(cudaDeviceSynchronize());
            if (p->d_tq_qs) cudaFree(p->d_tq_qs);
            p->d_tq_qs = nullptr;
            p->tq_qs_rows = 0;
            DENDRITE_CUDA(cudaMalloc(&p->d_tq_qs, cap * 2 * kTurboDim * sizeof(float)));
            p->tq_qs_rows = cap;
        }
    }
    AttnArgs a = attn_args(p, layer, Q, out);
    a.plan = pc.dev;
    a.part_acc = p->d_partial;
    a.part_ml = reinterpret_cast<float2*>(p->d_partial + p->partial_rows_cap * p->head_dim);
    if (!began) prof_begin(p, T_ATTN_TOTAL, s);
    return launch_attention(p, layer, a, s);
}

extern "C" int dendrite_last_plan_stats(dendrite_pool* p, dendrite_plan_stats* out) {
    if (!p || !out) return DENDRITE_EINVAL;
    if (!p->plan.valid) return DENDRITE_EINVAL;
    PlanCache& pc = p->plan;
    if (pc.device) {   // the CTA counts and partial rows were computed on the device
        int32_t c[4];
        DENDRITE_CUDA(cudaSetDevice(p->device));
        DENDRITE_CUDA(cudaDeviceSynchronize());
        DENDRITE_CUDA(cudaMemcpy(c, p->d_plan[pc.buf] + pc.sec_off[SEC_COUNTS], sizeof(c), cudaMemcpyDeviceToHost));
        pc.stats.n_ctas = c[0];
        pc.stats.n_tc_ctas = c[1];
        pc.stats.n_partials = c[2];
    }
    *out = pc.stats;
    return DENDRITE_OK;
}

// ====================================================== allocation-free variant
// Some callers cannot let a library allocate device memory while they decode:
// a serving process that has handed nearly all free device memory to its own
// caching allocator (a cudaMalloc here could fail or fragment that reserve),
// a latency-critical decode loop that cannot afford the device-wide
// synchronisation cudaMalloc/cudaFree may imply, or a deployment that gives
// each library a fixed memory budget at load time.  For them,
// dendrite_tree_attn_decode_noalloc keeps its scratch -- the uploaded plan and
// the partial (max, sum, acc) rows -- in one file-scope device array of fixed
// size instead of the pool's grow-only workspace.  Every GPU that loads this
// library holds that array until the process exits.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(DENDRITE_NOALLOC_SCRATCH_BYTES);
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Host staging of the plan upload: plain host memory, so cudaMemcpyAsync has
// finished reading it when it returns and the next call may overwrite it.
// One buffer serves every thread and device, so packing a plan into it and
// handing it to cudaMemcpyAsync happen under g_noalloc_host_mu: two threads
// that each drive their own pool never upload each other's plans.
alignas(256) unsigned char g_noalloc_host[kNoAllocScratchBytes];
std::mutex g_noalloc_host_mu;

constexpr int kNoAllocMaxDevices = 64;
void* g_noalloc_dev[kNoAllocMaxDevices] = {};

// Device address of the scratch array on `device` (the current device).  In
// host code the array's name is only a host-side stand-in, so the address is
// looked up once per device, on that device's first call.
int noalloc_scratch(int device, unsigned char** out) {
    if (device < 0 || device >= kNoAllocMaxDevices) return DENDRITE_EINVAL;
    if (!g_noalloc_dev[device]) {
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_err(e);
        if (!ptr) return DENDRITE_ECUDA;
        g_noalloc_dev[device] = ptr;
    }
    *out = static_cast<unsigned char*>(g_noalloc_dev[device]);
    return DENDRITE_OK;
}

}  // namespace

extern "C" int dendrite_tree_attn_decode_noalloc(dendrite_pool* p, const void* Q, int32_t n_q_heads,
                                                 int32_t q_len, const int32_t* branches, int32_t n, void* out,
                                                 void* stream) {
    if (!p) return DENDRITE_EINVAL;
    if (p->dtype == DENDRITE_TURBO) return DENDRITE_EDTYPE;   // needs the pool's query workspace
    if (p->poisoned) return p->poisoned;
    if (p->pending.active && !p->pending.layer_done[0]) return DENDRITE_EINVAL;
    DENDRITE_CUDA(cudaSetDevice(p->device));
    if (!Q || !out || !branches || n <= 0 || q_len <= 0 || n_q_heads <= 0) return DENDRITE_EINVAL;
    if (n_q_heads % p->n_kv) return DENDRITE_EINVAL;
    if (((uintptr_t)Q | (uintptr_t)out) & 15) return DENDRITE_EINVAL;
    if ((int64_t)n * q_len * n_q_heads >= INT32_MAX / 2) return DENDRITE_ELIMIT;
    static thread_local std::vector<uint8_t> seen;
    seen.assign(p->max_branches, 0);
    for (int32_t i = 0; i < n; ++i) {
        DENDRITE_TRY(check_live(p, branches[i]));
        if (p->br[branches[i]].len < q_len) return DENDRITE_EINVAL;
        if (seen[branches[i]]) return DENDRITE_EINVAL;
        seen[branches[i]] = 1;
    }
    cudaStream_t s = (cudaStream_t)stream;
    // a captured copy from the pageable host buffer would read it only when
    // the graph is replayed, after later calls have rewritten it
    cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &capturing) != cudaSuccess || capturing != cudaStreamCaptureStatusNone)
        return DENDRITE_EINVAL;
    unsigned char* scratch = nullptr;
    DENDRITE_TRY(noalloc_scratch(p->device, &scratch));
    static thread_local HostPlan hp;
    hp.clear();
    DENDRITE_TRY(build_plan(p, branches, n, q_len, n_q_heads, p->sm_count * p->attn_ctas_per_sm, tc_ctas(p), hp,
                            false));
    // scratch layout: plan sections, then partial acc rows, then partial (m, l)
    size_t off[kPlanSections + 1];
    const size_t b = plan_layout(hp, off);
    const size_t plan_bytes = (b + 255) & ~size_t(255);
    const size_t acc_bytes = hp.partial_rows * p->head_dim * sizeof(float);
    const size_t ml_bytes = hp.partial_rows * sizeof(float2);
    if (plan_bytes + acc_bytes + ml_bytes > kNoAllocScratchBytes) return DENDRITE_ELIMIT;
    prof_begin(p, T_ATTN_TOTAL, s);
    {
        std::lock_guard<std::mutex> lock(g_noalloc_host_mu);
        plan_pack(hp, off, reinterpret_cast<char*>(g_noalloc_host));
        DENDRITE_CUDA(cudaMemcpyAsync(scratch, g_noalloc_host, off[kPlanSections], cudaMemcpyHostToDevice, s));
    }
    AttnArgs a = attn_args(p, 0, Q, out);
    a.plan = plan_view(hp, off, reinterpret_cast<const char*>(scratch), n, q_len, n_q_heads, n_q_heads / p->n_kv);
    a.part_acc = reinterpret_cast<float*>(scratch + plan_bytes);
    a.part_ml = reinterpret_cast<float2*>(scratch + plan_bytes + acc_bytes);
    return launch_attention(p, 0, a, s);
}

// ====================================================== bounded-wait self-test
// One thread waits on an mbarrier that nothing arrives at, through the same
// bounded wait the attention kernels use.  The wait gives up after its time
// limit and the pool records DENDRITE_ETIMEOUT; the device itself never
// faults or hangs.
namespace {

__global__ void k_wait_selftest(DevMeta* meta) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(smem_u32(&bar), 0, &abort_flag))
        atomicCAS(&meta->status, 0, DENDRITE_ETIMEOUT);
}

}  // namespace

extern "C" int dendrite_selftest_bounded_wait(dendrite_pool* p, void* stream) {
    if (!p) return DENDRITE_EINVAL;
    if (p->poisoned) return p->poisoned;
    DENDRITE_CUDA(cudaSetDevice(p->device));
    k_wait_selftest<<<1, 32, 0, (cudaStream_t)stream>>>(p->d_meta);
    DENDRITE_CUDA(cudaGetLastError());
    return DENDRITE_OK;
}

