// Tensor-core (tcgen05) partial kernel for attention units of many query rows.
//
// A shared-prefix segment read by R query rows per KV head is a dense
// contraction of R rows against the segment's keys and values: R flops per
// byte of K + V.  Beyond about 64 rows the mma.sync kernel (16-row tiles,
// accumulators in registers) is bound by its tensor and softmax issue rate,
// not by HBM.  This kernel takes those units (up to 256 rows: two row tiles
// of 128) and runs both products on the fifth-generation tensor cores with
// the accumulators in tensor memory (TMEM):
//
//   S_r = Q_r K^T   M = 128 rows, N = 16..64 tokens, K = head_dim 128
//   O_r += P_r V    M = 128 rows, N = head_dim 128,  K = 16..64 tokens
//
// P_r is never staged in shared memory: the softmax writes it (bf16, two per
// 32-bit column) over the S buffer it was computed from, and the P V
// product reads its A operand from tensor memory.  Each row tile has two S/P
// buffers, so the softmax of stage k + 1 writes its P while P V of stage k
// still runs; an S buffer is reused for stage k + 2 once P V of stage k,
// which read P from it, has completed.
//
// Warp roles (448 threads, one CTA per SM):
//   warps 0, 11 TMA producers: stream 64-token stages (4 blocks of 16 tokens)
//               of K and of V into two 4-stage rings, block ids fetched 32
//               tiles at a time.
//   warps 1, 12 TMEM owner (warp 1); lane 0 issues the S MMAs of row tile
//               0 (warp 1) or 1 (warp 12) and their commits.
//   warps 10, 13 lane 0 issues the P V MMAs of row tile 0 or 1.
//   warps 2-9   softmax, one query row per thread (warps 2-5 row tile 0,
//               warps 6-9 row tile 1): read the row of S from TMEM, mask,
//               exponentiate (base 2), write P (bf16) back into the first 32
//               columns of the same S buffer, keep (m, l).
// TMEM (512 columns): row tile r holds O_r in columns [256 r, 256 r + 128)
// and two S/P buffers of 64 columns after it, so the MMA of S for the next
// stage overlaps the softmax of this one and P V of the previous one.
//
// Online softmax with a lazy reference: each row keeps a reference max m and
// rescales O (a TMEM read-modify-write) only when a stage's max exceeds m by
// more than 8 (base-2 units), so P <= 2^8 and the fp32 accumulators stay far
// from overflow; (m, l, O) is a valid partial for any reference m, so the
// log-sum-exp merge is unchanged.  P is rounded to bf16 before the MMA and
// the row sum l is taken over the rounded values, as in the mma.sync kernel.
//
// Work split: the plan's tensor-core class has its own tile list and CTA
// partition; a CTA walks its tile range unit by unit and writes one partial
// (m, l, acc) per row of every unit chunk it processed.
//
// Every mbarrier wait is bounded (about 2 s of %globaltimer).  On expiry the
// CTA records DENDRITE_ETIMEOUT, every role stops issuing work, the MMA warp
// waits (bounded) for its issued MMAs and the producer for its copies in
// flight, and the TMEM is freed before the CTA exits.
#include "attn_common.cuh"

using namespace dendrite;

namespace {

constexpr int TC_NSTAGE = 4;
constexpr int TC_TOK = 64;                                   // tokens per stage (4 blocks)
constexpr int TC_HALF = TC_TOK * 128;                        // 64 tokens x 64 columns bf16 = 8 KiB
constexpr int TC_RING_STAGE = 2 * TC_HALF;                   // K (or V) of a stage: half 0, half 1
constexpr int TC_QTILE = 128 * D * 2;                        // 128 rows x 128 columns bf16 = 32 KiB
constexpr int TC_ROWTILES = 2;
constexpr int TC_SOFTMAX_WARP0 = 2;
constexpr int TC_PV_WARP = TC_SOFTMAX_WARP0 + 4 * TC_ROWTILES;   // 10
constexpr int TC_V_WARP = TC_PV_WARP + 1;                          // 11
constexpr int TC_S1_WARP = TC_V_WARP + 1;                          // 12
constexpr int TC_PV1_WARP = TC_S1_WARP + 1;                        // 13
constexpr int TC_THREADS = (TC_PV1_WARP + 1) * 32;
// K ring, then V ring: each TC_NSTAGE stages of 64 tokens
constexpr int OFF_K = 0;
constexpr int OFF_V = TC_NSTAGE * TC_RING_STAGE;
constexpr int OFF_Q = 2 * TC_NSTAGE * TC_RING_STAGE;
constexpr int OFF_BAR = OFF_Q + TC_ROWTILES * TC_QTILE;
// mbarriers; S/P buffers are indexed 2 r + b (row tile r, buffer b):
// S_FULL when S is in the buffer, P_FULL when P overwrote it, PV_DONE when
// the P V product that read that P has completed (the buffer is free again)
enum {
    B_K_FULL = 0,
    B_K_EMPTY = B_K_FULL + TC_NSTAGE,
    B_V_FULL = B_K_EMPTY + TC_NSTAGE,
    B_V_EMPTY = B_V_FULL + TC_NSTAGE,
    B_S_FULL = B_V_EMPTY + TC_NSTAGE,
    B_P_FULL = B_S_FULL + 4,
    B_PV_DONE = B_P_FULL + 4,
    B_Q_FULL = B_PV_DONE + 4,
    B_FINAL = B_Q_FULL + 2,   // one per issuer: S0, PV0, S1, PV1
    B_COUNT = B_FINAL + 4
};
// a packed unit's extra tiles (logical block, member mask), per row tile
constexpr int OFF_XINFO = OFF_BAR + B_COUNT * 8 + 16;
constexpr int SMEM_TC = 1024 + OFF_XINFO + TC_ROWTILES * kMaxTcExtraTiles * 8;
static_assert(SMEM_TC <= 227 * 1024, "shared memory budget");
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_THRESHOLD = 8.f;

// ------------------------------------------------------------- tcgen05 helpers
// Shared-memory matrix descriptor, 128-byte swizzle: start >> 4 in bits
// [0, 14), leading byte offset >> 4 in [16, 30), stride byte offset >> 4 in
// [32, 46), descriptor version 1 at bit 46, swizzle mode 2 (128 B) at [61, 64).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | (uint64_t)((lbo >> 4) & 0x3FFF) << 16 |
           (uint64_t)((sbo >> 4) & 0x3FFF) << 32 | (uint64_t)1 << 46 | (uint64_t)2 << 61;
}
// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B,
// A/B major-ness (0 = K-major, 1 = MN-major), N >> 3, M >> 4.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)acc)
        : "memory");
}
// The same with A (M x K, two bf16 per 32-bit column, row i in lane i) read
// from tensor memory at a_tmem.
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"((uint32_t)acc)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
// 2^x by the SFU (PTX ex2.approx.ftz.f32: relative error about 2^-22,
// results below 2^-126 flushed to zero; 2^-inf = +0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

#define TC_R8(i) "=r"(v[i]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3]), \
                 "=r"(v[i + 4]), "=r"(v[i + 5]), "=r"(v[i + 6]), "=r"(v[i + 7])
#define TC_W8(i) "r"(v[i]), "r"(v[i + 1]), "r"(v[i + 2]), "r"(v[i + 3]), \
                 "r"(v[i + 4]), "r"(v[i + 5]), "r"(v[i + 6]), "r"(v[i + 7])

// 32 consecutive fp32 columns of this thread's TMEM lane (32x32b shape).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : TC_R8(0), TC_R8(8), TC_R8(16), TC_R8(24)
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        TC_W8(0), TC_W8(8), TC_W8(16), TC_W8(24)
        : "memory");
}
#define TC_RW8(i) "+r"(v[i]), "+r"(v[i + 1]), "+r"(v[i + 2]), "+r"(v[i + 3]), \
                  "+r"(v[i + 4]), "+r"(v[i + 5]), "+r"(v[i + 6]), "+r"(v[i + 7])
// Wait for this thread's tcgen05.ld results.  The registers pass through the
// statement so that no use of them is scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&v)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : TC_RW8(0), TC_RW8(8), TC_RW8(16), TC_RW8(24)::"memory");
}
// Orders later uses of v after the preceding statement (a wait issued for
// several loads at once).
__device__ __forceinline__ void reg_tie(uint32_t (&v)[32]) {
    asm volatile("" : TC_RW8(0), TC_RW8(8), TC_RW8(16), TC_RW8(24));
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait by one thread; on failure marks the CTA aborted and records
// DENDRITE_ETIMEOUT (a no-op when another error is already recorded).
__device__ __forceinline__ bool thread_wait(uint32_t bar, uint32_t parity, volatile int* abortp, DevMeta* meta) {
    if (mbar_test(bar, parity)) return true;   // usually complete already
    if (*abortp) return false;
    if (mbar_wait(bar, parity, abortp)) return true;
    *abortp = 1;
    atomicCAS(&meta->status, 0, DENDRITE_ETIMEOUT);
    return false;
}
// Bounded wait by a whole warp; the result is the same in every lane.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abortp, DevMeta* meta) {
    bool ok = !*abortp && mbar_wait(bar, parity, abortp);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && (threadIdx.x & 31) == 0 && !*abortp) {
        *abortp = 1;
        atomicCAS(&meta->status, 0, DENDRITE_ETIMEOUT);
    }
    return ok;
}
// Wait without an abort exit, used only to drain work already issued.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity) && globaltimer() - t0 < WAIT_LIMIT_NS) {
    }
}

__global__ void __launch_bounds__(TC_THREADS, 1)
k_attn_partial_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const AttnArgs a) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ int abort_flag;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* sm = smem_raw + (base - raw);
    const uint32_t bars = base + OFF_BAR;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + B_COUNT * 8);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [bars](int i) { return bars + 8u * (uint32_t)i; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < TC_NSTAGE; ++s) {
            mbar_init(bar(B_K_FULL + s), 1);
            mbar_init(bar(B_K_EMPTY + s), 2);    // both S issuers (row tiles 0 and 1)
            mbar_init(bar(B_V_FULL + s), 1);
            mbar_init(bar(B_V_EMPTY + s), 2);    // both PV issuers
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(bar(B_S_FULL + i), 1);
            mbar_init(bar(B_P_FULL + i), 4);     // the row tile's four softmax warps
            mbar_init(bar(B_PV_DONE + i), 1);
        }
        for (int r = 0; r < TC_ROWTILES; ++r) mbar_init(bar(B_Q_FULL + r), 4);
        for (int i = 0; i < 4; ++i) mbar_init(bar(B_FINAL + i), 1);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    pdl_trigger();
    if (a.plan.counts && (int32_t)blockIdx.x >= a.plan.counts[1]) return;   // past the device-expanded split
    if (threadIdx.x == 0) {
        abort_flag = a.meta->status != 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (abort_flag) return;
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const AttnPlanDev& pl = a.plan;
    const int c = blockIdx.x;
    const int32_t t_begin = pl.tc_cta_begin[c], t_end = pl.tc_cta_begin[c + 1];
    const int32_t u0 = pl.tc_cta_unit[c];
    volatile int* abortp = &abort_flag;

    if (warp == 0 || warp == TC_V_WARP) {
        // ------------------------------------------------------ producers
        // Warp 0 streams K into the K ring, warp 11 V into the V ring, so a
        // K slot is refilled as soon as its S is done and a V slot as soon as
        // its P V is done.  Lane i < ntiles issues tile i of the stage: two
        // 64-column halves at token offset 16 i of the stage's two 8 KiB halves.
        const bool k_role = warp == 0;
        const CUtensorMap* tmap = k_role ? &tmK : &tmV;
        const uint32_t ring = base + (k_role ? OFF_K : OFF_V);
        const int b_full = k_role ? B_K_FULL : B_V_FULL, b_empty = k_role ? B_K_EMPTY : B_V_EMPTY;
        uint32_t issued = 0, parity_bits = 0;
        int32_t g = 0;
        int32_t t = t_begin, u = u0;
        while (t < t_end && !*abortp) {
            const AttnUnit U = pl.units[u];
            const int32_t uend = U.tile_off + U.n_blk;
            if (t >= uend) { ++u; continue; }
            const int32_t cend = min(t_end, uend);
            const int32_t* trow = a.table + (int64_t)U.table_row * a.bpb + U.blk_start - U.tile_off;
            // block id of tile t: from the unit's table row, or for a packed
            // unit's extra tile through its entry in the plan
            auto blk_at = [&](int32_t tt) -> int32_t {
                const int32_t ti = tt - U.tile_off;
                if (ti < U.n_shared) return trow[tt];
                const AttnXTile e = pl.xtiles[U.x_off + ti - U.n_shared];
                return a.table[(int64_t)e.table_row * a.bpb + e.blk];
            };
            // block ids, 32 tiles per batch, the next batch loaded one batch ahead
            int32_t cur_base = t, nxt_base = t + 32;
            int32_t cur = t + lane < cend ? blk_at(t + lane) : 0;
            int32_t nxt = nxt_base + lane < cend ? blk_at(nxt_base + lane) : 0;
            for (int32_t st = t; st < cend; st += 4, ++g) {
                if (st >= cur_base + 32) {
                    cur = nxt;
                    cur_base = nxt_base;
                    nxt_base += 32;
                    nxt = nxt_base + lane < cend ? blk_at(nxt_base + lane) : 0;
                }
                int32_t blk = __shfl_sync(0xffffffffu, cur, (st - cur_base) + (lane & 3));
                const int slot = g % TC_NSTAGE;
                const uint32_t ph = (uint32_t)(g / TC_NSTAGE) & 1u;
                const int ntiles = min(4, cend - st);
                int ok = 1;
                if (lane == 0) ok = thread_wait(bar(b_empty + slot), ph ^ 1u, abortp, a.meta);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (lane == 0) mbar_expect_tx(bar(b_full + slot), (uint32_t)(ntiles * 2 * HALF_BYTES));
                __syncwarp();
                if (lane < ntiles) {
                    if ((uint32_t)blk >= (uint32_t)a.n_blocks) {   // broken table: poison, read zeros
                        atomicCAS(&a.meta->status, 0, DENDRITE_ECORRUPT);
                        blk = -1;
                    }
                    const int32_t row0 = (blk * a.n_kv + U.kv_head) * BS;
                    const uint32_t dst = ring + slot * TC_RING_STAGE + lane * HALF_BYTES;
                    const uint32_t fb = bar(b_full + slot);
                    tma_load_3d(dst, tmap, 0, 0, row0, fb);
                    tma_load_3d(dst + TC_HALF, tmap, 0, 1, row0, fb);
                }
                issued |= 1u << slot;
                parity_bits = (parity_bits & ~(1u << slot)) | (ph << slot);
            }
            t = cend;
            ++u;
        }
        if (lane == 0 && *abortp) {   // copies still in flight land before the CTA exits
            for (int s = 0; s < TC_NSTAGE; ++s)
                if (issued >> s & 1u) drain_wait(bar(b_full + s), parity_bits >> s & 1u);
        }
    } else if (warp == 1 || warp == TC_PV_WARP || warp == TC_S1_WARP || warp == TC_PV1_WARP) {
        // ------------------------------------------------------ MMA issuers
        // Four single-thread issuers, one chain of waits each: for row tile
        // r, an S issuer (warp 1 for r = 0, warp 12 for r = 1) issues
        // S_r(k) = Q_r K^T as soon as stage k's K landed and the P V of
        // stage k - 2, which read the buffer S_r(k) overwrites, completed;
        // a PV issuer (warp 10, warp 13) issues O_r += P_r V as soon as stage
        // k's V landed and P_r(k) is in tensor memory.  A ring
        // slot goes back to its producer once both issuers of its kind have
        // committed it; the issuer of a row tile a unit does not have simply
        // arrives.
        const bool s_role = warp == 1 || warp == TC_S1_WARP;
        const int my_r = (warp == 1 || warp == TC_PV_WARP) ? 0 : 1;
        if (lane == 0) {
            const uint32_t sQ = base + OFF_Q + my_r * TC_QTILE;
            int32_t g = 0, js = 0, qc = 0;
            bool ok = true, any = false;
            int32_t t = t_begin, u = u0;
            while (ok && t < t_end) {
                const AttnUnit U = pl.units[u];
                const int32_t uend = U.tile_off + U.n_blk;
                if (t >= uend) { ++u; continue; }
                const int32_t cend = min(t_end, uend);
                const bool active = my_r < U.rt;
                const int32_t nst = (cend - t + 3) >> 2;
                if (s_role && active) ok = thread_wait(bar(B_Q_FULL + my_r), (uint32_t)qc++ & 1u, abortp, a.meta);
                for (int32_t k = 0; k < nst && ok; ++k) {
                    const int32_t gg = g + k;
                    const int slot = gg % TC_NSTAGE;
                    const uint32_t ph = (uint32_t)(gg / TC_NSTAGE) & 1u;
                    const int ntiles = min(4, cend - (t + 4 * k));
                    if (s_role) {
                        ok = thread_wait(bar(B_K_FULL + slot), ph, abortp, a.meta);
                        if (ok && active) {
                            const int b = js & 1;
                            ok = thread_wait(bar(B_PV_DONE + 2 * my_r + b), ((uint32_t)(js >> 1) & 1u) ^ 1u, abortp,
                                             a.meta);
                            if (!ok) break;
                            tc_fence_after();
                            const uint32_t stage = base + OFF_K + slot * TC_RING_STAGE;
                            const uint32_t id = idesc_bf16(128, 16 * ntiles, 0, 0);
                            const uint32_t dS = tmem + my_r * 256 + 128 + b * 64;
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint32_t qoff = (kk >> 2) * 16384 + (kk & 3) * 32;
                                const uint32_t koff = (kk >> 2) * TC_HALF + (kk & 3) * 32;
                                umma_bf16(dS, sdesc(sQ + qoff, 16, 1024), sdesc(stage + koff, 16, 1024), id, kk > 0);
                            }
                            umma_commit(bar(B_S_FULL + 2 * my_r + b));
                            umma_commit(bar(B_K_EMPTY + slot));
                            ++js;
                            any = true;
                        } else if (ok) {
                            mbar_arrive(bar(B_K_EMPTY + slot));
                        }
                    } else {
                        ok = thread_wait(bar(B_V_FULL + slot), ph, abortp, a.meta);
                        if (ok && active) {
                            const int b = js & 1;
                            ok = thread_wait(bar(B_P_FULL + 2 * my_r + b), (uint32_t)(js >> 1) & 1u, abortp, a.meta);
                            if (!ok) break;
                            tc_fence_after();
                            const uint32_t vst = base + OFF_V + slot * TC_RING_STAGE;
                            const uint32_t id = idesc_bf16(128, 128, 0, 1);
                            const uint32_t tP = tmem + my_r * 256 + 128 + b * 64;   // 16 tokens per 8 columns
                            for (int kk = 0; kk < ntiles; ++kk)
                                umma_bf16_ta(tmem + my_r * 256, tP + kk * 8, sdesc(vst + kk * 2048, TC_HALF, 1024), id,
                                             kk > 0 || k > 0);
                            umma_commit(bar(B_PV_DONE + 2 * my_r + b));
                            umma_commit(bar(B_V_EMPTY + slot));
                            ++js;
                            any = true;
                        } else if (ok) {
                            mbar_arrive(bar(B_V_EMPTY + slot));
                        }
                    }
                }
                g += nst;
                t = cend;
                ++u;
            }
            if (any) {   // every MMA this thread issued has finished before the TMEM is freed
                const uint32_t fb = bar(B_FINAL + (s_role ? 0 : 1) + 2 * my_r);
                umma_commit(fb);
                drain_wait(fb, 0);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ softmax
        const int r = (warp - TC_SOFTMAX_WARP0) >> 2;
        const int sub = warp & 3;                 // TMEM lanes 32 sub .. 32 sub + 31
        const int trow = sub * 32 + lane;         // row within the row tile
        const uint32_t tl = tmem + ((uint32_t)(sub * 32) << 16) + r * 256;
        unsigned char* sQ = sm + OFF_Q + r * TC_QTILE;
        const __nv_bfloat16* Q = static_cast<const __nv_bfloat16*>(a.Q);
        const int row = r * 128 + trow;
        int2* xinfo = reinterpret_cast<int2*>(sm + OFF_XINFO) + r * kMaxTcExtraTiles;
        // This thread's row of a unit's Q into the K-major swizzled tile, and
        // the row's record.  A unit's Q is staged as soon as the previous
        // chunk's last S was read (no S MMA of it is pending then), before
        // that chunk's epilogue, so the next chunk's S overlaps the epilogue.
        auto stage_q = [&](const AttnUnit& V) -> AttnRow {
            const bool v_ok = row < V.n_rows;
            const AttnRow RR = v_ok ? unit_row(pl, V, row) : AttnRow{0, 0};
            const uint4* q = reinterpret_cast<const uint4*>(Q + (int64_t)RR.q_row * D);
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
                const uint4 v = v_ok ? __ldg(q + ch) : make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(sQ + (ch >> 3) * 16384 + trow * 128 + (((ch & 7) ^ (trow & 7)) << 4)) = v;
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_Q_FULL + r));
            return RR;
        };
        int32_t js = 0;
        bool ok = true;
        int32_t t = t_begin, u = u0;
        int32_t staged_u = -1;      // unit whose Q is already in the tile
        AttnRow staged_R{0, 0};
        while (ok && t < t_end) {
            const AttnUnit U = pl.units[u];
            const int32_t uend = U.tile_off + U.n_blk;
            if (t >= uend) { ++u; continue; }
            const int32_t cend = min(t_end, uend);
            if (r >= U.rt) {
                t = cend;
                ++u;
                continue;
            }
            const bool valid = row < U.n_rows;
            const AttnRow R = staged_u == u ? staged_R : stage_q(U);
            if (U.n_blk > U.n_shared) {
                // a packed unit: its extra tiles' logical blocks and member
                // masks into shared memory, once every warp of the row tile
                // is done with the previous unit's (the plan keeps them to
                // kMaxTcExtraTiles; a unit past that reads none and is flagged)
                const int32_t nx = U.n_blk - U.n_shared;
                if (nx > kMaxTcExtraTiles && trow == 0) atomicCAS(&a.meta->status, 0, DENDRITE_ECORRUPT);
                asm volatile("bar.sync %0, 128;" ::"r"(1 + r) : "memory");
                for (int32_t i = trow; i < min(nx, kMaxTcExtraTiles); i += 128)
                    xinfo[i] = *reinterpret_cast<const int2*>(pl.xtiles + U.x_off + i);
                asm volatile("bar.sync %0, 128;" ::"r"(1 + r) : "memory");
            }
            const int32_t nst = (cend - t + 3) >> 2;
            float m_ref = -INFINITY, l = 0.f;
            for (int32_t k = 0; k < nst && ok; ++k, ++js) {
                const int32_t st = t + 4 * k;
                const int ntiles = min(4, cend - st);
                const int b = js & 1;
                ok = warp_wait(bar(B_S_FULL + 2 * r + b), (uint32_t)(js >> 1) & 1u, abortp, a.meta);
                if (!ok) break;
                tc_fence_after();
                float s[64];
                {
                    uint32_t v0[32], v1[32];
                    tmem_ld32(tl + 128 + b * 64, v0);
                    tmem_ld32(tl + 128 + b * 64 + 32, v1);
                    tmem_wait_ld(v0);
                    reg_tie(v1);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        s[i] = __uint_as_float(v0[i]);
                        s[32 + i] = __uint_as_float(v1[i]);
                    }
                }
                // mask stage columns past the chunk and positions the row does
                // not see (only stages some row of the warp does not fully see)
                const int32_t ti0 = st - U.tile_off;
                if (ti0 + ntiles <= U.n_shared) {
                    const int32_t vis = min(ntiles * BS, R.limit - (U.blk_start + ti0) * BS);
                    if (!__all_sync(0xffffffffu, vis >= TC_TOK)) {
#pragma unroll
                        for (int i = 0; i < 64; ++i) s[i] = i < vis ? s[i] : -INFINITY;
                    }
                } else {
                    // a stage with a packed unit's extra tiles: each tile counts
                    // only for the rows of the members in its mask
                    const int32_t mi = div_rcp(U.row_lo + row, pl.q_len * pl.group, pl.rcp_rows_per_member);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int32_t tj = ti0 + j;
                        int32_t lb = U.blk_start + tj;
                        bool seen = j < ntiles;
                        if (seen && tj >= U.n_shared) {
                            const int2 e = xinfo[min(tj - U.n_shared, kMaxTcExtraTiles - 1)];
                            lb = e.x;
                            seen = ((uint32_t)e.y >> (mi & 31)) & 1u;
                        }
                        const int32_t v = seen ? min(BS, R.limit - lb * BS) : 0;
#pragma unroll
                        for (int c = 0; c < BS; ++c) s[BS * j + c] = c < v ? s[BS * j + c] : -INFINITY;
                    }
                }
                // row max of the raw scores (eight independent chains), then
                // in base-2 units (the scale is positive)
                float mx;
                {
                    float m8[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) m8[j] = s[j];
#pragma unroll
                    for (int i = 8; i < 64; ++i) m8[i & 7] = fmaxf(m8[i & 7], s[i]);
                    mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
                    mx *= a.scale_log2;
                }
                if (k == 0) {
                    m_ref = mx;   // this stage's PV overwrites O
                } else {
                    const bool need = mx > m_ref + RESCALE_THRESHOLD;
                    if (__any_sync(0xffffffffu, need)) {
                        // O holds the PV of the previous stage once it completes
                        ok = warp_wait(bar(B_PV_DONE + 2 * r + ((js - 1) & 1)), (uint32_t)((js - 1) >> 1) & 1u,
                                       abortp, a.meta);
                        if (!ok) break;
                        tc_fence_after();
                        const float alpha = need ? ex2_approx(m_ref - mx) : 1.f;
#pragma unroll 1
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t v[32];
                            tmem_ld32(tl + c0, v);
                            tmem_wait_ld(v);
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                            tmem_st32(tl + c0, v);
                        }
                        tmem_wait_st();
                        if (need) {
                            l *= alpha;
                            m_ref = mx;
                        }
                    }
                }
                // P = 2^(s * scale - m_ref) in bf16; the row sum is taken over
                // the rounded values (eight independent chains)
                const float nref = m_ref == -INFINITY ? 0.f : -m_ref;
                uint32_t pk[32];
                {
                    float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        pk[i] = pack_bf16(ex2_approx(fmaf(s[2 * i], a.scale_log2, nref)),
                                          ex2_approx(fmaf(s[2 * i + 1], a.scale_log2, nref)));
                        l8[(2 * i) & 7] += __uint_as_float(pk[i] << 16);
                        l8[(2 * i + 1) & 7] += __uint_as_float(pk[i] & 0xffff0000u);
                    }
                    l += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
                }
                // P over the S it came from (token 2 i in the low half of
                // column i); unused columns past the chunk hold P = 0
                tmem_st32(tl + 128 + b * 64, pk);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_P_FULL + 2 * r + b));
            }
            if (!ok) break;
            // the next chunk this row tile works on: stage its Q now
            {
                int32_t t2 = cend, u2 = u + 1;
                while (t2 < t_end) {
                    const AttnUnit& V = pl.units[u2];
                    const int32_t e2 = V.tile_off + V.n_blk;
                    if (t2 >= e2) { ++u2; continue; }
                    if (r < V.rt) break;
                    t2 = min(t_end, e2);
                    ++u2;
                }
                if (t2 < t_end) {
                    staged_R = stage_q(pl.units[u2]);
                    staged_u = u2;
                }
            }
            // chunk done: O after the last PV -> partial row
            ok = warp_wait(bar(B_PV_DONE + 2 * r + ((js - 1) & 1)), (uint32_t)((js - 1) >> 1) & 1u, abortp, a.meta);
            if (!ok) break;
            tc_fence_after();
            const int32_t prow = U.prow_base + (c - U.cfirst) * U.n_rows + row;
            float* dst = a.part_acc + (int64_t)(valid ? prow : 0) * D;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(tl + c0, v);
                tmem_wait_ld(v);
                if (valid) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<uint4*>(dst + c0 + i) = make_uint4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                }
            }
            if (valid) a.part_ml[prow] = make_float2(m_ref, l);
            tc_fence_before();
            t = cend;
            ++u;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
}

}  // namespace

namespace dendrite {

int attn_tc_setup() {
    if (cudaFuncSetAttribute(k_attn_partial_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TC) !=
        cudaSuccess)
        return DENDRITE_ECUDA;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_attn_partial_tc, TC_THREADS, SMEM_TC) != cudaSuccess ||
        occ != 1)
        return DENDRITE_ECUDA;   // the kernel's 512 TMEM columns need exactly one CTA per SM
    return DENDRITE_OK;
}

int launch_attn_tc(const CUtensorMap& mk, const CUtensorMap& mv, const AttnArgs& a, int n_ctas, cudaStream_t s) {
    k_attn_partial_tc<<<n_ctas, TC_THREADS, SMEM_TC, s>>>(mk, mv, a);
    return cudaGetLastError() == cudaSuccess ? DENDRITE_OK : DENDRITE_ECUDA;
}

}  // namespace dendrite
