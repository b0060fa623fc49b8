// Pieces shared by the attention kernels: the argument block every attention
// kernel receives, and the inline PTX wrappers (mbarrier, TMA, mma.sync,
// ldmatrix) they use.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "dendrite_internal.h"

namespace dendrite {

// Lets the next kernel in the stream, when launched as a programmatic
// dependent, start its prologue; it still waits (griddepcontrol.wait) for
// this whole grid to finish before it reads anything.  Every kernel of the
// library calls it only after its own griddepcontrol.wait, except the plan
// upload (see there), so when a kernel lets dependents launch, every kernel
// before it in the stream has finished.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Row r of unit U: segment row sr = row_lo + r belongs to member sr / (q_len G),
// query token j = (sr % (q_len G)) / G and head group g = sr % G; it reads the
// Q/out row (member, token, kv head, group) and sees positions
// < len - q_len + j + 1.
// The two divisions use the divisors' fp32 reciprocals (the host limits
// segment rows to 2^24, so sr converts exactly and the estimate is off by at
// most one, which one remainder test corrects): integer division by a
// run-time divisor would sit on the dependent chain from the unit record to
// the Q load.
__device__ __forceinline__ int32_t div_rcp(int32_t n, int32_t d, float rcp) {
    int32_t q = __float2int_rz(__int2float_rz(n) * rcp);
    const int32_t r = n - q * d;
    q += (r >= d) - (r < 0);
    return q;
}

__device__ __forceinline__ AttnRow unit_row(const AttnPlanDev& pl, const AttnUnit& U, int32_t r) {
    const int32_t G = pl.group, RM = pl.q_len * G;
    const int32_t sr = U.row_lo + r;
    const int32_t mi = div_rcp(sr, RM, pl.rcp_rows_per_member), rem = sr - mi * RM;
    const int32_t j = div_rcp(rem, G, pl.rcp_group), g = rem - j * G;
    const AttnMember M = pl.members[U.mem_off + mi];
    return AttnRow{(M.qi * pl.q_len + j) * pl.n_q_heads + U.kv_head * G + g, M.len - pl.q_len + j + 1, mi};
}

struct AttnArgs {
    AttnPlanDev plan;
    const void* Q;
    void* out;
    const int32_t* table;
    const float* pool_k;   // fp32 kernel
    const float* pool_v;
    float* part_acc;       // [partial rows][head_dim]
    float2* part_ml;       // [partial rows] (m, l)
    DevMeta* meta;
    int32_t bpb;
    int32_t n_kv;
    int32_t head_dim;
    int32_t n_blocks;
    float scale_log2;      // log2(e) / sqrt(head_dim)
    const float* tq_signs; // compressed pools: rotation signs [128] (the merge rotates rows back); else null
};

// Tensor-core (tcgen05) partial kernel for units of many query rows; see
// attn_tc.cu.  Units of the plan's tc class, CTAs [0, n_ctas).
int attn_tc_setup();
int launch_attn_tc(const CUtensorMap& mk, const CUtensorMap& mv, const AttnArgs& a, int n_ctas, cudaStream_t s);

}  // namespace dendrite

namespace {

using dendrite::AttnArgs;

constexpr int D = 128;
constexpr int BS = 16;
constexpr int HALF_BYTES = BS * 64 * 2;          // one 64-column half of a 16-token K or V tile
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;

// ------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: true when the phase with `parity` completed; false on
// timeout or when another role of the CTA already gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1; it < (1u << 30); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > WAIT_LIMIT_NS) return false;
        }
    }
    return false;
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
        "%4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16_pair_sum(uint32_t v) {
    return __uint_as_float(v << 16) + __uint_as_float(v & 0xffff0000u);
}
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Byte offset of element (token t, column d) inside one swizzled K or V tile:
// two 64-column halves of 16 rows x 128 bytes, 16-byte chunks XOR-ed with
// (row & 7) as TMA's 128-byte swizzle lays them out.
__device__ __forceinline__ uint32_t swz(int t, int d) {
    return (uint32_t)((d >> 6) * HALF_BYTES + t * 128 + ((((d & 63) >> 3) ^ (t & 7)) << 4) + (d & 7) * 2);
}

}  // namespace
