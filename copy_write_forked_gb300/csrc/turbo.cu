// Compressed KV blocks: TurboQuant rows (PolarQuant angle codes plus a one-bit
// QJL sketch of the key residual), encoded by the append and decoded inside
// the attention partial kernel.
//
// Method (dendrite demo.tape, section "TurboQuant": "TurboQuant KV
// compression (PolarQuant + QJL)"; the steps follow the published PolarQuant,
// QJL and TurboQuant methods the pages name):
//   - a row r (head_dim 128) is rotated, x = H (s * r) / sqrt(128) with H the
//     Walsh-Hadamard matrix and s the pool's random signs;
//   - the recursive polar transform turns x into 64 level-1 angles in
//     [0, 2 pi) (4-bit codes, 16 equal bins), 63 angles of levels 2..7 in
//     [0, pi/2] (3-bit codes, 8 equal bins of [pi/4 - w, pi/4 + w],
//     w = min(pi/4, 1.6 / sqrt(k - 1)) for halves of k = 2^(level-1)
//     coordinates) and the norm;
//   - a key also keeps sign(S e) (128 bits) and |e| for its residual
//     e = x - x_hat, S the pool's Gaussian 128 x 128 matrix, so that
//     <q', x> ~ <q', x_hat> + sqrt(pi/2)/128 |e| <S q', sign(S e)>.
// Records: value 64 bytes, key 96 bytes (layout below); attention runs in the
// rotated space and the merge rotates the output back.
//
// The encoder's decisions (bins, signs) are taken in fp32 with one rounded
// operation at a time (__fmul_rn / __fadd_rn / __fsqrt_rn, no contraction)
// in a fixed order, so the codes depend only on the input bits.
#include "attn_common.cuh"
#include "turbo.h"

#include <algorithm>
#include <cmath>

using namespace dendrite;

namespace {

struct TurboTables {
    float t1, t3;              // tan(pi/8), tan(3 pi/8): level-1 sub-bin boundaries
    float tan_up[6][7];        // levels 2..7: tangents of the 7 inner bin boundaries
    float cos1[16], sin1[16];  // level-1 bin centres
    float cos_up[6][8], sin_up[6][8];
};
__constant__ TurboTables c_tq;

constexpr int KREC = 96, VREC = 64;
constexpr unsigned FULL = 0xffffffffu;

__device__ __forceinline__ int tq_bin1(float a, float b) {
    if (a == 0.f && b == 0.f) return 0;
    int q;
    float x, y;
    if (a > 0.f && b >= 0.f) { q = 0; x = a; y = b; }
    else if (a <= 0.f && b > 0.f) { q = 1; x = b; y = -a; }
    else if (a < 0.f && b <= 0.f) { q = 2; x = -a; y = -b; }
    else { q = 3; x = -b; y = a; }
    const int sub = (y >= __fmul_rn(x, c_tq.t1)) + (y >= x) + (y >= __fmul_rn(x, c_tq.t3));
    return 4 * q + sub;
}

__device__ __forceinline__ int tq_bin2(float a, float b, int lv) {
    if (a == 0.f && b == 0.f) return 0;
    int c = 0;
#pragma unroll
    for (int k = 0; k < 7; ++k) c += b >= __fmul_rn(a, c_tq.tan_up[lv][k]);
    return c;
}

__device__ __forceinline__ float tq_radius(float a, float b) {
    return __fsqrt_rn(__fadd_rn(__fmul_rn(a, a), __fmul_rn(b, b)));
}

// PolarQuant of one rotated row held as x[4] per lane.  Lane l ends with the
// level-1 codes 2l, 2l+1 (returned in c1), the codes of the upper levels it
// holds (level L node j sits in lane j * 2^(L-2)) in cu[L-2] (-1 elsewhere),
// and lane 0 with the norm.
__device__ __forceinline__ void tq_polar_encode(const float (&x)[4], int lane, int& c1a, int& c1b, int (&cu)[6],
                                                float& norm) {
    c1a = tq_bin1(x[0], x[1]);
    c1b = tq_bin1(x[2], x[3]);
    const float r1a = tq_radius(x[0], x[1]), r1b = tq_radius(x[2], x[3]);
    // level 2: node l of lane l from (r1[2l], r1[2l+1])
    cu[0] = tq_bin2(r1a, r1b, 0);
    float r = tq_radius(r1a, r1b);
#pragma unroll
    for (int L = 3; L <= 7; ++L) {
        const int step = 1 << (L - 3);          // partner distance of the level-(L-1) holders
        const float o = __shfl_xor_sync(FULL, r, step);
        const bool holder = (lane & ((step << 1) - 1)) == 0;
        cu[L - 2] = holder ? tq_bin2(r, o, L - 2) : -1;
        r = holder ? tq_radius(r, o) : r;
    }
    norm = r;   // valid in lane 0
}

// The polar transform run backwards in fp32 (each product rounded), for the
// encoder's residual: x_hat[4] per lane from the norm (lane 0) and the codes
// laid out as tq_polar_encode leaves them.
__device__ __forceinline__ void tq_polar_decode32(float norm, int c1a, int c1b, const int (&cu)[6], int lane,
                                                  float (&xh)[4]) {
    float r = norm;   // holder of level 7: lane 0
#pragma unroll
    for (int L = 7; L >= 3; --L) {
        const int step = 1 << (L - 3);
        const bool holder = (lane & ((step << 1) - 1)) == 0;
        const int c = holder ? cu[L - 2] : 0;
        const float lo = __fmul_rn(r, c_tq.cos_up[L - 2][c]);
        const float hi = __fmul_rn(r, c_tq.sin_up[L - 2][c]);
        const float from = __shfl_xor_sync(FULL, hi, step);
        if (holder) r = lo;
        else if ((lane & ((step << 1) - 1)) == step) r = from;
    }
    // level 2 (lane l holds node l) into the two level-1 radii
    const float ra = __fmul_rn(r, c_tq.cos_up[0][cu[0]]);
    const float rb = __fmul_rn(r, c_tq.sin_up[0][cu[0]]);
    xh[0] = __fmul_rn(ra, c_tq.cos1[c1a]);
    xh[1] = __fmul_rn(ra, c_tq.sin1[c1a]);
    xh[2] = __fmul_rn(rb, c_tq.cos1[c1b]);
    xh[3] = __fmul_rn(rb, c_tq.sin1[c1b]);
}

// Writes the shared polar part of a record (64 bytes) into rec (words).
__device__ __forceinline__ void tq_pack_polar(uint32_t* rec, float norm, int c1a, int c1b, const int (&cu)[6],
                                              int lane) {
    // norm
    if (lane == 0) rec[0] = __float_as_uint(norm);
    // 64 level-1 nibbles: byte 4 + lane holds codes 2 lane (low) and 2 lane + 1
    const uint32_t byte = (uint32_t)(c1a & 15) | ((uint32_t)(c1b & 15) << 4);
    const uint32_t b1 = __shfl_down_sync(FULL, byte, 1), b2 = __shfl_down_sync(FULL, byte, 2),
                   b3 = __shfl_down_sync(FULL, byte, 3);
    if ((lane & 3) == 0) rec[1 + (lane >> 2)] = byte | (b1 << 8) | (b2 << 16) | (b3 << 24);
    // 63 three-bit codes of levels 2..7 (level order) in a little-endian bit
    // stream: level L node j is code (first index of L) + j
    uint32_t w[6] = {0, 0, 0, 0, 0, 0};
    const int first[6] = {0, 32, 48, 56, 60, 62};
#pragma unroll
    for (int L = 2; L <= 7; ++L) {
        const int c = cu[L - 2];
        if (c < 0) continue;
        const int j = lane >> (L - 2);
        const int p = 3 * (first[L - 2] + j);
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const int q = p + k;
            if ((c >> k) & 1) w[q >> 5] |= 1u << (q & 31);
        }
    }
#pragma unroll
    for (int k = 0; k < 6; ++k) {
        const uint32_t v = __reduce_or_sync(FULL, w[k]);
        if (lane == k) rec[9 + k] = v;
    }
    if (lane == 6) rec[15] = 0u;
}

// Encodes one row (x[4] per lane, the caller's values in fp32) into a value
// record (key == false) or a key record.
__device__ __forceinline__ void tq_encode_row(float (&x)[4], bool key, const float* __restrict__ signs,
                                              const float4* __restrict__ S4, uint32_t* rec, int lane) {
    const float4 sg = __ldg(reinterpret_cast<const float4*>(signs) + lane);
    x[0] = __fmul_rn(x[0], sg.x);
    x[1] = __fmul_rn(x[1], sg.y);
    x[2] = __fmul_rn(x[2], sg.z);
    x[3] = __fmul_rn(x[3], sg.w);
    tq_fwht(x, lane);
    const float inv = 0.0883883476483184405501055452631f;   // 1 / sqrt(128), rounded to fp32
#pragma unroll
    for (int k = 0; k < 4; ++k) x[k] = __fmul_rn(x[k], inv);
    int c1a, c1b, cu[6];
    float norm;
    tq_polar_encode(x, lane, c1a, c1b, cu, norm);
    tq_pack_polar(rec, norm, c1a, c1b, cu, lane);
    if (!key) return;
    float xh[4];
    tq_polar_decode32(norm, c1a, c1b, cu, lane, xh);
    float e[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) e[k] = __fsub_rn(x[k], xh[k]);
    // z_j = sum_i S[j][i] e_i in index order for j = 4 lane .. 4 lane + 3, and
    // |e|^2 in index order (lane 0's copy is kept)
    float z[4] = {0.f, 0.f, 0.f, 0.f}, n2 = 0.f;
#pragma unroll 1
    for (int src = 0; src < 32; ++src) {
        float ei[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) ei[k] = __shfl_sync(FULL, e[k], src);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 s = __ldg(S4 + (4 * lane + k) * 32 + src);
            z[k] = __fadd_rn(z[k], __fmul_rn(s.x, ei[0]));
            z[k] = __fadd_rn(z[k], __fmul_rn(s.y, ei[1]));
            z[k] = __fadd_rn(z[k], __fmul_rn(s.z, ei[2]));
            z[k] = __fadd_rn(z[k], __fmul_rn(s.w, ei[3]));
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) n2 = __fadd_rn(n2, __fmul_rn(ei[k], ei[k]));
    }
    const uint32_t nib = (uint32_t)(z[0] >= 0.f) | ((uint32_t)(z[1] >= 0.f) << 1) | ((uint32_t)(z[2] >= 0.f) << 2) |
                         ((uint32_t)(z[3] >= 0.f) << 3);
    // bit j = 4 lane + k at byte 64 + j / 8, bit j % 8: eight lanes per word
    uint32_t wv = nib << (4 * (lane & 7));
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) wv |= __shfl_xor_sync(FULL, wv, m);
    if ((lane & 7) == 0) rec[16 + (lane >> 3)] = wv;
    if (lane == 0) rec[20] = __float_as_uint(__fsqrt_rn(n2));
    if (lane >= 21 && lane < 24) rec[lane] = 0u;
}

// Unpacks the polar part of a record (words rec[0..15]) into the per-lane
// layout of tq_polar_encode: level-1 codes 2 lane, 2 lane + 1, the upper-level
// codes of the nodes this lane holds, the norm (every lane).
__device__ __forceinline__ void tq_unpack_polar(const uint32_t* rec, int lane, int& c1a, int& c1b, int (&cu)[6],
                                                float& norm) {
    norm = __uint_as_float(rec[0]);
    const uint32_t byte = (rec[1 + (lane >> 2)] >> (8 * (lane & 3))) & 0xFFu;
    c1a = (int)(byte & 15);
    c1b = (int)(byte >> 4);
    const int first[6] = {0, 32, 48, 56, 60, 62};
#pragma unroll
    for (int L = 2; L <= 7; ++L) {
        const bool holder = (lane & ((1 << (L - 2)) - 1)) == 0;
        const int j = lane >> (L - 2);
        const int q = 3 * (first[L - 2] + j);
        const uint64_t two = (uint64_t)rec[9 + (q >> 5)] | ((q >> 5) < 5 ? (uint64_t)rec[10 + (q >> 5)] << 32 : 0ull);
        cu[L - 2] = holder ? (int)((two >> (q & 31)) & 7u) : 0;
    }
}

// ------------------------------------------------------------------- append
// A grid of CTAs strides over the touched (branch, block, kv head) tiles of
// an append into a compressed pool, as the uncompressed copy kernel does; in
// each tile warp w takes slots w, w + 4, ...: slots before the new rows are
// copied record for record from a copied-on-write tail (nothing moves for an
// in-place tail), the others encode their new K row into a key record and V
// row into a value record.  args: branch[n], len[n], prefix of touched
// blocks per branch[n] (device); blockIdx.y selects the layer.
__global__ void __launch_bounds__(128) k_append_turbo(
    const int32_t* __restrict__ args, int32_t n, int32_t n_new, int32_t bs, int32_t bpb, int32_t n_kv,
    int32_t n_blocks, const int32_t* __restrict__ table, const int32_t* __restrict__ call,
    const __nv_bfloat16* __restrict__ Kin0, const __nv_bfloat16* __restrict__ Vin0, unsigned char* __restrict__ Kp0,
    unsigned char* __restrict__ Vp0, int64_t in_layer, int64_t kp_layer, int64_t vp_layer,
    const float* __restrict__ signs, const float* __restrict__ S, DevMeta* meta, int64_t n_tiles) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ uint32_t srec[4][40];   // per warp: a key record (24 words) and a value record (16)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const __nv_bfloat16* Kin = Kin0 + blockIdx.y * in_layer;
    const __nv_bfloat16* Vin = Vin0 + blockIdx.y * in_layer;
    unsigned char* Kp = Kp0 + blockIdx.y * kp_layer;
    unsigned char* Vp = Vp0 + blockIdx.y * vp_layer;
    const int32_t* cow_src = call + n;
    const float4* S4 = reinterpret_cast<const float4*>(S);
    if (meta->status) return;
    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int32_t h = (int32_t)(tile % n_kv);
        const int32_t t = (int32_t)(tile / n_kv);
        int32_t lo = 0, hi = n - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (args[2 * n + mid] <= t) lo = mid; else hi = mid - 1;
        }
        const int32_t i = lo;
        const int32_t L = args[n + i];
        const int32_t lblk = L / bs + (t - args[2 * n + i]);
        const int32_t s0 = lblk == L / bs ? L % bs : 0;
        const int32_t s1 = min(bs, L + n_new - lblk * bs);
        const int32_t dst = table[(int64_t)args[i] * bpb + lblk];
        const int32_t csrc = lblk == L / bs ? cow_src[i] : -1;
        if ((uint32_t)dst >= (uint32_t)n_blocks || csrc >= n_blocks) {
            if (threadIdx.x == 0) atomicCAS(&meta->status, 0, DENDRITE_ECORRUPT);
            return;
        }
        for (int32_t slot = warp; slot < s1; slot += 4) {
            uint4* kd = reinterpret_cast<uint4*>(Kp + (((int64_t)dst * n_kv + h) * bs + slot) * KREC);
            uint4* vd = reinterpret_cast<uint4*>(Vp + (((int64_t)dst * n_kv + h) * bs + slot) * VREC);
            if (slot < s0) {
                if (csrc < 0) continue;   // an in-place tail keeps its rows
                const uint4* ks = reinterpret_cast<const uint4*>(Kp + (((int64_t)csrc * n_kv + h) * bs + slot) * KREC);
                const uint4* vs = reinterpret_cast<const uint4*>(Vp + (((int64_t)csrc * n_kv + h) * bs + slot) * VREC);
                if (lane < 6) kd[lane] = ks[lane];
                else if (lane < 10) vd[lane - 6] = vs[lane - 6];
                continue;
            }
            const int64_t tok = (int64_t)lblk * bs + slot - L;
            const int64_t src = (((int64_t)i * n_new + tok) * n_kv + h) * 128 + 4 * lane;
            float x[4];
            {
                const uint2 kv = __ldg(reinterpret_cast<const uint2*>(Kin + src));
                x[0] = __uint_as_float(kv.x << 16);
                x[1] = __uint_as_float(kv.x & 0xffff0000u);
                x[2] = __uint_as_float(kv.y << 16);
                x[3] = __uint_as_float(kv.y & 0xffff0000u);
            }
            tq_encode_row(x, true, signs, S4, srec[warp], lane);
            {
                const uint2 vv = __ldg(reinterpret_cast<const uint2*>(Vin + src));
                x[0] = __uint_as_float(vv.x << 16);
                x[1] = __uint_as_float(vv.x & 0xffff0000u);
                x[2] = __uint_as_float(vv.y << 16);
                x[3] = __uint_as_float(vv.y & 0xffff0000u);
            }
            tq_encode_row(x, false, signs, S4, srec[warp] + 24, lane);
            __syncwarp();
            const uint4* r4 = reinterpret_cast<const uint4*>(srec[warp]);
            if (lane < 6) kd[lane] = r4[lane];
            else if (lane < 10) vd[lane - 6] = r4[lane];
            __syncwarp();
        }
    }
}

// ------------------------------------------------------------------ queries
// One warp per query row o: qs[o][0..128) = R q (rotated query),
// qs[o][128..256) = S R q (its QJL projections), fp32.
__global__ void __launch_bounds__(256) k_turbo_query(const __nv_bfloat16* __restrict__ Q, int32_t n_rows,
                                                      const float* __restrict__ signs, const float* __restrict__ S,
                                                      float* __restrict__ qs, const DevMeta* meta) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int32_t o = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (o >= n_rows || meta->status) return;
    float x[4];
    {
        const uint2 q = __ldg(reinterpret_cast<const uint2*>(Q + (int64_t)o * 128 + 4 * lane));
        const float4 sg = __ldg(reinterpret_cast<const float4*>(signs) + lane);
        x[0] = __uint_as_float(q.x << 16) * sg.x;
        x[1] = __uint_as_float(q.x & 0xffff0000u) * sg.y;
        x[2] = __uint_as_float(q.y << 16) * sg.z;
        x[3] = __uint_as_float(q.y & 0xffff0000u) * sg.w;
    }
    tq_fwht(x, lane);
    const float inv = 0.0883883476483184405501055452631f;
#pragma unroll
    for (int k = 0; k < 4; ++k) x[k] *= inv;
    float* dst = qs + (int64_t)o * 256;
    *reinterpret_cast<float4*>(dst + 4 * lane) = make_float4(x[0], x[1], x[2], x[3]);
    const float4* S4 = reinterpret_cast<const float4*>(S);
    float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int src = 0; src < 32; ++src) {
        float xi[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) xi[k] = __shfl_sync(FULL, x[k], src);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 s = __ldg(S4 + (4 * lane + k) * 32 + src);
            z[k] = fmaf(s.x, xi[0], fmaf(s.y, xi[1], fmaf(s.z, xi[2], fmaf(s.w, xi[3], z[k]))));
        }
    }
    *reinterpret_cast<float4*>(dst + 128 + 4 * lane) = make_float4(z[0], z[1], z[2], z[3]);
}

// ---------------------------------------------------------- partial kernel
// The plan's units (at most 16 rows) over compressed tiles.  Per tile the CTA
// loads the 16 key and 16 value records of the (block, kv head), decodes them
// into fp32 rows of the rotated space in shared memory (warp w decodes slots
// w, w + 4, ...), then warp w serves rows w, w + 4, w + 8, w + 12 of the unit:
// per position, the score <q', k_hat> + sqrt(pi/2)/128 |e| <S q', sign(S e)>
// (lane l takes columns l + 32 j of both sums), an online softmax in base 2,
// and acc += p v_hat.  Partial rows stay in the rotated space.
__global__ void __launch_bounds__(128) k_attn_partial_turbo(const AttnArgs a, const float* __restrict__ qs) {
    __shared__ __align__(16) uint32_t krec[16][24];
    __shared__ __align__(16) uint32_t vrec[16][16];
    __shared__ __align__(16) float kd[16][128];
    __shared__ __align__(16) float vd[16][128];
    __shared__ float enorm[16];
    __shared__ int st0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
    const unsigned char* KP = reinterpret_cast<const unsigned char*>(a.pool_k);
    const unsigned char* VP = reinterpret_cast<const unsigned char*>(a.pool_v);
    const float qjl_c = 0.0097916591f;   // sqrt(pi / 2) / 128
    while (t < t_end) {
        const AttnUnit U = pl.units[u];
        const int32_t uend = U.tile_off + U.n_blk;
        if (t >= uend) { ++u; continue; }
        const int32_t cend = min(t_end, uend);
        float qr[4][4], sq[4][4], acc[4][4], m[4], l[4];
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
            for (int j = 0; j < 4; ++j) {
                qr[rr][j] = v ? qs[(int64_t)R.q_row * 256 + lane + 32 * j] : 0.f;
                sq[rr][j] = v ? qs[(int64_t)R.q_row * 256 + 128 + lane + 32 * j] : 0.f;
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
            const uint4* kg = reinterpret_cast<const uint4*>(KP + ((int64_t)blk * a.n_kv + U.kv_head) * BS * KREC);
            const uint4* vg = reinterpret_cast<const uint4*>(VP + ((int64_t)blk * a.n_kv + U.kv_head) * BS * VREC);
            __syncthreads();
            for (int e = threadIdx.x; e < BS * KREC / 16; e += blockDim.x) reinterpret_cast<uint4*>(krec)[e] = kg[e];
            for (int e = threadIdx.x; e < BS * VREC / 16; e += blockDim.x) reinterpret_cast<uint4*>(vrec)[e] = vg[e];
            __syncthreads();
            for (int slot = warp; slot < BS; slot += 4) {
                int c1a, c1b, cu[6];
                float nrm, xh[4];
                tq_unpack_polar(krec[slot], lane, c1a, c1b, cu, nrm);
                tq_polar_decode32(nrm, c1a, c1b, cu, lane, xh);
                *reinterpret_cast<float4*>(&kd[slot][4 * lane]) = make_float4(xh[0], xh[1], xh[2], xh[3]);
                tq_unpack_polar(vrec[slot], lane, c1a, c1b, cu, nrm);
                tq_polar_decode32(nrm, c1a, c1b, cu, lane, xh);
                *reinterpret_cast<float4*>(&vd[slot][4 * lane]) = make_float4(xh[0], xh[1], xh[2], xh[3]);
                if (lane == 0) enorm[slot] = __uint_as_float(krec[slot][20]);
            }
            __syncthreads();
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                if (warp + 4 * rr >= U.n_rows) continue;
                for (int tok = 0; tok < BS; ++tok) {
                    if (lb * BS + tok >= lim[rr]) break;
                    float dq = 0.f, dj = 0.f;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        dq = fmaf(qr[rr][j], kd[tok][lane + 32 * j], dq);
                        const bool bit = (krec[tok][16 + j] >> lane) & 1u;
                        dj += bit ? sq[rr][j] : -sq[rr][j];
                    }
                    float dot = fmaf(qjl_c * enorm[tok], dj, dq);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(FULL, dot, o);
                    const float sc = dot * a.scale_log2;
                    const float mn = fmaxf(m[rr], sc);
                    const float al = exp2f(m[rr] - mn);
                    const float p = exp2f(sc - mn);
                    l[rr] = l[rr] * al + p;
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[rr][j] = fmaf(p, vd[tok][lane + 32 * j], acc[rr][j] * al);
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
            for (int j = 0; j < 4; ++j) a.part_acc[(int64_t)(prow0 + row) * D + lane + 32 * j] = acc[rr][j];
            if (lane == 0) a.part_ml[prow0 + row] = make_float2(m[rr], l[rr]);
        }
        t = cend;
        ++u;
    }
}

}  // namespace

namespace dendrite {

int launch_append_turbo(const TurboAppend& t, cudaStream_t s) {
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(t.n_tiles, (int64_t)t.sm_count * 16));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, (unsigned)t.n_layers_in);
    cfg.blockDim = dim3(128);
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_append_turbo, t.args, t.n, t.n_new, t.bs, t.bpb, t.n_kv, t.n_blocks, t.table,
                              t.call, t.K, t.V, t.kp, t.vp, t.in_layer, t.kp_layer, t.vp_layer, t.signs, t.S, t.meta,
                              t.n_tiles) == cudaSuccess
               ? DENDRITE_OK
               : DENDRITE_ECUDA;
}

int launch_turbo_partials(const AttnArgs& a, const void* Q, int32_t n_rows, const float* signs, const float* S,
                          float* qs, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cfg.stream = s;
    cfg.gridDim = dim3((unsigned)((n_rows + 7) / 8));
    cfg.blockDim = dim3(256);
    if (cudaLaunchKernelEx(&cfg, k_turbo_query, static_cast<const __nv_bfloat16*>(Q), n_rows, signs, S, qs,
                           (const DevMeta*)a.meta) != cudaSuccess)
        return DENDRITE_ECUDA;
    if (a.plan.n_ctas > 0) {
        cfg.gridDim = dim3((unsigned)a.plan.n_ctas);
        cfg.blockDim = dim3(128);
        if (cudaLaunchKernelEx(&cfg, k_attn_partial_turbo, a, (const float*)qs) != cudaSuccess) return DENDRITE_ECUDA;
    }
    return DENDRITE_OK;
}

int turbo_ctas_per_sm() {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_attn_partial_turbo, 128, 0) != cudaSuccess) return 1;
    return std::max(1, occ);
}

// ----------------------------------------------------------- host tables
int turbo_setup_tables() {
    static bool done_dev[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DENDRITE_ECUDA;
    if (done_dev[dev]) return DENDRITE_OK;
    TurboTables t{};
    const double pi = 3.14159265358979323846;
    t.t1 = (float)std::tan(pi / 8);
    t.t3 = (float)std::tan(3 * pi / 8);
    for (int c = 0; c < 16; ++c) {
        t.cos1[c] = (float)std::cos((c + 0.5) * pi / 8);
        t.sin1[c] = (float)std::sin((c + 0.5) * pi / 8);
    }
    for (int L = 2; L <= 7; ++L) {
        const double k = (double)(1 << (L - 1));
        const double w = std::min(pi / 4, 1.6 / std::sqrt(k - 1));
        const double lo = pi / 4 - w, hi = pi / 4 + w, bw = (hi - lo) / 8;
        for (int j = 1; j < 8; ++j) t.tan_up[L - 2][j - 1] = (float)std::tan(lo + j * bw);
        for (int c = 0; c < 8; ++c) {
            t.cos_up[L - 2][c] = (float)std::cos(lo + (c + 0.5) * bw);
            t.sin_up[L - 2][c] = (float)std::sin(lo + (c + 0.5) * bw);
        }
    }
    if (cudaMemcpyToSymbol(c_tq, &t, sizeof(t)) != cudaSuccess) return DENDRITE_ECUDA;
    done_dev[dev] = true;
    return DENDRITE_OK;
}

}  // namespace dendrite
