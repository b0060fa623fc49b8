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
#include <cuda_fp16.h>

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
// One warp per query row o.  With q' = R q (the rotated query) and z = S q'
// (its QJL projections), row o of qs (1024 bytes) holds q' / max|q'| and
// z / max|z| in fp16 (128 + 128 halves), then the two scales (float2).  The
// scaled halves lie in [-1, 1], so no query overflows fp16.
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
    float qm = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
    float zm = fmaxf(fmaxf(fabsf(z[0]), fabsf(z[1])), fmaxf(fabsf(z[2]), fabsf(z[3])));
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        qm = fmaxf(qm, __shfl_xor_sync(FULL, qm, m));
        zm = fmaxf(zm, __shfl_xor_sync(FULL, zm, m));
    }
    qm = qm > 0.f ? qm : 1.f;
    zm = zm > 0.f ? zm : 1.f;
    const float rq = 1.f / qm, rz = 1.f / zm;
    unsigned char* row = reinterpret_cast<unsigned char*>(qs) + (int64_t)o * 1024;
    const __half2 a = __floats2half2_rn(x[0] * rq, x[1] * rq), b = __floats2half2_rn(x[2] * rq, x[3] * rq);
    const __half2 c = __floats2half2_rn(z[0] * rz, z[1] * rz), d = __floats2half2_rn(z[2] * rz, z[3] * rz);
    *reinterpret_cast<uint2*>(row + 8 * lane) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
    *reinterpret_cast<uint2*>(row + 256 + 8 * lane) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&c), *reinterpret_cast<const uint32_t*>(&d));
    if (lane == 0) *reinterpret_cast<float2*>(row + 512) = make_float2(qm, zm);
}

// ---------------------------------------------------------- partial kernel
// The plan's units (at most 16 rows) over compressed tiles, on the tensor
// cores.  The CTA's four warps take the chunk's tiles in turn (warp w: tiles
// w, w + 4, ...), each with its own online-softmax state, and merge at the
// end of the chunk.  Per tile a warp
//   - copies the 16 key and 16 value records into shared memory (cp.async,
//     one tile ahead);
//   - decodes them into the unit-norm rows u = x_hat / |x_hat| in fp16 (a
//     lane expands one level-4 node: 16 coordinates, multiplying the angle
//     factors down from the root), swizzled for ldmatrix;
//   - S1 = Q' U_k^T and S2 = Z sign(S E)^T with mma.sync m16n8k16 (fp16 in,
//     fp32 accumulate; the sign matrix is built from the key bits in
//     registers), the score of row r and token t being
//     qmax_r |k_t| S1 + sqrt(pi/2)/128 zmax_r |e_t| S2 (times 1/sqrt(d),
//     in base 2), then the online softmax;
//   - acc += P' U_v with P' = p |v_t| / vs, vs the largest value norm the
//     warp has seen (a running scale folded into the softmax rescale), so P'
//     stays in [0, 1] in fp16 and acc = (sum p v_hat) / vs.
// Partial rows stay in the rotated space.
constexpr int TQ_WARPS = 4;
constexpr int TQ_REC_ROW = 96;                       // smem stride of a key or value record
constexpr int TQ_STAGE = 2 * BS * TQ_REC_ROW;        // key then value records of one tile
constexpr int TQ_DEC_TILE = BS * 256;                // one decoded 16 x 128 fp16 tile
constexpr int TQ_SCR_ROW = 136;                      // floats per row of the merge scratch
constexpr int TQ_DEC_BYTES = BS * TQ_SCR_ROW * 4;    // decoded K and V tiles, later the merge scratch
static_assert(TQ_DEC_BYTES >= 2 * TQ_DEC_TILE, "merge scratch overlays the decoded tiles");
constexpr int TQ_WARP_BYTES = 2 * TQ_STAGE + TQ_DEC_BYTES;
constexpr int TQ_Q_OFF = TQ_WARPS * TQ_WARP_BYTES;   // 16 query rows x 512 bytes (swizzled)
constexpr int TQ_TAB_OFF = TQ_Q_OFF + 16 * 512;      // 64 (cos, sin) pairs
constexpr int TQ_QSC_OFF = TQ_TAB_OFF + 64 * 8;      // per row (qmax, zmax) scales
constexpr int TQ_ML_OFF = TQ_QSC_OFF + 16 * 8;       // per warp and row (m, l)
constexpr int TQ_SMEM = TQ_ML_OFF + TQ_WARPS * 16 * 8;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void mma16816_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}
// Two QJL sign bits (bit 0: lower k) as a pair of fp16 +-1: a set bit is +1.
__device__ __forceinline__ uint32_t sign_pair(uint32_t x) {
    return 0xBC00BC00u ^ (((x & 3u) * 0x40008000u) & 0x80008000u);
}
// Byte offset of (row t, column d) in a decoded fp16 tile: 16-byte chunks
// XOR-ed with t & 7, so that ldmatrix's eight rows hit distinct banks.
__device__ __forceinline__ uint32_t tq_swz(int t, int d) {
    return (uint32_t)(t * 256 + ((((d >> 3) ^ (t & 7))) << 4) + (d & 7) * 2);
}

// Decodes coordinates 16 j .. 16 j + 15 of a record's unit-norm row: the
// product of the angle factors on the path from the root (level 7) to each
// coordinate, in that order.  tab: (cos, sin) of the bin centres, levels 7
// down to 2 (8 each) then level 1 (16).  The 3-bit codes come from two
// 16-byte loads of record words 8..15 (stream word k is record word 9 + k):
// level 2 nodes 4j..4j+3 at stream bit 12 j, level 3 nodes 2j, 2j+1 at
// 96 + 6 j, level 4 node j at 144 + 3 j, level 5 node j/2 at 168 + 3 (j/2),
// level 6 node j/4 at 180 + 3 (j/4), level 7 at 186.
__device__ __forceinline__ void tq_decode16(const uint32_t* rec, int j, const float2* tab, uint4& lo, uint4& hi) {
    const uint4 A = *reinterpret_cast<const uint4*>(rec + 8);
    const uint4 B = *reinterpret_cast<const uint4*>(rec + 12);
    const uint32_t s0 = A.y, s1 = A.z, s2 = A.w, s3 = B.x, s4 = B.y, s5 = B.z;
    const uint32_t c7 = (s5 >> 26) & 7u;
    const uint32_t c6 = (s5 >> (20 + 3 * (j >> 2))) & 7u;
    const uint32_t c5 = (s5 >> (8 + 3 * (j >> 1))) & 7u;
    const uint32_t c4 = (uint32_t)(((((uint64_t)s5) << 32) | s4) >> (16 + 3 * j)) & 7u;
    const uint32_t c3 = (uint32_t)(((((uint64_t)s4) << 32) | s3) >> (6 * j)) & 63u;
    const int p2 = 12 * j;
    const uint32_t lo2 = p2 < 32 ? s0 : (p2 < 64 ? s1 : s2), hi2 = p2 < 32 ? s1 : (p2 < 64 ? s2 : s3);
    const uint32_t c2 = __funnelshift_r(lo2, hi2, p2 & 31) & 0xFFFu;
    const uint32_t c1 = rec[1 + j];
    const float2 t7 = tab[c7], t6 = tab[8 + c6], t5 = tab[16 + c5], t4 = tab[24 + c4];
    float r = (j & 4) ? t7.y : t7.x;
    r *= (j & 2) ? t6.y : t6.x;
    r *= (j & 1) ? t5.y : t5.x;
    float r3[2] = {r * t4.x, r * t4.y};
    float r2[4], r1[8], x[16];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float2 t3 = tab[32 + ((c3 >> (3 * i)) & 7u)];
        r2[2 * i] = r3[i] * t3.x;
        r2[2 * i + 1] = r3[i] * t3.y;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t2 = tab[40 + ((c2 >> (3 * i)) & 7u)];
        r1[2 * i] = r2[i] * t2.x;
        r1[2 * i + 1] = r2[i] * t2.y;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float2 t1 = tab[48 + ((c1 >> (4 * k)) & 15u)];
        x[2 * k] = r1[k] * t1.x;
        x[2 * k + 1] = r1[k] * t1.y;
    }
    lo = make_uint4(pack_half2(x[0], x[1]), pack_half2(x[2], x[3]), pack_half2(x[4], x[5]), pack_half2(x[6], x[7]));
    hi = make_uint4(pack_half2(x[8], x[9]), pack_half2(x[10], x[11]), pack_half2(x[12], x[13]),
                    pack_half2(x[14], x[15]));
}

// One warp's rows against one tile: 16 query rows (fp16 at qrows, row stride
// 512 bytes, chunks XOR-ed with row & 7) against the tile's 16 tokens (key and
// value records at rk / rv, decoded unit rows at kt / vt).  pos0: position of
// the lane's first column; a0/a1, b0/b1: the rows' score scales.
struct TqRows {
    float o[16][4];
    float m0, m1, l0, l1, vs;
};

__device__ __forceinline__ void tq_tile(TqRows& st, uint32_t qrows, const unsigned char* rk,
                                        const unsigned char* rv, uint32_t kt, uint32_t vt, int32_t pos0,
                                        int32_t lim0, int32_t lim1, float a0, float a1, float b0, float b1,
                                        int lane) {
    const float NEG_INF = -INFINITY;
    // per-token scalars of this lane's columns: tokens 2 (lane % 4) + e + 8 nt
    float kn[2][2], en[2][2], vn[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int tok = 2 * (lane & 3) + e + 8 * nt;
            const uint32_t* kr = reinterpret_cast<const uint32_t*>(rk + tok * TQ_REC_ROW);
            kn[nt][e] = __uint_as_float(kr[0]);
            en[nt][e] = __uint_as_float(kr[20]);
            vn[nt][e] = __uint_as_float(reinterpret_cast<const uint32_t*>(rv + tok * TQ_REC_ROW)[0]);
        }
    }
    // the QJL bits of tokens lane / 4 and 8 + lane / 4
    uint32_t qb[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const uint32_t* kr = reinterpret_cast<const uint32_t*>(rk + ((lane >> 2) + 8 * nt) * TQ_REC_ROW);
#pragma unroll
        for (int w = 0; w < 4; ++w) qb[nt][w] = kr[16 + w] >> (2 * (lane & 3));
    }
    // S1 = Q' U_k^T, S2 = Z sign^T (16 rows x 16 tokens each)
    float s1[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
        const int mi = lane >> 3;
        const int tokl = (mi >> 1) * 8 + (lane & 7);
        const int qr = lane & 15, qh = lane >> 4;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t qa[4], za[4], kb0, kb1, kb2, kb3;
            ldsm_x4(qrows + qr * 512 + (((2 * ks + qh) ^ (qr & 7)) << 4), qa[0], qa[1], qa[2], qa[3]);
            ldsm_x4(qrows + qr * 512 + (((16 + 2 * ks + qh) ^ (qr & 7)) << 4), za[0], za[1], za[2], za[3]);
            ldsm_x4(kt + tq_swz(tokl, ks * 16 + (mi & 1) * 8), kb0, kb1, kb2, kb3);
            mma16816_f16(s1[0], qa, kb0, kb1);
            mma16816_f16(s1[1], qa, kb2, kb3);
            const int sh = (ks & 1) * 16;
            mma16816_f16(s2[0], za, sign_pair(qb[0][ks >> 1] >> sh), sign_pair(qb[0][ks >> 1] >> (sh + 8)));
            mma16816_f16(s2[1], za, sign_pair(qb[1][ks >> 1] >> sh), sign_pair(qb[1][ks >> 1] >> (sh + 8)));
        }
    }
    // scores, mask, online softmax
    float sc[2][4];
    float mx0 = NEG_INF, mx1 = NEG_INF, vmax = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int32_t pos = pos0 + 8 * nt + e;
            const float v0 = a0 * (kn[nt][e] * s1[nt][e]) + b0 * (en[nt][e] * s2[nt][e]);
            const float v1 = a1 * (kn[nt][e] * s1[nt][2 + e]) + b1 * (en[nt][e] * s2[nt][2 + e]);
            sc[nt][e] = pos < lim0 ? v0 : NEG_INF;
            sc[nt][2 + e] = pos < lim1 ? v1 : NEG_INF;
            mx0 = fmaxf(mx0, sc[nt][e]);
            mx1 = fmaxf(mx1, sc[nt][2 + e]);
            vmax = fmaxf(vmax, vn[nt][e]);
        }
    }
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(FULL, mx0, m));
        mx1 = fmaxf(mx1, __shfl_xor_sync(FULL, mx1, m));
        vmax = fmaxf(vmax, __shfl_xor_sync(FULL, vmax, m));
    }
    const float n0 = fmaxf(st.m0, mx0), n1 = fmaxf(st.m1, mx1);
    const float u0s = n0 == NEG_INF ? 0.f : n0, u1s = n1 == NEG_INF ? 0.f : n1;
    const float al0 = exp2f(st.m0 - u0s), al1 = exp2f(st.m1 - u1s);
    st.m0 = n0;
    st.m1 = n1;
    const float vs_new = fmaxf(fmaxf(st.vs, vmax), 1e-30f);
    const float rv_new = 1.f / vs_new;
    const float g = st.vs * rv_new;
    const float g0 = al0 * g, g1 = al1 * g;
    st.vs = vs_new;
    float ps0 = 0.f, ps1 = 0.f;
    uint32_t pa[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        float p[4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            p[e] = exp2f(sc[nt][e] - u0s);
            p[2 + e] = exp2f(sc[nt][2 + e] - u1s);
            ps0 += p[e];
            ps1 += p[2 + e];
        }
        const float w0 = vn[nt][0] * rv_new, w1 = vn[nt][1] * rv_new;
        pa[2 * nt] = pack_half2(p[0] * w0, p[1] * w1);
        pa[2 * nt + 1] = pack_half2(p[2] * w0, p[3] * w1);
    }
    st.l0 = st.l0 * al0 + ps0;
    st.l1 = st.l1 * al1 + ps1;
    if (!__all_sync(FULL, g0 == 1.f && g1 == 1.f)) {
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            st.o[n][0] *= g0;
            st.o[n][1] *= g0;
            st.o[n][2] *= g1;
            st.o[n][3] *= g1;
        }
    }
    // acc += P' U_v
    {
        const int mi = lane >> 3;
        const int tokl = (mi & 1) * 8 + (lane & 7);
#pragma unroll
        for (int np = 0; np < 8; ++np) {
            uint32_t v0r, v1r, v2r, v3r;
            ldsm_x4_t(vt + tq_swz(tokl, np * 16 + (mi >> 1) * 8), v0r, v1r, v2r, v3r);
            mma16816_f16(st.o[2 * np], pa, v0r, v1r);
            mma16816_f16(st.o[2 * np + 1], pa, v2r, v3r);
        }
    }
}

// Decodes rows 4 (pss % 4) + lane / 8 of the key (pss < 4) or value (pss >= 4)
// records of one tile into the decoded tiles dk / dv (lane % 8: level-4 node).
__device__ __forceinline__ void tq_decode_pass(int pss, const unsigned char* rk, const unsigned char* rv,
                                               unsigned char* dk, unsigned char* dv, const float2* tab, int lane) {
    const int j = lane & 7;
    const int row = (pss & 3) * 4 + (lane >> 3);
    const bool isv = pss >= 4;
    const uint32_t* rec = reinterpret_cast<const uint32_t*>((isv ? rv : rk) + row * TQ_REC_ROW);
    uint4 lo, hi;
    tq_decode16(rec, j, tab, lo, hi);
    unsigned char* d = isv ? dv : dk;
    // lanes 4..7 of a row store their upper chunk first: each quarter-warp's
    // eight 16-byte stores then fall in eight distinct bank groups
    const bool up = j >= 4;
    *reinterpret_cast<uint4*>(d + tq_swz(row, 16 * j + (up ? 8 : 0))) = up ? hi : lo;
    *reinterpret_cast<uint4*>(d + tq_swz(row, 16 * j + (up ? 0 : 8))) = up ? lo : hi;
}

// Units of more than 16 rows (up to 64) share each tile's decode: the CTA's
// four warps decode it together (two passes each; records double-buffered by
// cp.async at CTA level), then warp w runs rows 16 w .. 16 w + 15 over it and
// stores its rows' partials itself.  Shared memory of this mode (it reuses
// the space of the per-warp mode between units):
constexpr int TQB_Q_OFF = 0;                                   // 64 query rows x 512 bytes
constexpr int TQB_STAGE_OFF = 64 * 512;                        // 2 record stages
constexpr int TQB_DEC_OFF = TQB_STAGE_OFF + 2 * TQ_STAGE;      // decoded K then V tile
constexpr int TQB_QSC_OFF = TQB_DEC_OFF + 2 * TQ_DEC_TILE;     // 64 (qmax, zmax)
static_assert(TQB_QSC_OFF + 64 * 8 <= TQ_TAB_OFF, "the wide mode stays clear of the bin tables");

__global__ void __launch_bounds__(128, 3) k_attn_partial_turbo(const AttnArgs a, const float* __restrict__ qs) {
    extern __shared__ __align__(16) unsigned char tq_smem[];
    __shared__ int st0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    pdl_trigger();
    if (tid == 0) st0 = a.meta->status;
    float2* tab = reinterpret_cast<float2*>(tq_smem + TQ_TAB_OFF);
    if (tid < 64) {
        const int L = tid < 48 ? 7 - (tid >> 3) : 1;   // levels 7 .. 2, then level 1
        const int c = tid < 48 ? (tid & 7) : tid - 48;
        tab[tid] = L == 1 ? make_float2(c_tq.cos1[c], c_tq.sin1[c])
                          : make_float2(c_tq.cos_up[L - 2][c], c_tq.sin_up[L - 2][c]);
    }
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
    const uint32_t sbase = smem_u32(tq_smem);
    const float NEG_INF = -INFINITY;
    while (t < t_end) {
        const AttnUnit U = pl.units[u];
        const int32_t uend = U.tile_off + U.n_blk;
        if (t >= uend) { ++u; continue; }
        const int32_t cend = min(t_end, uend);
        const bool wide = U.n_rows > 16;
        const int qoff = wide ? TQB_Q_OFF : TQ_Q_OFF;
        float2* qsc = reinterpret_cast<float2*>(tq_smem + (wide ? TQB_QSC_OFF : TQ_QSC_OFF));
        const int q_rows = wide ? 64 : 16;
        // ---- the unit's query rows: fp16 tile (swizzled) and scales
        for (int e = tid; e < q_rows * 8; e += 128) {
            const int r = e >> 3, cc = e & 7;
            const bool v = r < U.n_rows;
            const AttnRow R = v ? unit_row(pl, U, r) : AttnRow{0, 0};
            const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned char*>(qs) +
                                                              (int64_t)R.q_row * 1024);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int ch = cc + 8 * k;
                const uint4 val = v ? src[ch] : make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(tq_smem + qoff + r * 512 + ((ch ^ (r & 7)) << 4)) = val;
            }
            if (cc == 0)
                qsc[r] = v ? *reinterpret_cast<const float2*>(reinterpret_cast<const unsigned char*>(src) + 512)
                           : make_float2(0.f, 0.f);
        }
        __syncthreads();
        // this warp's rows: 0..15 of a narrow unit, 16 w .. 16 w + 15 of a wide one
        const int rbase = wide ? 16 * warp : 0;
        const bool has_rows = rbase < U.n_rows;
        const int r0 = rbase + (lane >> 2), r1 = r0 + 8;
        int32_t lim0 = 0, lim1 = 0;
        if (r0 < U.n_rows) lim0 = unit_row(pl, U, r0).limit;
        if (r1 < U.n_rows) lim1 = unit_row(pl, U, r1).limit;
        const float2 sc0 = qsc[r0 < q_rows ? r0 : 0], sc1 = qsc[r1 < q_rows ? r1 : 0];
        const float a0 = sc0.x * a.scale_log2, a1 = sc1.x * a.scale_log2;
        const float b0 = qjl_c * sc0.y * a.scale_log2, b1 = qjl_c * sc1.y * a.scale_log2;
        TqRows st;
#pragma unroll
        for (int n = 0; n < 16; ++n) st.o[n][0] = st.o[n][1] = st.o[n][2] = st.o[n][3] = 0.f;
        st.m0 = st.m1 = NEG_INF;
        st.l0 = st.l1 = st.vs = 0.f;
        // the records of tile tt into the stage at dst: key rows then value rows
        // (96-byte smem rows), chunks k0, k0 + kstep, ... of the 160
        auto issue = [&](int32_t tt, uint32_t dst, int k0, int kstep) {
            const int32_t lb = U.blk_start + (tt - U.tile_off);
            int32_t blk = a.table[(int64_t)U.table_row * a.bpb + lb];
            if ((uint32_t)blk >= (uint32_t)a.n_blocks) {
                if (k0 == 0) atomicCAS(&a.meta->status, 0, DENDRITE_ECORRUPT);
                blk = 0;   // read a valid block; the pool is poisoned anyway
            }
            const unsigned char* kg = KP + ((int64_t)blk * a.n_kv + U.kv_head) * BS * KREC;
            const unsigned char* vg = VP + ((int64_t)blk * a.n_kv + U.kv_head) * BS * VREC;
            for (int ch = k0; ch < 160; ch += kstep) {
                if (ch < 96) {
                    const int row = ch / 6, col = ch - 6 * row;
                    cp_async16(dst + row * TQ_REC_ROW + col * 16, kg + ch * 16);
                } else {
                    const int v = ch - 96, row = v >> 2, col = v & 3;
                    cp_async16(dst + BS * TQ_REC_ROW + row * TQ_REC_ROW + col * 16, vg + v * 16);
                }
            }
        };
        const int32_t lpos = U.blk_start - U.tile_off;   // logical block of tile tt: lpos + tt
        if (!wide) {
            // ---- per-warp tiles (warp w: tiles w, w + 4, ...)
            const uint32_t wbase = sbase + warp * TQ_WARP_BYTES;
            unsigned char* wptr = tq_smem + warp * TQ_WARP_BYTES;
            int32_t tt = t + warp;
            if (tt < cend) issue(tt, wbase, lane, 32);
            cp_async_commit();
            for (int it = 0; tt < cend; tt += TQ_WARPS, ++it) {
                if (tt + TQ_WARPS < cend) issue(tt + TQ_WARPS, wbase + ((it + 1) & 1) * TQ_STAGE, lane, 32);
                cp_async_commit();
                cp_async_wait1();
                __syncwarp();
                const unsigned char* rk = wptr + (it & 1) * TQ_STAGE;
                const unsigned char* rv = rk + BS * TQ_REC_ROW;
                unsigned char* dk = wptr + 2 * TQ_STAGE;
                unsigned char* dv = dk + TQ_DEC_TILE;
#pragma unroll 2
                for (int pss = 0; pss < 8; ++pss) tq_decode_pass(pss, rk, rv, dk, dv, tab, lane);
                __syncwarp();
                tq_tile(st, sbase + TQ_Q_OFF, rk, rv, wbase + 2 * TQ_STAGE, wbase + 2 * TQ_STAGE + TQ_DEC_TILE,
                        (lpos + tt) * BS + 2 * (lane & 3), lim0, lim1, a0, a1, b0, b1, lane);
                __syncwarp();   // records and decoded tiles are reused by the next tile
            }
            cp_async_wait0();
            // ---- merge the four warps' states and write the partial rows
            float2* sml = reinterpret_cast<float2*>(tq_smem + TQ_ML_OFF);
            float l0 = st.l0, l1 = st.l1;
            l0 += __shfl_xor_sync(FULL, l0, 1);
            l0 += __shfl_xor_sync(FULL, l0, 2);
            l1 += __shfl_xor_sync(FULL, l1, 1);
            l1 += __shfl_xor_sync(FULL, l1, 2);
            if ((lane & 3) == 0) {
                sml[warp * 16 + r0] = make_float2(st.m0, l0);
                sml[warp * 16 + r1] = make_float2(st.m1, l1);
            }
            __syncthreads();
            {
                float M0 = NEG_INF, M1 = NEG_INF;
#pragma unroll
                for (int w = 0; w < TQ_WARPS; ++w) {
                    M0 = fmaxf(M0, sml[w * 16 + r0].x);
                    M1 = fmaxf(M1, sml[w * 16 + r1].x);
                }
                const float f0 = st.m0 == NEG_INF ? 0.f : exp2f(st.m0 - M0) * st.vs;
                const float f1 = st.m1 == NEG_INF ? 0.f : exp2f(st.m1 - M1) * st.vs;
                float* scr = reinterpret_cast<float*>(wptr + 2 * TQ_STAGE);
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    const int col = 8 * n + 2 * (lane & 3);
                    *reinterpret_cast<float2*>(scr + r0 * TQ_SCR_ROW + col) =
                        make_float2(st.o[n][0] * f0, st.o[n][1] * f0);
                    *reinterpret_cast<float2*>(scr + r1 * TQ_SCR_ROW + col) =
                        make_float2(st.o[n][2] * f1, st.o[n][3] * f1);
                }
            }
            __syncthreads();
            {
                const int r = tid >> 3, cc = tid & 7;
                const int32_t prow = U.prow_base + (c - U.cfirst) * U.n_rows + r;
                if (r < U.n_rows) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int col = 4 * cc + 32 * k;
                        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                        for (int w = 0; w < TQ_WARPS; ++w) {
                            const float4 v = *reinterpret_cast<const float4*>(
                                tq_smem + w * TQ_WARP_BYTES + 2 * TQ_STAGE + (r * TQ_SCR_ROW + col) * 4);
                            sum.x += v.x;
                            sum.y += v.y;
                            sum.z += v.z;
                            sum.w += v.w;
                        }
                        *reinterpret_cast<float4*>(a.part_acc + (int64_t)prow * D + col) = sum;
                    }
                    if (cc == 0) {
                        float M = NEG_INF, L = 0.f;
#pragma unroll
                        for (int w = 0; w < TQ_WARPS; ++w) M = fmaxf(M, sml[w * 16 + r].x);
#pragma unroll
                        for (int w = 0; w < TQ_WARPS; ++w) {
                            const float2 ml = sml[w * 16 + r];
                            L += ml.x == NEG_INF ? 0.f : ml.y * exp2f(ml.x - M);
                        }
                        a.part_ml[prow] = make_float2(M, L);
                    }
                }
            }
        } else {
            // ---- shared tiles: the CTA decodes, warp w runs its 16 rows
            const uint32_t stage0 = sbase + TQB_STAGE_OFF;
            unsigned char* sptr = tq_smem + TQB_STAGE_OFF;
            unsigned char* dk = tq_smem + TQB_DEC_OFF;
            unsigned char* dv = dk + TQ_DEC_TILE;
            issue(t, stage0, tid, 128);
            cp_async_commit();
            for (int32_t tt = t, it = 0; tt < cend; ++tt, ++it) {
                if (tt + 1 < cend) issue(tt + 1, stage0 + ((it + 1) & 1) * TQ_STAGE, tid, 128);
                cp_async_commit();
                cp_async_wait1();
                __syncthreads();   // the tile's records, from every thread's copies
                const unsigned char* rk = sptr + (it & 1) * TQ_STAGE;
                const unsigned char* rv = rk + BS * TQ_REC_ROW;
                tq_decode_pass(2 * warp, rk, rv, dk, dv, tab, lane);
                tq_decode_pass(2 * warp + 1, rk, rv, dk, dv, tab, lane);
                __syncthreads();   // the decoded tile
                if (has_rows)
                    tq_tile(st, sbase + TQB_Q_OFF + rbase * 512, rk, rv, sbase + TQB_DEC_OFF,
                            sbase + TQB_DEC_OFF + TQ_DEC_TILE, (lpos + tt) * BS + 2 * (lane & 3), lim0, lim1, a0,
                            a1, b0, b1, lane);
                __syncthreads();   // records and decoded tile are reused by the next tile
            }
            cp_async_wait0();
            if (has_rows) {
                float l0 = st.l0, l1 = st.l1;
                l0 += __shfl_xor_sync(FULL, l0, 1);
                l0 += __shfl_xor_sync(FULL, l0, 2);
                l1 += __shfl_xor_sync(FULL, l1, 1);
                l1 += __shfl_xor_sync(FULL, l1, 2);
                const int32_t pbase = U.prow_base + (c - U.cfirst) * U.n_rows;
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    const int col = 8 * n + 2 * (lane & 3);
                    if (r0 < U.n_rows)
                        *reinterpret_cast<float2*>(a.part_acc + (int64_t)(pbase + r0) * D + col) =
                            make_float2(st.o[n][0] * st.vs, st.o[n][1] * st.vs);
                    if (r1 < U.n_rows)
                        *reinterpret_cast<float2*>(a.part_acc + (int64_t)(pbase + r1) * D + col) =
                            make_float2(st.o[n][2] * st.vs, st.o[n][3] * st.vs);
                }
                if ((lane & 3) == 0) {
                    if (r0 < U.n_rows) a.part_ml[pbase + r0] = make_float2(st.m0, l0);
                    if (r1 < U.n_rows) a.part_ml[pbase + r1] = make_float2(st.m1, l1);
                }
            }
        }
        __syncthreads();   // the next unit rewrites the query tile and the scratch
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
        cfg.dynamicSmemBytes = TQ_SMEM;
        if (cudaLaunchKernelEx(&cfg, k_attn_partial_turbo, a, (const float*)qs) != cudaSuccess) return DENDRITE_ECUDA;
    }
    return DENDRITE_OK;
}

int turbo_ctas_per_sm() {
    int occ = 0;
    if (cudaFuncSetAttribute(k_attn_partial_turbo, cudaFuncAttributeMaxDynamicSharedMemorySize, TQ_SMEM) !=
        cudaSuccess)
        return 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_attn_partial_turbo, 128, TQ_SMEM) != cudaSuccess)
        return 1;
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
