// Compressed KV blocks (TurboQuant: PolarQuant + QJL); see turbo.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "attn_common.cuh"

namespace dendrite {

constexpr int kTurboKeyBytes = 96;     // one key row's record
constexpr int kTurboValueBytes = 64;   // one value row's record
constexpr int kTurboDim = 128;         // head_dim of compressed pools
constexpr int kTurboQjlBits = 128;     // rows of the QJL matrix

// An append's encode/copy work on a compressed pool (device pointers).
struct TurboAppend {
    const int32_t* args;   // branch[n], len[n], prefix of touched blocks per branch[n]
    int32_t n, n_new, bs, bpb, n_kv, n_blocks;
    const int32_t* table;
    const int32_t* call;   // the metadata kernel's per-call scratch (copy-on-write sources at [n, 2n))
    const __nv_bfloat16* K;
    const __nv_bfloat16* V;
    unsigned char* kp;     // layer 0 of the written layers: key records
    unsigned char* vp;     // value records
    int64_t in_layer;      // input elements per layer
    int64_t kp_layer, vp_layer;   // pool bytes per layer
    const float* signs;    // [128] rotation signs
    const float* S;        // [128][128] QJL matrix
    DevMeta* meta;
    int64_t n_tiles;
    int32_t n_layers_in;
    int sm_count;
};

int turbo_setup_tables();   // bin tables of the codec on the current device (once per device)
int turbo_ctas_per_sm();    // resident CTAs per SM of the compressed partial kernel
int launch_append_turbo(const TurboAppend& t, cudaStream_t s);
// Rotated queries and their QJL projections into qs [n_rows][256], then the
// partial kernel over the plan's units.
int launch_turbo_partials(const AttnArgs& a, const void* Q, int32_t n_rows, const float* signs, const float* S,
                          float* qs, cudaStream_t s);

}  // namespace dendrite

// In-warp Walsh-Hadamard transform of 128 values, lane l holding 4l..4l+3:
// for h = 1, 2, 4, ..., 64 the pair (i, i + h) with i & h == 0 becomes
// (u + v, u - v), each sum and difference rounded once.
__device__ __forceinline__ void tq_fwht(float (&x)[4], int lane) {
    const float a = __fadd_rn(x[0], x[1]), b = __fsub_rn(x[0], x[1]);
    const float c = __fadd_rn(x[2], x[3]), d = __fsub_rn(x[2], x[3]);
    x[0] = __fadd_rn(a, c);
    x[2] = __fsub_rn(a, c);
    x[1] = __fadd_rn(b, d);
    x[3] = __fsub_rn(b, d);
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = lane & m;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float o = __shfl_xor_sync(0xffffffffu, x[k], m);
            x[k] = upper ? __fsub_rn(o, x[k]) : __fadd_rn(x[k], o);
        }
    }
}
