// Shared device helpers of the MiTA CUDA library: I/O type traits, the
// correctly rounded pooled mean, orderable selection keys and the plan
// layout.  (This file belongs to the CUDA library only.)
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mita.h"

#define MITA_DEV __device__ __forceinline__

namespace mita {

// ---------------------------------------------------------------- I/O types
MITA_DEV float to_f32(float x) { return x; }
MITA_DEV float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> MITA_DEV T from_f32(float x);
template <> MITA_DEV float from_f32<float>(float x) { return x; }
template <> MITA_DEV __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Error-free sum of two fp32 values (Knuth's TwoSum): hi + lo == a + b exactly.
MITA_DEV void two_sum(float a, float b, float& hi, float& lo) {
    hi = a + b;
    float bb = hi - a;
    lo = (a - (hi - bb)) + (b - bb);
}

// Accumulate x into the unevaluated pair (hi, lo).
MITA_DEV void acc2(float& hi, float& lo, float x) {
    float h, l;
    two_sum(hi, x, h, l);
    hi = h;
    lo += l;
}

// The bf16 value nearest (ties to even) to the exact quotient (hi + lo) / c,
// for a positive integer count c.  A fp32 estimate gives a candidate b; the
// exact position of hi + lo against c times the midpoints next to b decides
// whether b, or a neighbour, is the correctly rounded result.  c * midpoint
// is computed by a fused multiply-add, so the comparison is exact while the
// sum has fewer than 24 significant bits beyond the midpoint's.
MITA_DEV __nv_bfloat16 mean_to_bf16(float hi, float lo, float c) {
    const bool neg = hi < 0.0f;
    if (neg) { hi = -hi; lo = -lo; }
    float q = __fdiv_rn(hi + lo, c);
    uint16_t b = __bfloat16_as_ushort(__float2bfloat16_rn(q));   // non-negative
    {   // above the upper midpoint?
        float v0 = __bfloat162float(__ushort_as_bfloat16(b));
        float v1 = __bfloat162float(__ushort_as_bfloat16((uint16_t)(b + 1)));
        float mid = 0.5f * (v0 + v1);
        float e = fmaf(-c, mid, hi) + lo;
        if (e > 0.0f || (e == 0.0f && (b & 1))) b = (uint16_t)(b + 1);
        else if (b > 0) {   // below the lower midpoint?
            float vm = __bfloat162float(__ushort_as_bfloat16((uint16_t)(b - 1)));
            float midl = 0.5f * (vm + v0);
            float el = fmaf(-c, midl, hi) + lo;
            if (el < 0.0f || (el == 0.0f && (b & 1))) b = (uint16_t)(b - 1);
        }
    }
    __nv_bfloat16 r = __ushort_as_bfloat16(b);
    return neg ? __hneg(r) : r;
}

template <typename T> MITA_DEV T pooled_mean(float hi, float lo, float c);
template <> MITA_DEV __nv_bfloat16 pooled_mean<__nv_bfloat16>(float hi, float lo, float c) {
    return mean_to_bf16(hi, lo, c);
}
template <> MITA_DEV float pooled_mean<float>(float hi, float lo, float c) {
    return __fdiv_rn(hi + lo, c);
}

// Adaptive average pooling bin of output cell i (G inputs -> P outputs).
MITA_DEV void pool_bin(int i, int G, int P, int& lo, int& hi) {
    lo = (i * G) / P;
    hi = ((i + 1) * G + P - 1) / P;
}

// Order-preserving map of a fp32 score to an unsigned key: a larger score
// gives a larger key, and -0.0 maps like +0.0.
MITA_DEV uint32_t order_key(float x) {
    uint32_t u = __float_as_uint(x == 0.0f ? 0.0f : x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inverse of order_key().
MITA_DEV float key_to_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxRoutes = 8;   // experts per query, at most

// ---------------------------------------------------------------- plan
struct Shape {
    int B, H, N, d, m, k;
    int gh, gw, ph, pw;
    __host__ __device__ int BH() const { return B * H; }
};

}  // namespace mita

struct mita_plan_s {
    mita::Shape s;
    mita_dtype_t dtype;
    int device;
    int path_opt;          // mita_path_t requested
    int keep_landmarks;
    int routing_only;      // 1: softmax over the routed keys alone (no shared expert)
    int routes_s;          // experts per query (0 or 1: one; up to kMaxRoutes)
    float* dQl;            // backward: gradients of Q_l and V_l [BH, m, d] fp32
    float* dVl;
    int landmarks_valid;
    // workspace: the core region (landmarks, experts, routes, buckets,
    // status) from mita_plan, and the regions only some paths need, each its
    // own allocation made when a path that needs it is first chosen
    void* ws;
    size_t ws_bytes;       // all regions held
    void* ws_S;            // raw scores (staged and tiled paths, backward)
    void* ws_tiled;        // tiled path's row keys, value partials, tile lists
    void* ws_grad;         // backward's fp32 region
    // completion of the plan's last eager launch, for mita_get_status()
    cudaEvent_t done;
    cudaStream_t aux;      // non-blocking stream for the status word's copy
    int done_valid;
    void* Ql;              // [BH, m, d] io type
    void* Vl;              // [BH, m, d] io type
    float* S;              // [BH, m, N] raw scores (staged path)
    int32_t* idx;          // [BH, m, k] when the caller passes none
    int32_t* route;        // [BH, N]    when the caller passes none
    int32_t* counts;       // [BH, m]
    int32_t* offsets;      // [BH, m + 1]
    int32_t* perm;         // [BH, N]
    int32_t* status;       // [1]
    // tiled path only (null otherwise)
    uint32_t* rowmax;      // [2, BH, m] order keys of each landmark's largest, then smallest, raw score
    float* vpart;          // [head group, splits, m, d + 1] landmark-value partials
    int32_t* cursor;       // [BH, m]   bucket scatter cursors
    int32_t* tiles;        // [BH, max tiles] int2 attention tiles (expert << 16 | queries, first position)
    int32_t* ntiles;       // [BH]
    uint64_t launches;     // kernels launched so far
    // mita_forward_host only: device staging for two chunks of heads (Q, K,
    // V, out, experts, routes and, where the tiled path applies, its value
    // partials), the two copy streams, and the events that order the chunks
    // across those streams and the caller's
    void* ws_host;
    size_t host_slot_bytes;
    int host_heads;        // heads per chunk
    cudaStream_t h2d, d2h;
    cudaEvent_t ev_start, ev_in[2], ev_comp[2], ev_out[2];
};
