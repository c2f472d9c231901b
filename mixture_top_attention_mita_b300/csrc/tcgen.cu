// tcgen05 kernels of the tiled MiTA path (sm_103a): the dense contractions
// run on the fifth-generation tensor cores with operands staged by TMA and
// fp32 accumulators in tensor memory.
//   tc_scores  S = Q_l . K^T: for m <= 256 the scores half of
//              tc_scores_route below (tokens as M, every store 128
//              consecutive bytes of one row); beyond, per (128 landmarks x
//              128 keys) tile with each epilogue thread owning one landmark
//              row, storing the row's scores and folding them into the row
//              max and min.
//   tc_values  split-K partials of V_l: numerators exp(S / sqrt d - max) are
//              computed from S straight into a 128-byte swizzled K-major A
//              tile, V comes by TMA as an M/N-major B tile, and the MMAs of a
//              split of 1024-4096 keys accumulate in tensor memory (two stages: the
//              next tile's numerators and V copy overlap the current MMAs).
//   tc_route   q . Q_l^T for 128 queries against all landmarks; each thread
//              owns one query and takes the first argmax (the route).
//   tc_scores_route  both of the above for one tile of 128 tokens when m <= 128
//              (S^T = K . Q_l^T and Q . Q_l^T side by side in tensor memory).
// Step numbers refer to the operator of 36Kr / 新智元 "注意力也是FFN？",
// section "用少量地标查询，同时构造全局概括与细节专家": scores are step 2,
// landmark values step 4, routes step 5.
#include <algorithm>
#include <type_traits>

#include "tc_util.cuh"
#include "tcgen.cuh"
#include "host_cache.cuh"
#include "launch.cuh"

namespace mita {
namespace tcg {

using bf16 = __nv_bfloat16;
using namespace tc;

constexpr uint32_t kChunk = 128 * 128;   // one 128-row x 64-column bf16 tile, bytes

// ---------------------------------------------------------------- scores
template <int D, bool VEC>
__global__ void __launch_bounds__(128) tc_scores(const __grid_constant__ CUtensorMap mQl,
                                                 const __grid_constant__ CUtensorMap mK, Shape s,
                                                 float* __restrict__ S, uint32_t* __restrict__ rowmax,
                                                 uint32_t* __restrict__ rowmin, int32_t* __restrict__ status) {
    chain_wait_and_trigger();
    constexpr int KC = D / 64;
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ uint32_t tslot;
    __shared__ __align__(8) uint64_t bars[2];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (smem_u32(smem) & 1023u) {   // the swizzled tiles need a 1024-byte aligned base
        if (tid == 0) atomicExch(status, (int)MITA_ERR_DEVICE);
        return;
    }
    const int n0 = blockIdx.x * 128, i0 = blockIdx.y * 128, bh = blockIdx.z;
    const uint32_t sA = smem_u32(smem), sB = sA + KC * kChunk;
    const uint32_t bar_ld = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[1]);
    if (tid == 0) {
        mbar_init(bar_ld, 1);
        mbar_init(bar_mma, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(&tslot), 128);
    __syncthreads();
    fence_after();
    const uint32_t tmem = tslot;
    if (tid == 0) {
        mbar_expect_tx(bar_ld, 2u * KC * kChunk);
        for (int kc = 0; kc < KC; ++kc) {
            tma_load_2d(sA + kc * kChunk, &mQl, kc * 64, bh * s.m + i0, bar_ld);
            tma_load_2d(sB + kc * kChunk, &mK, kc * 64, bh * s.N + n0, bar_ld);
        }
        if (mbar_wait_bounded(bar_ld, 0)) {
            fence_after();
            constexpr uint32_t idesc = idesc_bf16(128, 128, 0, 0);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
                mma_bf16(tmem, desc_kmajor(sA + off), desc_kmajor(sB + off), idesc, kk > 0);
            }
            mma_commit(bar_mma);
        }
    }
    if (!mbar_wait_bounded(bar_mma, 0)) {
        if (lane == 0) atomicExch(status, (int)MITA_ERR_TIMEOUT);
    } else {
        fence_after();
        const int i = i0 + warp * 32 + lane, nv = min(128, s.N - n0);
        const bool live = i < s.m;
        float* row = S + ((size_t)bh * s.m + (live ? i : 0)) * s.N + n0;
        float mx = -INFINITY, mn = INFINITY;
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
            float v[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
            if (live) {
                if (VEC && c0 + 32 <= nv) {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        *(float4*)(row + c0 + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        mx = fmaxf(mx, v[j]);
                        mn = fminf(mn, v[j]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c0 + j < nv) {
                            row[c0 + j] = v[j];
                            mx = fmaxf(mx, v[j]);
                            mn = fminf(mn, v[j]);
                        }
                }
            }
        }
        if (live && mx >= mn) {
            atomicMax(&rowmax[(size_t)bh * s.m + i], order_key(mx));
            atomicMin(&rowmin[(size_t)bh * s.m + i], order_key(mn));
        }
    }
    fence_before();
    __syncthreads();
    if (warp == 0) tmem_free(tmem, 128);
}

// ---------------------------------------------------------------- landmark values
// 512 threads, TPR of them a landmark row: thread t builds the numerators of
// row t % RPB (RPB = 512 / TPR rows) for keys [KPT (t / RPB), + KPT) of each
// 128-key tile (KPT = 128 / TPR), with the next tile's scores already loaded
// into registers.  TPR = 4 covers the 128 rows of the MMA tile; TPR = 8
// (few landmarks) puts every thread on the first 64 rows.
// Warps w, w + 4 (w < 4) read the same tensor-memory lanes and split the D
// output columns.
template <int D, bool VEC, int TPR>
__global__ void __launch_bounds__(512) tc_values(const __grid_constant__ CUtensorMap mV, Shape s,
                                                 const float* __restrict__ S, const uint32_t* __restrict__ rowmax,
                                                 float* __restrict__ part, float cs, int kcv,
                                                 int32_t* __restrict__ status) {
    chain_wait_and_trigger();
    constexpr int KC = D / 64;                       // 64-wide feature chunks of a V tile
    constexpr uint32_t PBYTES = 2 * kChunk;          // numerators: 128 rows x 128 keys
    constexpr uint32_t VBYTES = KC * kChunk;         // V: 128 keys x D
    constexpr uint32_t STAGE = PBYTES + VBYTES;
    constexpr uint32_t TCOLS = D;                    // fp32 accumulator columns
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ uint32_t tslot;
    __shared__ __align__(8) uint64_t bars[5];        // v_full[2], mma_done[2], final
    __shared__ float rsum[512];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (smem_u32(smem) & 1023u) {
        if (tid == 0) atomicExch(status, (int)MITA_ERR_DEVICE);
        return;
    }
    const int split = blockIdx.x, i0 = blockIdx.y * 128, bh = blockIdx.z, ns = gridDim.x;
    const int jb0 = split * kcv, je = min(s.N, jb0 + kcv), ntile = (je - jb0 + 127) / 128;
    const uint32_t base = smem_u32(smem);
    const uint32_t bar0 = smem_u32(&bars[0]);
    auto v_full = [&](int st) { return bar0 + 8u * st; };
    auto mma_done = [&](int st) { return bar0 + 16u + 8u * st; };
    const uint32_t bar_fin = bar0 + 32u;
    if (tid == 0) {
        for (int b = 0; b < 5; ++b) mbar_init(bar0 + 8u * b, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(&tslot), TCOLS);
    __syncthreads();
    fence_after();
    const uint32_t tmem = tslot;
    constexpr int RPB = 512 / TPR, KPT = 128 / TPR;   // rows a pass, keys a thread
    const int r = tid % RPB, q = tid / RPB, i = i0 + r;
    const bool live = i < s.m;
    const float mb = live ? key_to_float(rowmax[(size_t)bh * s.m + i]) * cs : 0.0f;
    const float* srow = S + ((size_t)bh * s.m + (live ? i : 0)) * s.N;
    float psum = 0.0f;
    bool ok = true;
    auto issue_v = [&](int t) {
        const int st = t & 1;
        mbar_expect_tx(v_full(st), VBYTES);
        for (int kc = 0; kc < KC; ++kc)
            tma_load_2d(base + st * STAGE + PBYTES + kc * kChunk, &mV, kc * 64, bh * s.N + jb0 + 128 * t, v_full(st));
    };
    // this thread's KPT scores of tile t
    auto load_s = [&](int t, float (&x)[KPT]) {
        const int j = jb0 + 128 * t + KPT * q;
        if (VEC && live && j + KPT <= je) {
#pragma unroll
            for (int c = 0; c < KPT / 4; ++c) {
                const float4 a = __ldg((const float4*)(srow + j + 4 * c));
                x[4 * c] = a.x; x[4 * c + 1] = a.y; x[4 * c + 2] = a.z; x[4 * c + 3] = a.w;
            }
        } else {
#pragma unroll
            for (int u = 0; u < KPT; ++u) x[u] = (live && j + u < je) ? __ldg(srow + j + u) : -INFINITY;
        }
    };
    // 16-byte piece c of this thread's numerators: piece pc of row r in chunk ch of the A tile
    auto piece_addr = [&](int st, int c) {
        const int pg = q * (KPT / 8) + c, ch = pg >> 3, pc = pg & 7;
        return smem + st * STAGE + ch * kChunk + r * 128 + ((pc ^ (r & 7)) << 4);
    };
    if (tid == 0) {
        issue_v(0);
        if (ntile > 1) issue_v(1);
    }
    if (!live) {   // padding rows: zero numerators in both stages, written once
        for (int st = 0; st < 2; ++st)
#pragma unroll
            for (int c = 0; c < KPT / 8; ++c) *(uint4*)piece_addr(st, c) = make_uint4(0u, 0u, 0u, 0u);
    }
    if constexpr (RPB < 128) {   // rows RPB .. 127 of the A tile hold no landmark: zero in both stages
        constexpr int kPieces = (128 - RPB) * 16;   // 16-byte pieces a stage
        for (int x = tid; x < 2 * kPieces; x += 512) {
            const int st = x / kPieces, y = x % kPieces, rr = RPB + y / 16, pg = y % 16;
            *(uint4*)(smem + st * STAGE + (pg >> 3) * kChunk + rr * 128 + (((pg & 7) ^ (rr & 7)) << 4)) =
                make_uint4(0u, 0u, 0u, 0u);
        }
    }
    float x[KPT];
    if (live) load_s(0, x);
    for (int t = 0; t < ntile; ++t) {
        const int st = t & 1;
        const uint32_t sP = base + st * STAGE, sV = sP + PBYTES;
        if (t >= 2) {   // the stage is free again once the MMAs of tile t - 2 are done
            if (!mbar_wait_bounded(mma_done(st), ((t - 2) >> 1) & 1)) ok = false;
            if (tid == 0 && ok) issue_v(t);
        }
        // numerators of row r, keys KPT q .. KPT q + KPT - 1 of the tile
        if (live) {
        uint32_t w[KPT / 2];
#pragma unroll
        for (int u = 0; u < KPT / 2; ++u) {
            float p0, p1;
            asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(p0) : "f"(fmaf(x[2 * u], cs, -mb)));
            asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(p1) : "f"(fmaf(x[2 * u + 1], cs, -mb)));
            const __nv_bfloat162 pp = __floats2bfloat162_rn(p0, p1);
            psum += __low2float(pp) + __high2float(pp);
            w[u] = *reinterpret_cast<const uint32_t*>(&pp);
        }
        if (t + 1 < ntile) load_s(t + 1, x);   // in flight while the stores and the MMAs proceed
#pragma unroll
        for (int c = 0; c < KPT / 8; ++c)
            *(uint4*)piece_addr(st, c) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        }
        fence_async_smem();   // the numerators are read next by the tensor core
        __syncthreads();
        if (tid == 0 && ok) {
            if (!mbar_wait_bounded(v_full(st), (t >> 1) & 1)) ok = false;
            if (ok) {
                fence_after();
                constexpr uint32_t idesc = idesc_bf16(128, D, 0, 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t da = desc_kmajor(sP + (kk >> 2) * kChunk + (kk & 3) * 32);
                    const uint64_t db = desc_mnmajor(sV + kk * 16 * 128, kChunk);
                    mma_bf16(tmem, da, db, idesc, t > 0 || kk > 0);
                }
                mma_commit(mma_done(st));
            }
        }
    }
    if (tid == 0) mma_commit(bar_fin);
    rsum[tid] = psum;
    __syncthreads();
    const bool fin = mbar_wait_bounded(bar_fin, 0);
    if (!fin || !ok) {
        if (lane == 0) atomicExch(status, (int)MITA_ERR_TIMEOUT);
    } else if (warp < 8) {
        fence_after();
        const int lr = (warp & 3) * 32 + lane, li = i0 + lr, cbase = (warp >> 2) * (D / 2);
        float* dst = part + (((size_t)bh * ns + split) * s.m + (li < s.m ? li : 0)) * (D + 1);
#pragma unroll
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
            float v[32];
            tmem_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + cbase + c0, v);
            if (li < s.m)
#pragma unroll
                for (int j = 0; j < 32; ++j) dst[cbase + c0 + j] = v[j];
        }
        if (warp < 4 && li < s.m) {
            float den = 0.0f;
#pragma unroll
            for (int u = 0; u < TPR; ++u) den += rsum[lr + RPB * u];
            dst[D] = den;
        }
    }
    fence_before();
    __syncthreads();
    if (warp == 0) tmem_free(tmem, TCOLS);
}

// ---------------------------------------------------------------- routes
template <int D>
__global__ void __launch_bounds__(128) tc_route(const __grid_constant__ CUtensorMap mQ,
                                                const __grid_constant__ CUtensorMap mQl, Shape s, int nb, int tcols,
                                                int32_t* __restrict__ route, int32_t* __restrict__ counts,
                                                int32_t* __restrict__ status) {
    chain_wait_and_trigger();
    constexpr int KC = D / 64;
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ uint32_t tslot;
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int hist[256];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (smem_u32(smem) & 1023u) {
        if (tid == 0) atomicExch(status, (int)MITA_ERR_DEVICE);
        return;
    }
    const int q0 = blockIdx.x * 128, bh = blockIdx.y;
    const uint32_t sA = smem_u32(smem), sB = sA + KC * kChunk;
    const uint32_t bchunk = (uint32_t)nb * 128u;   // bytes per 64-column chunk of the landmark tile
    const uint32_t bar_ld = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[1]);
    for (int e = tid; e < 256; e += 128) hist[e] = 0;
    if (tid == 0) {
        mbar_init(bar_ld, 1);
        mbar_init(bar_mma, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(&tslot), (uint32_t)tcols);
    __syncthreads();
    fence_after();
    const uint32_t tmem = tslot;
    if (tid == 0) {
        mbar_expect_tx(bar_ld, KC * (kChunk + bchunk));
        for (int kc = 0; kc < KC; ++kc) {
            tma_load_2d(sA + kc * kChunk, &mQ, kc * 64, bh * s.N + q0, bar_ld);
            tma_load_2d(sB + kc * bchunk, &mQl, kc * 64, bh * s.m, bar_ld);
        }
        if (mbar_wait_bounded(bar_ld, 0)) {
            fence_after();
            const uint32_t idesc = idesc_bf16(128, nb, 0, 0);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t da = desc_kmajor(sA + (kk >> 2) * kChunk + (kk & 3) * 32);
                const uint64_t db = desc_kmajor(sB + (kk >> 2) * bchunk + (kk & 3) * 32);
                mma_bf16(tmem, da, db, idesc, kk > 0);
            }
            mma_commit(bar_mma);
        }
    }
    if (!mbar_wait_bounded(bar_mma, 0)) {
        if (lane == 0) atomicExch(status, (int)MITA_ERR_TIMEOUT);
    } else {
        fence_after();
        const int q = q0 + warp * 32 + lane;
        float best = -INFINITY;
        int arg = 0;
        for (int c0 = 0; c0 < nb; c0 += 32) {
            float v[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (c0 + j < s.m && v[j] > best) {   // ascending landmarks, strict: first argmax
                    best = v[j];
                    arg = c0 + j;
                }
        }
        if (q < s.N) {
            route[(size_t)bh * s.N + q] = arg;
            atomicAdd(&hist[arg], 1);
        }
    }
    fence_before();
    __syncthreads();
    for (int e = tid; e < s.m; e += 128)
        if (hist[e]) atomicAdd(&counts[(size_t)bh * s.m + e], hist[e]);
    if (warp == 0) tmem_free(tmem, (uint32_t)tcols);
}

// ---------------------------------------------------------------- scores and routes
// Scores and routes of one tile of 128 tokens (m <= 128 landmarks): both
// contractions take the token rows as M and the landmarks as N, against the
// one Q_l tile, S^T = K . Q_l^T at tensor-memory column 0 and R = Q . Q_l^T at
// column tcols / 2 (ROUTE), or the scores alone for up to 256 landmarks
// (!ROUTE; the routes then come from tc_route).  Thread t of the epilogue owns token n0 + t: it stores its
// column of S (for each landmark the warp's 32 consecutive keys are one
// 128-byte store), the warp's max and min of each landmark's scores (one
// floating-point redux each) go into the block's row keys, and the thread takes the
// first argmax of its query's logits (the route).  The block then adds its
// row keys and route counts to the global ones.
template <int D, bool ROUTE>
__global__ void __launch_bounds__(128) tc_scores_route(const __grid_constant__ CUtensorMap mK,
                                                       const __grid_constant__ CUtensorMap mQ,
                                                       const __grid_constant__ CUtensorMap mQl, Shape s, int nb,
                                                       int tcols, float* __restrict__ S, uint32_t* __restrict__ rowmax,
                                                       uint32_t* __restrict__ rowmin, int32_t* __restrict__ route,
                                                       int32_t* __restrict__ counts, int32_t* __restrict__ status) {
    chain_wait_and_trigger();
    constexpr int KC = D / 64;
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ uint32_t tslot;
    __shared__ __align__(8) uint64_t bars[2];
    constexpr int kML = ROUTE ? 128 : 256;   // landmarks a block takes
    __shared__ uint32_t smax[kML], smin[kML];
    __shared__ int hist[kML];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (smem_u32(smem) & 1023u) {
        if (tid == 0) atomicExch(status, (int)MITA_ERR_DEVICE);
        return;
    }
    const int n0 = blockIdx.x * 128, bh = blockIdx.y, m = s.m, N = s.N;
    const uint32_t sK = smem_u32(smem), sQ = sK + KC * kChunk, sB = ROUTE ? sQ + KC * kChunk : sQ;
    const uint32_t bchunk = (uint32_t)nb * 128u;   // bytes per 64-column chunk of the landmark tile
    const uint32_t bar_ld = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[1]);
    for (int e = tid; e < kML; e += 128) {
        smax[e] = 0u;
        smin[e] = 0xffffffffu;
    }
    const bool seq = !ROUTE && route != nullptr;   // routes after the scores, same columns
    for (int e = tid; e < kML; e += 128) hist[e] = 0;
    if (tid == 0) {
        mbar_init(bar_ld, 1);
        mbar_init(bar_mma, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(&tslot), (uint32_t)tcols);
    __syncthreads();
    fence_after();
    const uint32_t tmem = tslot, tR = tmem + (uint32_t)(tcols / 2);
    if (tid == 0) {
        mbar_expect_tx(bar_ld, KC * ((ROUTE ? 2 : 1) * kChunk + bchunk));
        for (int kc = 0; kc < KC; ++kc) {
            tma_load_2d(sK + kc * kChunk, &mK, kc * 64, bh * N + n0, bar_ld);
            if (ROUTE) tma_load_2d(sQ + kc * kChunk, &mQ, kc * 64, bh * N + n0, bar_ld);
            tma_load_2d(sB + kc * bchunk, &mQl, kc * 64, bh * m, bar_ld);
        }
        if (mbar_wait_bounded(bar_ld, 0)) {
            fence_after();
            const uint32_t idesc = idesc_bf16(128, nb, 0, 0);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t oa = (kk >> 2) * kChunk + (kk & 3) * 32;
                const uint64_t db = desc_kmajor(sB + (kk >> 2) * bchunk + (kk & 3) * 32);
                mma_bf16(tmem, desc_kmajor(sK + oa), db, idesc, kk > 0);
                if (ROUTE) mma_bf16(tR, desc_kmajor(sQ + oa), db, idesc, kk > 0);
            }
            mma_commit(bar_mma);
            // the key tile's slot takes the query tile once the MMAs have read it
            if (seq && mbar_wait_bounded(bar_mma, 0)) {
                mbar_expect_tx(bar_ld, KC * kChunk);
                for (int kc = 0; kc < KC; ++kc) tma_load_2d(sK + kc * kChunk, &mQ, kc * 64, bh * N + n0, bar_ld);
            }
        }
    }
    const int n = n0 + warp * 32 + lane;
    const bool live = n < N;
    const uint32_t lanes = (uint32_t)(warp * 32) << 16;
    // first argmax over the landmarks of this thread's query logits at
    // tensor-memory column tr (ascending landmarks, strict compare)
    auto take_route = [&](uint32_t tr) {
        float best = -INFINITY;
        int arg = 0;
        for (int c0 = 0; c0 < nb; c0 += 32) {
            float v[32];
            tmem_ld32(tr + lanes + c0, v);
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (c0 + j < m && v[j] > best) {
                    best = v[j];
                    arg = c0 + j;
                }
        }
        if (live) {
            route[(size_t)bh * N + n] = arg;
            atomicAdd(&hist[arg], 1);
        }
    };
    const bool ok = mbar_wait_bounded(bar_mma, 0);
    if (!ok) {
        if (lane == 0) atomicExch(status, (int)MITA_ERR_TIMEOUT);
    } else {
        fence_after();
        float* sp = S + (size_t)bh * m * N + n;   // advances one row of S per landmark
        // one chunk of 32 landmarks; FULL: every token of the tile is in the
        // row (block-uniform), so no lane needs masking; ALL: all 32
        // landmarks of the chunk exist, so no landmark is checked
        auto chunk = [&](int c0, auto full_t, auto all_t) {
            constexpr bool FULL = decltype(full_t)::value, ALL = decltype(all_t)::value;
            float v[32];
            tmem_ld32(tmem + lanes + c0, v);
            const int cn = ALL ? 32 : min(32, m - c0);
            float mine_hi = -INFINITY, mine_lo = INFINITY;   // lane j keeps landmark c0 + j's
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (ALL || j < cn) {   // block-uniform
                    if (FULL || live) *sp = v[j];
                    sp += N;
                    const float xh = FULL || live ? v[j] : -INFINITY, xl = FULL || live ? v[j] : INFINITY;
                    float hi, lo;
                    asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(hi) : "f"(xh));
                    asm("redux.sync.min.f32 %0, %1, 0xffffffff;" : "=f"(lo) : "f"(xl));
                    mine_hi = lane == j ? hi : mine_hi;
                    mine_lo = lane == j ? lo : mine_lo;
                }
            }
            if (lane < cn) {
                atomicMax(&smax[c0 + lane], order_key(mine_hi));
                atomicMin(&smin[c0 + lane], order_key(mine_lo));
            }
        };
        const int mfull = m & ~31;   // landmarks in whole chunks of 32
        if (n0 + 128 <= N) {
            for (int c0 = 0; c0 < mfull; c0 += 32) chunk(c0, std::true_type{}, std::true_type{});
            if (mfull < m) chunk(mfull, std::true_type{}, std::false_type{});
        } else {
            for (int c0 = 0; c0 < mfull; c0 += 32) chunk(c0, std::false_type{}, std::true_type{});
            if (mfull < m) chunk(mfull, std::false_type{}, std::false_type{});
        }
        if (ROUTE) take_route(tR);
    }
    fence_before();
    if (seq) {
        // every score read from tensor memory: R = Q . Q_l^T into the same columns
        const bool all_ok = __syncthreads_and(ok);
        if (all_ok && tid == 0) {
            fence_after();
            if (mbar_wait_bounded(bar_ld, 1)) {
                const uint32_t idesc = idesc_bf16(128, nb, 0, 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t oa = (kk >> 2) * kChunk + (kk & 3) * 32;
                    mma_bf16(tmem, desc_kmajor(sK + oa), desc_kmajor(sB + (kk >> 2) * bchunk + (kk & 3) * 32), idesc,
                             kk > 0);
                }
                mma_commit(bar_mma);
            }
        }
        if (all_ok) {
            if (!mbar_wait_bounded(bar_mma, 1)) {
                if (lane == 0) atomicExch(status, (int)MITA_ERR_TIMEOUT);
            } else {
                fence_after();
                take_route(tmem);
            }
        }
        fence_before();
    }
    __syncthreads();
    for (int e = tid; e < m; e += 128) {
        const size_t r = (size_t)bh * m + e;
        if (smax[e] != 0u) atomicMax(&rowmax[r], smax[e]);
        if (smin[e] != 0xffffffffu) atomicMin(&rowmin[r], smin[e]);
        if ((ROUTE || seq) && hist[e]) atomicAdd(&counts[r], hist[e]);
    }
    if (warp == 0) tmem_free(tmem, (uint32_t)tcols);
}

}  // namespace tcg

// ---------------------------------------------------------------- host side
// 2-D map over `rows` rows of `d` bf16, boxes of 64 columns x box_rows rows,
// 128-byte swizzle (rows past the end read as zero).
static bool map_rows(CUtensorMap* map, const void* base, int d, size_t rows, int box_rows) {
    return tma_map_bf16(map, base, d, rows, 64, box_rows);
}

template <int D>
static cudaError_t tc_scores_t(const Shape& s, const void* Ql, const void* K, float* S, uint32_t* rowmax,
                               uint32_t* rowmin, int32_t* status, cudaStream_t st, bool chain) {
    CUtensorMap mq, mk;
    if (!map_rows(&mq, Ql, D, (size_t)s.BH() * s.m, 128) || !map_rows(&mk, K, D, (size_t)s.BH() * s.N, 128))
        return cudaErrorInvalidValue;
    const int smem = 2 * (D / 64) * (int)tcg::kChunk + 1024;
    const dim3 grid((s.N + 127) / 128, (s.m + 127) / 128, s.BH());
    if (s.N % 4 == 0) {
        ensure_smem_attr((const void*)tcg::tc_scores<D, true>, smem);
        cudaError_t le = launch_chained(chain, tcg::tc_scores<D, true>, grid, dim3(128), smem, st, mq, mk, s, S, rowmax, rowmin, status);
        if (le != cudaSuccess) return le;
    } else {
        ensure_smem_attr((const void*)tcg::tc_scores<D, false>, smem);
        cudaError_t le = launch_chained(chain, tcg::tc_scores<D, false>, grid, dim3(128), smem, st, mq, mk, s, S, rowmax, rowmin, status);
        if (le != cudaSuccess) return le;
    }
    return cudaGetLastError();
}

// Keys per landmark-values split: as many splits as let every block of the
// launch run in one wave (two 512-thread blocks per SM), but no split shorter
// than eight 128-key tiles (shorter splits add more partials than they save:
// one head of 16K keys, 77.7 against 85 us), the row split as evenly as that
// allows.
int tc_value_keys(const Shape& s) {
    int sms = 148;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long rows = (long long)((s.m + 127) / 128) * s.BH();
    const long long tiles = (s.N + 127) / 128;
    long long ns = std::min((2LL * sms) / rows, tiles / 8);
    ns = std::max(1LL, ns);
    return (int)(((tiles + ns - 1) / ns) * 128);
}

template <int D>
static cudaError_t tc_values_t(const Shape& s, const float* S, const uint32_t* rowmax, const void* V, float* part,
                               float cs, int32_t* status, cudaStream_t st, bool chain) {
    CUtensorMap mv;
    if (!map_rows(&mv, V, D, (size_t)s.BH() * s.N, 128)) return cudaErrorInvalidValue;
    const int smem = 2 * (2 * (int)tcg::kChunk + (D / 64) * (int)tcg::kChunk) + 1024;
    const int kcv = tc_value_keys(s);
    const dim3 grid((s.N + kcv - 1) / kcv, (s.m + 127) / 128, s.BH());
    // eight threads a landmark row for at most 32 landmarks (DeiT-S backward
    // recompute 963.6 -> 947.7 us); at 49 landmarks (56x56) four measure
    // faster (177.9 against 179.3 us)
    auto kern = s.N % 4 == 0 ? (s.m <= 32 ? tcg::tc_values<D, true, 8> : tcg::tc_values<D, true, 4>)
                             : (s.m <= 32 ? tcg::tc_values<D, false, 8> : tcg::tc_values<D, false, 4>);
    ensure_smem_attr((const void*)kern, smem);
    cudaError_t le = launch_chained(chain, kern, grid, dim3(512), smem, st, mv, s, S, rowmax, part, cs, kcv, status);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

template <int D>
static cudaError_t tc_route_t(const Shape& s, const void* Q, const void* Ql, int32_t* route, int32_t* counts,
                              int32_t* status, cudaStream_t st, bool chain) {
    const int nb = (s.m + 15) / 16 * 16;
    int tcols = 32;
    while (tcols < nb) tcols <<= 1;
    CUtensorMap mq, ml;
    if (!map_rows(&mq, Q, D, (size_t)s.BH() * s.N, 128) || !map_rows(&ml, Ql, D, (size_t)s.BH() * s.m, nb))
        return cudaErrorInvalidValue;
    const int smem = (D / 64) * ((int)tcg::kChunk + nb * 128) + 1024;
    ensure_smem_attr((const void*)tcg::tc_route<D>, smem);
    cudaError_t le = launch_chained(chain, tcg::tc_route<D>, dim3((s.N + 127) / 128, s.BH()), dim3(128), smem, st, mq, ml, s,
                                    nb, tcols, route, counts, status);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

// ROUTE: scores and routes side by side (m <= 128); else the scores (m <=
// 256) and, when route is given, the routes after them in the same
// tensor-memory columns.
template <int D, bool ROUTE>
static cudaError_t tc_scores_route_t(const Shape& s, const void* Ql, const void* K, const void* Q, float* S,
                                     uint32_t* rowmax, uint32_t* rowmin, int32_t* route, int32_t* counts,
                                     int32_t* status, cudaStream_t st, bool chain) {
    const int nb = (s.m + 15) / 16 * 16;
    int tcols = 32;
    while (tcols < (ROUTE ? 2 : 1) * nb) tcols <<= 1;
    CUtensorMap mk, mq, ml;
    if (!map_rows(&mk, K, D, (size_t)s.BH() * s.N, 128) || !map_rows(&ml, Ql, D, (size_t)s.BH() * s.m, nb))
        return cudaErrorInvalidValue;
    if (route != nullptr) {
        if (!map_rows(&mq, Q, D, (size_t)s.BH() * s.N, 128)) return cudaErrorInvalidValue;
    } else {
        mq = mk;   // not read
    }
    // scores alone: at most 512 / tcols blocks a SM (the 512 tensor-memory
    // columns); the shared-memory request keeps a further block, which would
    // only wait in its allocation, off the SM (228 KB of shared memory a SM).
    // With the routes the smaller request measures faster (56x56: 193.0
    // against 194.5 us with the cap).
    const int smem0 = (D / 64) * ((ROUTE ? 2 : 1) * (int)tcg::kChunk + nb * 128) + 1024;
    const int smem = ROUTE ? smem0 : std::max(smem0, 233472 / (512 / tcols + 1));
    auto kern = tcg::tc_scores_route<D, ROUTE>;
    ensure_smem_attr((const void*)kern, smem);
    cudaError_t le = launch_chained(chain, kern, dim3((s.N + 127) / 128, s.BH()), dim3(128), smem, st, mk, mq, ml, s,
                                    nb, tcols, S, rowmax, rowmin, route, counts, status);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

bool tc_scores_route_supported(const Shape& s) { return s.m <= 256; }

cudaError_t tc_scores_route(const Shape& s, const void* Ql, const void* K, const void* Q, float* S, uint32_t* rowmax,
                            uint32_t* rowmin, int32_t* route, int32_t* counts, int32_t* status, cudaStream_t st,
                            bool chain) {
    if (s.m > 128)   // 256 tensor-memory columns for the scores, then the routes in the same ones
        return s.d == 64 ? tc_scores_route_t<64, false>(s, Ql, K, Q, S, rowmax, rowmin, route, counts, status, st, chain)
                         : tc_scores_route_t<128, false>(s, Ql, K, Q, S, rowmax, rowmin, route, counts, status, st,
                                                         chain);
    return s.d == 64 ? tc_scores_route_t<64, true>(s, Ql, K, Q, S, rowmax, rowmin, route, counts, status, st, chain)
                     : tc_scores_route_t<128, true>(s, Ql, K, Q, S, rowmax, rowmin, route, counts, status, st, chain);
}

int tc_value_splits(const Shape& s) { return (s.N + tc_value_keys(s) - 1) / tc_value_keys(s); }

cudaError_t tc_scores(const Shape& s, const void* Ql, const void* K, float* S, uint32_t* rowmax, uint32_t* rowmin,
                      int32_t* status, cudaStream_t st, bool chain) {
    if (s.m <= 256)   // token-major tiles: every store is 128 consecutive bytes of one row
        return s.d == 64 ? tc_scores_route_t<64, false>(s, Ql, K, nullptr, S, rowmax, rowmin, nullptr, nullptr,
                                                        status, st, chain)
                         : tc_scores_route_t<128, false>(s, Ql, K, nullptr, S, rowmax, rowmin, nullptr, nullptr,
                                                         status, st, chain);
    return s.d == 64 ? tc_scores_t<64>(s, Ql, K, S, rowmax, rowmin, status, st, chain)
                     : tc_scores_t<128>(s, Ql, K, S, rowmax, rowmin, status, st, chain);
}
cudaError_t tc_values(const Shape& s, const float* S, const uint32_t* rowmax, const void* V, float* part, float cs,
                      int32_t* status, cudaStream_t st, bool chain) {
    return s.d == 64 ? tc_values_t<64>(s, S, rowmax, V, part, cs, status, st, chain)
                     : tc_values_t<128>(s, S, rowmax, V, part, cs, status, st, chain);
}
cudaError_t tc_route(const Shape& s, const void* Q, const void* Ql, int32_t* route, int32_t* counts, int32_t* status,
                     cudaStream_t st, bool chain) {
    return s.d == 64 ? tc_route_t<64>(s, Q, Ql, route, counts, status, st, chain)
                     : tc_route_t<128>(s, Q, Ql, route, counts, status, st, chain);
}

}  // namespace mita
