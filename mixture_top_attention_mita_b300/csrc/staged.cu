// Stage-by-stage MiTA forward kernels (any supported shape).
//
// One kernel per step of the operator (36Kr / 新智元 "注意力也是FFN？", section
// "用少量地标查询，同时构造全局概括与细节专家"):
//   pool_kernel      step 1, landmark queries by adaptive average pooling
//   scores_kernel    step 2, raw landmark scores S = Q_l . K^T (fp32, [m, N])
//   topk_kernel      step 3, per-landmark radix select of the k best keys
//                    (topk_warp_kernel: rows of up to 256 keys)
//   values_rows_kernel  step 4, landmark values V_l = softmax(S / sqrt d) . V
//   route_kernel     step 5, first argmax of q . Q_l per query
//   bucket_kernel    step 5, stable counting sort of the queries by route
//   attend_kernel    step 6, one softmax over m shared + k routed keys
// These kernels favour plain structure over speed; the fused and tensor-core
// kernels handle the shapes they cover faster.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "staged.cuh"
#include "fused.cuh"
#include "tcgen.cuh"
#include "tiled.cuh"
#include "host_cache.cuh"
#include "launch.cuh"
#include "mma_util.cuh"

namespace mita {

// ---------------------------------------------------------------- step 1
// grid (m, BH), block d threads: thread f sums feature f over the bin's
// tokens (coalesced row reads) and writes the correctly rounded mean.
template <typename T>
__global__ void pool_kernel(Shape s, const T* __restrict__ Q, T* __restrict__ Ql) {
    const int i = blockIdx.x, bh = blockIdx.y, f = threadIdx.x;
    const int r = i / s.pw, c = i % s.pw;
    int r0, r1, c0, c1;
    pool_bin(r, s.gh, s.ph, r0, r1);
    pool_bin(c, s.gw, s.pw, c0, c1);
    const T* q = Q + (size_t)bh * s.N * s.d;
    float hi = 0.0f, lo = 0.0f;
    for (int y = r0; y < r1; ++y)
        for (int x = c0; x < c1; ++x) acc2(hi, lo, to_f32(q[(size_t)(y * s.gw + x) * s.d + f]));
    const float cnt = (float)((r1 - r0) * (c1 - c0));
    Ql[((size_t)bh * s.m + i) * s.d + f] = pooled_mean<T>(hi, lo, cnt);
}

// ---------------------------------------------------------------- step 2
// S[bh, i, j] = sum_f Q_l[i, f] K[j, f] in fp32.  Block tile: 32 landmarks x
// 128 keys, features staged through shared memory 32 at a time.
template <typename T>
__global__ void __launch_bounds__(256) scores_kernel(Shape s, const T* __restrict__ Ql,
                                                     const T* __restrict__ K, float* __restrict__ S) {
    __shared__ float a_s[32][33];
    __shared__ float b_s[128][33];
    const int bh = blockIdx.z, i0 = blockIdx.y * 32, j0 = blockIdx.x * 128;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 8 x 32
    const T* a = Ql + (size_t)bh * s.m * s.d;
    const T* b = K + (size_t)bh * s.N * s.d;
    float acc[4][4] = {};
    for (int f0 = 0; f0 < s.d; f0 += 32) {
        for (int e = threadIdx.x; e < 32 * 32; e += 256) {
            int r = e >> 5, f = e & 31;
            a_s[r][f] = (i0 + r < s.m) ? to_f32(a[(size_t)(i0 + r) * s.d + f0 + f]) : 0.0f;
        }
        for (int e = threadIdx.x; e < 128 * 32; e += 256) {
            int r = e >> 5, f = e & 31;
            b_s[r][f] = (j0 + r < s.N) ? to_f32(b[(size_t)(j0 + r) * s.d + f0 + f]) : 0.0f;
        }
        __syncthreads();
#pragma unroll 4
        for (int f = 0; f < 32; ++f) {
            float av[4], bv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) av[u] = a_s[ty * 4 + u][f];
#pragma unroll
            for (int u = 0; u < 4; ++u) bv[u] = b_s[tx + 32 * u][f];
#pragma unroll
            for (int p = 0; p < 4; ++p)
#pragma unroll
                for (int u = 0; u < 4; ++u) acc[p][u] = fmaf(av[p], bv[u], acc[p][u]);
        }
        __syncthreads();
    }
    float* out = S + (size_t)bh * s.m * s.N;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        int i = i0 + ty * 4 + p;
        if (i >= s.m) continue;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            int j = j0 + tx + 32 * u;
            if (j < s.N) out[(size_t)i * s.N + j] = acc[p][u];
        }
    }
}

// ---------------------------------------------------------------- block scan helper
// Exclusive prefix sum of one int per thread over a block of kThreads
// threads; returns the block total through *total.
template <int kThreads>
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    if (w == 0) {
        int t = lane < kThreads / 32 ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < kThreads / 32) warp_sums[lane] = t;   // inclusive
    }
    __syncthreads();
    int base = w ? warp_sums[w - 1] : 0;
    *total = warp_sums[kThreads / 32 - 1];
    __syncthreads();
    return base + x - v;
}

// ---------------------------------------------------------------- step 3
// One block per (landmark, head).  Radix select, 8 bits per pass from the
// top, finds the k-th largest order key T and how many keys equal to T are
// needed; a final pass in index order emits keys > T plus the lowest-index
// keys == T, which yields the expert in ascending index order with ties to
// the lower index.
constexpr int kTopkThreads = 512;

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(Shape s, const float* __restrict__ S,
                                                           int32_t* __restrict__ idx) {
    chain_wait_and_trigger();
    __shared__ int hist[256];
    __shared__ int warp_sums[32];
    __shared__ uint32_t sh_prefix;
    __shared__ int sh_need;
    const int i = blockIdx.x, bh = blockIdx.y;
    const float* row = S + ((size_t)bh * s.m + i) * s.N;
    uint32_t prefix = 0, mask = 0;
    int need = s.k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int e = threadIdx.x; e < 256; e += kTopkThreads) hist[e] = 0;
        __syncthreads();
        for (int j = threadIdx.x; j < s.N; j += kTopkThreads) {
            uint32_t key = order_key(row[j]);
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255], 1);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // lane L holds digits 255-8L .. 248-8L (descending)
            const int lane = threadIdx.x;
            int c[8], tot = 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) { c[u] = hist[255 - 8 * lane - u]; tot += c[u]; }
            int incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            int above = incl - tot;   // count in strictly higher digits
            // the lane whose range crosses `need`
            bool mine = above < need && incl >= need;
            if (mine) {
                int run = above, digit = 0, rem = need;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (run + c[u] >= need) { digit = 255 - 8 * lane - u; rem = need - run; break; }
                    run += c[u];
                }
                sh_prefix = prefix | ((uint32_t)digit << shift);
                sh_need = rem;
            }
        }
        __syncthreads();
        prefix = sh_prefix;
        need = sh_need;
        mask |= 255u << shift;
        __syncthreads();
    }
    // prefix == T; `need` keys equal to T are taken, lowest index first.
    int32_t* out = idx + ((size_t)bh * s.m + i) * s.k;
    int taken = 0, eq_seen = 0;
    for (int j0 = 0; j0 < s.N; j0 += kTopkThreads) {
        int j = j0 + threadIdx.x;
        uint32_t key = j < s.N ? order_key(row[j]) : 0u;
        int is_eq = (j < s.N && key == prefix) ? 1 : 0;
        int eq_tot;
        int eq_rank = eq_seen + block_exclusive_scan<kTopkThreads>(is_eq, warp_sums, &eq_tot);
        int sel = (j < s.N) && (key > prefix || (is_eq && eq_rank < need));
        int sel_tot;
        int pos = taken + block_exclusive_scan<kTopkThreads>(sel, warp_sums, &sel_tot);
        if (sel) out[pos] = j;
        taken += sel_tot;
        eq_seen += eq_tot;
    }
}

// Rows of up to kWarpTopkN keys: a warp per (landmark, head) with the row's
// order keys in registers (key lane + 32 u).  The k-th largest order key T is
// built bit by bit from the top (a warp-wide count of keys >= each
// candidate); the expert is every key above T plus the lowest-index keys
// equal to T, emitted in index order through ballots: the selection of
// topk_kernel, without its block-wide passes.
constexpr int kWarpTopkN = 256;

__global__ void __launch_bounds__(256) topk_warp_kernel(Shape s, const float* __restrict__ S,
                                                        int32_t* __restrict__ idx) {
    constexpr int U = kWarpTopkN / 32;
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * 8 + (threadIdx.x >> 5), bh = blockIdx.y;
    if (i >= s.m) return;
    const float* row = S + ((size_t)bh * s.m + i) * s.N;
    uint32_t key[U];   // 0 marks a slot past the row (no finite score maps to 0)
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int j = lane + 32 * u;
        key[u] = j < s.N ? order_key(row[j]) : 0u;
    }
    uint32_t T = 0;
    for (int b = 31; b >= 0; --b) {
        const uint32_t cand = T | (1u << b);
        int c = 0;
#pragma unroll
        for (int u = 0; u < U; ++u) c += key[u] >= cand ? 1 : 0;
        if (__reduce_add_sync(0xffffffffu, c) >= s.k) T = cand;
    }
    int gt = 0;
#pragma unroll
    for (int u = 0; u < U; ++u) gt += key[u] > T ? 1 : 0;
    const int need = s.k - __reduce_add_sync(0xffffffffu, gt);
    int32_t* out = idx + ((size_t)bh * s.m + i) * s.k;
    const unsigned lt = (1u << lane) - 1u;
    int taken = 0, eq_seen = 0;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const bool eq = key[u] == T;
        const unsigned be = __ballot_sync(0xffffffffu, eq);
        const bool sel = key[u] > T || (eq && eq_seen + __popc(be & lt) < need);
        const unsigned bs = __ballot_sync(0xffffffffu, sel);
        if (sel) out[taken + __popc(bs & lt)] = lane + 32 * u;
        taken += __popc(bs);
        eq_seen += __popc(be);
    }
}

// The expert lists of all landmarks from S (topk_warp_kernel on short rows).
static void launch_topk(const Shape& s, const float* S, int32_t* idx, cudaStream_t st) {
    if (s.N <= kWarpTopkN)
        topk_warp_kernel<<<dim3((s.m + 7) / 8, s.BH()), 256, 0, st>>>(s, S, idx);
    else
        topk_kernel<<<dim3(s.m, s.BH()), kTopkThreads, 0, st>>>(s, S, idx);
}

// ---------------------------------------------------------------- step 4
// Landmark values: values_rows_kernel (below, with the backward's kernels).

// ---------------------------------------------------------------- step 5
// One thread per query: raw scores q . Q_l[i] over all landmarks, first
// argmax.  Landmarks are staged through shared memory 32 at a time.
template <typename T, int D>
__global__ void __launch_bounds__(128) route_kernel(Shape s, const T* __restrict__ Q,
                                                   const T* __restrict__ Ql, int32_t* __restrict__ route, int ns,
                                                   int32_t* __restrict__ tops) {
    __shared__ float l_s[32][D];
    const int bh = blockIdx.y;
    const int qi = blockIdx.x * 128 + threadIdx.x;
    const bool live = qi < s.N;
    float q[D];
    const T* qp = Q + ((size_t)bh * s.N + (live ? qi : 0)) * D;
#pragma unroll
    for (int f = 0; f < D; ++f) q[f] = to_f32(qp[f]);
    float best = -INFINITY;
    int arg = 0;
    // s > 1: the ns best landmarks, best first (a later landmark displaces an
    // earlier one only with a strictly larger score: ties go to the lower index)
    float tv[kMaxRoutes];
    int ti[kMaxRoutes];
#pragma unroll
    for (int r = 0; r < kMaxRoutes; ++r) {
        tv[r] = -INFINITY;
        ti[r] = -1;
    }
    const T* lp = Ql + (size_t)bh * s.m * D;
    for (int i0 = 0; i0 < s.m; i0 += 32) {
        const int n = min(32, s.m - i0);
        __syncthreads();
        for (int e = threadIdx.x; e < n * D; e += 128) l_s[e / D][e % D] = to_f32(lp[(size_t)i0 * D + e]);
        __syncthreads();
        for (int u = 0; u < n; ++u) {
            float a = 0.0f;
#pragma unroll
            for (int f = 0; f < D; ++f) a = fmaf(q[f], l_s[u][f], a);
            if (i0 + u == 0 || a > best) { best = a; arg = i0 + u; }
            if (ns > 1) {
                int pos = ns;   // first place whose entry this score beats
#pragma unroll
                for (int r = kMaxRoutes - 1; r >= 0; --r)
                    if (r < ns && (ti[r] < 0 || a > tv[r])) pos = r;
                if (pos < ns) {
#pragma unroll
                    for (int r = kMaxRoutes - 1; r > 0; --r)
                        if (r < ns && r > pos) {
                            tv[r] = tv[r - 1];
                            ti[r] = ti[r - 1];
                        }
#pragma unroll
                    for (int r = 0; r < kMaxRoutes; ++r)
                        if (r == pos) {
                            tv[r] = a;
                            ti[r] = i0 + u;
                        }
                }
            }
        }
    }
    if (live) {
        route[(size_t)bh * s.N + qi] = arg;
        if (ns > 1)
#pragma unroll
            for (int r = 0; r < kMaxRoutes; ++r)
                if (r < ns) tops[((size_t)bh * s.N + qi) * ns + r] = ti[r];
    }
}

// One warp per head: per-landmark counts, exclusive offsets, and the
// queries listed bucket by bucket in ascending query order (stable).
__global__ void bucket_kernel(Shape s, const int32_t* __restrict__ route, int32_t* __restrict__ counts,
                              int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                              int32_t* __restrict__ status) {
    const int bh = blockIdx.x, lane = threadIdx.x;
    const int32_t* r = route + (size_t)bh * s.N;
    int32_t* cnt = counts + (size_t)bh * s.m;
    int32_t* off = offsets + (size_t)bh * (s.m + 1);
    int32_t* p = perm + (size_t)bh * s.N;
    for (int i = lane; i < s.m; i += 32) cnt[i] = 0;
    __syncwarp();
    for (int q = lane; q < s.N; q += 32) {
        int b = r[q];
        if (b < 0 || b >= s.m) { atomicExch(status, (int)MITA_ERR_DEVICE); continue; }
        atomicAdd(&cnt[b], 1);
    }
    __syncwarp();
    __threadfence_block();
    int carry = 0;
    for (int i0 = 0; i0 < s.m; i0 += 32) {
        int i = i0 + lane;
        int v = i < s.m ? __ldcg(&cnt[i]) : 0, x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (i < s.m) off[i] = carry + x - v;
        carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) off[s.m] = carry;
    __syncwarp();
    __threadfence_block();
    // cursor per bucket reuses counts
    for (int i = lane; i < s.m; i += 32) cnt[i] = off[i];
    __syncwarp();
    __threadfence_block();
    for (int q0 = 0; q0 < s.N; q0 += 32) {
        int q = q0 + lane;
        int b = q < s.N ? r[q] : -1;
        bool ok = b >= 0 && b < s.m;
        unsigned peers = __match_any_sync(0xffffffffu, ok ? b : -1);
        unsigned lower = peers & ((1u << lane) - 1u);
        int leader = __ffs(peers) - 1;
        int base = 0;
        if (ok && lane == leader) base = atomicAdd(&cnt[b], __popc(peers));
        base = __shfl_sync(peers, base, leader);
        if (ok) p[base + __popc(lower)] = q;
        __syncwarp();
    }
    // restore counts
    for (int i = lane; i < s.m; i += 32) cnt[i] = off[i + 1] - off[i];
}

// Longer rows, m <= kBucketMaxM: a block of 32 warps per head, warp w taking
// the queries of its contiguous segment.  Per-(bucket, warp) counts, one
// block-wide exclusive scan over them in (bucket, warp) order, then each warp
// places its segment again: the same stable listing as bucket_kernel.
constexpr int kBucketMaxM = 256;

__global__ void __launch_bounds__(1024) bucket_block_kernel(Shape s, const int32_t* __restrict__ route,
                                                            int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                            int32_t* __restrict__ perm, int32_t* __restrict__ status) {
    __shared__ int wc[kBucketMaxM * 32];   // [bucket][warp]: counts, then cursors
    __shared__ int warp_sums[32];
    const int bh = blockIdx.x, tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int32_t* r = route + (size_t)bh * s.N;
    int32_t* cnt = counts + (size_t)bh * s.m;
    int32_t* off = offsets + (size_t)bh * (s.m + 1);
    int32_t* p = perm + (size_t)bh * s.N;
    const int seg = (s.N + 1023) / 1024 * 32;   // queries per warp, whole 32-query steps
    const int q_beg = w * seg, q_end = min(s.N, q_beg + seg);
    for (int u = tid; u < s.m * 32; u += 1024) wc[u] = 0;
    __syncthreads();
    for (int q0 = q_beg; q0 < q_end; q0 += 32) {
        const int q = q0 + lane;
        const int b = q < q_end ? r[q] : -1;
        const bool ok = b >= 0 && b < s.m;
        if (q < q_end && !ok) atomicExch(status, (int)MITA_ERR_DEVICE);
        const unsigned peers = __match_any_sync(0xffffffffu, ok ? b : -1);
        if (ok && lane == __ffs(peers) - 1) wc[b * 32 + w] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    for (int b = tid; b < s.m; b += 1024) {
        int c = 0;
        for (int x = 0; x < 32; ++x) c += wc[b * 32 + x];
        cnt[b] = c;
    }
    const int E = (s.m * 32 + 1023) / 1024;   // entries per thread, <= 8
    int loc[8], sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int u = tid * E + j;
        loc[j] = j < E && u < s.m * 32 ? wc[u] : 0;
        sum += loc[j];
    }
    int total;
    int run = block_exclusive_scan<1024>(sum, warp_sums, &total);   // its barriers order the reads above
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int u = tid * E + j;
        if (j < E && u < s.m * 32) {
            wc[u] = run;
            run += loc[j];
        }
    }
    __syncthreads();
    for (int b = tid; b < s.m; b += 1024) off[b] = wc[b * 32];
    if (tid == 0) off[s.m] = total;
    for (int q0 = q_beg; q0 < q_end; q0 += 32) {
        const int q = q0 + lane;
        const int b = q < q_end ? r[q] : -1;
        const bool ok = b >= 0 && b < s.m;
        const unsigned peers = __match_any_sync(0xffffffffu, ok ? b : -1);
        const unsigned lower = peers & ((1u << lane) - 1u);
        const int leader = __ffs(peers) - 1;
        int base = 0;
        if (ok && lane == leader) {
            base = wc[b * 32 + w];
            wc[b * 32 + w] = base + __popc(peers);
        }
        base = __shfl_sync(peers, base, leader);
        if (ok) p[base + __popc(lower)] = q;
        __syncwarp();
    }
}

static void launch_bucket(const Shape& s, const int32_t* route, int32_t* counts, int32_t* offsets, int32_t* perm,
                          int32_t* status, cudaStream_t st) {
    if (s.N >= 2048 && s.m <= kBucketMaxM)
        bucket_block_kernel<<<s.BH(), 1024, 0, st>>>(s, route, counts, offsets, perm, status);
    else
        bucket_kernel<<<s.BH(), 32, 0, st>>>(s, route, counts, offsets, perm, status);
}

// The bucketing step alone, on a caller-made route array (test entry point).
cudaError_t testing_bucket(mita_plan_s* p, const int32_t* route, cudaStream_t st) {
    launch_bucket(p->s, route, p->counts, p->offsets, p->perm, p->status, st);
    return cudaGetLastError();
}

// Small vector helpers: a 4-term fused dot product and 4 elements of a row as
// fp32 (a bf16 is the upper half of the fp32 with the same value).
MITA_DEV float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
MITA_DEV float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

MITA_DEV float dot4(float4 a, float4 b, float acc) {
    return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, fmaf(a.x, b.x, acc))));
}

template <typename T>
MITA_DEV float4 load4(const T* p) {
    if constexpr (sizeof(T) == 4) {
        return *reinterpret_cast<const float4*>(p);
    } else {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
    }
}

// ---------------------------------------------------------------- step 6
// One warp per query, queries taken in bucket order so that neighbouring
// warps share an expert.  The query's slots (m shared, then the k keys of
// each of its ns experts) are listed in shared memory first: the landmark or
// key row of each, or -1 for a slot without weight (routing only, or a key
// an earlier expert of the query already holds, found by binary search in
// that expert's ascending list).  Logits and the output then take 4 slots per
// step, 8 lanes per slot, each lane D/8 features of the row (16-byte loads);
// the softmax is exact (max, exp, sum) in fp32.
constexpr int kAttendWarps = 4;

template <typename T, int F>
MITA_DEV void load_feats(const T* p, float (&v)[F]) {   // F consecutive elements, 16-byte aligned
    if constexpr (sizeof(T) == 2) {
#pragma unroll
        for (int i = 0; i < F; i += 8) {
            const uint4 u = *reinterpret_cast<const uint4*>(p + i);
            v[i] = bf16_lo(u.x); v[i + 1] = bf16_hi(u.x); v[i + 2] = bf16_lo(u.y); v[i + 3] = bf16_hi(u.y);
            v[i + 4] = bf16_lo(u.z); v[i + 5] = bf16_hi(u.z); v[i + 6] = bf16_lo(u.w); v[i + 7] = bf16_hi(u.w);
        }
    } else {
#pragma unroll
        for (int i = 0; i < F; i += 4) {
            const float4 x = load4(p + i);
            v[i] = x.x; v[i + 1] = x.y; v[i + 2] = x.z; v[i + 3] = x.w;
        }
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(32 * kAttendWarps)
    attend_kernel(Shape s, const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                  const T* __restrict__ Ql, const T* __restrict__ Vl, const int32_t* __restrict__ idx,
                  const int32_t* __restrict__ route, const int32_t* __restrict__ perm, T* __restrict__ out,
                  int shared, int ns, const int32_t* __restrict__ tops, int32_t* __restrict__ status) {
    constexpr int FPL = D / 8;   // features per lane
    extern __shared__ float smem[];
    __shared__ int r_s[kAttendWarps][kMaxRoutes];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, grp = lane >> 3, sub = lane & 7;
    const int L = s.m + ns * s.k;   // shared slots, then the k keys of each of the ns experts
    float* l_s = smem + (size_t)w * 2 * L;
    int* c_s = reinterpret_cast<int*>(l_s + L);
    const int bh = blockIdx.y;
    const int slot = blockIdx.x * kAttendWarps + w;
    if (slot >= s.N) return;
    const int qi = perm[(size_t)bh * s.N + slot];
    if (qi < 0 || qi >= s.N) { if (lane == 0) atomicExch(status, (int)MITA_ERR_DEVICE); return; }
    const int r = route[(size_t)bh * s.N + qi];
    if (r < 0 || r >= s.m) { if (lane == 0) atomicExch(status, (int)MITA_ERR_DEVICE); return; }
    // expert e of this query (e = 0: the route); an invalid landmark falls back to the route
    if (lane < ns) {
        int re = lane == 0 ? r : tops[((size_t)bh * s.N + qi) * ns + lane];
        if (re < 0 || re >= s.m) { atomicExch(status, (int)MITA_ERR_DEVICE); re = r; }
        r_s[w][lane] = re;
    }
    __syncwarp();
    for (int t = lane; t < L; t += 32) {
        int c;
        if (t < s.m) {
            c = shared ? t : -1;   // routing only: the shared slots take no weight
        } else {
            const int u = t - s.m, e = u / s.k;
            c = idx[((size_t)bh * s.m + r_s[w][e]) * s.k + (u - e * s.k)];
            if (c < 0 || c >= s.N) { atomicExch(status, (int)MITA_ERR_DEVICE); c = 0; }
        }
        c_s[t] = c;
    }
    __syncwarp();
    if (ns > 1) {   // a key already held by an earlier expert of this query takes part once
        for (int t = s.m + s.k + lane; t < L; t += 32) {
            const int u = t - s.m, e = u / s.k, j = c_s[t];
            bool dup = false;
            for (int e2 = 0; e2 < e && !dup; ++e2) {
                const int* E2 = c_s + s.m + e2 * s.k;
                int lo = 0, hi = s.k - 1;
                while (lo <= hi) {
                    const int mid = (lo + hi) >> 1;
                    if (E2[mid] == j) { dup = true; break; }
                    if (E2[mid] < j) lo = mid + 1; else hi = mid - 1;
                }
            }
            l_s[t] = dup ? 1.0f : 0.0f;
        }
        __syncwarp();
        for (int t = s.m + s.k + lane; t < L; t += 32)
            if (l_s[t] != 0.0f) c_s[t] = -1;
        __syncwarp();
    }
    const size_t hoff = (size_t)bh * s.N * D;
    const T* lq = Ql + (size_t)bh * s.m * D;
    const T* lv = Vl + (size_t)bh * s.m * D;
    float qf[FPL];
    load_feats<T, FPL>(Q + hoff + (size_t)qi * D + sub * FPL, qf);
    const float scale = rsqrtf((float)D);
    float mx = -INFINITY;
    for (int t0 = 0; t0 < L; t0 += 4) {
        const int t = t0 + grp;
        const int c = t < L ? c_s[t] : -1;
        float a = 0.0f;
        if (c >= 0) {
            float kf[FPL];
            load_feats<T, FPL>((t < s.m ? lq : K + hoff) + (size_t)c * D + sub * FPL, kf);
#pragma unroll
            for (int i = 0; i < FPL; ++i) a = fmaf(qf[i], kf[i], a);
        }
        a += __shfl_xor_sync(0xffffffffu, a, 1);
        a += __shfl_xor_sync(0xffffffffu, a, 2);
        a += __shfl_xor_sync(0xffffffffu, a, 4);
        const float lg = c >= 0 ? a * scale : -INFINITY;
        if (sub == 0 && t < L) l_s[t] = lg;
        mx = fmaxf(mx, lg);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    __syncwarp();
    float den = 0.0f;
    for (int t = lane; t < L; t += 32) {
        const float p = exp2f((l_s[t] - mx) * kLog2e);
        l_s[t] = p;
        den += p;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    __syncwarp();
    float acc[FPL];
#pragma unroll
    for (int i = 0; i < FPL; ++i) acc[i] = 0.0f;
    for (int t0 = 0; t0 < L; t0 += 4) {
        const int t = t0 + grp;
        if (t >= L) continue;
        const float p = l_s[t];
        const int c = c_s[t];
        if (p == 0.0f || c < 0) continue;   // no weight (or an underflow: none either way)
        float vf[FPL];
        load_feats<T, FPL>((t < s.m ? lv : V + hoff) + (size_t)c * D + sub * FPL, vf);
#pragma unroll
        for (int i = 0; i < FPL; ++i) acc[i] = fmaf(p, vf[i], acc[i]);
    }
#pragma unroll
    for (int i = 0; i < FPL; ++i) {
        acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 8);
        acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 16);
    }
    if (grp == 0) {
        const float inv = 1.0f / den;
        T* o = out + hoff + (size_t)qi * D + sub * FPL;
#pragma unroll
        for (int i = 0; i < FPL; ++i) o[i] = from_f32<T>(acc[i] * inv);
    }
}

size_t staged_attend_smem(const Shape& s, int ns) {
    return (size_t)kAttendWarps * 2 * (s.m + (size_t)ns * s.k) * sizeof(float);
}

// ---------------------------------------------------------------- launcher
template <typename T, int D>
static int launch_values_rows(const Shape& s, const float* S, const T* V, T* Vl, float* Vl32, float* stats,
                              float* scratch, size_t scratch_bytes, cudaStream_t st);

template <typename T, int D>
static cudaError_t run_staged_t(mita_plan_s* p, const T* Q, const T* K, const T* V, T* out, int32_t* idx,
                                int32_t* route, cudaStream_t st) {
    const Shape& s = p->s;
    const int BH = s.BH();
    T* Ql = (T*)p->Ql;
    T* Vl = (T*)p->Vl;
    int nv = 0;
    bool one_kernel = false;   // landmarks, experts and landmark values from the one-kernel path
    if constexpr (std::is_same<T, __nv_bfloat16>::value)
        one_kernel = p->routes_s > 1 && fused_supported(s, MITA_BF16);
    if (one_kernel) {
        // its output (one expert per query) is overwritten by the attention below
        cudaError_t e = run_fused(p, Q, K, V, out, idx, route, 1, st);
        if (e != cudaSuccess) return e;
        nv = -3;   // run_fused counts its own launch; route, bucket and attention follow
    } else {
        pool_kernel<T><<<dim3(s.m, BH), D, 0, st>>>(s, Q, Ql);
        scores_kernel<T><<<dim3((s.N + 127) / 128, (s.m + 31) / 32, BH), 256, 0, st>>>(s, Ql, K, p->S);
        launch_topk(s, p->S, idx, st);
        // key-split partial sums (if any) use the output as scratch before the attention writes it
        nv = launch_values_rows<T, D>(s, p->S, V, Vl, nullptr, nullptr, reinterpret_cast<float*>(out),
                                      (size_t)BH * s.N * D * sizeof(T), st);
    }
    // s > 1: each query's landmark list goes into the score buffer, free once
    // the landmark values are done (BH x N x s <= BH x m x N entries)
    const int ns = p->routes_s > 1 ? p->routes_s : 1;
    int32_t* tops = (int32_t*)p->S;
    route_kernel<T, D><<<dim3((s.N + 127) / 128, BH), 128, 0, st>>>(s, Q, Ql, route, ns, tops);
    launch_bucket(s, route, p->counts, p->offsets, p->perm, p->status, st);
    const size_t smem = staged_attend_smem(s, ns);
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    ensure_smem_attr((const void*)attend_kernel<T, D>, (int)smem);
    attend_kernel<T, D><<<dim3((s.N + kAttendWarps - 1) / kAttendWarps, BH), 32 * kAttendWarps, smem, st>>>(
        s, Q, K, V, Ql, Vl, idx, route, p->perm, out, p->routing_only ? 0 : 1, ns, tops, p->status);
    p->launches += 6 + nv;
    return cudaGetLastError();
}

// ---------------------------------------------------------------- backward
// The backward pass of the operator with the experts and routes held as
// constants (see mita.h).  The output softmax: expert_bwd_mma_kernel (bf16,
// d = 64) or expert_bwd_kernel (fp32 I/O, d = 128), a block per expert, where
// the expert's m + k slots fit on chip; attend_bwd_kernel (warp per query)
// otherwise.  The landmark values: values_bwd_tile_kernel (block per 64-key
// tile).  The bin means: pool_bwd_kernel.  Gradients are fp32; the slot and
// landmark gradients are added with atomics.

// Warp per query: the forward's logits and weights again, dw = dOut . v,
// dlogit = w (dw - w . dw); the query's own gradient is stored, the shared
// keys' and values' (dQ_l, dV_l) and the routed rows' (dK, dV) are added.
template <typename T, int D>
__global__ void __launch_bounds__(32 * kAttendWarps)
    attend_bwd_kernel(Shape s, const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                      const T* __restrict__ Ql, const T* __restrict__ Vl, const int32_t* __restrict__ idx,
                      const int32_t* __restrict__ route, const T* __restrict__ dOut, float* __restrict__ dQ,
                      float* __restrict__ dK, float* __restrict__ dV, float* __restrict__ dQl,
                      float* __restrict__ dVl, int shared, int32_t* __restrict__ status) {
    extern __shared__ float smem[];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = s.m + s.k;
    float* q_s = smem + w * (2 * D + 2 * L);
    float* g_s = q_s + D;     // dOut row
    float* l_s = g_s + D;     // weights
    float* d_s = l_s + L;     // logit gradients
    const int bh = blockIdx.y, qi = blockIdx.x * kAttendWarps + w;
    if (qi >= s.N) return;
    const int r = route[(size_t)bh * s.N + qi];
    if (r < 0 || r >= s.m) { if (lane == 0) atomicExch(status, (int)MITA_ERR_DEVICE); return; }
    const size_t hoff = (size_t)bh * s.N * D;
    for (int f = lane; f < D; f += 32) {
        q_s[f] = to_f32(Q[hoff + (size_t)qi * D + f]);
        g_s[f] = to_f32(dOut[hoff + (size_t)qi * D + f]);
    }
    __syncwarp();
    const T* lq = Ql + (size_t)bh * s.m * D;
    const T* lv = Vl + (size_t)bh * s.m * D;
    const int32_t* E = idx + ((size_t)bh * s.m + r) * s.k;
    auto key_row = [&](int t) -> int {   // routed slot t: its key, checked
        int j = E[t - s.m];
        if (j < 0 || j >= s.N) { atomicExch(status, (int)MITA_ERR_DEVICE); j = 0; }
        return j;
    };
    const float scale = rsqrtf((float)D);
    float mx = -INFINITY;
    for (int t = lane; t < L; t += 32) {
        float a = -INFINITY;
        if (t >= s.m || shared) {
            const T* key = t < s.m ? lq + (size_t)t * D : K + hoff + (size_t)key_row(t) * D;
            a = 0.0f;
#pragma unroll 8
            for (int f = 0; f < D; ++f) a = fmaf(q_s[f], to_f32(key[f]), a);
            a *= scale;
        }
        l_s[t] = a;
        mx = fmaxf(mx, a);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    __syncwarp();
    float den = 0.0f;
    for (int t = lane; t < L; t += 32) {
        const float p = exp2f((l_s[t] - mx) * kLog2e);
        l_s[t] = p;
        den += p;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    const float inv = 1.0f / den;
    float wdw = 0.0f;
    for (int t = lane; t < L; t += 32) {
        const float wt = l_s[t] * inv;
        l_s[t] = wt;
        float dw = 0.0f;
        if (wt != 0.0f) {
            const T* v = t < s.m ? lv + (size_t)t * D : V + hoff + (size_t)key_row(t) * D;
#pragma unroll 8
            for (int f = 0; f < D; ++f) dw = fmaf(g_s[f], to_f32(v[f]), dw);
        }
        d_s[t] = dw;
        wdw = fmaf(wt, dw, wdw);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wdw += __shfl_xor_sync(0xffffffffu, wdw, o);
    for (int t = lane; t < L; t += 32) d_s[t] = l_s[t] * (d_s[t] - wdw);
    __syncwarp();
    float dq[D / 32];
#pragma unroll
    for (int u = 0; u < D / 32; ++u) dq[u] = 0.0f;
    for (int t = 0; t < L; ++t) {
        const float c = d_s[t], wt = l_s[t];
        if (c == 0.0f && wt == 0.0f) continue;
        const bool sh = t < s.m;
        const int j = sh ? t : key_row(t);
        const T* key = sh ? lq + (size_t)j * D : K + hoff + (size_t)j * D;
        float* gk = sh ? dQl + ((size_t)bh * s.m + j) * D : dK + hoff + (size_t)j * D;
        float* gv = sh ? dVl + ((size_t)bh * s.m + j) * D : dV + hoff + (size_t)j * D;
#pragma unroll
        for (int u = 0; u < D / 32; ++u) {
            const int f = lane + 32 * u;
            dq[u] = fmaf(c, to_f32(key[f]), dq[u]);
            if (c != 0.0f) atomicAdd(gk + f, c * q_s[f] * scale);
            if (wt != 0.0f) atomicAdd(gv + f, wt * g_s[f]);
        }
    }
#pragma unroll
    for (int u = 0; u < D / 32; ++u) dQ[hoff + (size_t)qi * D + lane + 32 * u] = dq[u] * scale;
}

// Block of NW warps per (expert e, head): the queries routed to e, in bucket
// order and in chunks of QW NW, against the expert's m + k keys and values, which stay in
// shared memory as fp32 for the whole block.  Per chunk: logits and dw =
// dOut . v (lane per key; warp w takes rows w, w + NW, ... so that a short
// chunk still gives every warp a row), the softmax and dlogit =
// w (dw - w . dw) in registers, the chunk's dQ rows (stored: a query has one
// expert), and the key and value gradients of the chunk added to per-thread
// 4 x 4 tiles.  Those are summed over all of e's queries on chip and leave
// with one float4 atomic add per (slot, 4 features): to dQ_l / dV_l for the
// shared slots, to dK / dV for the routed keys.  Slots are padded to LP =
// 32 JT; a padded slot reads the last real row and is masked out.


inline size_t expert_bwd_bytes(int D, int L, int LP, int QC) {
    return (2 * (size_t)L * (D + 4) + 2 * (size_t)QC * D + 2 * (size_t)QC * LP) * sizeof(float);
}

template <typename T, int D, int JT, int NW, int QW>
__global__ void __launch_bounds__(32 * NW, NW == 8 ? 3 : 1)
    expert_bwd_kernel(Shape s, const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                      const T* __restrict__ Ql, const T* __restrict__ Vl, const int32_t* __restrict__ idx,
                      const int32_t* __restrict__ offsets, const int32_t* __restrict__ perm,
                      const T* __restrict__ dOut, float* __restrict__ dQ, float* __restrict__ dK,
                      float* __restrict__ dV, float* __restrict__ dQl, float* __restrict__ dVl, int shared,
                      int32_t* __restrict__ status) {
    constexpr int kEbThreads = 32 * NW, kEbQ = QW * NW;
    constexpr int KS = D + 4;                  // key / value row stride (floats)
    constexpr int LP = 32 * JT;                // padded slots
    constexpr int NC = D / 4;                  // float4 columns
    constexpr int RG = kEbThreads / NC;        // row groups of the tiles
    constexpr int QPT = kEbQ / RG;             // dQ rows per thread
    constexpr int TR = (LP / 4 + RG - 1) / RG; // 4-slot gradient tiles per thread
    static_assert(kEbQ % RG == 0 && kEbQ >= RG, "tile split");
    extern __shared__ float4 eb_smem[];
    __shared__ int32_t qid[kEbQ];
    __shared__ int32_t kid[LP];
    const int e = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int L = s.m + s.k;
    const int32_t* off = offsets + (size_t)bh * (s.m + 1);
    const int beg = off[e], cnt = off[e + 1] - beg;
    if (cnt <= 0) return;
    float* Ks = reinterpret_cast<float*>(eb_smem);
    float* Vs = Ks + (size_t)L * KS;
    float* Qs = Vs + (size_t)L * KS;   // [kEbQ][D]
    float* Gs = Qs + kEbQ * D;         // dOut rows
    float* Ws = Gs + kEbQ * D;         // [kEbQ][LP] weights
    float* Cs = Ws + kEbQ * LP;        // [kEbQ][LP] logit gradients
    const size_t hoff = (size_t)bh * s.N * D;
    const int32_t* E = idx + ((size_t)bh * s.m + e) * s.k;
    const int32_t* P = perm + (size_t)bh * s.N + beg;
    // query ids of the chunk at c0, then its Q and dOut rows (after a barrier)
    auto load_ids = [&](int c0) {
        const int nq = min(kEbQ, cnt - c0);
        if (tid < kEbQ) {
            int q = tid < nq ? P[c0 + tid] : -1;
            if (tid < nq && (q < 0 || q >= s.N)) { atomicExch(status, (int)MITA_ERR_DEVICE); q = -1; }
            qid[tid] = q;
        }
    };
    auto stage_rows = [&]() {
        for (int u = tid; u < kEbQ * NC; u += kEbThreads) {
            const int r = u / NC, c = 4 * (u % NC);
            float4 qv = make_float4(0.f, 0.f, 0.f, 0.f), g = qv;
            if (qid[r] >= 0) {
                qv = load4(Q + hoff + (size_t)qid[r] * D + c);
                g = load4(dOut + hoff + (size_t)qid[r] * D + c);
            }
            *reinterpret_cast<float4*>(Qs + r * D + c) = qv;
            *reinterpret_cast<float4*>(Gs + r * D + c) = g;
        }
    };
    // slot keys and the first chunk's ids in one round trip, then the slot
    // rows and the first chunk's rows in another
    for (int t = tid; t < LP; t += kEbThreads) {
        int j = -1;
        if (t >= s.m && t < L) {
            j = E[t - s.m];
            if (j < 0 || j >= s.N) { atomicExch(status, (int)MITA_ERR_DEVICE); j = -1; }
        }
        kid[t] = j;
    }
    load_ids(0);
    __syncthreads();   // ids ready
    for (int u = tid; u < L * NC; u += kEbThreads) {
        const int t = u / NC, c = 4 * (u % NC);
        float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
        if (t < s.m) {
            kv = load4(Ql + ((size_t)bh * s.m + t) * D + c);
            vv = load4(Vl + ((size_t)bh * s.m + t) * D + c);
        } else if (kid[t] >= 0) {
            kv = load4(K + hoff + (size_t)kid[t] * D + c);
            vv = load4(V + hoff + (size_t)kid[t] * D + c);
        }
        *reinterpret_cast<float4*>(Ks + t * KS + c) = kv;
        *reinterpret_cast<float4*>(Vs + t * KS + c) = vv;
    }
    const float scale = rsqrtf((float)D);
    const int tc = tid % NC, rg = tid / NC;
    float gk[TR][4][4], gv[TR][4][4];
#pragma unroll
    for (int r = 0; r < TR; ++r)
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) gk[r][a][b] = gv[r][a][b] = 0.0f;
    for (int c0 = 0;;) {
        const int nq = min(kEbQ, cnt - c0);
        stage_rows();      // the first chunk's rows load with the slot rows
        __syncthreads();
        // logits and dw: warp w takes chunk rows w + NW i (i < n), lane the slots lane + 32j
        auto rows = [&](auto nc) {
            constexpr int n = decltype(nc)::value;
            float a[n][JT], dw[n][JT];
#pragma unroll
            for (int i = 0; i < n; ++i)
#pragma unroll
                for (int j = 0; j < JT; ++j) a[i][j] = dw[i][j] = 0.0f;
#pragma unroll 1
            for (int f = 0; f < D; f += 4) {
                float4 qv[n], g[n];
#pragma unroll
                for (int i = 0; i < n; ++i) {
                    qv[i] = *reinterpret_cast<const float4*>(Qs + (w + NW * i) * D + f);
                    g[i] = *reinterpret_cast<const float4*>(Gs + (w + NW * i) * D + f);
                }
#pragma unroll
                for (int j = 0; j < JT; ++j) {
                    const int t = min(lane + 32 * j, L - 1);
                    const float4 kv = *reinterpret_cast<const float4*>(Ks + t * KS + f);
                    const float4 vv = *reinterpret_cast<const float4*>(Vs + t * KS + f);
#pragma unroll
                    for (int i = 0; i < n; ++i) {
                        a[i][j] = dot4(qv[i], kv, a[i][j]);
                        dw[i][j] = dot4(g[i], vv, dw[i][j]);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < n; ++i) {
                const int r = w + NW * i;
                float mx = -INFINITY;
#pragma unroll
                for (int j = 0; j < JT; ++j) {
                    const int t = lane + 32 * j;
                    const bool live = t < L && (t >= s.m ? kid[t] >= 0 : shared != 0);
                    a[i][j] = live ? a[i][j] * scale : -INFINITY;
                    mx = fmaxf(mx, a[i][j]);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                float den = 0.0f;
#pragma unroll
                for (int j = 0; j < JT; ++j) {
                    a[i][j] = exp2f((a[i][j] - mx) * kLog2e);
                    den += a[i][j];
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
                const float inv = 1.0f / den;
                float wdw = 0.0f;
#pragma unroll
                for (int j = 0; j < JT; ++j) {
                    a[i][j] *= inv;
                    wdw = fmaf(a[i][j], dw[i][j], wdw);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) wdw += __shfl_xor_sync(0xffffffffu, wdw, o);
#pragma unroll
                for (int j = 0; j < JT; ++j) {
                    Ws[r * LP + lane + 32 * j] = a[i][j];
                    Cs[r * LP + lane + 32 * j] = a[i][j] * (dw[i][j] - wdw);
                }
            }
        };
        {
            const int nrow = w < nq ? min(QW, (nq - w + NW - 1) / NW) : 0;   // rows of this warp
            if (nrow == 1) rows(std::integral_constant<int, 1>{});
            else if (nrow == 2 || (QW == 2 && nrow > 0)) rows(std::integral_constant<int, 2>{});
            else if (nrow > 2) rows(std::integral_constant<int, QW>{});
        }
        __syncthreads();
        // dQ rows rg + RG u: sum over slots of dlogit . key, 4 features per thread
        {
            float acc[QPT][4];
#pragma unroll
            for (int u = 0; u < QPT; ++u)
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[u][b] = 0.0f;
            if (rg < nq) {
                for (int t = 0; t < L; ++t) {
                    const float4 kv = *reinterpret_cast<const float4*>(Ks + t * KS + 4 * tc);
#pragma unroll
                    for (int u = 0; u < QPT; ++u) {
                        const float c = Cs[(rg + RG * u) * LP + t];
                        acc[u][0] = fmaf(c, kv.x, acc[u][0]);
                        acc[u][1] = fmaf(c, kv.y, acc[u][1]);
                        acc[u][2] = fmaf(c, kv.z, acc[u][2]);
                        acc[u][3] = fmaf(c, kv.w, acc[u][3]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < QPT; ++u) {
                const int r = rg + RG * u;
                if (r < nq && qid[r] >= 0)
                    *reinterpret_cast<float4*>(dQ + hoff + (size_t)qid[r] * D + 4 * tc) =
                        make_float4(acc[u][0] * scale, acc[u][1] * scale, acc[u][2] * scale, acc[u][3] * scale);
            }
        }
        // key and value gradients of the slot tiles (rg + RG r), features 4 tc..
        for (int q = 0; q < nq; ++q) {
            const float4 qv = *reinterpret_cast<const float4*>(Qs + q * D + 4 * tc);
            const float4 g = *reinterpret_cast<const float4*>(Gs + q * D + 4 * tc);
#pragma unroll
            for (int r = 0; r < TR; ++r) {
                const int t0 = 4 * (rg + RG * r);
                if (t0 < LP) {
                    const float4 c = *reinterpret_cast<const float4*>(Cs + q * LP + t0);
                    const float4 wt = *reinterpret_cast<const float4*>(Ws + q * LP + t0);
                    const float cc[4] = {c.x, c.y, c.z, c.w}, ww[4] = {wt.x, wt.y, wt.z, wt.w};
                    const float qq[4] = {qv.x, qv.y, qv.z, qv.w}, gg[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
                    for (int a = 0; a < 4; ++a)
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            gk[r][a][b] = fmaf(cc[a], qq[b], gk[r][a][b]);
                            gv[r][a][b] = fmaf(ww[a], gg[b], gv[r][a][b]);
                        }
                }
            }
        }
        c0 += kEbQ;
        if (c0 >= cnt) break;
        __syncthreads();   // the chunk's tiles are consumed
        load_ids(c0);
        __syncthreads();
    }
#pragma unroll
    for (int r = 0; r < TR; ++r) {
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int t = 4 * (rg + RG * r) + a;
            if (t >= L) continue;
            float* rk;
            float* rv;
            if (t < s.m) {
                if (!shared) continue;
                rk = dQl + ((size_t)bh * s.m + t) * D;
                rv = dVl + ((size_t)bh * s.m + t) * D;
            } else {
                if (kid[t] < 0) continue;
                rk = dK + hoff + (size_t)kid[t] * D;
                rv = dV + hoff + (size_t)kid[t] * D;
            }
            atomicAdd(reinterpret_cast<float4*>(rk + 4 * tc),
                      make_float4(gk[r][a][0] * scale, gk[r][a][1] * scale, gk[r][a][2] * scale,
                                  gk[r][a][3] * scale));
            atomicAdd(reinterpret_cast<float4*>(rv + 4 * tc),
                      make_float4(gv[r][a][0], gv[r][a][1], gv[r][a][2], gv[r][a][3]));
        }
    }
}

// expert_bwd_kernel for bf16 I/O at d = 64 with the five products on
// mma.sync (m16n8k16, fp32 accumulation): logits = Q . K_slots^T and
// dw = dOut . V_slots^T take the bf16 rows as they are (exact products);
// dQ = C . K_slots, dK_slots = C^T . Q and dV_slots = W^T . dOut take the
// fp32 weights W and logit gradients C as a bf16 pair hi + lo (about 16
// mantissa bits).  The softmax between them runs per row on the fp32 logits
// (lane per slot).  Tiles are bf16 rows with XOR-swizzled 16-byte chunks;
// rows past the chunk's queries and slots past the expert are zero.  Chunks
// hold QC queries; the slot gradients stay in registers (warp w: slot tile
// w % (LP/16)) until one float2 atomic add per (slot, 2 features).
template <int LP, int QC, int NW>
__global__ void __launch_bounds__(32 * NW, NW == 8 ? 3 : 1)
    expert_bwd_mma_kernel(Shape s, const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K,
                          const __nv_bfloat16* __restrict__ V, const __nv_bfloat16* __restrict__ Ql,
                          const __nv_bfloat16* __restrict__ Vl, const int32_t* __restrict__ idx,
                          const int32_t* __restrict__ offsets, const int32_t* __restrict__ perm,
                          const __nv_bfloat16* __restrict__ dOut, float* __restrict__ dQ, float* __restrict__ dK,
                          float* __restrict__ dV, float* __restrict__ dQl, float* __restrict__ dVl, int shared,
                          int32_t* __restrict__ status) {
    using namespace mx;
    constexpr int D = 64, NT = 32 * NW;
    constexpr int RBk = D * 2;    // bytes per row of the K, V, Q, dOut tiles
    constexpr int RBc = LP * 2;   // bytes per row of the C and W tiles
    constexpr int FS = LP + 8;    // fp32 row stride of the logit tiles
    constexpr int MT1 = QC / 16, N1 = (LP / 8) / (NW / MT1);
    constexpr int MTq = QC / 16, Nq = (D / 8) / (NW / MTq);
    constexpr int MTk = LP / 16, Nk = (D / 8) / (NW / MTk);
    static_assert(NW % MT1 == 0 && NW % MTk == 0 && N1 % 2 == 0 && Nq % 2 == 0 && Nk % 2 == 0, "warp split");
    extern __shared__ __align__(128) uint8_t ebm_raw[];
    uint8_t* Kb = ebm_raw;           // [LP][D]
    uint8_t* Vb = Kb + LP * RBk;
    uint8_t* Qb = Vb + LP * RBk;     // [QC][D]
    uint8_t* Gb = Qb + QC * RBk;
    uint8_t* Ch = Gb + QC * RBk;     // [QC][LP] C hi, C lo, W hi, W lo
    uint8_t* Cl = Ch + QC * RBc;
    uint8_t* Wh = Cl + QC * RBc;
    uint8_t* Wl = Wh + QC * RBc;
    float* Af = reinterpret_cast<float*>(Wl + QC * RBc);   // [QC][FS] logits
    float* Df = Af + QC * FS;                              // [QC][FS] dw
    __shared__ int32_t qid[QC];
    __shared__ int32_t kid[LP];
    const int e = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int L = s.m + s.k;
    const int32_t* off = offsets + (size_t)bh * (s.m + 1);
    const int beg = off[e], cnt = off[e + 1] - beg;
    if (cnt <= 0) return;
    const size_t hoff = (size_t)bh * s.N * D;
    const int32_t* E = idx + ((size_t)bh * s.m + e) * s.k;
    const int32_t* P = perm + (size_t)bh * s.N + beg;
    auto load_ids = [&](int c0) {
        const int nq = min(QC, cnt - c0);
        if (tid < QC) {
            int q = tid < nq ? P[c0 + tid] : -1;
            if (tid < nq && (q < 0 || q >= s.N)) { atomicExch(status, (int)MITA_ERR_DEVICE); q = -1; }
            qid[tid] = q;
        }
    };
    auto stage_rows = [&]() {
        for (int u = tid; u < QC * (D / 8); u += NT) {
            const int r = u >> 3, c = u & 7, q = qid[r];
            const size_t o = hoff + (size_t)(q >= 0 ? q : 0) * D + 8 * c;
            cp_async16(smem_u32(Qb + swz<RBk>(r, c)), Q + o, q >= 0 ? 16u : 0u);
            cp_async16(smem_u32(Gb + swz<RBk>(r, c)), dOut + o, q >= 0 ? 16u : 0u);
        }
        cp_async_commit();
    };
    for (int t = tid; t < LP; t += NT) {
        int j = -1;
        if (t >= s.m && t < L) {
            j = E[t - s.m];
            if (j < 0 || j >= s.N) { atomicExch(status, (int)MITA_ERR_DEVICE); j = -1; }
        }
        kid[t] = j;
    }
    load_ids(0);
    __syncthreads();
    for (int u = tid; u < LP * (D / 8); u += NT) {
        const int t = u >> 3, c = u & 7;
        const __nv_bfloat16 *sk = K + hoff, *sv = V + hoff;
        uint32_t bytes = 0;
        if (t < s.m) {
            sk = Ql + ((size_t)bh * s.m + t) * D + 8 * c;
            sv = Vl + ((size_t)bh * s.m + t) * D + 8 * c;
            bytes = 16;
        } else if (t < L && kid[t] >= 0) {
            sk = K + hoff + (size_t)kid[t] * D + 8 * c;
            sv = V + hoff + (size_t)kid[t] * D + 8 * c;
            bytes = 16;
        }
        cp_async16(smem_u32(Kb + swz<RBk>(t, c)), sk, bytes);
        cp_async16(smem_u32(Vb + swz<RBk>(t, c)), sv, bytes);
    }
    const float scale = rsqrtf((float)D);
    const int g8 = lane >> 2, q2 = 2 * (lane & 3);
    float kacc[Nk][4], vacc[Nk][4];
#pragma unroll
    for (int n = 0; n < Nk; ++n)
#pragma unroll
        for (int v = 0; v < 4; ++v) kacc[n][v] = vacc[n][v] = 0.0f;
    for (int c0 = 0;;) {
        const int nq = min(QC, cnt - c0), nm = (nq + 15) >> 4;
        stage_rows();   // the first chunk's rows load with the slot rows
        cp_async_wait<0>();
        __syncthreads();
        // logits and dw: warp w takes row tile w % MT1 and N1 slot tiles
        {
            const int mt = w % MT1, n0 = (w / MT1) * N1;
            if (mt < nm) {
                float a[N1][4], g[N1][4];
#pragma unroll
                for (int n = 0; n < N1; ++n)
#pragma unroll
                    for (int v = 0; v < 4; ++v) a[n][v] = g[n][v] = 0.0f;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    uint32_t qa[4], ga[4];
                    ldsm_x4(smem_u32(Qb + swz<RBk>(mt * 16 + (lane & 15), 2 * kk + (lane >> 4))), qa[0], qa[1], qa[2], qa[3]);
                    ldsm_x4(smem_u32(Gb + swz<RBk>(mt * 16 + (lane & 15), 2 * kk + (lane >> 4))), ga[0], ga[1], ga[2], ga[3]);
#pragma unroll
                    for (int np = 0; np < N1; np += 2) {
                        const int row = (n0 + np) * 8 + (lane & 7) + ((lane >> 4) << 3);
                        const int ch = 2 * kk + ((lane >> 3) & 1);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(smem_u32(Kb + swz<RBk>(row, ch)), b0, b1, b2, b3);
                        mma16816(a[np], qa[0], qa[1], qa[2], qa[3], b0, b1);
                        mma16816(a[np + 1], qa[0], qa[1], qa[2], qa[3], b2, b3);
                        ldsm_x4(smem_u32(Vb + swz<RBk>(row, ch)), b0, b1, b2, b3);
                        mma16816(g[np], ga[0], ga[1], ga[2], ga[3], b0, b1);
                        mma16816(g[np + 1], ga[0], ga[1], ga[2], ga[3], b2, b3);
                    }
                }
#pragma unroll
                for (int n = 0; n < N1; ++n) {
                    const int col = (n0 + n) * 8 + q2, r0 = mt * 16 + g8;
                    *reinterpret_cast<float2*>(Af + r0 * FS + col) = make_float2(a[n][0], a[n][1]);
                    *reinterpret_cast<float2*>(Af + (r0 + 8) * FS + col) = make_float2(a[n][2], a[n][3]);
                    *reinterpret_cast<float2*>(Df + r0 * FS + col) = make_float2(g[n][0], g[n][1]);
                    *reinterpret_cast<float2*>(Df + (r0 + 8) * FS + col) = make_float2(g[n][2], g[n][3]);
                }
            }
        }
        __syncthreads();
        // softmax per row (lane per slot); W and C leave as bf16 hi / lo pairs
        for (int r = w; r < nm * 16; r += NW) {
            constexpr int JT = LP / 32;
            float x[JT], dw[JT];
            const bool row = r < nq;
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < JT; ++j) {
                const int t = lane + 32 * j;
                const bool live = row && t < L && (t >= s.m ? kid[t] >= 0 : shared != 0);
                x[j] = live ? Af[r * FS + t] * scale : -INFINITY;
                dw[j] = Df[r * FS + t];
                mx = fmaxf(mx, x[j]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            float den = 0.0f;
#pragma unroll
            for (int j = 0; j < JT; ++j) {
                x[j] = row ? exp2f((x[j] - mx) * kLog2e) : 0.0f;
                den += x[j];
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
            const float inv = row ? 1.0f / den : 0.0f;
            float wdw = 0.0f;
#pragma unroll
            for (int j = 0; j < JT; ++j) {
                x[j] *= inv;
                wdw = fmaf(x[j], dw[j], wdw);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) wdw += __shfl_xor_sync(0xffffffffu, wdw, o);
#pragma unroll
            for (int j = 0; j < JT; ++j) {
                const int t = lane + 32 * j;
                const float c = x[j] * (dw[j] - wdw);
                const uint32_t o = swz<RBc>(r, t >> 3) + 2 * (t & 7);
                const __nv_bfloat16 wh = __float2bfloat16_rn(x[j]), chi = __float2bfloat16_rn(c);
                *reinterpret_cast<__nv_bfloat16*>(Wh + o) = wh;
                *reinterpret_cast<__nv_bfloat16*>(Wl + o) = __float2bfloat16_rn(x[j] - __bfloat162float(wh));
                *reinterpret_cast<__nv_bfloat16*>(Ch + o) = chi;
                *reinterpret_cast<__nv_bfloat16*>(Cl + o) = __float2bfloat16_rn(c - __bfloat162float(chi));
            }
        }
        __syncthreads();
        // dQ = C . K_slots: warp w takes row tile w % MTq and Nq feature tiles
        {
            const int mt = w % MTq, n0 = (w / MTq) * Nq;
            if (mt < nm) {
                float acc[Nq][4];
#pragma unroll
                for (int n = 0; n < Nq; ++n)
#pragma unroll
                    for (int v = 0; v < 4; ++v) acc[n][v] = 0.0f;
#pragma unroll
                for (int kk = 0; kk < LP / 16; ++kk) {
                    uint32_t h[4], l[4];
                    ldsm_x4(smem_u32(Ch + swz<RBc>(mt * 16 + (lane & 15), 2 * kk + (lane >> 4))), h[0], h[1], h[2], h[3]);
                    ldsm_x4(smem_u32(Cl + swz<RBc>(mt * 16 + (lane & 15), 2 * kk + (lane >> 4))), l[0], l[1], l[2], l[3]);
#pragma unroll
                    for (int np = 0; np < Nq; np += 2) {
                        const int krow = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(smem_u32(Kb + swz<RBk>(krow, n0 + np + (lane >> 4))), b0, b1, b2, b3);
                        mma16816(acc[np], h[0], h[1], h[2], h[3], b0, b1);
                        mma16816(acc[np], l[0], l[1], l[2], l[3], b0, b1);
                        mma16816(acc[np + 1], h[0], h[1], h[2], h[3], b2, b3);
                        mma16816(acc[np + 1], l[0], l[1], l[2], l[3], b2, b3);
                    }
                }
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = mt * 16 + g8 + 8 * hh;
                    if (r < nq && qid[r] >= 0) {
                        float* dst = dQ + hoff + (size_t)qid[r] * D;
#pragma unroll
                        for (int n = 0; n < Nq; ++n)
                            *reinterpret_cast<float2*>(dst + (n0 + n) * 8 + q2) =
                                make_float2(acc[n][2 * hh] * scale, acc[n][2 * hh + 1] * scale);
                    }
                }
            }
        }
        // dK_slots += C^T . Q, dV_slots += W^T . dOut: warp w takes slot tile w % MTk
        {
            const int mt = w % MTk, n0 = (w / MTk) * Nk;
            for (int kk = 0; kk < nm; ++kk) {
                uint32_t ch4[4], cl4[4], wh4[4], wl4[4];
                const int arow = kk * 16 + (lane & 7) + ((lane >> 4) << 3);
                const int ach = 2 * mt + ((lane >> 3) & 1);
                ldsm_x4_t(smem_u32(Ch + swz<RBc>(arow, ach)), ch4[0], ch4[1], ch4[2], ch4[3]);
                ldsm_x4_t(smem_u32(Cl + swz<RBc>(arow, ach)), cl4[0], cl4[1], cl4[2], cl4[3]);
                ldsm_x4_t(smem_u32(Wh + swz<RBc>(arow, ach)), wh4[0], wh4[1], wh4[2], wh4[3]);
                ldsm_x4_t(smem_u32(Wl + swz<RBc>(arow, ach)), wl4[0], wl4[1], wl4[2], wl4[3]);
#pragma unroll
                for (int np = 0; np < Nk; np += 2) {
                    const int brow = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                    const int bch = n0 + np + (lane >> 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(smem_u32(Qb + swz<RBk>(brow, bch)), b0, b1, b2, b3);
                    mma16816(kacc[np], ch4[0], ch4[1], ch4[2], ch4[3], b0, b1);
                    mma16816(kacc[np], cl4[0], cl4[1], cl4[2], cl4[3], b0, b1);
                    mma16816(kacc[np + 1], ch4[0], ch4[1], ch4[2], ch4[3], b2, b3);
                    mma16816(kacc[np + 1], cl4[0], cl4[1], cl4[2], cl4[3], b2, b3);
                    ldsm_x4_t(smem_u32(Gb + swz<RBk>(brow, bch)), b0, b1, b2, b3);
                    mma16816(vacc[np], wh4[0], wh4[1], wh4[2], wh4[3], b0, b1);
                    mma16816(vacc[np], wl4[0], wl4[1], wl4[2], wl4[3], b0, b1);
                    mma16816(vacc[np + 1], wh4[0], wh4[1], wh4[2], wh4[3], b2, b3);
                    mma16816(vacc[np + 1], wl4[0], wl4[1], wl4[2], wl4[3], b2, b3);
                }
            }
        }
        c0 += QC;
        if (c0 >= cnt) break;
        __syncthreads();   // the chunk's tiles are consumed
        load_ids(c0);
        __syncthreads();
    }
    {
        const int mt = w % MTk, n0 = (w / MTk) * Nk;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int t = mt * 16 + g8 + 8 * hh;
            if (t >= L) continue;
            float* rk;
            float* rv;
            if (t < s.m) {
                if (!shared) continue;
                rk = dQl + ((size_t)bh * s.m + t) * D;
                rv = dVl + ((size_t)bh * s.m + t) * D;
            } else {
                if (kid[t] < 0) continue;
                rk = dK + hoff + (size_t)kid[t] * D;
                rv = dV + hoff + (size_t)kid[t] * D;
            }
#pragma unroll
            for (int n = 0; n < Nk; ++n) {
                const int col = (n0 + n) * 8 + q2;
                atomicAdd(reinterpret_cast<float2*>(rk + col),
                          make_float2(kacc[n][2 * hh] * scale, kacc[n][2 * hh + 1] * scale));
                atomicAdd(reinterpret_cast<float2*>(rv + col), make_float2(vacc[n][2 * hh], vacc[n][2 * hh + 1]));
            }
        }
    }
}

inline size_t expert_bwd_mma_bytes(int LP, int QC) {
    return (size_t)2 * LP * 128 + (size_t)2 * QC * 128 + (size_t)4 * QC * LP * 2 + (size_t)2 * QC * (LP + 8) * 4;
}

// Landmark values again for the backward, a block per (32 landmarks, head,
// key split): row maxima of S over the split's keys, then 64-key chunks of V
// staged once in shared memory for all 32 rows, weights
// w = exp((S - max) / sqrt d) and their sums.  One split writes V_l in the
// I/O type (as the forward uses it) and, where Vl32 is not null, V_l in fp32
// and per row {max S, sum w} for values_bwd_tile_kernel; several write
// {sums, sum w, max} per split to `part` for values_rows_fin_kernel.
constexpr int kVrRows = 32, kVrKeys = 64;

template <typename T, int D>
__global__ void __launch_bounds__(256) values_rows_kernel(Shape s, const float* __restrict__ S,
                                                          const T* __restrict__ V, T* __restrict__ Vl,
                                                          float* __restrict__ Vl32, float* __restrict__ stats,
                                                          int ksplit, float* __restrict__ part) {
    constexpr int NC = D / 4, KS = D + 4, WS = kVrKeys + 1;
    constexpr int RG = 256 / NC, RPT = kVrRows / RG;
    __shared__ __align__(16) float Vt[kVrKeys * KS];
    __shared__ float Wt[kVrRows * WS];
    __shared__ float mx_s[kVrRows], den_s[kVrRows];
    const int i0 = blockIdx.x * kVrRows, bh = blockIdx.y, tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int nr = min(kVrRows, s.m - i0);
    const int cps = ((s.N + kVrKeys - 1) / kVrKeys + ksplit - 1) / ksplit;   // chunks per split
    const int k_lo = blockIdx.z * cps * kVrKeys, k_hi = min(s.N, k_lo + cps * kVrKeys);
    const float* Sh = S + ((size_t)bh * s.m + i0) * s.N;
    for (int r = w; r < kVrRows; r += 8) {
        float mx = -INFINITY;
        if (r < nr)
            for (int j = k_lo + lane; j < k_hi; j += 32) mx = fmaxf(mx, Sh[(size_t)r * s.N + j]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) mx_s[r] = mx;
    }
    const float c = rsqrtf((float)D) * kLog2e;
    const int tc = tid % NC, rg = tid / NC, wr = tid >> 3, wk = tid & 7;
    float acc[RPT][4] = {};
    float den = 0.0f;
    const T* Vh = V + (size_t)bh * s.N * D;
    for (int j0 = k_lo; j0 < k_hi; j0 += kVrKeys) {
        const int nk = min(kVrKeys, k_hi - j0);
        __syncthreads();   // row maxima ready; the previous chunk consumed
        for (int u = tid; u < kVrKeys * NC; u += 256) {
            const int r = u / NC, c4 = 4 * (u % NC);
            *reinterpret_cast<float4*>(Vt + r * KS + c4) =
                r < nk ? load4(Vh + (size_t)(j0 + r) * D + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const int key = wk + 8 * v;
            float x = 0.0f;
            if (wr < nr && key < nk) x = exp2f((Sh[(size_t)wr * s.N + j0 + key] - mx_s[wr]) * c);
            Wt[wr * WS + key] = x;
            den += x;
        }
        __syncthreads();
        for (int key = 0; key < nk; ++key) {
            const float4 vv = *reinterpret_cast<const float4*>(Vt + key * KS + 4 * tc);
#pragma unroll
            for (int u = 0; u < RPT; ++u) {
                const float x = Wt[(rg + RG * u) * WS + key];
                acc[u][0] = fmaf(x, vv.x, acc[u][0]);
                acc[u][1] = fmaf(x, vv.y, acc[u][1]);
                acc[u][2] = fmaf(x, vv.z, acc[u][2]);
                acc[u][3] = fmaf(x, vv.w, acc[u][3]);
            }
        }
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    if (wk == 0) den_s[wr] = den;
    __syncthreads();
    if (ksplit > 1) {
#pragma unroll
        for (int u = 0; u < RPT; ++u) {
            const int r = rg + RG * u;
            if (r >= nr) continue;
            float* pr = part + (((size_t)bh * s.m + i0 + r) * ksplit + blockIdx.z) * (D + 2);
            *reinterpret_cast<float2*>(pr + 4 * tc) = make_float2(acc[u][0], acc[u][1]);
            *reinterpret_cast<float2*>(pr + 4 * tc + 2) = make_float2(acc[u][2], acc[u][3]);
            if (tc == 0) {
                pr[D] = den_s[r];
                pr[D + 1] = mx_s[r];
            }
        }
        return;
    }
#pragma unroll
    for (int u = 0; u < RPT; ++u) {
        const int r = rg + RG * u;
        if (r >= nr) continue;
        const size_t o = ((size_t)bh * s.m + i0 + r) * D + 4 * tc;
        const float rsum = den_s[r];
        float y[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            y[b] = acc[u][b] / rsum;
            Vl[o + b] = from_f32<T>(y[b]);
        }
        if (Vl32 == nullptr) continue;
        *reinterpret_cast<float4*>(Vl32 + o) = make_float4(y[0], y[1], y[2], y[3]);
        if (tc == 0) {
            stats[2 * ((size_t)bh * s.m + i0 + r)] = mx_s[r];
            stats[2 * ((size_t)bh * s.m + i0 + r) + 1] = rsum;
        }
    }
}

// Combines values_rows_kernel's key splits: thread per (landmark row, 4
// features); the splits' sums are rescaled to the row's largest max.  The
// fp32 copy and row stats are written where Vl32 is not null.
template <typename T, int D>
__global__ void __launch_bounds__(256) values_rows_fin_kernel(Shape s, int ksplit, const float* __restrict__ part,
                                                              T* __restrict__ Vl, float* __restrict__ Vl32,
                                                              float* __restrict__ stats) {
    constexpr int NC = D / 4;
    const size_t e = (size_t)blockIdx.x * 256 + threadIdx.x;
    if (e >= (size_t)s.BH() * s.m * NC) return;
    const size_t row = e / NC;
    const int tc = (int)(e % NC);
    const float* pr = part + row * ksplit * (D + 2);
    const float c = rsqrtf((float)D) * kLog2e;
    float M = -INFINITY;
    for (int z = 0; z < ksplit; ++z) M = fmaxf(M, pr[z * (D + 2) + D + 1]);
    float den = 0.0f, a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int z = 0; z < ksplit; ++z) {
        const float* q = pr + z * (D + 2);
        const float f = exp2f((q[D + 1] - M) * c);
        den = fmaf(q[D], f, den);
#pragma unroll
        for (int b = 0; b < 4; ++b) a[b] = fmaf(q[4 * tc + b], f, a[b]);
    }
    const size_t o = row * D + 4 * tc;
    float y[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        y[b] = a[b] / den;
        Vl[o + b] = from_f32<T>(y[b]);
    }
    if (Vl32 == nullptr) return;
    *reinterpret_cast<float4*>(Vl32 + o) = make_float4(y[0], y[1], y[2], y[3]);
    if (tc == 0) {
        stats[2 * row] = M;
        stats[2 * row + 1] = den;
    }
}

// Landmark-value backward, a block per (64-key tile, head); the block owns its
// keys' rows of dK and dV.  With P = softmax(S / sqrt d) per landmark row
// (max and sum from values_rows_kernel), per chunk of 32 landmarks:
// dP = dV_l . V_tile^T, dR = P (dP - dV_l . V_l) / sqrt d (the row's
// P . dP is dV_l . V_l), then dV_tile += P^T dV_l and dK_tile += dR^T Q_l in
// 4 x 4 register tiles, and dQ_l += dR . K_tile by float4 atomics.  The tile's
// dK, dV rows are added once at the end.
template <typename T, int D>
__global__ void __launch_bounds__(256, D == 64 ? 3 : 1) values_bwd_tile_kernel(Shape s, const float* __restrict__ S,
                                                              const float* __restrict__ stats,
                                                              const float* __restrict__ Vl32,
                                                              const T* __restrict__ K, const T* __restrict__ V,
                                                              const T* __restrict__ Ql,
                                                              const float* __restrict__ dVl, float* __restrict__ dK,
                                                              float* __restrict__ dV, float* __restrict__ dQl) {
    constexpr int KT = kVrKeys, RT = kVrRows, NC = D / 4, KS = D + 4, PS = KT + 8;
    constexpr int TT = (KT / 4) * NC / 256;   // 4 x 4 gradient tiles per thread
    constexpr int RG = 256 / NC, RPT = RT / RG;
    extern __shared__ float4 vb_smem[];
    float* Kt = reinterpret_cast<float*>(vb_smem);   // [KT][KS]
    float* Vt = Kt + KT * KS;
    float* Gl = Vt + KT * KS;   // [RT][KS] dV_l rows
    float* Qc = Gl + RT * KS;   // [RT][KS] Q_l rows
    float* Pt = Qc + RT * KS;   // [RT][PS]
    float* Rt = Pt + RT * PS;   // [RT][PS]
    float* Dr = Rt + RT * PS;   // [RT] dV_l . V_l
    const int j0 = blockIdx.x * KT, bh = blockIdx.y, tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int nk = min(KT, s.N - j0);
    const size_t hoff = (size_t)bh * s.N * D;
    for (int u = tid; u < KT * NC; u += 256) {
        const int r = u / NC, c4 = 4 * (u % NC);
        const bool in = r < nk;
        *reinterpret_cast<float4*>(Kt + r * KS + c4) =
            in ? load4(K + hoff + (size_t)(j0 + r) * D + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(Vt + r * KS + c4) =
            in ? load4(V + hoff + (size_t)(j0 + r) * D + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float scale = rsqrtf((float)D), c = scale * kLog2e;
    float gk[TT][4][4], gv[TT][4][4];
#pragma unroll
    for (int t = 0; t < TT; ++t)
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) gk[t][a][b] = gv[t][a][b] = 0.0f;
    const int pr = tid >> 3, pk = tid & 7;     // P / dR entries: row pr, keys pk + 8 v
    const int tc = tid % NC, rg = tid / NC;    // dQ_l rows rg + RG u, features 4 tc
    for (int i0 = 0; i0 < s.m; i0 += RT) {
        const int nr = min(RT, s.m - i0);
        if (i0 > 0) __syncthreads();   // the previous chunk consumed
        // the chunk's scores go to Pt (turned into P in place below)
        for (int u = tid; u < RT * KT; u += 256) {
            const int r = u / KT, key = u % KT;
            Pt[r * PS + key] = r < nr && key < nk ? S[((size_t)bh * s.m + i0 + r) * s.N + j0 + key] : 0.0f;
        }
        const bool row = pr < nr;
        const size_t so = ((size_t)bh * s.m + i0 + pr);
        const float mx = row ? stats[2 * so] : 0.0f, den = row ? stats[2 * so + 1] : 1.0f;
        for (int u = tid; u < RT * NC; u += 256) {
            const int r = u / NC, c4 = 4 * (u % NC);
            const size_t o = ((size_t)bh * s.m + i0 + r) * D + c4;
            const bool in = r < nr;
            *reinterpret_cast<float4*>(Gl + r * KS + c4) =
                in ? *reinterpret_cast<const float4*>(dVl + o) : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(Qc + r * KS + c4) = in ? load4(Ql + o) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int r = w; r < RT; r += 8) {
            float x = 0.0f;
            if (r < nr) {
                const size_t o = ((size_t)bh * s.m + i0 + r) * D;
                for (int f = lane; f < D; f += 32) x = fmaf(dVl[o + f], Vl32[o + f], x);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
            if (lane == 0) Dr[r] = x;
        }
        __syncthreads();
        {
            float dp[8] = {};
#pragma unroll 2
            for (int f = 0; f < D; f += 4) {
                const float4 g = *reinterpret_cast<const float4*>(Gl + pr * KS + f);
#pragma unroll
                for (int v = 0; v < 8; ++v) dp[v] = dot4(g, *reinterpret_cast<const float4*>(Vt + (pk + 8 * v) * KS + f), dp[v]);
            }
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const int key = pk + 8 * v;
                float p = 0.0f;
                if (row && key < nk) p = exp2f((Pt[pr * PS + key] - mx) * c) / den;
                Pt[pr * PS + key] = p;
                Rt[pr * PS + key] = p * (dp[v] - Dr[pr]) * scale;
            }
        }
        __syncthreads();
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            const int tile = tid + 256 * t, kg = tile / NC, fc = tile % NC;
            for (int r = 0; r < nr; ++r) {
                const float4 p4 = *reinterpret_cast<const float4*>(Pt + r * PS + 4 * kg);
                const float4 d4 = *reinterpret_cast<const float4*>(Rt + r * PS + 4 * kg);
                const float4 g4 = *reinterpret_cast<const float4*>(Gl + r * KS + 4 * fc);
                const float4 q4 = *reinterpret_cast<const float4*>(Qc + r * KS + 4 * fc);
                const float pp[4] = {p4.x, p4.y, p4.z, p4.w}, dd[4] = {d4.x, d4.y, d4.z, d4.w};
                const float gg[4] = {g4.x, g4.y, g4.z, g4.w}, qq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        gv[t][a][b] = fmaf(pp[a], gg[b], gv[t][a][b]);
                        gk[t][a][b] = fmaf(dd[a], qq[b], gk[t][a][b]);
                    }
            }
        }
        {
            float acc[RPT][4] = {};
            for (int key = 0; key < nk; ++key) {
                const float4 kv = *reinterpret_cast<const float4*>(Kt + key * KS + 4 * tc);
#pragma unroll
                for (int u = 0; u < RPT; ++u) {
                    const float x = Rt[(rg + RG * u) * PS + key];
                    acc[u][0] = fmaf(x, kv.x, acc[u][0]);
                    acc[u][1] = fmaf(x, kv.y, acc[u][1]);
                    acc[u][2] = fmaf(x, kv.z, acc[u][2]);
                    acc[u][3] = fmaf(x, kv.w, acc[u][3]);
                }
            }
#pragma unroll
            for (int u = 0; u < RPT; ++u) {
                const int r = rg + RG * u;
                if (r < nr)
                    atomicAdd(reinterpret_cast<float4*>(dQl + ((size_t)bh * s.m + i0 + r) * D + 4 * tc),
                              make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]));
            }
        }
    }
#pragma unroll
    for (int t = 0; t < TT; ++t) {
        const int tile = tid + 256 * t, kg = tile / NC, fc = tile % NC;
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int key = 4 * kg + a;
            if (key >= nk) continue;
            const size_t o = hoff + (size_t)(j0 + key) * D + 4 * fc;
            float4 k4 = *reinterpret_cast<float4*>(dK + o), v4 = *reinterpret_cast<float4*>(dV + o);
            k4.x += gk[t][a][0]; k4.y += gk[t][a][1]; k4.z += gk[t][a][2]; k4.w += gk[t][a][3];
            v4.x += gv[t][a][0]; v4.y += gv[t][a][1]; v4.z += gv[t][a][2]; v4.w += gv[t][a][3];
            *reinterpret_cast<float4*>(dK + o) = k4;
            *reinterpret_cast<float4*>(dV + o) = v4;
        }
    }
}

// values_bwd_tile_kernel for bf16 I/O at d = 64 with its products on
// mma.sync (m16n8k16, fp32 accumulation), per chunk of 32 landmark rows:
// dP = dV_l . V_tile^T, then per element P (from the scores and the row's
// max and sum) and dR = P (dP - dV_l . V_l) / sqrt d, then dV_tile += P^T
// dV_l, dK_tile += dR^T Q_l and dQ_l += dR . K_tile.  The fp32 operands (dV_l,
// P, dR) enter as bf16 pairs hi + lo (about 16 mantissa bits; the lo x lo
// term of P^T dV_l is dropped).  Warp w keeps the dK and dV accumulators of
// keys 16 (w % 4) .. + 15 and features 32 (w / 4) .. + 31 over all chunks;
// the tile's rows are added once at the end.  Tiles are bf16 rows of 64 with
// XOR-swizzled 16-byte chunks; rows past the landmarks or keys are zero.
constexpr int kVmKeys = 64, kVmRows = 32;

MITA_DEV void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const __nv_bfloat162 l = __floats2bfloat162_rn(a - __low2float(h), b - __high2float(h));
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

__global__ void __launch_bounds__(256, 3)
    values_bwd_mma_kernel(Shape s, const float* __restrict__ S, const float* __restrict__ stats,
                          const float* __restrict__ Vl32, const __nv_bfloat16* __restrict__ K,
                          const __nv_bfloat16* __restrict__ V, const __nv_bfloat16* __restrict__ Ql,
                          const float* __restrict__ dVl, float* __restrict__ dK, float* __restrict__ dV,
                          float* __restrict__ dQl) {
    using namespace mx;
    constexpr int D = 64, RB = 128;   // bytes per bf16 row of 64
    extern __shared__ __align__(128) uint8_t vm_raw[];
    uint8_t* Kt = vm_raw;             // [64 keys][64 features]
    uint8_t* Vt = Kt + kVmKeys * RB;
    uint8_t* Qc = Vt + kVmKeys * RB;  // [32 rows][64 features]: Q_l, dV_l hi, dV_l lo
    uint8_t* Gh = Qc + kVmRows * RB;
    uint8_t* Gl = Gh + kVmRows * RB;
    uint8_t* Ph = Gl + kVmRows * RB;  // [32 rows][64 keys]: P hi, P lo, dR hi, dR lo
    uint8_t* Pl = Ph + kVmRows * RB;
    uint8_t* Rh = Pl + kVmRows * RB;
    uint8_t* Rl = Rh + kVmRows * RB;
    __shared__ float mx_s[kVmRows], den_s[kVmRows], dr_s[kVmRows];
    const int j0 = blockIdx.x * kVmKeys, bh = blockIdx.y, tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int nk = min(kVmKeys, s.N - j0);
    const size_t hoff = (size_t)bh * s.N * D;
    const int g8 = lane >> 2, q2 = 2 * (lane & 3);
    for (int u = tid; u < kVmKeys * 8; u += 256) {
        const int r = u >> 3, c = u & 7;
        const size_t o = hoff + (size_t)(j0 + (r < nk ? r : 0)) * D + 8 * c;
        cp_async16(smem_u32(Kt + swz<RB>(r, c)), K + o, r < nk ? 16u : 0u);
        cp_async16(smem_u32(Vt + swz<RB>(r, c)), V + o, r < nk ? 16u : 0u);
    }
    cp_async_commit();
    const float scale = rsqrtf((float)D), c2 = scale * kLog2e;
    float kacc[4][4], vacc[4][4];   // key tile w % 4, feature tiles 4 (w / 4) + n
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int v = 0; v < 4; ++v) kacc[n][v] = vacc[n][v] = 0.0f;
    for (int i0 = 0; i0 < s.m; i0 += kVmRows) {
        const int nr = min(kVmRows, s.m - i0);
        if (i0 > 0) __syncthreads();   // the previous chunk's tiles consumed
        for (int u = tid; u < kVmRows * 8; u += 256) {
            const int r = u >> 3, c = u & 7;
            const size_t o = ((size_t)bh * s.m + i0 + (r < nr ? r : 0)) * D + 8 * c;
            cp_async16(smem_u32(Qc + swz<RB>(r, c)), Ql + o, r < nr ? 16u : 0u);
            uint32_t hw[4] = {0u, 0u, 0u, 0u}, lw[4] = {0u, 0u, 0u, 0u};
            if (r < nr) {
                const float4 a = *reinterpret_cast<const float4*>(dVl + o);
                const float4 b = *reinterpret_cast<const float4*>(dVl + o + 4);
                split_bf16x2(a.x, a.y, hw[0], lw[0]);
                split_bf16x2(a.z, a.w, hw[1], lw[1]);
                split_bf16x2(b.x, b.y, hw[2], lw[2]);
                split_bf16x2(b.z, b.w, hw[3], lw[3]);
            }
            *reinterpret_cast<uint4*>(Gh + swz<RB>(r, c)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(Gl + swz<RB>(r, c)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        cp_async_commit();
        if (tid < kVmRows) {
            const size_t so = (size_t)bh * s.m + i0 + tid;
            mx_s[tid] = tid < nr ? stats[2 * so] : 0.0f;
            den_s[tid] = tid < nr ? stats[2 * so + 1] : 1.0f;
        }
        for (int r = w; r < kVmRows; r += 8) {   // dV_l . V_l, the row's P . dP
            float x = 0.0f;
            if (r < nr) {
                const size_t o = ((size_t)bh * s.m + i0 + r) * D;
                for (int f = lane; f < D; f += 32) x = fmaf(dVl[o + f], Vl32[o + f], x);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
            if (lane == 0) dr_s[r] = x;
        }
        cp_async_wait<0>();
        __syncthreads();
        // dP = dV_l . V^T (warp w: row tile w % 2, key tiles 2 (w / 2), + 1), then P and dR
        {
            const int mt = w & 1, nt = 2 * (w >> 1);
            float sv[2][2][2];   // the scores of this lane's elements, loaded before the products
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int r = mt * 16 + g8 + 8 * hh, key = (nt + n) * 8 + q2 + e;
                        sv[n][hh][e] = r < nr && key < nk ? S[((size_t)bh * s.m + i0 + r) * s.N + j0 + key] : 0.0f;
                    }
            float p[2][4];
#pragma unroll
            for (int n = 0; n < 2; ++n) p[n][0] = p[n][1] = p[n][2] = p[n][3] = 0.0f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t ah[4], al[4], b0, b1, b2, b3;
                const uint32_t ao = swz<RB>(mt * 16 + (lane & 15), 2 * kk + (lane >> 4));
                ldsm_x4(smem_u32(Gh + ao), ah[0], ah[1], ah[2], ah[3]);
                ldsm_x4(smem_u32(Gl + ao), al[0], al[1], al[2], al[3]);
                ldsm_x4(smem_u32(Vt + swz<RB>(nt * 8 + (lane & 7) + ((lane >> 4) << 3), 2 * kk + ((lane >> 3) & 1))), b0,
                        b1, b2, b3);
                mma16816(p[0], ah[0], ah[1], ah[2], ah[3], b0, b1);
                mma16816(p[0], al[0], al[1], al[2], al[3], b0, b1);
                mma16816(p[1], ah[0], ah[1], ah[2], ah[3], b2, b3);
                mma16816(p[1], al[0], al[1], al[2], al[3], b2, b3);
            }
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = mt * 16 + g8 + 8 * hh, key = (nt + n) * 8 + q2;
                    float pv[2], rv[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float pe = r < nr && key + e < nk ? exp2f((sv[n][hh][e] - mx_s[r]) * c2) / den_s[r] : 0.0f;
                        pv[e] = pe;
                        rv[e] = pe * (p[n][2 * hh + e] - dr_s[r]) * scale;
                    }
                    const uint32_t o = swz<RB>(r, key >> 3) + (uint32_t)(key & 7) * 2u;
                    uint32_t h, l;
                    split_bf16x2(pv[0], pv[1], h, l);
                    *reinterpret_cast<uint32_t*>(Ph + o) = h;
                    *reinterpret_cast<uint32_t*>(Pl + o) = l;
                    split_bf16x2(rv[0], rv[1], h, l);
                    *reinterpret_cast<uint32_t*>(Rh + o) = h;
                    *reinterpret_cast<uint32_t*>(Rl + o) = l;
                }
        }
        __syncthreads();
        // dV += P^T dV_l, dK += dR^T Q_l (warp w: key tile w % 4, feature tiles 4 (w / 4) .. + 3)
        {
            const int mt = w & 3, n0 = 4 * (w >> 2);
#pragma unroll
            for (int kk = 0; kk < kVmRows / 16; ++kk) {
                const int arow = kk * 16 + (lane & 7) + ((lane >> 4) << 3);
                const int ach = 2 * mt + ((lane >> 3) & 1);
                uint32_t ph[4], pl[4], rh[4], rl[4];
                ldsm_x4_t(smem_u32(Ph + swz<RB>(arow, ach)), ph[0], ph[1], ph[2], ph[3]);
                ldsm_x4_t(smem_u32(Pl + swz<RB>(arow, ach)), pl[0], pl[1], pl[2], pl[3]);
                ldsm_x4_t(smem_u32(Rh + swz<RB>(arow, ach)), rh[0], rh[1], rh[2], rh[3]);
                ldsm_x4_t(smem_u32(Rl + swz<RB>(arow, ach)), rl[0], rl[1], rl[2], rl[3]);
#pragma unroll
                for (int np = 0; np < 4; np += 2) {
                    const int brow = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                    const int bch = n0 + np + (lane >> 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(smem_u32(Gh + swz<RB>(brow, bch)), b0, b1, b2, b3);
                    mma16816(vacc[np], ph[0], ph[1], ph[2], ph[3], b0, b1);
                    mma16816(vacc[np], pl[0], pl[1], pl[2], pl[3], b0, b1);
                    mma16816(vacc[np + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
                    mma16816(vacc[np + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
                    ldsm_x4_t(smem_u32(Gl + swz<RB>(brow, bch)), b0, b1, b2, b3);
                    mma16816(vacc[np], ph[0], ph[1], ph[2], ph[3], b0, b1);
                    mma16816(vacc[np + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
                    ldsm_x4_t(smem_u32(Qc + swz<RB>(brow, bch)), b0, b1, b2, b3);
                    mma16816(kacc[np], rh[0], rh[1], rh[2], rh[3], b0, b1);
                    mma16816(kacc[np], rl[0], rl[1], rl[2], rl[3], b0, b1);
                    mma16816(kacc[np + 1], rh[0], rh[1], rh[2], rh[3], b2, b3);
                    mma16816(kacc[np + 1], rl[0], rl[1], rl[2], rl[3], b2, b3);
                }
            }
        }
        // dQ_l += dR . K (warp w: row tile w % 2, feature tiles 2 (w / 2), + 1)
        {
            const int mt = w & 1, nt = 2 * (w >> 1);
            float a[2][4];
#pragma unroll
            for (int n = 0; n < 2; ++n) a[n][0] = a[n][1] = a[n][2] = a[n][3] = 0.0f;
#pragma unroll
            for (int kk = 0; kk < kVmKeys / 16; ++kk) {
                uint32_t rh[4], rl[4], b0, b1, b2, b3;
                const uint32_t ao = swz<RB>(mt * 16 + (lane & 15), 2 * kk + (lane >> 4));
                ldsm_x4(smem_u32(Rh + ao), rh[0], rh[1], rh[2], rh[3]);
                ldsm_x4(smem_u32(Rl + ao), rl[0], rl[1], rl[2], rl[3]);
                const int brow = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                ldsm_x4_t(smem_u32(Kt + swz<RB>(brow, nt + (lane >> 4))), b0, b1, b2, b3);
                mma16816(a[0], rh[0], rh[1], rh[2], rh[3], b0, b1);
                mma16816(a[0], rl[0], rl[1], rl[2], rl[3], b0, b1);
                mma16816(a[1], rh[0], rh[1], rh[2], rh[3], b2, b3);
                mma16816(a[1], rl[0], rl[1], rl[2], rl[3], b2, b3);
            }
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = mt * 16 + g8 + 8 * hh;
                    if (r < nr)
                        atomicAdd(reinterpret_cast<float2*>(dQl + ((size_t)bh * s.m + i0 + r) * D + (nt + n) * 8 + q2),
                                  make_float2(a[n][2 * hh], a[n][2 * hh + 1]));
                }
        }
    }
    // the tile's rows of dK and dV
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int key = (w & 3) * 16 + g8 + 8 * hh, f = (4 * (w >> 2) + n) * 8 + q2;
            if (key >= nk) continue;
            const size_t o = hoff + (size_t)(j0 + key) * D + f;
            float2 k2 = *reinterpret_cast<float2*>(dK + o), v2 = *reinterpret_cast<float2*>(dV + o);
            k2.x += kacc[n][2 * hh];
            k2.y += kacc[n][2 * hh + 1];
            v2.x += vacc[n][2 * hh];
            v2.y += vacc[n][2 * hh + 1];
            *reinterpret_cast<float2*>(dK + o) = k2;
            *reinterpret_cast<float2*>(dV + o) = v2;
        }
}

constexpr size_t values_bwd_mma_bytes() { return (size_t)(2 * kVmKeys + 7 * kVmRows) * 128; }

template <int D>
constexpr size_t values_bwd_tile_bytes() {
    return ((size_t)2 * kVrKeys * (D + 4) + 2 * kVrRows * (D + 4) + 2 * kVrRows * (kVrKeys + 8) + kVrRows) *
           sizeof(float);
}

// Thread per (token, 4 features): dQ[t] += dQ_l[i] / |bin i| over the (at
// most two per axis) bins that hold token t.  Each block first tabulates the
// bins' row and column ranges in shared memory (ph + pw <= 2048 entries).
constexpr int kPoolBwdTab = 2048;

template <int D>
__global__ void __launch_bounds__(256) pool_bwd_kernel(Shape s, const float* __restrict__ dQl, float* __restrict__ dQ) {
    constexpr int NC = D / 4;
    __shared__ int2 rng[kPoolBwdTab];   // rows [0, ph), then columns [ph, ph + pw)
    for (int u = threadIdx.x; u < s.ph + s.pw; u += 256) {
        int lo, hi;
        if (u < s.ph) pool_bin(u, s.gh, s.ph, lo, hi);
        else pool_bin(u - s.ph, s.gw, s.pw, lo, hi);
        rng[u] = make_int2(lo, hi);
    }
    __syncthreads();
    const int e = blockIdx.x * 256 + threadIdx.x;
    const int bh = blockIdx.y;
    if (e >= s.N * NC) return;
    const int t = e / NC, c4 = 4 * (e % NC), y = t / s.gw, x = t - y * s.gw;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const int rc = y * s.ph / s.gh, cc = x * s.pw / s.gw;
    for (int r = max(0, rc - 1); r <= min(s.ph - 1, rc + 1); ++r) {
        const int2 rr = rng[r];
        if (y < rr.x || y >= rr.y) continue;
        for (int c = max(0, cc - 1); c <= min(s.pw - 1, cc + 1); ++c) {
            const int2 cr = rng[s.ph + c];
            if (x < cr.x || x >= cr.y) continue;
            // one correctly rounded reciprocal of the bin's size per bin, then products
            const float rn = __frcp_rn((float)((rr.y - rr.x) * (cr.y - cr.x)));
            const float4 g = *reinterpret_cast<const float4*>(dQl + ((size_t)bh * s.m + r * s.pw + c) * D + c4);
            acc.x = fmaf(g.x, rn, acc.x); acc.y = fmaf(g.y, rn, acc.y);
            acc.z = fmaf(g.z, rn, acc.z); acc.w = fmaf(g.w, rn, acc.w);
        }
    }
    float4* o = reinterpret_cast<float4*>(dQ + ((size_t)bh * s.N + t) * D + c4);
    float4 q = *o;
    q.x += acc.x; q.y += acc.y; q.z += acc.z; q.w += acc.w;
    *o = q;
}

// Landmark values V_l (with their fp32 copy and row stats where Vl32 is not
// null) by values_rows_kernel, with key splits when the row tiles alone give
// fewer than two blocks per SM; the splits' partial sums go to `scratch`
// (bytes available: scratch_bytes).  Returns the number of launches.
template <typename T, int D>
static int launch_values_rows(const Shape& s, const float* S, const T* V, T* Vl, float* Vl32, float* stats,
                              float* scratch, size_t scratch_bytes, cudaStream_t st) {
    const int BH = s.BH();
    const int row_tiles = (s.m + kVrRows - 1) / kVrRows;
    int ksplit = 1;
    if ((size_t)row_tiles * BH < 296) {
        ksplit = std::min(8, (s.N + 511) / 512);
        while (ksplit > 1 && (size_t)BH * s.m * ksplit * (D + 2) * sizeof(float) > scratch_bytes) --ksplit;
    }
    values_rows_kernel<T, D><<<dim3(row_tiles, BH, ksplit), 256, 0, st>>>(s, S, V, Vl, Vl32, stats, ksplit,
                                                                          scratch);
    if (ksplit == 1) return 1;
    values_rows_fin_kernel<T, D><<<(unsigned)(((size_t)BH * s.m * (D / 4) + 255) / 256), 256, 0, st>>>(
        s, ksplit, scratch, Vl, Vl32, stats);
    return 2;
}

template <typename T, int D>
static cudaError_t run_backward_t(mita_plan_s* p, const T* Q, const T* K, const T* V, const T* dOut, float* dQ,
                                  float* dK, float* dV, cudaStream_t st) {
    const Shape& s = p->s;
    const int BH = s.BH();
    T* Ql = (T*)p->Ql;
    T* Vl = (T*)p->Vl;
    const size_t nbytes = (size_t)BH * s.N * D * sizeof(float);
    cudaError_t e;
    if ((e = cudaMemsetAsync(p->dQl, 0, (size_t)2 * BH * s.m * D * sizeof(float), st)) != cudaSuccess) return e;
    // the forward's landmarks, scores, experts, landmark values and routes; at
    // bf16 with the tiled path's workspace (m <= 128), its pool and its
    // one-kernel scores and routes (the same Q_l, scores and first argmax)
    bool tiled_recompute = false;
    if constexpr (std::is_same<T, __nv_bfloat16>::value)
        tiled_recompute = p->rowmax != nullptr && s.m <= 128 && tc_scores_route_supported(s);
    if (tiled_recompute) {
        uint32_t* rowmin = p->rowmax + (size_t)BH * s.m;
        if (s.N <= 32 * s.m) {   // bins of about 32 tokens or fewer: a block of D threads per landmark
            pool_kernel<T><<<dim3(s.m, BH), D, 0, st>>>(s, Q, Ql);
            if ((e = cudaMemsetAsync(p->rowmax, 0, (size_t)BH * s.m * 4, st)) != cudaSuccess) return e;
            if ((e = cudaMemsetAsync(rowmin, 0xff, (size_t)BH * s.m * 4, st)) != cudaSuccess) return e;
        } else if ((e = tiled_pool(s, Q, Ql, p->rowmax, p->counts, st)) != cudaSuccess) {
            return e;
        }
        if ((e = tc_scores_route(s, Ql, K, Q, p->S, p->rowmax, rowmin, p->route, p->counts, p->status, st, false)) !=
            cudaSuccess)
            return e;
    } else {
        pool_kernel<T><<<dim3(s.m, BH), D, 0, st>>>(s, Q, Ql);
        scores_kernel<T><<<dim3((s.N + 127) / 128, (s.m + 31) / 32, BH), 256, 0, st>>>(s, Ql, K, p->S);
        p->launches += 1;   // and the route kernel below
    }
    if (tiled_recompute && s.N > 256 && tiled_topk_supported(s)) {   // long rows: the register-resident select
        if ((e = tiled_topk(s, p->S, p->rowmax, p->idx, st)) != cudaSuccess) return e;
    } else {
        launch_topk(s, p->S, p->idx, st);
    }
    float* Vl32 = p->dVl + (size_t)BH * s.m * D;   // fp32 landmark values, then per-row {max S, sum w}
    float* stats = Vl32 + (size_t)BH * s.m * D;
    if (tiled_recompute) {   // the tiled path's tensor-core landmark values, with the row stats
        if ((e = tiled_values_stats(s, p->S, p->rowmax, V, p->vpart, Vl, Vl32, stats, p->status, st)) != cudaSuccess)
            return e;
        p->launches += 1;   // two launches in place of one
    } else {
        // key-split partial sums use dK as scratch before it is cleared
        p->launches += launch_values_rows<T, D>(s, p->S, V, Vl, Vl32, stats, dK, nbytes, st) - 1;
    }
    if (!tiled_recompute)
        route_kernel<T, D><<<dim3((s.N + 127) / 128, BH), 128, 0, st>>>(s, Q, Ql, p->route, 1, nullptr);
    if ((e = cudaMemsetAsync(dK, 0, nbytes, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dV, 0, nbytes, st)) != cudaSuccess) return e;
    const int L = s.m + s.k;
    const int shared = p->routing_only ? 0 : 1;
    // expert-major output softmax where the expert's slots fit (L <= 128 at
    // d = 64, L <= 64 at d = 128; 16 warps where a thread would otherwise hold
    // more than 32 gradient accumulators, 16-query chunks on 8 warps for the
    // short experts of small images); the warp-per-query kernel otherwise
    auto expert_launch = [&](auto kern, int LP, int NW, int QC) -> bool {
        const size_t bytes = expert_bwd_bytes(D, L, LP, QC);
        if (bytes > 200 * 1024) return false;
        ensure_smem_attr((const void*)kern, (int)bytes);
        launch_bucket(s, p->route, p->counts, p->offsets, p->perm, p->status, st);
        kern<<<dim3(s.m, BH), 32 * NW, bytes, st>>>(s, Q, K, V, Ql, Vl, p->idx, p->offsets, p->perm, dOut, dQ,
                                                       dK, dV, p->dQl, p->dVl, shared, p->status);
        p->launches += 2;
        return true;
    };
    bool done = false;
    if constexpr (D == 64 && std::is_same<T, __nv_bfloat16>::value) {
        auto mma_launch = [&](auto kern, int LP, int QC, int NW) {
            const size_t bytes = expert_bwd_mma_bytes(LP, QC);
            ensure_smem_attr((const void*)kern, (int)bytes);
            launch_bucket(s, p->route, p->counts, p->offsets, p->perm, p->status, st);
            kern<<<dim3(s.m, BH), 32 * NW, bytes, st>>>(s, Q, K, V, Ql, Vl, p->idx, p->offsets, p->perm, dOut, dQ,
                                                         dK, dV, p->dQl, p->dVl, shared, p->status);
            p->launches += 2;
            return true;
        };
        if (L <= 64) done = mma_launch(expert_bwd_mma_kernel<64, 32, 8>, 64, 32, 8);
        else if (L <= 128) done = mma_launch(expert_bwd_mma_kernel<128, 64, 16>, 128, 64, 16);
    } else if constexpr (D == 64) {
        if (L <= 64) done = expert_launch(expert_bwd_kernel<T, D, 2, 8, 2>, 64, 8, 16);
        else if (L <= 128) done = expert_launch(expert_bwd_kernel<T, D, 4, 16, 4>, 128, 16, 64);
    } else {
        if (L <= 64) done = expert_launch(expert_bwd_kernel<T, D, 2, 16, 4>, 64, 16, 64);
    }
    if (!done) {
        const size_t smem = (size_t)kAttendWarps * (2 * D + 2 * L) * sizeof(float);
        if (smem > 227 * 1024) return cudaErrorInvalidValue;
        ensure_smem_attr((const void*)attend_bwd_kernel<T, D>, (int)smem);
        attend_bwd_kernel<T, D><<<dim3((s.N + kAttendWarps - 1) / kAttendWarps, BH), 32 * kAttendWarps, smem, st>>>(
            s, Q, K, V, Ql, Vl, p->idx, p->route, dOut, dQ, dK, dV, p->dQl, p->dVl, shared, p->status);
        p->launches += 1;
    }
    bool vmma = false;   // bf16 at d = 64: the landmark-value backward on mma.sync
    if constexpr (D == 64 && std::is_same<T, __nv_bfloat16>::value) {
        ensure_smem_attr((const void*)values_bwd_mma_kernel, (int)values_bwd_mma_bytes());
        values_bwd_mma_kernel<<<dim3((s.N + kVmKeys - 1) / kVmKeys, BH), 256, values_bwd_mma_bytes(), st>>>(
            s, p->S, stats, Vl32, K, V, Ql, p->dVl, dK, dV, p->dQl);
        vmma = true;
    }
    if (!vmma) {
        const size_t vb_bytes = values_bwd_tile_bytes<D>();
        ensure_smem_attr((const void*)values_bwd_tile_kernel<T, D>, (int)vb_bytes);
        values_bwd_tile_kernel<T, D><<<dim3((s.N + kVrKeys - 1) / kVrKeys, BH), 256, vb_bytes, st>>>(
            s, p->S, stats, Vl32, K, V, Ql, p->dVl, dK, dV, p->dQl);
    }
    pool_bwd_kernel<D><<<dim3((unsigned)((s.N * (D / 4) + 255) / 256), BH), 256, 0, st>>>(s, p->dQl, dQ);
    p->launches += 6;   // pool, scores (and routes), top-k, one value recompute, value backward, pool backward
    return cudaGetLastError();
}

cudaError_t run_backward(mita_plan_s* p, const void* Q, const void* K, const void* V, const void* dOut, float* dQ,
                         float* dK, float* dV, cudaStream_t st) {
    if (p->dtype == MITA_BF16) {
        using T = __nv_bfloat16;
        if (p->s.d == 64)
            return run_backward_t<T, 64>(p, (const T*)Q, (const T*)K, (const T*)V, (const T*)dOut, dQ, dK, dV, st);
        return run_backward_t<T, 128>(p, (const T*)Q, (const T*)K, (const T*)V, (const T*)dOut, dQ, dK, dV, st);
    }
    using T = float;
    if (p->s.d == 64)
        return run_backward_t<T, 64>(p, (const T*)Q, (const T*)K, (const T*)V, (const T*)dOut, dQ, dK, dV, st);
    return run_backward_t<T, 128>(p, (const T*)Q, (const T*)K, (const T*)V, (const T*)dOut, dQ, dK, dV, st);
}

cudaError_t staged_topk(const Shape& s, const float* S, int32_t* idx, cudaStream_t st, bool chained) {
    return launch_chained(chained, topk_kernel, dim3(s.m, s.BH()), dim3(kTopkThreads), 0, st, s, S, idx);
}

cudaError_t run_staged(mita_plan_s* p, const void* Q, const void* K, const void* V, void* out, int32_t* idx,
                       int32_t* route, cudaStream_t st) {
    if (p->dtype == MITA_BF16) {
        using T = __nv_bfloat16;
        if (p->s.d == 64) return run_staged_t<T, 64>(p, (const T*)Q, (const T*)K, (const T*)V, (T*)out, idx, route, st);
        return run_staged_t<T, 128>(p, (const T*)Q, (const T*)K, (const T*)V, (T*)out, idx, route, st);
    }
    using T = float;
    if (p->s.d == 64) return run_staged_t<T, 64>(p, (const T*)Q, (const T*)K, (const T*)V, (T*)out, idx, route, st);
    return run_staged_t<T, 128>(p, (const T*)Q, (const T*)K, (const T*)V, (T*)out, idx, route, st);
}

}  // namespace mita
