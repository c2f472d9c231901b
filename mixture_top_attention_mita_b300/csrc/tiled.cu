// Tensor-core tiled MiTA forward for long sequences (bf16, d in {64, 128},
// m <= 256, k <= 1024): the 56x56 vision layer and the 64K-token sequence.
//
// The steps of the operator (36Kr / 新智元 "注意力也是FFN？", section
// "用少量地标查询，同时构造全局概括与细节专家") as a chain of kernels on one
// stream; the landmark scores, landmark values and routes run on tcgen05
// (tcgen.cu), the grouped attention on bf16 mma.sync:
//   tl_pool         Q_l, correctly rounded bin means (16-byte loads, TwoSum
//                   partials per token lane combined error-free)
//   tc_scores       S = Q_l . K^T (fp32, workspace) and each landmark's row
//                   max and min (with the routes, tc_scores_route, when
//                   m <= 256)
//   tl_topk_reg     per landmark the k best keys (ties to the lower index),
//                   rows up to 4096 keys held in registers: a 256-bin
//                   histogram over [min, max], an exact rank of the boundary
//                   bin's members, the expert as a bitmap over the row read
//                   out in key order
//   tl_topk_cb      the same for rows up to 64K keys (N a multiple of 4)
//                   with 2048 bins, the row read once: each key's coarse bin
//                   kept as a byte in shared memory for the second pass
//   tl_topk_bits    the same reading the row twice (other lengths up to
//                   64K keys; longer rows use the staged path's radix select)
//   tc_values       split-K partial sums of exp(S / sqrt d - max) . V and of
//                   the row sums, per split of 1024-4096 keys
//   tl_values_fin   V_l = sum of partials / sum of row sums, bf16
//   tc_route        q . Q_l^T per query tile, first argmax (the route), and
//                   per-landmark query counts (m > 256 only)
//   tl_bucket_off   per head: bucket offsets, cursors and the list of
//                   attention tiles (expert, queries, first bucket position)
//   tl_bucket_put   queries scattered to their bucket
//   tl_attend       per tile: the 64 queries of one expert against the m
//                   shared slots (Q_l, V_l) and the k routed slots (the
//                   expert's K, V rows), streamed through shared memory in
//                   64-slot blocks with an online softmax
#include "mma_util.cuh"
#include "staged.cuh"
#include "tcgen.cuh"
#include "tiled.cuh"
#include "host_cache.cuh"
#include "launch.cuh"

namespace mita {
namespace tl {

using bf16 = __nv_bfloat16;
using namespace mx;

// Queries per attention tile (16 per warp): 64 at both head sizes.  128-query
// tiles at d = 128 gather each routed K, V block once for twice the queries
// but measured slower on the 64K-token rows (3481 vs 3390 us per forward):
// one 8-warp block per SM hides the gathers worse than two 4-warp blocks.
constexpr int qt_of(int) { return 64; }
constexpr int kMaxK = 1024;  // routed keys per expert

int nsplit(const Shape& s) { return tc_value_splits(s); }
int max_tiles(const Shape& s) { return (s.N + qt_of(s.d) - 1) / qt_of(s.d) + s.m; }


// ---------------------------------------------------------------- pool
// Q_l (bf16): block per (landmark i, head bh), 128 threads; the block also
// resets the landmark's row max, row min and query count for the kernels
// after it (in place of three memsets).  Thread t sums the
// 8 features of 16-byte group t % G (G = D / 8) over the bin's tokens
// t / G, t / G + 128 / G, ... (one 16-byte load per token, four in flight),
// each feature with TwoSum compensation; the 128 / G partial (hi, lo) pairs of
// a feature are then combined the same way and the correctly rounded mean is
// decided exactly against c times the midpoints (mean_to_bf16).
template <int D>
__global__ void __launch_bounds__(128) tl_pool(Shape s, const bf16* __restrict__ Q, bf16* __restrict__ Ql,
                                               uint32_t* __restrict__ rowmax, uint32_t* __restrict__ rowmin,
                                               int32_t* __restrict__ counts) {
    chain_wait_and_trigger();
    constexpr int G = D / 8, TL = 128 / G;   // feature groups, token lanes
    __shared__ float2 part[TL][D];
    const int i = blockIdx.x, bh = blockIdx.y, t = threadIdx.x, fg = t % G, tln = t / G;
    if (t == 0) {
        const size_t r = (size_t)bh * s.m + i;
        rowmax[r] = 0u;             // below every score's order key
        rowmin[r] = 0xffffffffu;    // above every score's order key
        counts[r] = 0;
    }
    int r0, r1, c0, c1;
    pool_bin(i / s.pw, s.gh, s.ph, r0, r1);
    pool_bin(i % s.pw, s.gw, s.pw, c0, c1);
    const int w = c1 - c0, cnt = (r1 - r0) * w;
    // token e of the bin is at row e / w, column e % w: the quotient as
    // floor((e + 1/2) / w) in fp32, exact while e < 2^21 (the fraction of
    // (e + 1/2) / w stays 1 / (2 w) from an integer, above the product's
    // relative error of 2^-22); bins hold at most 65536 tokens here
    const float rw = 1.0f / (float)w;
    const bf16* q = Q + (size_t)bh * s.N * D + fg * 8;
    float hi[8], lo[8];
#pragma unroll
    for (int f = 0; f < 8; ++f) hi[f] = lo[f] = 0.0f;
    for (int e0 = tln; e0 < cnt; e0 += 4 * TL) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * TL;
            v[u] = make_uint4(0u, 0u, 0u, 0u);
            if (e < cnt) {
                const int yq = __float2int_rz(((float)e + 0.5f) * rw);
                const int y = r0 + yq, x = c0 + (e - yq * w);
                v[u] = *(const uint4*)(q + (size_t)(y * s.gw + x) * D);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (e0 + u * TL < cnt) {
                const uint32_t pv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    acc2(hi[2 * h], lo[2 * h], __uint_as_float(pv[h] << 16));
                    acc2(hi[2 * h + 1], lo[2 * h + 1], __uint_as_float(pv[h] & 0xffff0000u));
                }
            }
    }
#pragma unroll
    for (int f = 0; f < 8; ++f) part[tln][fg * 8 + f] = make_float2(hi[f], lo[f]);
    __syncthreads();
    for (int f = t; f < D; f += 128) {
        float h = 0.0f, l = 0.0f;
        for (int u = 0; u < TL; ++u) {
            const float2 p = part[u][f];
            float sh, se;
            two_sum(h, p.x, sh, se);
            h = sh;
            l += se + p.y;
        }
        Ql[((size_t)bh * s.m + i) * D + f] = mean_to_bf16(h, l, (float)cnt);
    }
}

// ---------------------------------------------------------------- top-k
constexpr int kTB = 256;          // threads per top-k block
constexpr int kNB = 2048;         // histogram bins of tl_topk_bits (rows past 4096 keys)
constexpr int kCandMax = 1024;    // boundary members ranked exactly

// Block-wide exclusive prefix sum of one int per thread (NT threads);
// *total receives the block total.
template <int NT = kTB>
MITA_DEV int block_excl_scan(int x, int* wsum, int* total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    __syncthreads();
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    int base = 0, tot = 0;
#pragma unroll
    for (int u = 0; u < NT / 32; ++u) {
        const int v = wsum[u];
        base += u < w ? v : 0;
        tot += v;
    }
    *total = tot;
    return base + incl - x;
}

// Block per (landmark i, head bh), rows up to kBitsMaxN keys: the k keys
// with the largest raw scores S[bh, i, :], ties to the lower key index, in
// ascending order.  NB bins of equal width over [row min, row max] (2048 on
// the rows past 4096 keys it is launched for) find the bin
// bin* holding the k-th largest score; every pass over the row is coalesced.
// Pass 1 builds the histogram; pass 2 marks the keys of the bins above bin* in a bitmap
// over the row (one ballot word per 32 keys) and lists bin*'s members with
// their indices; the listed members are ranked exactly (score desc, index
// asc) and the chosen ones join the bitmap; the bitmap, read word by word
// with one block scan, gives the expert in ascending key order.  A bin* with
// more than kCandMax members (ties, flat rows) is resolved by bisecting the
// order key of its need-th best member.
constexpr int kBitsMaxN = 65536;
constexpr int kChainMaxN = 16384;   // rows up to this length: overlapped (chained) launches

template <int NB>
__global__ void __launch_bounds__(kTB) tl_topk_bits(Shape s, const float* __restrict__ S,
                                                    const uint32_t* __restrict__ rowmax,
                                                    const uint32_t* __restrict__ rowmin, int32_t* __restrict__ idx) {
    chain_wait_and_trigger();
    constexpr int BPT = NB / kTB;   // bins per thread in the boundary search
    __shared__ int hist[NB];
    __shared__ uint32_t bits[kBitsMaxN / 32];
    __shared__ float cval[kCandMax];
    __shared__ int cidx[kCandMax];
    __shared__ int wsum[kTB / 32];
    __shared__ int sh[4];
    const int i = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int N = s.N, k = s.k, nw = (N + 31) >> 5;
    const float* row = S + ((size_t)bh * s.m + i) * N;
    const float mx = key_to_float(rowmax[(size_t)bh * s.m + i]);
    const float mn = key_to_float(rowmin[(size_t)bh * s.m + i]);
    const float range = mx - mn;
    const float sc = range > 0.0f ? (float)NB / range : 0.0f;
    auto bin_of = [&](float v) { return min(NB - 1, (int)((v - mn) * sc)); };
    for (int b = tid; b < NB; b += kTB) hist[b] = 0;
    for (int w = tid; w < nw; w += kTB) bits[w] = 0u;
    if (tid == 0) sh[3] = 0;
    __syncthreads();
    if ((N & 3) == 0) {   // 16-byte loads, two in flight per thread
        const float4* row4 = (const float4*)row;
        const int n4 = N >> 2;
        int j = tid;
        for (; j + kTB < n4; j += 2 * kTB) {
            const float4 a = row4[j], b = row4[j + kTB];
            atomicAdd(&hist[bin_of(a.x)], 1);
            atomicAdd(&hist[bin_of(a.y)], 1);
            atomicAdd(&hist[bin_of(a.z)], 1);
            atomicAdd(&hist[bin_of(a.w)], 1);
            atomicAdd(&hist[bin_of(b.x)], 1);
            atomicAdd(&hist[bin_of(b.y)], 1);
            atomicAdd(&hist[bin_of(b.z)], 1);
            atomicAdd(&hist[bin_of(b.w)], 1);
        }
        for (; j < n4; j += kTB) {
            const float4 a = row4[j];
            atomicAdd(&hist[bin_of(a.x)], 1);
            atomicAdd(&hist[bin_of(a.y)], 1);
            atomicAdd(&hist[bin_of(a.z)], 1);
            atomicAdd(&hist[bin_of(a.w)], 1);
        }
    } else {
        for (int j = tid; j < N; j += kTB) atomicAdd(&hist[bin_of(row[j])], 1);
    }
    __syncthreads();
    // thread t holds bins [BPT t, BPT t + BPT); counts of bins above, from the top down
    {
        int c[BPT], tot = 0;
#pragma unroll
        for (int u = 0; u < BPT; ++u) { c[u] = hist[BPT * tid + u]; tot += c[u]; }
        int all;
        const int below = block_excl_scan(tot, wsum, &all);
        const int above = all - below - tot;
        if (above < k && above + tot >= k) {
            int run = above;
#pragma unroll
            for (int u = BPT - 1; u >= 0; --u) {
                if (run < k && run + c[u] >= k) {
                    sh[0] = BPT * tid + u;
                    sh[1] = k - run;
                    sh[2] = c[u];
                }
                run += c[u];
            }
        }
    }
    __syncthreads();
    const int bstar = sh[0], need = sh[1], cstar = sh[2];
    const bool take_all = need >= cstar;            // every member of bin* is in the expert
    const bool listed = !take_all && cstar <= kCandMax;
    // pass 2: warp w walks words w, w + 8, ... (32 consecutive keys per word),
    // four words per step with their loads in flight together
    constexpr int kWS = kTB / 32;
    for (int w = warp; w < nw; w += 4 * kWS) {
        float v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = 32 * (w + u * kWS) + lane;
            v[u] = j < N ? row[j] : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int wu = w + u * kWS;
            if (wu < nw) {   // warp-uniform
                const int j = 32 * wu + lane;
                const int b = j < N ? bin_of(v[u]) : -1;
                const uint32_t sel = __ballot_sync(0xffffffffu, b > bstar || (take_all && b == bstar));
                if (lane == 0) bits[wu] = sel;
                if (listed && b == bstar) {
                    const int p = atomicAdd(&sh[3], 1);
                    cval[p] = v[u];
                    cidx[p] = j;
                }
            }
        }
    }
    __syncthreads();
    if (listed) {
        for (int p = tid; p < cstar; p += kTB) {
            const float v = cval[p];
            const int jp = cidx[p];
            int rank = 0;
            for (int q = 0; q < cstar; ++q) {
                const float w = cval[q];
                rank += (w > v || (w == v && cidx[q] < jp)) ? 1 : 0;
            }
            if (rank < need) atomicOr(&bits[jp >> 5], 1u << (jp & 31));
        }
        __syncthreads();
    } else if (!take_all) {
        // many members: the need-th best member's order key T by bisection, then
        // members above T and, in key order, those equal to T until need is met
        uint32_t T = 0u;
        for (int bb = 31; bb >= 0; --bb) {
            const uint32_t ct = T | (1u << bb);
            int cnt = 0;
            for (int j = tid; j < N; j += kTB) {
                const float v = row[j];
                cnt += (bin_of(v) == bstar && order_key(v) >= ct) ? 1 : 0;
            }
            int total;
            block_excl_scan(cnt, wsum, &total);
            if (total >= need) T = ct;
        }
        int gt = 0;
        for (int j = tid; j < N; j += kTB) {
            const float v = row[j];
            gt += (bin_of(v) == bstar && order_key(v) > T) ? 1 : 0;
        }
        int gt_all;
        block_excl_scan(gt, wsum, &gt_all);
        if (warp == 0) {   // one warp, in key order: members above T, and the first ones equal to T
            int eq_left = need - gt_all;
            for (int w = 0; w < nw; ++w) {
                const int j = 32 * w + lane;
                bool above = false, eq = false;
                if (j < N) {
                    const float v = row[j];
                    if (bin_of(v) == bstar) {
                        const uint32_t kv = order_key(v);
                        above = kv > T;
                        eq = kv == T;
                    }
                }
                const uint32_t eqm = __ballot_sync(0xffffffffu, eq);
                const int r = __popc(eqm & ((1u << lane) - 1u));
                const uint32_t add = __ballot_sync(0xffffffffu, above || (eq && r < eq_left));
                eq_left -= min(eq_left, __popc(eqm));
                if (lane == 0) bits[w] |= add;
            }
        }
        __syncthreads();
    }
    // the expert in ascending key order: thread t reads words [t*wpt, (t+1)*wpt)
    const int wpt = (nw + kTB - 1) / kTB, w0 = min(nw, tid * wpt), w1 = min(nw, w0 + wpt);
    int cnt = 0;
    for (int w = w0; w < w1; ++w) cnt += __popc(bits[w]);
    int total;
    int pos = block_excl_scan(cnt, wsum, &total);
    int32_t* out = idx + ((size_t)bh * s.m + i) * k;
    for (int w = w0; w < w1; ++w) {
        uint32_t b = bits[w];
        while (b) {
            const int x = __ffs(b) - 1;
            b &= b - 1u;
            if (pos < k) out[pos] = 32 * w + x;
            ++pos;
        }
    }
}

// Rows of 4097 .. kBitsMaxN keys, N a multiple of 4: the select of
// tl_topk_bits with the row read from memory once.  Pass 1 builds the
// histogram of kCNB fine bins and keeps each key's coarse bin (fine bin / 8)
// as one byte in shared memory (N bytes); pass 2 decides every key from its
// byte and reads back from the score matrix only the keys of the coarse bin
// that holds bin* (a few dozen per row on these inputs, still in L2).  Two
// blocks of kCT threads per SM: one streams its row while the other works
// from shared memory.
constexpr int kCT = 512;
constexpr int kCNB = 2048;

__global__ void __launch_bounds__(kCT, 2) tl_topk_cb(Shape s, const float* __restrict__ S,
                                                  const uint32_t* __restrict__ rowmax,
                                                  const uint32_t* __restrict__ rowmin, int32_t* __restrict__ idx) {
    chain_wait_and_trigger();
    constexpr int BPT = kCNB / kCT;   // bins per thread in the boundary search
    extern __shared__ __align__(16) unsigned char cbin_raw[];   // coarse bin of every key
    __shared__ int hist[kCNB];
    __shared__ uint32_t bits[kBitsMaxN / 32];
    __shared__ float cval[kCandMax];
    __shared__ int cidx[kCandMax];
    __shared__ int wsum[kCT / 32];
    __shared__ int sh[4];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int N = s.N, k = s.k, nw = (N + 31) >> 5, n4 = N >> 2;
    const size_t r = (size_t)blockIdx.y * s.m + blockIdx.x;
    const float* row = S + r * N;
    uint32_t* cb4 = (uint32_t*)cbin_raw;   // four keys' coarse bins per word
    const float mx = key_to_float(rowmax[r]), mn = key_to_float(rowmin[r]);
    float sc = mx > mn ? (float)kCNB / (mx - mn) : 0.0f;
    float off = -mn * sc;
    if (!(fabsf(off) <= 3.0e38f)) sc = off = 0.0f;   // overflow: one bin, resolved by bisection
    // a monotone function of the score; the unsigned conversion takes
    // negatives and NaN to 0
    auto bin_of = [&](float v) { return (int)min((unsigned)(kCNB - 1), __float2uint_rz(fmaf(v, sc, off))); };
    for (int b = tid; b < kCNB; b += kCT) hist[b] = 0;
    for (int w = tid; w < nw; w += kCT) bits[w] = 0u;
    if (tid == 0) sh[3] = 0;
    __syncthreads();
    auto put4 = [&](int j, const float4& a) {
        const int b0 = bin_of(a.x), b1 = bin_of(a.y), b2 = bin_of(a.z), b3 = bin_of(a.w);
        atomicAdd(&hist[b0], 1);
        atomicAdd(&hist[b1], 1);
        atomicAdd(&hist[b2], 1);
        atomicAdd(&hist[b3], 1);
        cb4[j] = (uint32_t)(b0 >> 3) | ((uint32_t)(b1 >> 3) << 8) | ((uint32_t)(b2 >> 3) << 16) |
                 ((uint32_t)(b3 >> 3) << 24);
    };
    {   // pass 1: 16-byte loads, kU in flight per thread
        constexpr int kU = 8;
        const float4* row4 = (const float4*)row;
        int j = tid;
        for (; j + (kU - 1) * kCT < n4; j += kU * kCT) {
            float4 a[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) a[u] = __ldg(row4 + j + u * kCT);
#pragma unroll
            for (int u = 0; u < kU; ++u) put4(j + u * kCT, a[u]);
        }
        for (; j < n4; j += kCT) put4(j, __ldg(row4 + j));
    }
    __syncthreads();
    {   // thread t holds bins [BPT t, BPT t + BPT); counts of bins above, from the top down
        int c[BPT], tot = 0;
#pragma unroll
        for (int u = 0; u < BPT; ++u) { c[u] = hist[BPT * tid + u]; tot += c[u]; }
        int all;
        const int below = block_excl_scan<kCT>(tot, wsum, &all);
        const int above = all - below - tot;
        if (above < k && above + tot >= k) {
            int run = above;
#pragma unroll
            for (int u = BPT - 1; u >= 0; --u) {
                if (run < k && run + c[u] >= k) {
                    sh[0] = BPT * tid + u;
                    sh[1] = k - run;
                    sh[2] = c[u];
                }
                run += c[u];
            }
        }
    }
    __syncthreads();
    const int bstar = sh[0], need = sh[1], cstar = sh[2];
    const bool take_all = need >= cstar;            // every member of bin* is in the expert
    const bool listed = !take_all && cstar <= kCandMax;
    const uint32_t c4 = ((uint32_t)bstar >> 3) * 0x01010101u;   // bin*'s coarse bin in every byte
    // pass 2: warp w's lanes hold the 128 consecutive keys of bitmap words
    // 4c .. 4c + 3 (c = w, w + 16, ...), four keys (one word of bytes) a
    // lane, compared four at a time; the keys of bin*'s coarse bin (rare) are
    // read back for their fine bin
    for (int c = warp; 32 * c < n4; c += kCT / 32) {
        const int q = 32 * c + lane;
        uint32_t nib = 0u;
        if (q < n4) {
            const uint32_t cbw = cb4[q];
            // one bit per byte above bin*'s coarse bin, gathered into bits 24 .. 27
            nib = (((__vcmpgtu4(cbw, c4) & 0x01010101u) * 0x01020408u) >> 24) & 0xfu;
            const uint32_t eq = __vcmpeq4(cbw, c4);
            if (eq) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if ((eq >> (8 * u)) & 1u) {
                        const float v = row[4 * q + u];
                        const int b = bin_of(v);
                        if (b > bstar || (take_all && b == bstar)) nib |= 1u << u;
                        if (listed && b == bstar) {
                            const int p = atomicAdd(&sh[3], 1);
                            cval[p] = v;
                            cidx[p] = 4 * q + u;
                        }
                    }
                }
            }
        }
        uint32_t word = nib << (4 * (lane & 7));
        word |= __shfl_xor_sync(0xffffffffu, word, 1);
        word |= __shfl_xor_sync(0xffffffffu, word, 2);
        word |= __shfl_xor_sync(0xffffffffu, word, 4);
        const int wi = 4 * c + (lane >> 3);
        if ((lane & 7) == 0 && wi < nw) bits[wi] = word;
    }
    __syncthreads();
    if (listed) {
        for (int p = tid; p < cstar; p += kCT) {
            const float x = cval[p];
            const int jp = cidx[p];
            int rank = 0;
            for (int q = 0; q < cstar; ++q) {
                const float w = cval[q];
                rank += (w > x || (w == x && cidx[q] < jp)) ? 1 : 0;
            }
            if (rank < need) atomicOr(&bits[jp >> 5], 1u << (jp & 31));
        }
        __syncthreads();
    } else if (!take_all) {
        // many members (ties, flat rows): the need-th best member's order key T
        // by bisection over the row, then members above T and, in key order,
        // those equal to T until need is met
        uint32_t T = 0u;
        for (int bb = 31; bb >= 0; --bb) {
            const uint32_t ct = T | (1u << bb);
            int cnt = 0;
            for (int j = tid; j < N; j += kCT) {
                const float v = row[j];
                cnt += (bin_of(v) == bstar && order_key(v) >= ct) ? 1 : 0;
            }
            int total;
            block_excl_scan<kCT>(cnt, wsum, &total);
            if (total >= need) T = ct;
        }
        int gt = 0;
        for (int j = tid; j < N; j += kCT) {
            const float v = row[j];
            gt += (bin_of(v) == bstar && order_key(v) > T) ? 1 : 0;
        }
        int gt_all;
        block_excl_scan<kCT>(gt, wsum, &gt_all);
        if (warp == 0) {
            int eq_left = need - gt_all;
            for (int w = 0; w < nw; ++w) {
                const int j = 32 * w + lane;
                bool above = false, eq = false;
                if (j < N) {
                    const float v = row[j];
                    if (bin_of(v) == bstar) {
                        const uint32_t kv = order_key(v);
                        above = kv > T;
                        eq = kv == T;
                    }
                }
                const uint32_t eqm = __ballot_sync(0xffffffffu, eq);
                const int rr = __popc(eqm & ((1u << lane) - 1u));
                const uint32_t add = __ballot_sync(0xffffffffu, above || (eq && rr < eq_left));
                eq_left -= min(eq_left, __popc(eqm));
                if (lane == 0) bits[w] |= add;
            }
        }
        __syncthreads();
    }
    // the expert in ascending key order: thread t reads words [t*wpt, (t+1)*wpt)
    const int wpt = (nw + kCT - 1) / kCT, w0 = min(nw, tid * wpt), w1 = min(nw, w0 + wpt);
    int cnt = 0;
    for (int w = w0; w < w1; ++w) cnt += __popc(bits[w]);
    int total;
    int pos = block_excl_scan<kCT>(cnt, wsum, &total);
    int32_t* out = idx + r * k;
    for (int w = w0; w < w1; ++w) {
        uint32_t b = bits[w];
        while (b) {
            const int x = __ffs(b) - 1;
            b &= b - 1u;
            if (pos < k) out[pos] = 32 * w + x;
            ++pos;
        }
    }
}

size_t topk_cb_smem(int N) { return ((size_t)N + 15) / 16 * 16; }

// Rows up to kRegRowN keys (the 56x56 layer's 3136): the expert of
// tl_topk_bits with 256 bins, with thread t holding keys t, t + kTB, ... of
// the row in registers.  The row is read once; the second pass recomputes
// each key's bin (one fused multiply-add) from its register, and warp w's
// lanes hold the 32 consecutive keys of bitmap word 8u + w in register u.
// VPT = ceil(N / kTB) keys a thread: every thread's first VPT - 1 keys are in
// the row, so only the last one is checked.
constexpr int kRegVPT = 16;
constexpr int kRegRowN = kRegVPT * kTB;

template <int VPT>
__global__ void __launch_bounds__(kTB, 6) tl_topk_reg(Shape s, const float* __restrict__ S,
                                                   const uint32_t* __restrict__ rowmax,
                                                   const uint32_t* __restrict__ rowmin, int32_t* __restrict__ idx) {
    chain_wait_and_trigger();
    constexpr int NB = 256;   // one bin per thread in the boundary search
    __shared__ int hist[NB];
    __shared__ uint32_t bits[kRegRowN / 32];
    __shared__ float cval[kCandMax];
    __shared__ int cidx[kCandMax];
    __shared__ int wsum[kTB / 32];
    __shared__ int sh[4];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int N = s.N, k = s.k, nw = (N + 31) >> 5;
    const size_t r = (size_t)blockIdx.y * s.m + blockIdx.x;
    const float* row = S + r * N;
    const float mx = key_to_float(rowmax[r]), mn = key_to_float(rowmin[r]);
    float sc = mx > mn ? (float)NB / (mx - mn) : 0.0f;
    float off = -mn * sc;
    if (!(fabsf(off) <= 3.0e38f)) sc = off = 0.0f;   // overflow: one bin, resolved by bisection
    // a monotone function of the score; the conversion takes negatives to 0
    auto bin_of = [&](float v) { return min(NB - 1, (int)fmaf(v, sc, off)); };
    // key u of this thread is in the row (only the last can fall past it)
    auto in_row = [&](int u) { return u < VPT - 1 || tid + kTB * u < N; };
    float v[VPT];
#pragma unroll
    for (int u = 0; u < VPT; ++u) v[u] = in_row(u) ? __ldg(row + tid + kTB * u) : 0.0f;
    hist[tid] = 0;
    for (int w = tid; w < nw; w += kTB) bits[w] = 0u;
    if (tid == 0) sh[3] = 0;
    __syncthreads();
#pragma unroll
    for (int u = 0; u < VPT; ++u)
        if (in_row(u)) atomicAdd(&hist[bin_of(v[u])], 1);
    __syncthreads();
    {   // bin* holds the k-th best score: counts of the bins above, from the top down
        const int c = hist[tid];
        int all;
        const int below = block_excl_scan(c, wsum, &all);
        const int above = all - below - c;
        if (above < k && above + c >= k) {
            sh[0] = tid;
            sh[1] = k - above;
            sh[2] = c;
        }
    }
    __syncthreads();
    const int bstar = sh[0], need = sh[1], cstar = sh[2];
    const bool take_all = need >= cstar;            // every member of bin* is in the expert
    const bool listed = !take_all && cstar <= kCandMax;
    const int bsel = take_all ? bstar - 1 : bstar;   // keys of bins above bsel are in the expert
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
        const int j0 = kTB * u + 32 * warp;
        if (u < VPT - 1 || j0 < N) {   // warp-uniform
            const int j = j0 + lane;
            const int b = in_row(u) ? bin_of(v[u]) : -1;
            const uint32_t sel = __ballot_sync(0xffffffffu, b > bsel);
            if (lane == 0) bits[j0 >> 5] = sel;
            if (listed && b == bstar) {
                const int p = atomicAdd(&sh[3], 1);
                cval[p] = v[u];
                cidx[p] = j;
            }
        }
    }
    __syncthreads();
    if (listed) {
        for (int p = tid; p < cstar; p += kTB) {
            const float x = cval[p];
            const int jp = cidx[p];
            int rank = 0;
            for (int q = 0; q < cstar; ++q) {
                const float w = cval[q];
                rank += (w > x || (w == x && cidx[q] < jp)) ? 1 : 0;
            }
            if (rank < need) atomicOr(&bits[jp >> 5], 1u << (jp & 31));
        }
        __syncthreads();
    } else if (!take_all) {
        // many members: the need-th best member's order key T by bisection, then
        // members above T and, in key order, those equal to T until need is met
        uint32_t T = 0u;
        for (int bb = 31; bb >= 0; --bb) {
            const uint32_t ct = T | (1u << bb);
            int cnt = 0;
#pragma unroll
            for (int u = 0; u < VPT; ++u)
                cnt += (in_row(u) && bin_of(v[u]) == bstar && order_key(v[u]) >= ct) ? 1 : 0;
            int total;
            block_excl_scan(cnt, wsum, &total);
            if (total >= need) T = ct;
        }
        int gt = 0;
#pragma unroll
        for (int u = 0; u < VPT; ++u)
            gt += (in_row(u) && bin_of(v[u]) == bstar && order_key(v[u]) > T) ? 1 : 0;
        int gt_all;
        block_excl_scan(gt, wsum, &gt_all);
        if (warp == 0) {   // one warp, in key order: members above T, and the first ones equal to T
            int eq_left = need - gt_all;
            for (int w = 0; w < nw; ++w) {
                const int j = 32 * w + lane;
                bool above = false, eq = false;
                if (j < N) {
                    const float x = row[j];
                    if (bin_of(x) == bstar) {
                        const uint32_t kv = order_key(x);
                        above = kv > T;
                        eq = kv == T;
                    }
                }
                const uint32_t eqm = __ballot_sync(0xffffffffu, eq);
                const int rr = __popc(eqm & ((1u << lane) - 1u));
                const uint32_t add = __ballot_sync(0xffffffffu, above || (eq && rr < eq_left));
                eq_left -= min(eq_left, __popc(eqm));
                if (lane == 0) bits[w] |= add;
            }
        }
        __syncthreads();
    }
    // the expert in ascending key order: thread t reads words [t*wpt, (t+1)*wpt)
    const int wpt = (nw + kTB - 1) / kTB, w0 = min(nw, tid * wpt), w1 = min(nw, w0 + wpt);
    int cnt = 0;
    for (int w = w0; w < w1; ++w) cnt += __popc(bits[w]);
    int total;
    int pos = block_excl_scan(cnt, wsum, &total);
    int32_t* out = idx + r * k;
    for (int w = w0; w < w1; ++w) {
        uint32_t b = bits[w];
        while (b) {
            const int x = __ffs(b) - 1;
            b &= b - 1u;
            if (pos < k) out[pos] = 32 * w + x;
            ++pos;
        }
    }
}

// tl_topk_reg for N <= kRegRowN keys with VPT = ceil(N / kTB).
template <int VPT = kRegVPT>
cudaError_t launch_topk_reg(bool chain, const Shape& s, dim3 grid, cudaStream_t st, const float* S,
                            const uint32_t* rowmax, const uint32_t* rowmin, int32_t* idx) {
    if constexpr (VPT > 1) {
        if ((s.N + kTB - 1) / kTB < VPT) return launch_topk_reg<VPT - 1>(chain, s, grid, st, S, rowmax, rowmin, idx);
    }
    return launch_chained(chain, tl_topk_reg<VPT>, grid, dim3(kTB), 0, st, s, S, rowmax, rowmin, idx);
}

// V_l[i] = (sum over splits of the partial row) / (sum of the partial row sums).
template <int D>
__global__ void tl_values_fin(Shape s, const float* __restrict__ part, int ns, bf16* __restrict__ Vl) {
    chain_wait_and_trigger();
    const int i = blockIdx.x, bh = blockIdx.y, f = threadIdx.x;
    const float* src = part + ((size_t)bh * ns * s.m + i) * (D + 1);
    float num = 0.0f, den = 0.0f;
    for (int sp = 0; sp < ns; ++sp) {
        num += src[(size_t)sp * s.m * (D + 1) + f];
        den += src[(size_t)sp * s.m * (D + 1) + D];
    }
    Vl[((size_t)bh * s.m + i) * D + f] = __float2bfloat16_rn(num / den);
}

// As tl_values_fin, also keeping V_l in fp32 and each row's softmax stats
// {max raw score, sum of the numerators} for the backward.
template <int D>
__global__ void tl_values_fin_stats(Shape s, const float* __restrict__ part, int ns, const uint32_t* __restrict__ rowmax,
                                    bf16* __restrict__ Vl, float* __restrict__ Vl32, float* __restrict__ stats) {
    const int i = blockIdx.x, bh = blockIdx.y, f = threadIdx.x;
    const float* src = part + ((size_t)bh * ns * s.m + i) * (D + 1);
    float num = 0.0f, den = 0.0f;
    for (int sp = 0; sp < ns; ++sp) {
        num += src[(size_t)sp * s.m * (D + 1) + f];
        den += src[(size_t)sp * s.m * (D + 1) + D];
    }
    const size_t row = (size_t)bh * s.m + i;
    const float y = num / den;
    Vl[row * D + f] = __float2bfloat16_rn(y);
    Vl32[row * D + f] = y;
    if (f == 0) {
        stats[2 * row] = key_to_float(rowmax[row]);
        stats[2 * row + 1] = den;
    }
}

// ---------------------------------------------------------------- buckets
// One warp per head: bucket offsets (exclusive scan of the counts), the
// scatter cursors and the attention tile list: per tile (expert << 16 |
// queries, first position in the head's bucketed query order).
__global__ void tl_bucket_off(Shape s, const int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                              int32_t* __restrict__ cursor, int2* __restrict__ tiles,
                              int32_t* __restrict__ ntiles, int maxt, int qt) {
    chain_wait_and_trigger();
    const int bh = blockIdx.x, lane = threadIdx.x;
    const int32_t* cnt = counts + (size_t)bh * s.m;
    int carry = 0, tcarry = 0;
    for (int i0 = 0; i0 < s.m; i0 += 32) {
        const int i = i0 + lane;
        const int c = i < s.m ? cnt[i] : 0, nt = (c + qt - 1) / qt;
        int x = c, y = nt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, x, o), b = __shfl_up_sync(0xffffffffu, y, o);
            if (lane >= o) { x += a; y += b; }
        }
        if (i < s.m) {
            offsets[(size_t)bh * (s.m + 1) + i] = carry + x - c;
            cursor[(size_t)bh * s.m + i] = carry + x - c;
            for (int e = 0; e < nt; ++e) {
                const int tt = tcarry + y - nt + e;
                if (tt < maxt)
                    tiles[(size_t)bh * maxt + tt] = make_int2((i << 16) | min(qt, c - e * qt), carry + x - c + e * qt);
            }
        }
        carry += __shfl_sync(0xffffffffu, x, 31);
        tcarry += __shfl_sync(0xffffffffu, y, 31);
    }
    if (lane == 0) {
        offsets[(size_t)bh * (s.m + 1) + s.m] = carry;
        ntiles[bh] = min(tcarry, maxt);
    }
}

__global__ void tl_bucket_put(Shape s, const int32_t* __restrict__ route, int32_t* __restrict__ cursor,
                              int32_t* __restrict__ perm, int32_t* __restrict__ status) {
    chain_wait_and_trigger();
    const int bh = blockIdx.y, q = blockIdx.x * blockDim.x + threadIdx.x, lane = threadIdx.x & 31;
    int r = q < s.N ? route[(size_t)bh * s.N + q] : -1;
    if (q < s.N && (r < 0 || r >= s.m)) {
        atomicExch(status, (int)MITA_ERR_DEVICE);
        r = -1;
    }
    // lanes of the warp with the same route take their places with one atomic:
    // the group's lowest lane adds the group size, the others add their rank
    const unsigned grp = __match_any_sync(0xffffffffu, r);
    if (r < 0) return;
    const int leader = __ffs(grp) - 1;
    int base = 0;
    if (lane == leader) base = atomicAdd(&cursor[(size_t)bh * s.m + r], __popc(grp));
    base = __shfl_sync(grp, base, leader);
    perm[(size_t)bh * s.N + base + __popc(grp & ((1u << lane) - 1u))] = q;
}

// ---------------------------------------------------------------- attention
// Block: one tile = up to QT queries of one expert (QT / 16 warps x 16 rows).
// Slots 0..m-1 are the shared pairs (Q_l, V_l), slots m..m+k-1 the routed
// pairs (K, V rows of the expert's keys); 64-slot blocks are staged by
// cp.async into a double buffer and folded in by an online softmax.
template <int D, int QT>
__global__ void __launch_bounds__(2 * QT, D == 64 ? 4 : 1)
    tl_attend(Shape s, const bf16* __restrict__ Q, const bf16* __restrict__ K, const bf16* __restrict__ V,
              const bf16* __restrict__ Ql, const bf16* __restrict__ Vl, const int32_t* __restrict__ idx,
              const int32_t* __restrict__ perm, const int2* __restrict__ tiles,
              const int32_t* __restrict__ ntiles, int maxt,
              bf16* __restrict__ out, float cs, int shared, int32_t* __restrict__ status) {
    chain_wait_and_trigger();
    constexpr int RB = 2 * D, CH = D / 8, KS = D / 16, NT = D / 8;
    extern __shared__ __align__(128) unsigned char sm[];
    constexpr int NTH = 2 * QT;   // threads
    __shared__ int rows_s[QT];
    __shared__ int E_s[kMaxK];   // the expert's key indices (read once per tile, not per staged row)
    const int bh = blockIdx.y, tile = blockIdx.x;
    if (tile >= ntiles[bh]) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, t = lane & 3;
    const int2 td = tiles[(size_t)bh * maxt + tile];
    const int e = td.x >> 16, nq = td.x & 0xffff, qstart = td.y;
    const int L = s.m + s.k, nblk = (L + 63) / 64;
    const int32_t* E = idx + ((size_t)bh * s.m + e) * s.k;
    const uint32_t uq = smem_u32(sm), ukv = uq + QT * RB;   // kv buffer b: K at ukv + b*2*64*RB, V after it
    const size_t hoff = (size_t)bh * s.N * D;
    if (tid < QT) {
        int q = perm[(size_t)bh * s.N + qstart + min(tid, nq - 1)];
        if (q < 0 || q >= s.N) { atomicExch(status, (int)MITA_ERR_DEVICE); q = 0; }
        rows_s[tid] = q;
    }
    for (int x = tid; x < s.k; x += NTH) {
        int j = E[x];
        if (j < 0 || j >= s.N) { atomicExch(status, (int)MITA_ERR_DEVICE); j = 0; }
        E_s[x] = j;
    }
    __syncthreads();
    // thread t copies 16-byte chunk cc = t % CH of rows r0 + RS i (r0 = t / CH);
    // RS is a multiple of 8, so the rows' swizzle term is the same for every
    // i and the shared-memory offsets are soff + RS RB i
    constexpr int RS = NTH / CH;   // rows per pass: 16 at d = 64, 8 at d = 128
    static_assert(RS % 8 == 0, "rows per pass keep the swizzle term");
    const int cc = tid % CH, r0 = tid / CH;
    const uint32_t soff = swz<RB>(r0, cc);
#pragma unroll
    for (int i = 0; i < QT / RS; ++i)
        cp_async16(uq + soff + (uint32_t)(i * RS * RB), Q + hoff + (size_t)rows_s[r0 + RS * i] * D + 8 * cc, 16u);
    const bf16* qlb = Ql + (size_t)bh * s.m * D + 8 * cc;
    const bf16* vlb = Vl + (size_t)bh * s.m * D + 8 * cc;
    const bf16* kgb = K + hoff + 8 * cc;
    const bf16* vgb = V + hoff + 8 * cc;
    auto stage = [&](int b) {
        const uint32_t kb = ukv + (uint32_t)(b & 1) * 2u * 64u * RB + soff, vb = kb + 64u * RB;
#pragma unroll
        for (int i = 0; i < 64 / RS; ++i) {
            const int slot = b * 64 + r0 + RS * i;
            const bf16 *ks = qlb, *vs = vlb;
            uint32_t nbytes = 16u;
            if (slot < s.m) {
                ks = qlb + (size_t)slot * D;
                vs = vlb + (size_t)slot * D;
            } else if (slot < L) {
                const size_t j = (size_t)E_s[slot - s.m] * D;
                ks = kgb + j;
                vs = vgb + j;
            } else {
                nbytes = 0u;   // zero rows past the last slot
            }
            cp_async16(kb + (uint32_t)(i * RS * RB), ks, nbytes);
            cp_async16(vb + (uint32_t)(i * RS * RB), vs, nbytes);
        }
        cp_async_commit();
    };
    stage(0);

    const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, brow = (lane & 7) + (lane >> 4) * 8;
    uint32_t qa[KS][4];
    float o[NT][4], osum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
    float m0 = -INFINITY, m1 = -INFINITY;   // running max (raw logits) of rows g, g+8
    const bool active = warp * 16 < nq;     // the warp's 16 rows hold at least one query
    for (int b = 0; b < nblk; ++b) {
        if (b + 1 < nblk) {
            stage(b + 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (active) {   // warps past the tile's queries only stage rows and wait
            if (b == 0) {
#pragma unroll
                for (int kk = 0; kk < KS; ++kk)
                    ldsm_x4(uq + swz<RB>(warp * 16 + arow, 2 * kk + (lane >> 4)), qa[kk][0], qa[kk][1], qa[kk][2],
                            qa[kk][3]);
            }
            const uint32_t kb = ukv + (uint32_t)(b & 1) * 2u * 64u * RB, vb = kb + 64u * RB;
            float sc[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.0f;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk)
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kb + swz<RB>(np * 16 + brow, 2 * kk + ((lane >> 3) & 1)), b0, b1, b2, b3);
                    mma16816(sc[2 * np], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                    mma16816(sc[2 * np + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
                }
            if (b * 64 + 64 > L) {   // padding slots of the last block
#pragma unroll
                for (int n = 0; n < 8; ++n)
#pragma unroll
                    for (int x = 0; x < 4; ++x)
                        if (b * 64 + 8 * n + 2 * t + (x & 1) >= L) sc[n][x] = -INFINITY;
            }
            if (!shared && b * 64 < s.m) {   // routing only: the shared slots take no weight
#pragma unroll
                for (int n = 0; n < 8; ++n)
#pragma unroll
                    for (int x = 0; x < 4; ++x)
                        if (b * 64 + 8 * n + 2 * t + (x & 1) < s.m) sc[n][x] = -INFINITY;
            }
            float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                bm0 = fmaxf(bm0, fmaxf(sc[n][0], sc[n][1]));
                bm1 = fmaxf(bm1, fmaxf(sc[n][2], sc[n][3]));
            }
#pragma unroll
            for (int x = 1; x <= 2; x <<= 1) {
                bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, x));
                bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, x));
            }
            const float n0 = fmaxf(m0, bm0), n1 = fmaxf(m1, bm1);
            const float f0 = ex2((m0 - n0) * cs), f1 = ex2((m1 - n1) * cs);   // 0 on the first block
            m0 = n0;
            m1 = n1;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                o[n][0] *= f0;
                o[n][1] *= f0;
                o[n][2] *= f1;
                o[n][3] *= f1;
            }
            osum[0] *= f0;
            osum[1] *= f0;
            osum[2] *= f1;
            osum[3] *= f1;
            const float mb0 = n0 * cs, mb1 = n1 * cs;
            uint32_t pa[4][4];
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                pa[n >> 1][(n & 1) * 2 + 0] = pack2(ex2(fmaf(sc[n][0], cs, -mb0)), ex2(fmaf(sc[n][1], cs, -mb0)));
                pa[n >> 1][(n & 1) * 2 + 1] = pack2(ex2(fmaf(sc[n][2], cs, -mb1)), ex2(fmaf(sc[n][3], cs, -mb1)));
            }
            const int vrow = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                mma16816(osum, pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], kOnes2, kOnes2);
#pragma unroll
                for (int np = 0; np < NT / 2; ++np) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(vb + swz<RB>(ks * 16 + vrow, 2 * np + (lane >> 4)), b0, b1, b2, b3);
                    mma16816(o[2 * np], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], b0, b1);
                    mma16816(o[2 * np + 1], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], b2, b3);
                }
            }
        }
        __syncthreads();   // this buffer is restaged two blocks later
    }
    // normalise; the rows go over the warp's own query rows, then out
    if (active) {
        const float inv0 = rcp(osum[0]), inv1 = rcp(osum[2]);
        const int srow = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
            const uint32_t r0 = pack2(o[2 * np][0] * inv0, o[2 * np][1] * inv0);
            const uint32_t r1 = pack2(o[2 * np][2] * inv1, o[2 * np][3] * inv1);
            const uint32_t r2 = pack2(o[2 * np + 1][0] * inv0, o[2 * np + 1][1] * inv0);
            const uint32_t r3 = pack2(o[2 * np + 1][2] * inv1, o[2 * np + 1][3] * inv1);
            stsm_x4(uq + swz<RB>(srow, 2 * np + (lane >> 4)), r0, r1, r2, r3);
        }
    }
    __syncthreads();
    for (int x = tid; x < nq * CH; x += NTH) {
        const int r = x / CH, c = x % CH;
        *(uint4*)(out + hoff + (size_t)rows_s[r] * D + 8 * c) = *(const uint4*)(sm + swz<RB>(r, c));
    }
}

// Heads per landmark-stage launch.  All heads at once: grouping heads so
// that a group's raw scores stay in L2 starves the launches of blocks at
// these head counts (measured slower at both long shapes).
int head_group(const Shape& s) { return s.BH(); }

template <int D>
cudaError_t run_t(mita_plan_s* p, const bf16* Q, const bf16* K, const bf16* V, bf16* out, int32_t* idx,
                  int32_t* route, cudaStream_t st) {
    const Shape& s = p->s;
    const int BH = s.BH();
    constexpr int RB = 2 * D;
    const float cs = kLog2e / sqrtf((float)D);
    bf16* Ql = (bf16*)p->Ql;
    bf16* Vl = (bf16*)p->Vl;
    uint32_t* rowmin = p->rowmax + (size_t)BH * s.m;
    cudaError_t err;
    // launches overlap their predecessor's tail on short rows, where launch
    // latency is a visible share of the chain; on long rows (kernels of
    // hundreds of microseconds) the overlap measured slower and is off
    const bool chain = s.N <= kChainMaxN;
    if ((err = launch_chained(chain, tl_pool<D>, dim3(s.m, BH), dim3(128), 0, st, s, Q, Ql, p->rowmax, rowmin,
                              p->counts)) != cudaSuccess)
        return err;
    const int ns = nsplit(s), G = head_group(s);
    // up to 128 landmarks: scores and routes from one kernel per token tile
    const bool scores_route = tc_scores_route_supported(s) && G == BH;
    for (int h0 = 0; h0 < BH; h0 += G) {
        Shape sg = s;
        sg.B = 1;
        sg.H = min(G, BH - h0);
        const size_t mo = (size_t)h0 * s.m, no = (size_t)h0 * s.N;
        if (scores_route) {
            if ((err = tc_scores_route(s, Ql, K, Q, p->S, p->rowmax, rowmin, route, p->counts, p->status, st, chain)) !=
                cudaSuccess)
                return err;
        } else if ((err = tc_scores(sg, Ql + mo * D, K + no * D, p->S, p->rowmax + mo, rowmin + mo, p->status, st,
                                    chain)) != cudaSuccess) {
            return err;
        }
        if (s.N > kRegRowN && s.N <= kBitsMaxN && (s.N & 3) == 0) {
            const size_t smem = topk_cb_smem(s.N);
            if ((err = ensure_smem_attr((const void*)tl_topk_cb, smem)) != cudaSuccess) return err;
            if ((err = launch_chained(chain, tl_topk_cb, dim3(s.m, sg.H), dim3(kCT), smem, st, sg, (const float*)p->S,
                                      (const uint32_t*)(p->rowmax + mo), (const uint32_t*)(rowmin + mo),
                                      idx + mo * s.k)) != cudaSuccess)
                return err;
        } else if (s.N <= kRegRowN) {
            if ((err = launch_topk_reg(chain, sg, dim3(s.m, sg.H), st, (const float*)p->S,
                                       (const uint32_t*)(p->rowmax + mo), (const uint32_t*)(rowmin + mo),
                                       idx + mo * s.k)) != cudaSuccess)
                return err;
        } else if (s.N <= kBitsMaxN) {
            if ((err = launch_chained(chain, tl_topk_bits<kNB>, dim3(s.m, sg.H), dim3(kTB), 0, st, sg,
                                      (const float*)p->S, (const uint32_t*)(p->rowmax + mo),
                                      (const uint32_t*)(rowmin + mo), idx + mo * s.k)) != cudaSuccess)
                return err;
        } else {   // rows past the bitmap: the staged path's radix select
            if ((err = staged_topk(sg, p->S, idx + mo * s.k, st, chain)) != cudaSuccess) return err;
        }
        if ((err = tc_values(sg, p->S, p->rowmax + mo, V + no * D, p->vpart, cs, p->status, st, chain)) != cudaSuccess)
            return err;
        if ((err = launch_chained(chain, tl_values_fin<D>, dim3(s.m, sg.H), dim3(D), 0, st, sg, (const float*)p->vpart, ns,
                                  Vl + mo * D)) != cudaSuccess)
            return err;
        p->launches += 4;
    }
    if (!scores_route) {
        if ((err = tc_route(s, Q, Ql, route, p->counts, p->status, st, chain)) != cudaSuccess) return err;
        p->launches += 1;
    }
    const int maxt = max_tiles(s);
    constexpr int QT = qt_of(D);
    if ((err = launch_chained(chain, tl_bucket_off, dim3(BH), dim3(32), 0, st, s, (const int32_t*)p->counts, p->offsets,
                              p->cursor, (int2*)p->tiles, p->ntiles, maxt, QT)) != cudaSuccess)
        return err;
    if ((err = launch_chained(chain, tl_bucket_put, dim3((s.N + 255) / 256, BH), dim3(256), 0, st, s, (const int32_t*)route,
                              p->cursor, p->perm, p->status)) != cudaSuccess)
        return err;
    {
        const int smem = (QT + 4 * 64) * RB;
        auto kern = tl_attend<D, QT>;
        ensure_smem_attr((const void*)kern, smem);
        if ((err = launch_chained(chain, kern, dim3(maxt, BH), dim3(2 * QT), smem, st, s, Q, K, V, (const bf16*)Ql,
                                  (const bf16*)Vl, (const int32_t*)idx, (const int32_t*)p->perm,
                                  (const int2*)p->tiles, (const int32_t*)p->ntiles, maxt,
                                  out, cs, p->routing_only ? 0 : 1, p->status)) != cudaSuccess)
            return err;
    }
    p->launches += 4;
    return cudaGetLastError();
}

}  // namespace tl

bool tiled_supported(const Shape& s, mita_dtype_t dtype) {
    return dtype == MITA_BF16 && (s.d == 64 || s.d == 128) && s.m <= 256 && s.k <= tl::kMaxK && s.N < (1 << 24);
}

size_t tiled_part_bytes(const Shape& s) {
    return (size_t)tl::head_group(s) * tl::nsplit(s) * s.m * (s.d + 1) * sizeof(float);
}

int tiled_max_tiles(const Shape& s) { return tl::max_tiles(s); }

bool tiled_topk_supported(const Shape& s) { return s.N <= tl::kRegRowN; }

cudaError_t tiled_values_stats(const Shape& s, const float* S, const uint32_t* rowmax, const void* V, float* part,
                               void* Vl, float* Vl32, float* stats, int32_t* status, cudaStream_t st) {
    const float cs = kLog2e / sqrtf((float)s.d);
    cudaError_t err = tc_values(s, S, rowmax, V, part, cs, status, st, false);
    if (err != cudaSuccess) return err;
    const int ns = tl::nsplit(s);
    using T = __nv_bfloat16;
    if (s.d == 64)
        return launch_chained(false, tl::tl_values_fin_stats<64>, dim3(s.m, s.BH()), dim3(64), 0, st, s,
                              (const float*)part, ns, rowmax, (T*)Vl, Vl32, stats);
    return launch_chained(false, tl::tl_values_fin_stats<128>, dim3(s.m, s.BH()), dim3(128), 0, st, s,
                          (const float*)part, ns, rowmax, (T*)Vl, Vl32, stats);
}

cudaError_t tiled_topk(const Shape& s, const float* S, const uint32_t* rowmax, int32_t* idx, cudaStream_t st) {
    const uint32_t* rowmin = rowmax + (size_t)s.BH() * s.m;
    return tl::launch_topk_reg(false, s, dim3(s.m, s.BH()), st, S, rowmax, rowmin, idx);
}

cudaError_t tiled_pool(const Shape& s, const void* Q, void* Ql, uint32_t* rowmax, int32_t* counts, cudaStream_t st) {
    using T = __nv_bfloat16;
    uint32_t* rowmin = rowmax + (size_t)s.BH() * s.m;
    if (s.d == 64)
        return launch_chained(false, tl::tl_pool<64>, dim3(s.m, s.BH()), dim3(128), 0, st, s, (const T*)Q, (T*)Ql,
                              rowmax, rowmin, counts);
    return launch_chained(false, tl::tl_pool<128>, dim3(s.m, s.BH()), dim3(128), 0, st, s, (const T*)Q, (T*)Ql, rowmax,
                          rowmin, counts);
}

cudaError_t run_tiled(mita_plan_s* p, const void* Q, const void* K, const void* V, void* out, int32_t* idx,
                      int32_t* route, cudaStream_t st) {
    using T = __nv_bfloat16;
    if (p->s.d == 64) return tl::run_t<64>(p, (const T*)Q, (const T*)K, (const T*)V, (T*)out, idx, route, st);
    return tl::run_t<128>(p, (const T*)Q, (const T*)K, (const T*)V, (T*)out, idx, route, st);
}

}  // namespace mita
