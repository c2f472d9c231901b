// One-kernel MiTA forward for short sequences (bf16, d = 64, N <= 256,
// m <= 32, k <= 32): the DeiT-T / DeiT-S layer shapes.
//
// The six steps of the operator (36Kr / 新智元 "注意力也是FFN？", section
// "用少量地标查询，同时构造全局概括与细节专家") run per head inside one CTA of
// 8 warps, from shared memory:
//   load      TMA (128-byte swizzle) of the head's Q, K and V tiles
//   phase A   pool        Q_l = correctly rounded bin means of Q (warp per
//                         landmark, two features per lane)
//   phase B   contraction [K ; Q] . Q_l^T with mma.sync: raw landmark scores
//                         (fp32, shared memory) and each query's first argmax
//                         landmark (the route)
//   phase C   select      per landmark (an 8-lane group per landmark, four
//                         per warp) the k best keys, ties to the lower index,
//                         by a monotone 64-bin histogram and an exact rank of
//                         the boundary bin's members; the bf16 softmax
//                         numerators overwrite the scores; one warp
//                         bucket-sorts the queries by route
//   phase D   values      V_l = P . V with mma.sync, normalised, bf16
//   phase E   attention   per (expert, 16 queries) tile: logits against the
//                         32 shared slots (Q_l) and 32 routed slots (the
//                         expert's keys, gathered row by row by ldmatrix), one
//                         softmax over both, output = P . [V_l ; V_E]; the
//                         output rows overwrite the tile's own query rows
//   store     TMA store of the head's output tile, then the next head's load
// Two CTAs share an SM (about 110 KB of shared memory each), so one CTA's
// loads and stores overlap the other's arithmetic.  Heads are strided over a
// persistent grid.
#include <cuda.h>

#include <algorithm>

#include "fused.cuh"
#include "host_cache.cuh"

namespace mita {
namespace fz {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kD = 64;
constexpr int kSlots = 32;      // shared slots (m <= 32) and routed slots (k <= 32)
constexpr int kMaxN = 256;
constexpr int kBins = 64;       // histogram bins of the select
constexpr int kCandG = 16;      // boundary-bin members ranked exactly per landmark
constexpr int kTile = 16;       // queries per attention tile
constexpr int kMaxSmem = 232448;
constexpr int kTokMax = 1024;   // bin memberships of all landmarks (the pool's token table)

// Select layout: one landmark per 8-lane group, lane g of the group holding
// the NV = 4 * NV4 consecutive keys [g * NV, g * NV + NV) of the landmark's
// score row, stored from column g * nvp (nvp = NV, or NV + 4 when NV is a
// multiple of 8, so that the 16-byte loads of the 8 lanes hit distinct banks).
constexpr int nv4_of(int N) { return ((N + 7) / 8 + 3) / 4; }
constexpr int nvp_of(int nv4) { return (4 * nv4) % 8 == 0 ? 4 * nv4 + 4 : 4 * nv4; }
// Per-landmark scratch inside the landmark's own score row (fp32 words), used
// after its scores are in registers and before its numerators overwrite it:
constexpr int kRowHist = 0;                 // 64 bin counts
constexpr int kRowCand = kBins;             // kCandG (score, key) pairs
constexpr int kRowTJ = kBins + 2 * kCandG;  // the threshold (score, key)
constexpr int kRowCnt = kRowTJ + 2;         // members of b* listed so far
constexpr int kRowScratch = kRowCnt + 1;

struct Layout {
    int N, np16, nk16, sstr, nvp, qkv;
    int oQ, oK, oV, oQl, oVl, oS, oIdx, oRoute, oPerm, oCnt, oOff, oTiles, oCtl, oBar, oTok, total;
};

static int align_to(int x, int a) { return (x + a - 1) / a * a; }

static Layout make_layout(int N, int m, int ntok) {
    Layout L{};
    L.N = N;
    L.np16 = align_to(N, 16);
    L.nk16 = L.np16 / 16;
    L.nvp = nvp_of(nv4_of(N));
    // fp32 words per score row: the 8 lanes' segments and the row scratch, a
    // multiple of 4 (16-byte rows) that is 4 mod 8, so that the 8 rows of a
    // phase-D ldmatrix fall in distinct banks
    int sstr = std::max(8 * L.nvp, kRowScratch);
    sstr = align_to(sstr, 4);
    if (sstr % 8 == 0) sstr += 4;
    L.sstr = sstr;
    L.qkv = align_to(N * 128, 1024);
    int o = 0;
    auto take = [&](int bytes, int al) { o = align_to(o, al); int r = o; o += bytes; return r; };
    L.oQ = take(L.qkv, 1024);
    L.oK = take(L.qkv, 1024);
    L.oV = take(N * 128, 1024);
    L.oQl = take(kSlots * 128, 128);
    L.oVl = take(kSlots * 128, 128);
    L.oS = take(std::max(m * L.sstr * 4, m * 128), 128);   // scores / numerators, or the pool's fallback list
    L.oIdx = take(kSlots * kSlots, 16);
    L.oRoute = take(kMaxN, 16);
    L.oPerm = take(kMaxN, 16);
    L.oCnt = take((kSlots + 1) * 4, 16);
    L.oOff = take((kSlots + 1) * 4, 16);
    L.oTiles = take((kMaxN / kTile + kSlots) * 4, 16);
    L.oCtl = take(16, 16);
    L.oBar = take(16, 16);
    L.oTok = take((ntok + kSlots + 1) * 2, 16);   // the pool's token table, then its landmark starts
    L.total = o + 1024;                  // slack to align the dynamic base to 1024
    return L;
}

struct Params {
    Shape s;
    Layout L;
    const unsigned char* Qg;  // inputs, for the L2 prefetch of the next head
    const unsigned char* Kg;
    const unsigned char* Vg;
    int32_t* idx;
    int32_t* route;
    __nv_bfloat16* Ql_keep;   // nullptr unless landmarks are kept
    __nv_bfloat16* Vl_keep;
    int32_t* status;
    float scale_log2;         // log2(e) / sqrt(d)
    int shared;               // 1: the m shared slots join the softmax; 0: routing only
    float rcnt[kSlots];       // 1 / (tokens in the bin of landmark i)
    float cnt[kSlots];        // tokens in the bin of landmark i
    uint32_t wpair[kSlots];   // 128 win in both 16-bit halves: the exact-sum exponent span test
    long long offset_cycles;  // start offset of the second CTA of each SM (0: none)
    int ntok;                 // entries of the token table
    int ptasks;               // pool tasks: four landmarks each, the largest bins first
    uint8_t ptask[kWarps][4]; // landmarks of pool task t (0xff: none)
    uint16_t tstart[kSlots + 1];   // landmark i pools tokens toff[tstart[i] .. tstart[i + 1])
    uint16_t toff[kTokMax];        // byte offset of a token's row in the swizzled Q tile, r*128 + (r%8)*16
};

// ---------------------------------------------------------------- PTX helpers
MITA_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// byte offset of 16-byte chunk `c` of row `r` in a 128-byte-swizzled tile
MITA_DEV uint32_t swz(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

MITA_DEV void ldsm_x4(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a));
}
MITA_DEV void ldsm_x4_t(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a));
}
MITA_DEV void stsm_x4(uint32_t a, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};\n"
                 ::"r"(a), "r"(r0), "r"(r1), "r"(r2), "r"(r3) : "memory");
}
MITA_DEV void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                       uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
MITA_DEV uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
MITA_DEV float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
MITA_DEV float bf_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

MITA_DEV float ex2(float x) {   // hardware 2^x (PTX ex2.approx), -inf -> 0
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
MITA_DEV float rcp(float x) {   // hardware reciprocal (PTX rcp.approx)
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
MITA_DEV float max3(float a, float b, float c) {
    float y;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
    return y;
}
MITA_DEV float min3(float a, float b, float c) {
    float y;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
    return y;
}

MITA_DEV void mbar_init(uint32_t bar, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count));
}
MITA_DEV void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
MITA_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
// As mbar_try_wait, but the thread may sleep up to `ns` nanoseconds for the phase.
MITA_DEV bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(bar), "r"(parity), "r"(ns) : "memory");
    return ok != 0;
}
MITA_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];\n" ::"r"(dst), "l"(map), "r"(x), "r"(y), "r"(bar) : "memory");
}
MITA_DEV void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];\n" ::"l"(map),
                 "r"(x), "r"(y), "r"(src) : "memory");
}
MITA_DEV void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}
MITA_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
MITA_DEV void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
MITA_DEV void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }
MITA_DEV void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// ---------------------------------------------------------------- pooled mean
// bf16 nearest (ties to even) to (hi + lo) / c for the exact bin sum hi + lo
// and a positive integer count c (rc ~ 1/c).  The fp32 quotient picks a
// candidate b; the exact position of the sum against c times the midpoints
// next to b (c * midpoint is exact, the fused multiply-add keeps the sign)
// decides between b and its neighbours.
MITA_DEV __nv_bfloat16 round_mean(float hi, float lo, float c, float rc) {
    const bool neg = hi < 0.0f;
    if (neg) { hi = -hi; lo = -lo; }
    uint16_t b = __bfloat16_as_ushort(__float2bfloat16_rn((hi + lo) * rc));
    const float v0 = __bfloat162float(__ushort_as_bfloat16(b));
    const float v1 = __bfloat162float(__ushort_as_bfloat16((uint16_t)(b + 1)));
    const float e_up = fmaf(-c, 0.5f * (v0 + v1), hi) + lo;
    if (e_up > 0.0f || (e_up == 0.0f && (b & 1))) {
        b = (uint16_t)(b + 1);
    } else if (b > 0) {
        const float vm = __bfloat162float(__ushort_as_bfloat16((uint16_t)(b - 1)));
        const float e_dn = fmaf(-c, 0.5f * (vm + v0), hi) + lo;
        if (e_dn < 0.0f || (e_dn == 0.0f && (b & 1))) b = (uint16_t)(b - 1);
    }
    const __nv_bfloat16 r = __ushort_as_bfloat16(b);
    return neg ? __hneg(r) : r;
}

MITA_DEV uint32_t umax16x2(uint32_t a, uint32_t b) {
    uint32_t y;
    asm("max.u16x2 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
    return y;
}
MITA_DEV uint32_t umin16x2(uint32_t a, uint32_t b) {
    uint32_t y;
    asm("min.u16x2 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
    return y;
}

// ---------------------------------------------------------------- the select
// Expert of one landmark (step 3) and its softmax numerators (for step 4), by
// the 8-lane group that owns the landmark's score row `srow`.  Lane g holds
// the raw scores of keys [g NV, g NV + NV) (NaN past key N).  A 64-bin
// histogram of equal-width bins over [row min, row max] (the bin is a
// monotone function of the score) finds the bin b* holding the k-th best
// score; the members of b* are ranked exactly (score descending, key
// ascending) and the need-th of them is the threshold (T, J).  The expert is
// every key with (score, key) at or above (T, J) in that order, written in
// ascending key order to `irow` and `grow`.  The histogram, the members of
// b* and (T, J) live in the row itself once its scores are in registers; the
// bf16 numerators exp(s/sqrt d - max) (0 past key N) overwrite its start.
template <int NV4>
MITA_DEV void select_landmark(float* srow, int nvp, int N, int k, float cs, uint8_t* irow, int32_t* grow) {
    constexpr int NV = 4 * NV4;
    const int lane = threadIdx.x & 31, gl = lane & 7;
    const unsigned gmask = 0xffu << (lane & 24);
    const int jbase = gl * NV;
    float v[NV];
#pragma unroll
    for (int u = 0; u < NV4; ++u) {
        const float4 x = *(const float4*)(srow + gl * nvp + 4 * u);
        v[4 * u] = x.x;
        v[4 * u + 1] = x.y;
        v[4 * u + 2] = x.z;
        v[4 * u + 3] = x.w;
    }
    // row max and min (max and min ignore the NaN padding)
    float mx = v[0], mn = v[0];
#pragma unroll
    for (int e = 1; e < NV; e += 2) {
        const float b = e + 1 < NV ? v[e + 1] : v[e];
        mx = max3(mx, v[e], b);
        mn = min3(mn, v[e], b);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(gmask, mx, o));
        mn = fminf(mn, __shfl_xor_sync(gmask, mn, o));
    }
    float sc = mx > mn ? (float)kBins / (mx - mn) : 0.0f;
    float off = -mn * sc;
    if (!(fabsf(off) <= 3.0e38f)) sc = off = 0.0f;   // overflow: one bin, ranked exactly below
    // bins: the unsigned conversion takes negatives and NaN to 0
    int bin[NV];
#pragma unroll
    for (int e = 0; e < NV; ++e) bin[e] = (int)min((unsigned)(kBins - 1), __float2uint_rz(fmaf(v[e], sc, off)));
    int* hist = (int*)srow + kRowHist;
    __syncwarp(gmask);   // every lane has loaded its scores: the row is scratch now
    ((int4*)hist)[2 * gl] = make_int4(0, 0, 0, 0);
    ((int4*)hist)[2 * gl + 1] = make_int4(0, 0, 0, 0);
    __syncwarp(gmask);
#pragma unroll
    for (int e = 0; e < NV; ++e) atomicAdd(&hist[bin[e]], 1);
    __syncwarp(gmask);
    // lane g holds bins [8g, 8g + 8); the padding past key N fell into bin 0
    const int4 h0 = ((const int4*)hist)[2 * gl], h1 = ((const int4*)hist)[2 * gl + 1];
    int c[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    if (gl == 0) c[0] -= 8 * NV - N;
    int tot = 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) tot += c[b];
    int suf = tot;   // members of this lane's bins and of every higher lane's
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
        const int y = __shfl_down_sync(gmask, suf, o, 8);
        if (gl + o < 8) suf += y;
    }
    const int above = suf - tot;
    const bool mine = above < k && suf >= k;   // exactly one lane: the suffix counts fall from N
    int bstar = 0, need = 0, cstar = 0;
    if (mine) {
        int run = above;
#pragma unroll
        for (int b = 7; b >= 0; --b) {
            if (run < k && run + c[b] >= k) {
                bstar = 8 * gl + b;
                need = k - run;
                cstar = c[b];
            }
            run += c[b];
        }
    }
    const int src = __ffs(__ballot_sync(gmask, mine)) - 1;
    bstar = __shfl_sync(gmask, bstar, src);
    need = __shfl_sync(gmask, need, src);
    cstar = __shfl_sync(gmask, cstar, src);
    // (T, J): the need-th best member of bin b*
    float T;
    int J;
    float* tj = srow + kRowTJ;
    if (cstar <= kCandG) {
        float2* cand = (float2*)(srow + kRowCand);
        int* ccnt = (int*)srow + kRowCnt;
        if (gl == 0) *ccnt = 0;
        __syncwarp(gmask);
#pragma unroll
        for (int e = 0; e < NV; ++e)
            if (bin[e] == bstar && jbase + e < N) cand[atomicAdd(ccnt, 1)] = make_float2(v[e], __int_as_float(jbase + e));
        __syncwarp(gmask);
        for (int ci = gl; ci < cstar; ci += 8) {
            const float2 me = cand[ci];
            const int jm = __float_as_int(me.y);
            int rank = 0;
            for (int e = 0; e < cstar; ++e) {
                const float2 o = cand[e];
                rank += (o.x > me.x || (o.x == me.x && __float_as_int(o.y) < jm)) ? 1 : 0;
            }
            if (rank == need - 1) {
                tj[0] = me.x;
                tj[1] = me.y;
            }
        }
        __syncwarp(gmask);
        T = tj[0];
        J = __float_as_int(tj[1]);
    } else {
        // many members (flat or tied rows): the need-th best member's order key
        // by bisection, then the key of the last one taken among its equals
        uint32_t key[NV];
#pragma unroll
        for (int e = 0; e < NV; ++e) key[e] = (bin[e] == bstar && jbase + e < N) ? order_key(v[e]) : 0u;
        uint32_t TK = 0u;
        for (int bb = 31; bb >= 0; --bb) {
            const uint32_t ct = TK | (1u << bb);
            int n = 0;
#pragma unroll
            for (int e = 0; e < NV; ++e) n += key[e] >= ct ? 1 : 0;
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) n += __shfl_xor_sync(gmask, n, o);
            if (n >= need) TK = ct;
        }
        int gt = 0, eq = 0;
#pragma unroll
        for (int e = 0; e < NV; ++e) {
            gt += key[e] > TK ? 1 : 0;
            eq += key[e] == TK ? 1 : 0;
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) gt += __shfl_xor_sync(gmask, gt, o);
        const int eq_left = need - gt;   // >= 1 members equal to TK are taken, the lowest keys first
        int x = eq;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            const int y = __shfl_up_sync(gmask, x, o, 8);
            if (gl >= o) x += y;
        }
        const int before = x - eq;
        int jl = 0;
        const bool has = before < eq_left && x >= eq_left;
        if (has) {
            int r = eq_left - before;
#pragma unroll
            for (int e = 0; e < NV; ++e)
                if (key[e] == TK && r > 0 && --r == 0) jl = jbase + e;
        }
        J = __shfl_sync(gmask, jl, __ffs(__ballot_sync(gmask, has)) - 1);
        T = key_to_float(TK);
    }
    // the expert: every key at or above (T, J), in ascending key order; keys
    // tied with T past J are dropped only when the row has such ties
    uint32_t sel = 0u;
#pragma unroll
    for (int e = 0; e < NV; ++e)
        if (v[e] >= T) sel |= 1u << e;
    int ns = __popc(sel);
    int pos = ns;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
        const int y = __shfl_up_sync(gmask, pos, o, 8);
        if (gl >= o) pos += y;
    }
    if (__shfl_sync(gmask, pos, (lane & 24) | 7) != k) {   // ties at T past J
        const int Jr = J - jbase;
        sel = 0u;
#pragma unroll
        for (int e = 0; e < NV; ++e)
            if (v[e] > T || (v[e] == T && e <= Jr)) sel |= 1u << e;
        ns = __popc(sel);
        pos = ns;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            const int y = __shfl_up_sync(gmask, pos, o, 8);
            if (gl >= o) pos += y;
        }
    }
    pos -= ns;
    while (sel) {
        const int e = __ffs(sel) - 1;
        sel &= sel - 1u;
        irow[pos] = (uint8_t)(jbase + e);
        grow[pos] = jbase + e;
        ++pos;
    }
    // softmax numerators over the row's own start, bf16 as the MMA reads them
    const float mb = mx * cs;
    __syncwarp(gmask);   // every lane has read (T, J) from the row
    uint2* prow = (uint2*)((__nv_bfloat16*)srow + jbase);
#pragma unroll
    for (int u = 0; u < NV4; ++u) {
        float p[4];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) p[c4] = ex2(fmaxf(fmaf(v[4 * u + c4], cs, -mb), -INFINITY));   // NaN -> 0
        prow[u] = make_uint2(pack2(p[0], p[1]), pack2(p[2], p[3]));
    }
}

// ---------------------------------------------------------------- the kernel
template <int NV4>   // the select's score float4s per lane: nv4_of(N)
__global__ void __launch_bounds__(kThreads, 2)
    fused_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                 const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapO,
                 const __grid_constant__ Params P) {
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte aligned base (128-byte swizzle), derived from the shared array by
    // pointer arithmetic so that every access below stays a shared-space access
    unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const Shape& s = P.s;
    const Layout& L = P.L;
    const int N = s.N, m = s.m, k = s.k;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;

    const uint32_t sbase = smem_u32(sm);
    const uint32_t uQ = sbase + L.oQ, uK = sbase + L.oK, uV = sbase + L.oV;
    const uint32_t uQl = sbase + L.oQl, uVl = sbase + L.oVl, uS = sbase + L.oS;
    const uint32_t sstrB = (uint32_t)L.sstr * 4u;
    const unsigned char* Qb = sm + L.oQ;
    float* S_s = (float*)(sm + L.oS);
    uint8_t* idx_s = sm + L.oIdx;
    uint8_t* route_s = sm + L.oRoute;
    uint8_t* perm_s = sm + L.oPerm;
    int* cnt_s = (int*)(sm + L.oCnt);
    int* off_s = (int*)(sm + L.oOff);
    int* tiles_s = (int*)(sm + L.oTiles);
    int* ctl = (int*)(sm + L.oCtl);     // [0] tile count, [1] abort flag
    const uint32_t uBar = sbase + L.oBar;

    // one-time set-up: landmark slots past m stay zero (finite) for the MMAs
    for (int e = tid; e < kSlots * 128 / 4; e += kThreads) {
        ((uint32_t*)(sm + L.oQl))[e] = 0u;
        ((uint32_t*)(sm + L.oVl))[e] = 0u;
    }
    uint16_t* toff_s = (uint16_t*)(sm + L.oTok);
    uint16_t* tstart_s = toff_s + P.ntok;
    for (int e = tid; e < P.ntok; e += kThreads) toff_s[e] = P.toff[e];
    for (int e = tid; e <= m; e += kThreads) tstart_s[e] = P.tstart[e];
    if (tid == 0) {
        mbar_init(uBar, 1);
        ctl[1] = 0;
        ctl[2] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();

    const int BH = s.BH();
    const uint32_t bytes_per_head = 3u * (uint32_t)N * 128u;
    if (tid == 0 && (int)blockIdx.x < BH) {
        mbar_expect_tx(uBar, bytes_per_head);
        tma_load_2d(uQ, &mapQ, 0, blockIdx.x * N, uBar);
        tma_load_2d(uK, &mapK, 0, blockIdx.x * N, uBar);
        tma_load_2d(uV, &mapV, 0, blockIdx.x * N, uBar);
    }

    // The two CTAs of an SM run the same phases on equal heads; started
    // together they stay in step and contend for the same units phase after
    // phase.  The second CTA of each SM (blocks are placed breadth first)
    // starts about a quarter of a head later, so that one CTA's selection and
    // pooling overlap the other's tensor-core phases (measured at DeiT-S:
    // 111.4 -> 109.7 us per forward; offsets of a tenth or a whole head gain
    // nothing).
    if (P.offset_cycles > 0 && (int)blockIdx.x >= (int)gridDim.x / 2) {
        const long long t0 = clock64();
        while (clock64() - t0 < P.offset_cycles) {}
    }
    const float cs = P.scale_log2;
    int it = 0;
    for (int head = blockIdx.x; head < BH; head += gridDim.x, ++it) {
        const uint32_t parity = it & 1;
        if (tid == 0) {
            // bounded wait for this head's tiles (about one second)
            const long long t0 = clock64();
            bool ok = false;
            while (!(ok = mbar_try_wait_sleep(uBar, parity, 20000u))) {
                if (clock64() - t0 > 2000000000LL) break;
            }
            if (!ok) {
                atomicExch(P.status, (int)MITA_ERR_TIMEOUT);
                ctl[1] = 1;
            }
        }
        __syncthreads();
        if (ctl[1]) break;
        while (!mbar_try_wait(uBar, parity)) {}   // completes at once: acquire for every thread

        if (tid == 0 && head + (int)gridDim.x < BH) {
            // the next head's tiles into L2 now, so that their TMA load at the end of
            // this head is short
            const size_t off = (size_t)(head + gridDim.x) * N * 128;
            prefetch_l2(P.Qg + off, (uint32_t)N * 128u);
            prefetch_l2(P.Kg + off, (uint32_t)N * 128u);
            prefetch_l2(P.Vg + off, (uint32_t)N * 128u);
        }

        // ---------------- phase A: landmark queries (8-lane group per landmark)
        // Lane g of a group sums features 8g .. 8g + 7 over the bin's tokens
        // (one 16-byte load of the swizzled row per token) in fp32, and keeps
        // the largest and smallest magnitude of each feature.  A bin of c
        // bf16 values whose exponents span at most win = 16 - ceil(log2 c)
        // binades sums exactly in fp32 (every partial sum is a multiple of the
        // smallest value's last bit and below 2^24 of them), tested on the
        // packed exponent fields of the largest and smallest magnitude.
        // The mean of an exact sum s: q1 = s * (1/c), then one correction step
        // q = q1 + (s - q1 c) (1/c) with both steps fused multiply-adds gives
        // the correctly rounded fp32 quotient s / c (checked exhaustively over
        // every fp32 significand of s for every count c up to 256; s normal),
        // and its bf16 rounding is the bf16 rounding of s / c (24 >= 2 * 8 + 2
        // bits: double rounding is innocuous).  A feature without the exactness
        // certificate is summed again error-free (TwoSum) by its group, each
        // lane taking every eighth token, and decided exactly (mean_to_bf16).
        {
            const int grp = lane >> 3, gl = lane & 7;
            const unsigned gmask = 0xffu << (lane & 24);
            const uint32_t lx = (uint32_t)gl << 4;   // the lane's 16-byte chunk of a row
            for (int task = warp; task < P.ptasks; task += kWarps) {
                const int i = P.ptask[task][grp];
                if (i >= m) continue;
                const int e0 = tstart_s[i], e1 = tstart_s[i + 1];
                float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                uint32_t mhi[4] = {0u, 0u, 0u, 0u};
                uint32_t mlo[4] = {0x7fff7fffu, 0x7fff7fffu, 0x7fff7fffu, 0x7fff7fffu};
#pragma unroll 2
                for (int e = e0; e < e1; ++e) {
                    const uint4 q = *(const uint4*)(Qb + ((uint32_t)toff_s[e] ^ lx));
                    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        sum[2 * h] += __uint_as_float(w[h] << 16);
                        sum[2 * h + 1] += __uint_as_float(w[h] & 0xffff0000u);
                        const uint32_t a = w[h] & 0x7fff7fffu;
                        mhi[h] = umax16x2(mhi[h], a);
                        mlo[h] = umin16x2(mlo[h], a);
                    }
                }
                const float rc = P.rcnt[i], cnt = P.cnt[i];
                const uint32_t wpair = P.wpair[i];
                uint32_t outw[4], bad = 0u;
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    // exponent fields; no carry: both halves stay below 2^16
                    const uint32_t lim = (mlo[h] & 0x7f807f80u) + wpair;
                    const uint32_t over = umax16x2(mhi[h] & 0x7f807f80u, lim) ^ lim;   // nonzero half: span too wide
                    float q[2];
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        const float q1 = sum[2 * h + x] * rc;
                        q[x] = fmaf(fmaf(-q1, cnt, sum[2 * h + x]), rc, q1);
                    }
                    outw[h] = pack2(q[0], q[1]);
                    bad |= ((over & 0xffffu) ? 1u : 0u) << (2 * h);
                    bad |= ((over >> 16) ? 1u : 0u) << (2 * h + 1);
                }
                // uncertified features (rare): the group sums each one again error-free
                unsigned lanes = __ballot_sync(gmask, bad != 0u);
                while (lanes) {
                    const int src = __ffs(lanes) - 1;
                    lanes &= lanes - 1u;
                    uint32_t fb = __shfl_sync(gmask, bad, src);
                    while (fb) {
                        const int f = __ffs(fb) - 1;
                        fb &= fb - 1u;
                        const int feat = 8 * (src & 7) + f;
                        const uint32_t fx = ((uint32_t)(feat >> 3) << 4) | ((uint32_t)(feat & 7) * 2u);
                        float hi = 0.0f, lo = 0.0f;
                        for (int e = e0 + gl; e < e1; e += 8)
                            acc2(hi, lo, __uint_as_float((uint32_t)*(const uint16_t*)(Qb + ((uint32_t)toff_s[e] ^ fx)) << 16));
#pragma unroll
                        for (int o = 1; o < 8; o <<= 1) {
                            const float oh = __shfl_xor_sync(gmask, hi, o), ol = __shfl_xor_sync(gmask, lo, o);
                            float sh, se;
                            two_sum(hi, oh, sh, se);
                            hi = sh;
                            lo += ol + se;
                        }
                        const uint32_t hb = __bfloat16_as_ushort(mean_to_bf16(hi, lo, cnt));
                        const uint32_t sh = (f & 1) ? 16u : 0u, keep = ~(0xffffu << sh), put = hb << sh;
                        const int h = f >> 1;
                        const bool me = lane == src;
                        outw[0] = me && h == 0 ? (outw[0] & keep) | put : outw[0];
                        outw[1] = me && h == 1 ? (outw[1] & keep) | put : outw[1];
                        outw[2] = me && h == 2 ? (outw[2] & keep) | put : outw[2];
                        outw[3] = me && h == 3 ? (outw[3] & keep) | put : outw[3];
                    }
                }
                *(uint4*)(sm + L.oQl + ((uint32_t)(i * 128 + (i & 7) * 16) ^ lx)) =
                    make_uint4(outw[0], outw[1], outw[2], outw[3]);
            }
            __syncthreads();
            if (P.Ql_keep)
                for (int x = tid; x < m * 32; x += kThreads) {
                    const int i = x >> 5, fp = x & 31;
                    *(uint32_t*)(P.Ql_keep + ((size_t)head * m + i) * kD + 2 * fp) =
                        *(const uint32_t*)(sm + L.oQl + swz(i, fp >> 2) + (fp & 3) * 4);
                }
        }
        __syncthreads();

        // ---------------- phase B: [K ; Q] . Q_l^T  -> scores and routes
        {
            // score columns of keys N .. 8 NV - 1 hold NaN (the select's padding)
            constexpr int NV = 4 * NV4;
            for (int i = warp; i < m; i += kWarps)
                for (int j = N + lane; j < 8 * NV; j += 32)
                    S_s[i * L.sstr + (j / NV) * L.nvp + j % NV] = __int_as_float(0x7fc00000);
            uint32_t bq[4][4][2];   // Q_l as B operand: [n8 tile][k16 step][2]
#pragma unroll
            for (int n = 0; n < 4; n += 2)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const int row = 8 * (n + (lane >> 4)) + (lane & 7);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(uQl + swz(row, 2 * kk + ((lane >> 3) & 1)), r0, r1, r2, r3);
                    bq[n][kk][0] = r0;
                    bq[n][kk][1] = r1;
                    bq[n + 1][kk][0] = r2;
                    bq[n + 1][kk][1] = r3;
                }
            const int nT = (N + 15) >> 4;
            for (int task = warp; task < 2 * nT; task += kWarps) {
                const bool isK = task < nT;
                const int r0 = 16 * (isK ? task : task - nT);
                const uint32_t base = isK ? uK : uQ;
                float acc[4][4];
#pragma unroll
                for (int n = 0; n < 4; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;
                const int arow = min(r0 + (lane & 7) + ((lane >> 3) & 1) * 8, N - 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(base + swz(arow, 2 * kk + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
                    for (int n = 0; n < 4; ++n) mma16816(acc[n], a0, a1, a2, a3, bq[n][kk][0], bq[n][kk][1]);
                }
                if (isK) {
#pragma unroll
                    for (int n = 0; n < 4; ++n)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int j = r0 + g + 8 * h;
                            const int i = 8 * n + 2 * t;
                            const int cj = (nvp_of(NV4) == 4 * NV4) ? j : (j / (4 * NV4)) * L.nvp + j % (4 * NV4);
                            if (j < N) {
                                if (i < m) S_s[i * L.sstr + cj] = acc[n][2 * h];
                                if (i + 1 < m) S_s[(i + 1) * L.sstr + cj] = acc[n][2 * h + 1];
                            }
                        }
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float best = -INFINITY;
                        int arg = kSlots;
#pragma unroll
                        for (int n = 0; n < 4; ++n)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int i = 8 * n + 2 * t + e;
                                const float v = acc[n][2 * h + e];
                                if (i < m && v > best) { best = v; arg = i; }
                            }
#pragma unroll
                        for (int o = 1; o <= 2; o <<= 1) {
                            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
                            const int oa = __shfl_xor_sync(0xffffffffu, arg, o);
                            if (ob > best || (ob == best && oa < arg)) { best = ob; arg = oa; }
                        }
                        if (arg >= m) arg = 0;   // no finite score (undefined inputs): keep the bucket valid
                        const int q = r0 + g + 8 * h;
                        if (t == 0 && q < N) {
                            route_s[q] = (uint8_t)arg;
                            P.route[(size_t)head * N + q] = arg;
                        }
                    }
                }
            }
        }
        __syncthreads();

        // ---------------- phase C: experts and numerators (8-lane group per landmark)
        {
            const int ntask = (m + 3) >> 2;
            for (int task = warp; task < ntask; task += kWarps) {
                const int i = 4 * task + (lane >> 3);
                if (i < m)
                    select_landmark<NV4>(S_s + i * L.sstr, L.nvp, N, k, cs, idx_s + i * kSlots,
                                         P.idx + ((size_t)head * m + i) * k);
            }
        }
        if (warp == kWarps - 1) {
            // bucket sort of the queries by route; tiles of up to kTile queries
            for (int b = lane; b <= kSlots; b += 32) cnt_s[b] = 0;
            __syncwarp();
            for (int q = lane; q < N; q += 32) atomicAdd(&cnt_s[route_s[q]], 1);
            __syncwarp();
            const int c = lane < m ? cnt_s[lane] : 0;
            int x = c, nt = (c + kTile - 1) / kTile, y = nt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int a = __shfl_up_sync(0xffffffffu, x, o);
                const int b = __shfl_up_sync(0xffffffffu, y, o);
                if (lane >= o) { x += a; y += b; }
            }
            const int excl = x - c, texcl = y - nt;
            __syncwarp();
            if (lane < m) {
                off_s[lane] = excl;
                cnt_s[lane] = excl;        // cursor
                for (int e = 0; e < nt; ++e) tiles_s[texcl + e] = (lane << 8) | (kTile * e);
            }
            if (lane == 31) {
                ctl[0] = y;
                off_s[m] = N;
            }
            __syncwarp();
            for (int q = lane; q < N; q += 32) {
                const int b = route_s[q];
                perm_s[atomicAdd(&cnt_s[b], 1)] = (uint8_t)q;
            }
        }
        // phase D's m16 tile mt = warp / 4 reads the numerators of landmarks
        // 16 mt .. 16 mt + 15, written by the selects of warps 4 mt .. 4 mt + 3:
        // each half of the warps waits for its own half only
        asm volatile("bar.sync %0, 128;\n" ::"r"(1 + (warp >> 2)) : "memory");

        // ---------------- phase D: landmark values V_l = P . V / (P . 1)
        {
            const int mt = warp >> 2, np = warp & 3;   // 2 x 4 (two n8 tiles each) over the 8 warps
            const uint32_t ones = 0x3F803F80u;         // bf16 pair (1, 1): B operand of the row sums
            float acc[3][4] = {};
            const int prow = min(mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, m - 1);
            const uint32_t pa = uS + (uint32_t)prow * sstrB + (uint32_t)(lane >> 4) * 16u;
            for (int kk = 0; kk < L.nk16; ++kk) {
                uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
                ldsm_x4(pa + kk * 32, a0, a1, a2, a3);
                const int vrow = min(kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, N - 1);
                ldsm_x4_t(uV + swz(vrow, 2 * np + (lane >> 4)), b0, b1, b2, b3);
                mma16816(acc[0], a0, a1, a2, a3, b0, b1);
                mma16816(acc[1], a0, a1, a2, a3, b2, b3);
                mma16816(acc[2], a0, a1, a2, a3, ones, ones);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = mt * 16 + g + 8 * h;
                if (i < m) {
                    const float inv = 1.0f / acc[2][2 * h];
#pragma unroll
                    for (int n = 0; n < 2; ++n) {
                        const uint32_t pk = pack2(acc[n][2 * h] * inv, acc[n][2 * h + 1] * inv);
                        *(uint32_t*)(sm + L.oVl + swz(i, 2 * np + n) + 4 * t) = pk;
                        if (P.Vl_keep)
                            *(uint32_t*)(P.Vl_keep + ((size_t)head * m + i) * kD + 16 * np + 8 * n + 2 * t) = pk;
                    }
                }
            }
        }
        __syncthreads();

        // ---------------- phase E: grouped attention, kTile queries per tile
        const int ntiles = ctl[0];
        for (int tile = warp; tile < ntiles; tile += kWarps) {
            const int b = tiles_s[tile] >> 8, st = tiles_s[tile] & 255;
            const int qbase = off_s[b] + st;
            const int nq = min(kTile, off_s[b + 1] - qbase);
            const uint8_t* E = idx_s + b * kSlots;
            // A operand: the tile's query rows (row r of the tile = query perm[qbase + r])
            const int arow = (lane & 7) + ((lane >> 3) & 1) * 8;
            const int qa_row = perm_s[qbase + min(arow, nq - 1)];
            uint32_t qa[4][4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                ldsm_x4(uQ + swz(qa_row, 2 * kk + (lane >> 4)), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
            // logits: 8 n8 slot tiles (0-3 shared Q_l, 4-7 routed keys) x 16 queries
            float sc[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.0f;
            const int brow = (lane & 7) + (lane >> 4) * 8;   // slot of this lane within an n8 pair
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t rowbase;
                int rsw;
                if (np < 2) {
                    const int slot = 16 * np + brow;
                    rowbase = uQl + (uint32_t)slot * 128u;
                    rsw = slot & 7;
                } else {
                    const int slot = 16 * (np - 2) + brow;
                    const int j = E[slot < k ? slot : 0];
                    rowbase = uK + (uint32_t)j * 128u;
                    rsw = j & 7;
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(rowbase + (uint32_t)(((2 * kk + ((lane >> 3) & 1)) ^ rsw) << 4), b0, b1, b2, b3);
                    mma16816(sc[2 * np], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                    mma16816(sc[2 * np + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
                }
            }
            // mask the padding slots, then one softmax per query row
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const int lim = n < 4 ? (P.shared ? m : 0) : k;
                const int s0 = 8 * (n & 3);
                if (s0 + 8 > lim) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (s0 + 2 * t + (e & 1) >= lim) sc[n][e] = -INFINITY;
                }
            }
            float mx0 = fmaxf(sc[0][0], sc[0][1]), mx1 = fmaxf(sc[0][2], sc[0][3]);
#pragma unroll
            for (int n = 1; n < 8; ++n) {
                mx0 = max3(mx0, sc[n][0], sc[n][1]);
                mx1 = max3(mx1, sc[n][2], sc[n][3]);
            }
#pragma unroll
            for (int o = 1; o <= 2; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            const float mb0 = mx0 * cs, mb1 = mx1 * cs;
            uint32_t pa[4][4];   // P as A operand per k16 slot step
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                pa[n >> 1][(n & 1) * 2 + 0] = pack2(ex2(fmaf(sc[n][0], cs, -mb0)), ex2(fmaf(sc[n][1], cs, -mb0)));
                pa[n >> 1][(n & 1) * 2 + 1] = pack2(ex2(fmaf(sc[n][2], cs, -mb1)), ex2(fmaf(sc[n][3], cs, -mb1)));
            }
            // out = P . [V_l ; V_E] : 8 n8 feature tiles x 16 queries
            float o8[8][4], osum[4] = {0.0f, 0.0f, 0.0f, 0.0f};   // osum: row sums of P (ones column)
#pragma unroll
            for (int n = 0; n < 8; ++n) o8[n][0] = o8[n][1] = o8[n][2] = o8[n][3] = 0.0f;
            const int vslot = (lane & 7) + ((lane >> 3) & 1) * 8;   // slot of this lane within a k16 step
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint32_t rowbase;
                int rsw;
                if (ks < 2) {
                    const int slot = 16 * ks + vslot;
                    rowbase = uVl + (uint32_t)slot * 128u;
                    rsw = slot & 7;
                } else {
                    const int slot = 16 * (ks - 2) + vslot;
                    const int j = E[slot < k ? slot : 0];
                    rowbase = uV + (uint32_t)j * 128u;
                    rsw = j & 7;
                }
                const uint32_t a0 = pa[ks][0], a1 = pa[ks][1], a2 = pa[ks][2], a3 = pa[ks][3];
                mma16816(osum, a0, a1, a2, a3, 0x3F803F80u, 0x3F803F80u);
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(rowbase + (uint32_t)(((2 * np + (lane >> 4)) ^ rsw) << 4), b0, b1, b2, b3);
                    mma16816(o8[2 * np], a0, a1, a2, a3, b0, b1);
                    mma16816(o8[2 * np + 1], a0, a1, a2, a3, b2, b3);
                }
            }
            // normalise; write the rows over the tile's own query rows
            const float inv0 = rcp(osum[0]), inv1 = rcp(osum[2]);
            const int srow_t = (lane & 7) + ((lane >> 3) & 1) * 8;
            const int qs_row = perm_s[qbase + min(srow_t, nq - 1)];
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                const uint32_t r0 = pack2(o8[2 * np][0] * inv0, o8[2 * np][1] * inv0);
                const uint32_t r1 = pack2(o8[2 * np][2] * inv1, o8[2 * np][3] * inv1);
                const uint32_t r2 = pack2(o8[2 * np + 1][0] * inv0, o8[2 * np + 1][1] * inv0);
                const uint32_t r3 = pack2(o8[2 * np + 1][2] * inv1, o8[2 * np + 1][3] * inv1);
                stsm_x4(uQ + swz(qs_row, 2 * np + (lane >> 4)), r0, r1, r2, r3);
            }
        }
        fence_async_smem();   // the output rows are read next by the TMA store
        __syncthreads();
        if (tid == 0) {
            tma_store_2d(&mapO, uQ, 0, head * N);
            bulk_commit();
            const int nxt = head + gridDim.x;
            if (nxt < BH) {
                mbar_expect_tx(uBar, bytes_per_head);
                tma_load_2d(uK, &mapK, 0, nxt * N, uBar);
                tma_load_2d(uV, &mapV, 0, nxt * N, uBar);
                bulk_wait_read0();   // the output tile has left Q's buffer
                tma_load_2d(uQ, &mapQ, 0, nxt * N, uBar);
            }
        }
    }
    if (tid == 0) bulk_wait0();
}

}  // namespace fz

// ---------------------------------------------------------------- host side
static bool make_map(CUtensorMap* map, const void* base, int rows, int box_rows) {
    return tma_map_bf16(map, base, fz::kD, (size_t)rows, fz::kD, box_rows);
}

// Entries of the pool's token table: the tokens of every landmark's bin.
static int pool_tokens(const Shape& s) {
    int n = 0;
    for (int i = 0; i < s.m; ++i) {
        const int r = i / s.pw, c = i % s.pw;
        const int r0 = r * s.gh / s.ph, r1 = ((r + 1) * s.gh + s.ph - 1) / s.ph;
        const int c0 = c * s.gw / s.pw, c1 = ((c + 1) * s.gw + s.pw - 1) / s.pw;
        n += (r1 - r0) * (c1 - c0);
    }
    return n;
}

bool fused_supported(const Shape& s, mita_dtype_t dtype) {
    if (dtype != MITA_BF16 || s.d != fz::kD) return false;
    if (s.N > fz::kMaxN || s.m > fz::kSlots || s.k > fz::kSlots) return false;
    const int ntok = pool_tokens(s);
    return ntok <= fz::kTokMax && fz::make_layout(s.N, s.m, ntok).total <= fz::kMaxSmem;
}

template <int NV4>
static cudaError_t launch_nv(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                             const CUtensorMap& mo, const fz::Params& prm, int device, cudaStream_t st) {
    auto kern = fz::fused_kernel<NV4>;
    cudaError_t e = ensure_smem_attr((const void*)kern, prm.L.total);
    if (e != cudaSuccess) return e;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    const int per_sm = blocks_per_sm((const void*)kern, fz::kThreads, prm.L.total);
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int slots = sms * per_sm;
    const int grid = prm.s.BH() < slots ? prm.s.BH() : slots;
    fz::Params p2 = prm;
    p2.offset_cycles = grid > sms ? 50LL * prm.s.N : 0;   // ~a quarter of a head's time
    kern<<<grid, fz::kThreads, prm.L.total, st>>>(mq, mk, mv, mo, p2);
    return cudaGetLastError();
}

cudaError_t run_fused(mita_plan_s* p, const void* Q, const void* K, const void* V, void* out, int32_t* idx,
                      int32_t* route, int keep_landmarks, cudaStream_t st) {
    const Shape& s = p->s;
    const int rows = s.BH() * s.N;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, Q, rows, s.N) || !make_map(&mk, K, rows, s.N) || !make_map(&mv, V, rows, s.N) ||
        !make_map(&mo, out, rows, s.N))
        return cudaErrorInvalidValue;
    fz::Params prm{};
    prm.s = s;
    prm.L = fz::make_layout(s.N, s.m, pool_tokens(s));
    prm.Qg = (const unsigned char*)Q;
    prm.Kg = (const unsigned char*)K;
    prm.Vg = (const unsigned char*)V;
    prm.idx = idx;
    prm.route = route;
    prm.Ql_keep = keep_landmarks ? (__nv_bfloat16*)p->Ql : nullptr;
    prm.Vl_keep = keep_landmarks ? (__nv_bfloat16*)p->Vl : nullptr;
    prm.status = p->status;
    prm.scale_log2 = kLog2e / sqrtf((float)s.d);
    prm.shared = p->routing_only ? 0 : 1;
    int ntok = 0;
    for (int i = 0; i < s.m; ++i) {
        // adaptive average pooling bins [floor(r*G/P), ceil((r+1)*G/P)) per axis
        const int r = i / s.pw, c = i % s.pw;
        const int r0 = r * s.gh / s.ph, r1 = ((r + 1) * s.gh + s.ph - 1) / s.ph;
        const int c0 = c * s.gw / s.pw, c1 = ((c + 1) * s.gw + s.pw - 1) / s.pw;
        prm.tstart[i] = (uint16_t)ntok;
        for (int y = r0; y < r1; ++y)
            for (int x = c0; x < c1; ++x) {
                const int t = y * s.gw + x;
                if (ntok >= fz::kTokMax) return cudaErrorInvalidValue;
                prm.toff[ntok++] = (uint16_t)(t * 128 + (t & 7) * 16);
            }
        const int n = (r1 - r0) * (c1 - c0);
        prm.cnt[i] = (float)n;
        prm.rcnt[i] = 1.0f / (float)n;
        // a bin of n bf16 values sums exactly in fp32 when their exponents span
        // at most win = 16 - ceil(log2 n) binades
        int lg = 0;
        while ((1 << lg) < n) ++lg;
        const int w = 128 * (16 - lg);
        prm.wpair[i] = w > 0 ? ((uint32_t)w | ((uint32_t)w << 16)) : 0u;
    }
    prm.tstart[s.m] = (uint16_t)ntok;
    prm.ntok = ntok;
    {   // pool tasks: landmarks by bin size, largest first, four per task
        int order[fz::kSlots];
        for (int i = 0; i < s.m; ++i) order[i] = i;
        std::stable_sort(order, order + s.m, [&](int a, int b) { return prm.cnt[a] > prm.cnt[b]; });
        prm.ptasks = (s.m + 3) / 4;
        for (int t = 0; t < fz::kWarps; ++t)
            for (int g = 0; g < 4; ++g) prm.ptask[t][g] = 4 * t + g < s.m ? (uint8_t)order[4 * t + g] : 0xff;
    }
    cudaError_t e;
    switch (fz::nv4_of(s.N)) {
        case 1: e = launch_nv<1>(mq, mk, mv, mo, prm, p->device, st); break;
        case 2: e = launch_nv<2>(mq, mk, mv, mo, prm, p->device, st); break;
        case 3: e = launch_nv<3>(mq, mk, mv, mo, prm, p->device, st); break;
        case 4: e = launch_nv<4>(mq, mk, mv, mo, prm, p->device, st); break;
        case 5: e = launch_nv<5>(mq, mk, mv, mo, prm, p->device, st); break;
        case 6: e = launch_nv<6>(mq, mk, mv, mo, prm, p->device, st); break;
        case 7: e = launch_nv<7>(mq, mk, mv, mo, prm, p->device, st); break;
        default: e = launch_nv<8>(mq, mk, mv, mo, prm, p->device, st); break;
    }
    p->launches += 1;
    return e;
}

}  // namespace mita
