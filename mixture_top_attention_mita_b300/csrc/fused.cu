// One-kernel MiTA forward for short sequences (bf16, d = 64, N <= 256,
// m <= 32, k <= 32): the DeiT-T / DeiT-S layer shapes.
//
// The six steps of the operator (36Kr / 新智元 "注意力也是FFN？", section
// "用少量地标查询，同时构造全局概括与细节专家") run per head inside one CTA, from
// shared memory:
//   phase 1  pool        Q_l = correctly rounded bin means of Q
//   phase 2  contraction [K ; Q] . Q_l^T with mma.sync: raw landmark scores
//                        (kept in shared memory) and each query's first
//                        argmax landmark (the route)
//   phase 3  select      per landmark, the k best keys (ties to the lower
//                        index) by a monotone 128-bin histogram + exact
//                        resolution of the boundary bin; softmax numerators
//                        of the landmark row; bucket sort of the queries
//   phase 4  values      V_l = P . V with mma.sync, normalised, bf16
//   phase 5  attention   per (expert, 8 queries) tile: logits against the 32
//                        shared slots (Q_l) and 32 routed slots (the
//                        expert's keys, gathered row by row with ldmatrix),
//                        one softmax over both, output = P . [V_l ; V_E]
// The kernel is persistent (one CTA per SM, heads strided by the grid) and
// loads the next head's Q, K, V with TMA (128-byte swizzle) into the second
// half of a double buffer while it computes the current head, so the HBM
// stream of inputs and outputs never waits for the arithmetic.
#include <cuda.h>

#include "fused.cuh"

namespace mita {
namespace fz {

constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kD = 64;
constexpr int kSlots = 32;      // shared slots (m <= 32) and routed slots (k <= 32)
constexpr int kMaxN = 256;
constexpr int kBins = 128;
constexpr int kCand = 32;       // boundary-bin candidates resolved by rank
constexpr int kMaxSmem = 232448;

struct Layout {
    int N, np16, nk16, sstr, pstrB, qkv;
    int oBuf0, oBuf1, oQl, oVl, oS, oP, oHist, oCand, oIdx, oRoute, oPerm, oCnt, oOff, oCur,
        oTiles, oPsum, oCtl, oBar, total;
};

static int align_to(int x, int a) { return (x + a - 1) / a * a; }

static Layout make_layout(int N) {
    Layout L{};
    L.N = N;
    L.np16 = align_to(N, 16);
    L.nk16 = L.np16 / 16;
    L.sstr = L.np16 + 4;                 // fp32 words per score row (conflict-free stores)
    L.pstrB = 2 * (L.np16 + 8);          // bytes per numerator row (conflict-free ldmatrix)
    L.qkv = align_to(N * 128, 1024);
    int o = 0;
    auto take = [&](int bytes, int al) { o = align_to(o, al); int r = o; o += bytes; return r; };
    L.oBuf0 = take(3 * L.qkv, 1024);
    L.oBuf1 = take(3 * L.qkv, 1024);
    L.oQl = take(kSlots * 128, 1024);
    L.oVl = take(kSlots * 128, 1024);
    L.oS = take(kSlots * L.sstr * 4, 16);
    L.oP = take(kSlots * L.pstrB, 16);
    L.oHist = take(kWarps * kBins * 4, 16);
    L.oCand = take(kWarps * kCand * 8, 16);
    L.oIdx = take(kSlots * kSlots, 16);
    L.oRoute = take(kMaxN, 16);
    L.oPerm = take(kMaxN, 16);
    L.oCnt = take((kSlots + 1) * 4, 16);
    L.oOff = take((kSlots + 1) * 4, 16);
    L.oCur = take(kSlots * 4, 16);
    L.oTiles = take((kMaxN / 8 + kSlots) * 4, 16);
    L.oPsum = take(kSlots * 4, 16);
    L.oCtl = take(16, 16);
    L.oBar = take(16, 16);
    L.total = o + 1024;                  // slack to align the dynamic base to 1024
    return L;
}

struct Params {
    Shape s;
    Layout L;
    __nv_bfloat16* out;
    int32_t* idx;
    int32_t* route;
    __nv_bfloat16* Ql_keep;   // nullptr unless landmarks are kept
    __nv_bfloat16* Vl_keep;
    int32_t* status;
    float scale_log2;         // log2(e) / sqrt(d)
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
MITA_DEV void ldsm_x2_t(uint32_t a, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];\n" : "=r"(r0), "=r"(r1) : "r"(a));
}
MITA_DEV void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                       uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
MITA_DEV uint32_t movm_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}
MITA_DEV uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
MITA_DEV float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
MITA_DEV float bf_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

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
MITA_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];\n" ::"r"(dst), "l"(map), "r"(x), "r"(y), "r"(bar) : "memory");
}

// ---------------------------------------------------------------- the kernel
__global__ void __launch_bounds__(kThreads, 1)
    fused_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                 const __grid_constant__ CUtensorMap mapV, const __grid_constant__ Params P) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const Shape& s = P.s;
    const Layout& L = P.L;
    const int N = s.N, m = s.m, k = s.k;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;

    const uint32_t sbase = smem_u32(sm);
    const uint32_t uBuf[2] = {sbase + L.oBuf0, sbase + L.oBuf1};
    const uint32_t uQl = sbase + L.oQl, uVl = sbase + L.oVl, uP = sbase + L.oP;
    float* S_s = (float*)(sm + L.oS);
    int* hist = (int*)(sm + L.oHist) + warp * kBins;
    float2* cand = (float2*)(sm + L.oCand) + warp * kCand;
    uint8_t* idx_s = sm + L.oIdx;
    uint8_t* route_s = sm + L.oRoute;
    uint8_t* perm_s = sm + L.oPerm;
    int* cnt_s = (int*)(sm + L.oCnt);
    int* off_s = (int*)(sm + L.oOff);
    int* cur_s = (int*)(sm + L.oCur);
    int* tiles_s = (int*)(sm + L.oTiles);
    float* psum_s = (float*)(sm + L.oPsum);
    int* ctl = (int*)(sm + L.oCtl);     // [0] tile count, [1] abort flag
    const uint32_t uBar = sbase + L.oBar;

    // one-time set-up: zero the padding that later phases rely on
    for (int e = tid; e < kSlots * 128 / 4; e += kThreads) {
        ((uint32_t*)(sm + L.oQl))[e] = 0u;
        ((uint32_t*)(sm + L.oVl))[e] = 0u;
    }
    for (int e = tid; e < kSlots * L.pstrB / 4; e += kThreads) ((uint32_t*)(sm + L.oP))[e] = 0u;
    for (int e = tid; e < kWarps * kBins; e += kThreads) ((int*)(sm + L.oHist))[e] = 0;
    if (tid == 0) {
        mbar_init(uBar, 1);
        mbar_init(uBar + 8, 1);
        ctl[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();

    const int BH = s.BH();
    const uint32_t bytes_per_head = 3u * (uint32_t)N * 128u;
    auto issue = [&](int head, int buf) {
        const uint32_t bar = uBar + 8 * buf;
        mbar_expect_tx(bar, bytes_per_head);
        tma_load_2d(uBuf[buf], &mapQ, 0, head * N, bar);
        tma_load_2d(uBuf[buf] + L.qkv, &mapK, 0, head * N, bar);
        tma_load_2d(uBuf[buf] + 2 * L.qkv, &mapV, 0, head * N, bar);
    };
    if (tid == 0 && (int)blockIdx.x < BH) issue(blockIdx.x, 0);

    const float cs = P.scale_log2;
    int it = 0;
    for (int head = blockIdx.x; head < BH; head += gridDim.x, ++it) {
        const int buf = it & 1;
        const uint32_t parity = (it >> 1) & 1;
        if (tid == 0) {
            const int nxt = head + gridDim.x;
            if (nxt < BH) {
                asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                issue(nxt, buf ^ 1);
            }
            // bounded wait for this head's tiles (about one second)
            const long long t0 = clock64();
            bool ok = false;
            while (!(ok = mbar_try_wait(uBar + 8 * buf, parity))) {
                if (clock64() - t0 > 2000000000LL) break;
            }
            if (!ok) {
                atomicExch(P.status, (int)MITA_ERR_TIMEOUT);
                ctl[1] = 1;
            }
        }
        __syncthreads();
        if (ctl[1]) return;
        while (!mbar_try_wait(uBar + 8 * buf, parity)) {}   // completes at once: acquire for every thread
        const uint32_t uQ = uBuf[buf], uK = uBuf[buf] + L.qkv, uV = uBuf[buf] + 2 * L.qkv;
        const unsigned char* Qb = sm + (uQ - sbase);

        // ---------------- phase 1: landmark queries
        for (int task = tid; task < m * 32; task += kThreads) {
            const int i = task >> 5, fp = task & 31;
            const int r = i / s.pw, c = i - r * s.pw;
            int r0, r1, c0, c1;
            pool_bin(r, s.gh, s.ph, r0, r1);
            pool_bin(c, s.gw, s.pw, c0, c1);
            float a0 = 0.0f, a1 = 0.0f;
            for (int y = r0; y < r1; ++y)
                for (int x = c0; x < c1; ++x) {
                    const int tok = y * s.gw + x;
                    const uint32_t v = *(const uint32_t*)(Qb + swz(tok, fp >> 2) + (fp & 3) * 4);
                    a0 += bf_lo(v);
                    a1 += bf_hi(v);
                }
            const float cnt = (float)((r1 - r0) * (c1 - c0));
            __nv_bfloat162 q2;
            q2.x = mean_to_bf16(a0, 0.0f, cnt);
            q2.y = mean_to_bf16(a1, 0.0f, cnt);
            *(__nv_bfloat162*)(sm + L.oQl + swz(i, fp >> 2) + (fp & 3) * 4) = q2;
            if (P.Ql_keep) *(__nv_bfloat162*)(P.Ql_keep + ((size_t)head * m + i) * kD + 2 * fp) = q2;
        }
        __syncthreads();

        // ---------------- phase 2: [K ; Q] . Q_l^T  -> scores and routes
        {
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
                            if (j < N) {
                                if (i < m) S_s[i * L.sstr + j] = acc[n][2 * h];
                                if (i + 1 < m) S_s[(i + 1) * L.sstr + j] = acc[n][2 * h + 1];
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

        // ---------------- phase 3: experts, numerators, buckets
        for (int i = warp; i < m; i += kWarps) {
            const float* srow = S_s + i * L.sstr;
            float v[8];
            float mx = -INFINITY, mn = INFINITY;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = lane + 32 * u;
                v[u] = j < N ? srow[j] : 0.0f;
                if (j < N) { mx = fmaxf(mx, v[u]); mn = fminf(mn, v[u]); }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            }
            // monotone binning: a larger score never lands in a lower bin
            const float range = mx - mn;
            const float sc = range > 0.0f ? (float)kBins / range : 0.0f;
            int bin[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = lane + 32 * u;
                bin[u] = -1;
                if (j < N) {
                    bin[u] = min(kBins - 1, (int)((v[u] - mn) * sc));
                    atomicAdd(&hist[bin[u]], 1);
                }
            }
            __syncwarp();
            int hc[4], tot = 0;
#pragma unroll
            for (int u = 0; u < 4; ++u) { hc[u] = hist[kBins - 1 - 4 * lane - u]; tot += hc[u]; }
            int incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int above = incl - tot;
            const bool mine = above < k && incl >= k;
            int bstar = 0, need = 0, cstar = 0;
            if (mine) {
                int run = above;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (run + hc[u] >= k && need == 0) {
                        bstar = kBins - 1 - 4 * lane - u;
                        need = k - run;
                        cstar = hc[u];
                    }
                    run += hc[u];
                }
            }
            const int src = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
            bstar = __shfl_sync(0xffffffffu, bstar, src);
            need = __shfl_sync(0xffffffffu, need, src);
            cstar = __shfl_sync(0xffffffffu, cstar, src);
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 4; ++u) hist[4 * lane + u] = 0;   // ready for the next landmark
            // boundary bin: pick the `need` best of its `cstar` members
            uint32_t bsel = 0;   // bit u: member lane + 32u is taken
            if (need < cstar) {
                if (cstar <= kCand) {
                    int base = 0;
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const bool isb = bin[u] == bstar;
                        const unsigned bal = __ballot_sync(0xffffffffu, isb);
                        if (isb) cand[base + __popc(bal & ((1u << lane) - 1u))] =
                                     make_float2(v[u], __int_as_float(lane + 32 * u));
                        base += __popc(bal);
                    }
                    __syncwarp();
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        if (bin[u] != bstar) continue;
                        const int j = lane + 32 * u;
                        int rank = 0;
                        for (int e = 0; e < cstar; ++e) {
                            const float2 ce = cand[e];
                            const int je = __float_as_int(ce.y);
                            rank += (ce.x > v[u] || (ce.x == v[u] && je < j)) ? 1 : 0;
                        }
                        if (rank < need) bsel |= 1u << u;
                    }
                    __syncwarp();
                } else {
                    // many members (degenerate scores): bisect the order key
                    uint32_t key[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) key[u] = order_key(v[u]);
                    uint32_t T = 0;
                    for (int b = 31; b >= 0; --b) {
                        const uint32_t cand_t = T | (1u << b);
                        int c = 0;
#pragma unroll
                        for (int u = 0; u < 8; ++u) c += (bin[u] == bstar && key[u] >= cand_t) ? 1 : 0;
                        c = __reduce_add_sync(0xffffffffu, c);
                        if (c >= need) T = cand_t;
                    }
                    int gt = 0;
#pragma unroll
                    for (int u = 0; u < 8; ++u) gt += (bin[u] == bstar && key[u] > T) ? 1 : 0;
                    gt = __reduce_add_sync(0xffffffffu, gt);
                    int eq_left = need - gt, base = 0;
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const bool isb = bin[u] == bstar;
                        const bool eq = isb && key[u] == T;
                        const unsigned bal = __ballot_sync(0xffffffffu, eq);
                        const int r = base + __popc(bal & ((1u << lane) - 1u));
                        if ((isb && key[u] > T) || (eq && r < eq_left)) bsel |= 1u << u;
                        base += __popc(bal);
                    }
                }
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (bin[u] == bstar) bsel |= 1u << u;
            }
            // write the expert in ascending key order
            int pos = 0;
            uint8_t* irow = idx_s + i * kSlots;
            int32_t* grow = P.idx + ((size_t)head * m + i) * k;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const bool sel = bin[u] > bstar || (bsel >> u & 1u);
                const unsigned bal = __ballot_sync(0xffffffffu, sel);
                if (sel) {
                    const int p = pos + __popc(bal & ((1u << lane) - 1u));
                    irow[p] = (uint8_t)(lane + 32 * u);
                    grow[p] = lane + 32 * u;
                }
                pos += __popc(bal);
            }
            // softmax numerators of the landmark row (bf16, as the MMA reads them)
            __nv_bfloat16* prow = (__nv_bfloat16*)(sm + L.oP + i * L.pstrB);
            float ps = 0.0f;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = lane + 32 * u;
                if (j < N) {
                    const __nv_bfloat16 pb = __float2bfloat16_rn(exp2f((v[u] - mx) * cs));
                    prow[j] = pb;
                    ps += __bfloat162float(pb);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
            if (lane == 0) psum_s[i] = ps;
            __syncwarp();   // histogram and candidate list are reused by the next landmark
        }
        if (warp == kWarps - 1) {
            // bucket sort of the queries by route; tiles of up to 8 queries
            for (int b = lane; b <= kSlots; b += 32) cnt_s[b] = 0;
            __syncwarp();
            for (int q = lane; q < N; q += 32) atomicAdd(&cnt_s[route_s[q]], 1);
            __syncwarp();
            const int c = lane < m ? cnt_s[lane] : 0;
            int x = c, nt = (c + 7) >> 3, y = nt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int a = __shfl_up_sync(0xffffffffu, x, o);
                const int b = __shfl_up_sync(0xffffffffu, y, o);
                if (lane >= o) { x += a; y += b; }
            }
            const int excl = x - c, texcl = y - nt;
            if (lane < m) {
                off_s[lane] = excl;
                cur_s[lane] = excl;
                for (int e = 0; e < nt; ++e) tiles_s[texcl + e] = (lane << 8) | (8 * e);
            }
            if (lane == 31) ctl[0] = y;
            __syncwarp();
            for (int q = lane; q < N; q += 32) {
                const int b = route_s[q];
                perm_s[atomicAdd(&cur_s[b], 1)] = (uint8_t)q;
            }
        }
        __syncthreads();

        // ---------------- phase 4: landmark values V_l = P . V
        {
            const int mt = warp >> 3, n = warp & 7;   // 2 x 8 tiles over the 16 warps
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            const int prow = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            for (int kk = 0; kk < L.nk16; ++kk) {
                uint32_t a0, a1, a2, a3, b0, b1;
                ldsm_x4(uP + prow * L.pstrB + (kk * 16 + (lane >> 4) * 8) * 2, a0, a1, a2, a3);
                const int vrow = min(kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, N - 1);
                ldsm_x2_t(uV + swz(vrow, n), b0, b1);
                mma16816(acc, a0, a1, a2, a3, b0, b1);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = mt * 16 + g + 8 * h;
                if (i < m) {
                    const float inv = 1.0f / psum_s[i];
                    const uint32_t pk = pack2(acc[2 * h] * inv, acc[2 * h + 1] * inv);
                    *(uint32_t*)(sm + L.oVl + swz(i, n) + 4 * t) = pk;
                    if (P.Vl_keep) *(uint32_t*)(P.Vl_keep + ((size_t)head * m + i) * kD + 8 * n + 2 * t) = pk;
                }
            }
        }
        __syncthreads();

        // ---------------- phase 5: grouped attention, 8 queries per tile
        const int ntiles = ctl[0];
        for (int tile = warp; tile < ntiles; tile += kWarps) {
            const int b = tiles_s[tile] >> 8, st = tiles_s[tile] & 255;
            const int nq = min(8, (b + 1 < m ? off_s[b + 1] : N) - off_s[b] - st);
            const int qbase = off_s[b] + st;
            const uint8_t* E = idx_s + b * kSlots;
            // B operand of the logits: the tile's queries (rows of Q)
            uint32_t bq[4][2];
            {
                const int qc = perm_s[qbase + min(lane & 7, nq - 1)];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(uQ + swz(qc, 4 * hh + (lane >> 3)), r0, r1, r2, r3);
                    bq[2 * hh][0] = r0;
                    bq[2 * hh][1] = r1;
                    bq[2 * hh + 1][0] = r2;
                    bq[2 * hh + 1][1] = r3;
                }
            }
            // logits: 4 key tiles (2 shared + 2 routed) x 8 queries
            float sc4[4][4];
            const int lr = (lane & 7) + ((lane >> 3) & 1) * 8;   // A row of this lane
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                sc4[mt][0] = sc4[mt][1] = sc4[mt][2] = sc4[mt][3] = 0.0f;
                uint32_t rowaddr;
                if (mt < 2) rowaddr = uQl + (uint32_t)((mt * 16 + lr) * 128);
                else {
                    const int slot = (mt - 2) * 16 + lr;
                    rowaddr = uK + (uint32_t)(E[slot < k ? slot : 0] * 128);
                }
                const int rsw = mt < 2 ? (mt * 16 + lr) & 7 : E[((mt - 2) * 16 + lr) < k ? (mt - 2) * 16 + lr : 0] & 7;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(rowaddr + (((2 * kk + (lane >> 4)) ^ rsw) << 4), a0, a1, a2, a3);
                    mma16816(sc4[mt], a0, a1, a2, a3, bq[kk][0], bq[kk][1]);
                }
            }
            // one softmax per query column over the m + k valid slots
            float cmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int slot = (mt & 1) * 16 + g + 8 * h;
                    const bool valid = mt < 2 ? slot < m : slot < k;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float x = valid ? sc4[mt][2 * h + e] * cs : -INFINITY;
                        sc4[mt][2 * h + e] = x;
                        cmax[e] = fmaxf(cmax[e], x);
                    }
                }
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) cmax[e] = fmaxf(cmax[e], __shfl_xor_sync(0xffffffffu, cmax[e], o));
            float csum[2] = {0.0f, 0.0f};
            uint32_t pb[4][2];   // P^T as B operand per key k16 step
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float p0 = exp2f(sc4[mt][2 * h] - cmax[0]);
                    const float p1 = exp2f(sc4[mt][2 * h + 1] - cmax[1]);
                    const __nv_bfloat162 pp = __floats2bfloat162_rn(p0, p1);
                    csum[0] += __low2float(pp);
                    csum[1] += __high2float(pp);
                    pb[mt][h] = movm_t(*reinterpret_cast<const uint32_t*>(&pp));
                }
            }
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) csum[e] += __shfl_xor_sync(0xffffffffu, csum[e], o);
            const float inv0 = 1.0f / csum[0], inv1 = 1.0f / csum[1];
            // out^T = [V_l ; V_E]^T . P^T : 4 feature tiles x 8 queries
            const int vr = (lane & 7) + (lane >> 4) * 8;   // key row of this lane within a k16 step
            uint32_t vaddr[4];
            int vsw[4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                if (kk < 2) {
                    vaddr[kk] = uVl + (uint32_t)((kk * 16 + vr) * 128);
                    vsw[kk] = (kk * 16 + vr) & 7;
                } else {
                    const int slot = (kk - 2) * 16 + vr;
                    const int j = E[slot < k ? slot : 0];
                    vaddr[kk] = uV + (uint32_t)(j * 128);
                    vsw[kk] = j & 7;
                }
            }
            const int qg = perm_s[qbase + min(g, nq - 1)];
            __nv_bfloat16* orow = P.out + ((size_t)head * N + qg) * kD;
#pragma unroll
            for (int fm = 0; fm < 4; ++fm) {
                float o4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(vaddr[kk] + (((2 * fm + ((lane >> 3) & 1)) ^ vsw[kk]) << 4), a0, a1, a2, a3);
                    mma16816(o4, a0, a1, a2, a3, pb[kk][0], pb[kk][1]);
                }
                const uint32_t y0 = movm_t(pack2(o4[0] * inv0, o4[1] * inv1));
                const uint32_t y1 = movm_t(pack2(o4[2] * inv0, o4[3] * inv1));
                if (g < nq) {
                    *(uint32_t*)(orow + 16 * fm + 2 * t) = y0;
                    *(uint32_t*)(orow + 16 * fm + 8 + 2 * t) = y1;
                }
            }
        }
        __syncthreads();
    }
}

}  // namespace fz

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    }
    return fn;
}

static bool make_map(CUtensorMap* map, const void* base, int rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)fz::kD, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)fz::kD * 2};
    const cuuint32_t box[2] = {(cuuint32_t)fz::kD, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool fused_supported(const Shape& s, mita_dtype_t dtype) {
    if (dtype != MITA_BF16 || s.d != fz::kD) return false;
    if (s.N > fz::kMaxN || s.m > fz::kSlots || s.k > fz::kSlots) return false;
    return fz::make_layout(s.N).total <= fz::kMaxSmem;
}

cudaError_t run_fused(mita_plan_s* p, const void* Q, const void* K, const void* V, void* out, int32_t* idx,
                      int32_t* route, int keep_landmarks, cudaStream_t st) {
    const Shape& s = p->s;
    const int rows = s.BH() * s.N;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, Q, rows, s.N) || !make_map(&mk, K, rows, s.N) || !make_map(&mv, V, rows, s.N))
        return cudaErrorInvalidValue;
    fz::Params prm{};
    prm.s = s;
    prm.L = fz::make_layout(s.N);
    prm.out = (__nv_bfloat16*)out;
    prm.idx = idx;
    prm.route = route;
    prm.Ql_keep = keep_landmarks ? (__nv_bfloat16*)p->Ql : nullptr;
    prm.Vl_keep = keep_landmarks ? (__nv_bfloat16*)p->Vl : nullptr;
    prm.status = p->status;
    prm.scale_log2 = kLog2e / sqrtf((float)s.d);
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device);
    cudaError_t e = cudaFuncSetAttribute(fz::fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         prm.L.total);
    if (e != cudaSuccess) return e;
    const int grid = s.BH() < sms ? s.BH() : sms;
    fz::fused_kernel<<<grid, fz::kThreads, prm.L.total, st>>>(mq, mk, mv, prm);
    p->launches += 1;
    return cudaGetLastError();
}

}  // namespace mita
