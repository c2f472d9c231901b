/*
 * MiTA forward oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded fp64 restatement of the Mixture-of-Top-k
 * Attention forward operator, written from the method description in
 * "NeurIPS'26：注意力也是FFN？从快权重出发，重新理解高效注意力" (36Kr / 新智元,
 * section "用少量地标查询，同时构造全局概括与细节专家") and its English version
 * "Is Attention Also FFN? ..." (section "Construct global generalization and
 * detail experts at the same time with a small number of landmark queries").
 *
 * Only tests, the smoke check and the CPU-baseline leg of the benchmark may
 * load this code.  The CUDA library never links, includes or calls it, and
 * this file includes nothing from the CUDA library.
 *
 * Every step is the plain definition, one head at a time, no blocking and no
 * fusion.  Accumulation is fp64.  The only rounding is the explicit rounding
 * of the landmark queries, the landmark values and the output to the I/O type
 * (the reading of the text for a bf16 pipeline, see round_io()).
 *
 * Steps (per head; Q, K, V are [N, d] row-major):
 *   1. pool      Q_l[i] = mean of Q over adaptive-average-pooling bin i
 *   2. scores    R[i, j] = Q_l[i] . K[j]            (raw, unscaled)
 *   3. top-k     E_i = k largest R[i, .], ties to the lower key index,
 *                stored in ascending key order
 *   4. values    V_l[i] = sum_j softmax_j(R[i, .] / sqrt(d)) V[j]
 *   5. route     A[q, i] = q . Q_l[i]; r(q) = first argmax_i A[q, i]
 *   6. attend    out_q = softmax over the m shared logits A[q, .]/sqrt(d)
 *                and the k routed logits q . K[j]/sqrt(d), j in E_r(q),
 *                applied to [V_l ; V[E_r(q)]]
 * Routing-only variant (shared = 0; the ablation in the same article, section
 * "长序列建模：训练时间从10.6小时降至2.4小时", that drops the shared expert):
 * step 6 takes one softmax over the k routed logits alone; steps 1-5 are
 * unchanged.
 * Routing to s > 1 experts (the article's routing keeps s as a parameter and
 * uses s = 1): a query is routed to its s best landmarks (A descending, ties
 * to the lower landmark index) and takes one softmax over the m shared logits
 * and the union of those s experts' keys, each key once.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* I/O types: the values the caller's tensors hold and the type the three
 * rounded intermediates/outputs are rounded to. */
enum { ORACLE_IO_F64 = 0, ORACLE_IO_F32 = 1, ORACLE_IO_BF16 = 2 };

/* Round x to the nearest bfloat16 value, ties to even (8 significant bits).
 * Written from the definition: scale x so that it has 8 integer bits, round
 * to the nearest integer with ties to even, scale back.  Results below the
 * bf16 normal range or above its largest finite value do not occur for the
 * inputs this operator is checked on and are not treated specially. */
double oracle_round_bf16(double x) {
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    frexp(x, &e);                       /* |x| = f * 2^e, f in [0.5, 1) */
    double y = ldexp(x, 8 - e);         /* |y| in [128, 256)            */
    double r = nearbyint(y);            /* default mode: nearest, even  */
    return ldexp(r, e - 8);
}

/* Round to the I/O type.  fp32: the C conversion rounds to nearest even. */
static double round_io(double x, int io) {
    if (io == ORACLE_IO_F32) return (double)(float)x;
    if (io == ORACLE_IO_BF16) return oracle_round_bf16(x);
    return x;
}

/* Adaptive average pooling bin of output cell i when G input cells are
 * pooled to P output cells: [floor(i*G/P), ceil((i+1)*G/P)). */
void oracle_bin(int i, int G, int P, int* lo, int* hi) {
    *lo = (i * G) / P;
    *hi = ((i + 1) * G + P - 1) / P;
}

/* Step 1: landmark queries by local average pooling of Q over the gh x gw
 * token grid (token t = row * gw + col) into ph x pw landmarks (landmark
 * i = r * pw + c).  Q_l is rounded to the I/O type. */
void oracle_pool(int gh, int gw, int ph, int pw, int d, int io,
                 const double* Q, double* Ql) {
    for (int r = 0; r < ph; ++r) {
        int r0, r1;
        oracle_bin(r, gh, ph, &r0, &r1);
        for (int c = 0; c < pw; ++c) {
            int c0, c1;
            oracle_bin(c, gw, pw, &c0, &c1);
            double count = (double)((r1 - r0) * (c1 - c0));
            double* dst = Ql + (size_t)(r * pw + c) * d;
            for (int f = 0; f < d; ++f) {
                double s = 0.0;
                for (int y = r0; y < r1; ++y)
                    for (int x = c0; x < c1; ++x)
                        s += Q[(size_t)(y * gw + x) * d + f];
                /* The fp64 sum s is exact while the bin's values, of p
                 * significant bits each (8 for bf16, 24 for fp32), span at
                 * most 53 - p - ceil(log2 count) binades; the checked inputs
                 * stay far inside that.  The exact quotient is then rounded
                 * twice, to fp64 and to the I/O type, and with 53 >= 2p + 2
                 * that gives the rounding of the exact mean itself
                 * (Figueroa, "When is double rounding innocuous?", 1995). */
                double mean = s / count;
                dst[f] = round_io(mean, io);
            }
        }
    }
}

/* Step 2: raw landmark scores R[i, j] = Q_l[i] . K[j]  ([m, N]). */
void oracle_scores(int N, int d, int m, const double* Ql, const double* K, double* R) {
    for (int i = 0; i < m; ++i)
        for (int j = 0; j < N; ++j) {
            double s = 0.0;
            for (int f = 0; f < d; ++f) s += Ql[(size_t)i * d + f] * K[(size_t)j * d + f];
            R[(size_t)i * N + j] = s;
        }
}

/* Order used by the top-k: higher score first, then lower index first.
 * -0.0 and +0.0 compare equal in C, so they tie and the index decides. */
static _Thread_local const double* g_sort_row;   /* one per thread: heads and rows run in parallel */
static int cmp_desc_then_index(const void* a, const void* b) {
    int ia = *(const int32_t*)a, ib = *(const int32_t*)b;
    double sa = g_sort_row[ia], sb = g_sort_row[ib];
    if (sa > sb) return -1;
    if (sa < sb) return 1;
    return (ia > ib) - (ia < ib);
}
static int cmp_int(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/* Step 3: routed expert i = the k key positions with the largest R[i, .],
 * ties to the lower index, stored ascending.  idx is [m, k]. */
void oracle_topk(int N, int m, int k, const double* R, int32_t* idx) {
    int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
    for (int i = 0; i < m; ++i) {
        for (int j = 0; j < N; ++j) order[j] = j;
        g_sort_row = R + (size_t)i * N;
        qsort(order, (size_t)N, sizeof(int32_t), cmp_desc_then_index);
        qsort(order, (size_t)k, sizeof(int32_t), cmp_int);
        memcpy(idx + (size_t)i * k, order, sizeof(int32_t) * (size_t)k);
    }
    free(order);
}

/* Step 4: landmark values by cross-attention of the landmark queries over
 * the whole sequence: V_l[i] = sum_j softmax_j(R[i, .] / sqrt(d)) V[j],
 * rounded to the I/O type.  Together with Q_l as keys, these are the shared
 * expert's key-value pairs. */
void oracle_landmark_values(int N, int d, int m, int io, const double* R, const double* V,
                            double* Vl) {
    double scale = 1.0 / sqrt((double)d);
    double* acc = (double*)malloc(sizeof(double) * (size_t)d);
    for (int i = 0; i < m; ++i) {
        const double* row = R + (size_t)i * N;
        double mx = -INFINITY;
        for (int j = 0; j < N; ++j) if (row[j] * scale > mx) mx = row[j] * scale;
        double den = 0.0;
        for (int f = 0; f < d; ++f) acc[f] = 0.0;
        for (int j = 0; j < N; ++j) {
            double w = exp(row[j] * scale - mx);
            den += w;
            for (int f = 0; f < d; ++f) acc[f] += w * V[(size_t)j * d + f];
        }
        for (int f = 0; f < d; ++f) Vl[(size_t)i * d + f] = round_io(acc[f] / den, io);
    }
    free(acc);
}

/* Step 5 (one query): raw query-landmark scores A[i] = q . Q_l[i] and the
 * route r(q) = the first i with the largest A[i] (s = 1). */
int oracle_route_one(int d, int m, const double* q, const double* Ql, double* A) {
    int best = 0;
    for (int i = 0; i < m; ++i) {
        double s = 0.0;
        for (int f = 0; f < d; ++f) s += q[f] * Ql[(size_t)i * d + f];
        A[i] = s;
        if (s > A[best]) best = i;
    }
    return best;
}

/* Step 6 (one query): one softmax over the concatenation of the m shared
 * logits (q . Q_l[i] / sqrt(d)) and the k routed logits (q . K[j] / sqrt(d),
 * j in E_r), applied to [V_l ; V[E_r]].  With shared = 0 (routing only) the
 * shared entries are left out of the softmax: their weights are zero and the
 * softmax runs over the k routed logits alone.  W (if not NULL) receives the
 * m + k weights in that order; out is rounded to the I/O type. */
void oracle_attend_one(int d, int m, int k, int io, int shared, const double* q, const double* A,
                       const int32_t* E, const double* K, const double* V,
                       const double* Vl, double* out, double* W) {
    double scale = 1.0 / sqrt((double)d);
    int L = m + k;
    double* logit = (double*)malloc(sizeof(double) * (size_t)L);
    for (int i = 0; i < m; ++i) logit[i] = shared ? A[i] * scale : -INFINITY;
    for (int t = 0; t < k; ++t) {
        const double* key = K + (size_t)E[t] * d;
        double s = 0.0;
        for (int f = 0; f < d; ++f) s += q[f] * key[f];
        logit[m + t] = s * scale;
    }
    double mx = -INFINITY;
    for (int l = 0; l < L; ++l) if (logit[l] > mx) mx = logit[l];
    double den = 0.0;
    for (int l = 0; l < L; ++l) { logit[l] = exp(logit[l] - mx); den += logit[l]; }
    for (int f = 0; f < d; ++f) {
        double s = 0.0;
        for (int i = 0; i < m; ++i) s += logit[i] * Vl[(size_t)i * d + f];
        for (int t = 0; t < k; ++t) s += logit[m + t] * V[(size_t)E[t] * d + f];
        out[f] = round_io(s / den, io);
    }
    if (W) for (int l = 0; l < L; ++l) W[l] = logit[l] / den;
    free(logit);
}

/* Step 5 for s > 1 (one query): the s landmarks with the largest A[i], ties
 * to the lower index, best first, in top[0 .. s-1]. */
void oracle_route_top(int m, int s, const double* A, int32_t* top) {
    for (int r = 0; r < s; ++r) {
        int best = -1;
        for (int i = 0; i < m; ++i) {
            int taken = 0;
            for (int u = 0; u < r; ++u) taken |= top[u] == i;
            if (!taken && (best < 0 || A[i] > A[best])) best = i;
        }
        top[r] = best;
    }
}

/* Step 6 for s > 1 (one query): one softmax over the m shared logits (none
 * with shared = 0) and the logits of every key in the union of the experts
 * E_top[0], ..., E_top[s-1], each key once; out is rounded to the I/O type. */
void oracle_attend_multi(int N, int d, int m, int k, int s, int io, int shared, const double* q,
                         const double* A, const int32_t* idx, const int32_t* top, const double* K,
                         const double* V, const double* Vl, double* out) {
    double scale = 1.0 / sqrt((double)d);
    char* in_union = (char*)calloc((size_t)N, 1);
    for (int r = 0; r < s; ++r)
        for (int t = 0; t < k; ++t) in_union[idx[(size_t)top[r] * k + t]] = 1;
    double* w = (double*)malloc(sizeof(double) * (size_t)(m + N));
    double mx = -INFINITY;
    for (int i = 0; i < m; ++i) {
        w[i] = shared ? A[i] * scale : -INFINITY;
        if (w[i] > mx) mx = w[i];
    }
    for (int j = 0; j < N; ++j) {
        w[m + j] = -INFINITY;
        if (!in_union[j]) continue;
        double s2 = 0.0;
        for (int f = 0; f < d; ++f) s2 += q[f] * K[(size_t)j * d + f];
        w[m + j] = s2 * scale;
        if (w[m + j] > mx) mx = w[m + j];
    }
    double den = 0.0;
    for (int l = 0; l < m + N; ++l) { w[l] = exp(w[l] - mx); den += w[l]; }
    for (int f = 0; f < d; ++f) {
        double acc = 0.0;
        for (int i = 0; i < m; ++i) acc += w[i] * Vl[(size_t)i * d + f];
        for (int j = 0; j < N; ++j) if (in_union[j]) acc += w[m + j] * V[(size_t)j * d + f];
        out[f] = round_io(acc / den, io);
    }
    free(w);
    free(in_union);
}

/* The whole operator for one head.  qlist (nq entries, NULL = all N queries
 * in order) selects the queries whose route and output are produced; the
 * landmarks, experts and landmark values always cover the whole head.
 * Optional outputs (NULL to skip): Ql [m,d], Vl [m,d], R [m,N], A [nq,m],
 * W [nq, m+k] (s = 1 only).  s: experts per query (1 <= s <= m); route[]
 * holds each query's best landmark.  Returns 0, or -1 on invalid sizes. */
int oracle_head(int N, int d, int gh, int gw, int ph, int pw, int m, int k, int io, int shared, int s,
                const double* Q, const double* K, const double* V,
                int nq, const int32_t* qlist,
                double* out, int32_t* idx, int32_t* route,
                double* Ql_out, double* Vl_out, double* R_out, double* A_out, double* W_out) {
    if (N < 1 || d < 1 || gh * gw != N || ph * pw != m || ph > gh || pw > gw || k < 1 || k > N)
        return -1;
    if (s < 1 || s > m || (s > 1 && W_out)) return -1;
    int32_t* top = (int32_t*)malloc(sizeof(int32_t) * (size_t)s);
    double* Ql = Ql_out ? Ql_out : (double*)malloc(sizeof(double) * (size_t)m * d);
    double* Vl = Vl_out ? Vl_out : (double*)malloc(sizeof(double) * (size_t)m * d);
    double* R = R_out ? R_out : (double*)malloc(sizeof(double) * (size_t)m * N);
    double* A = (double*)malloc(sizeof(double) * (size_t)m);

    oracle_pool(gh, gw, ph, pw, d, io, Q, Ql);
    oracle_scores(N, d, m, Ql, K, R);
    oracle_topk(N, m, k, R, idx);
    oracle_landmark_values(N, d, m, io, R, V, Vl);
    for (int n = 0; n < nq; ++n) {
        int qi = qlist ? qlist[n] : n;
        const double* q = Q + (size_t)qi * d;
        int r = oracle_route_one(d, m, q, Ql, A);
        route[n] = r;
        if (A_out) memcpy(A_out + (size_t)n * m, A, sizeof(double) * (size_t)m);
        if (s == 1) {
            oracle_attend_one(d, m, k, io, shared, q, A, idx + (size_t)r * k, K, V, Vl,
                              out + (size_t)n * d, W_out ? W_out + (size_t)n * (m + k) : NULL);
        } else {
            oracle_route_top(m, s, A, top);
            oracle_attend_multi(N, d, m, k, s, io, shared, q, A, idx, top, K, V, Vl, out + (size_t)n * d);
        }
    }
    free(top);
    free(A);
    if (!Ql_out) free(Ql);
    if (!Vl_out) free(Vl);
    if (!R_out) free(R);
    return 0;
}

/* Backward of one head (s = 1; `shared` as in step 6), fp64.  The experts
 * and routes are constants of the forward (their selection has no gradient);
 * the roundings of Q_l, V_l and out to the I/O type pass gradients through
 * unchanged.  Given dOut [N, d], writes dQ, dK, dV [N, d].  The chain rule
 * taken step by step, in reverse order:
 *   6  per query: w = softmax(logits); dw_l = dOut . v_l; dlogit = w (dw - w.dw);
 *      value gradients to V_l (shared) and V (routed); logit gradients to the
 *      query, to Q_l (shared keys) and to K (routed keys), all over sqrt(d)
 *   4  V_l = P V with P = softmax(R / sqrt(d)): dP = dV_l V^T, dV += P^T dV_l,
 *      dR = P (dP - rowsum(P dP)) / sqrt(d)
 *   2  R = Q_l K^T: dQ_l += dR K, dK += dR^T Q_l
 *   1  Q_l = bin means of Q: each token of bin i gets dQ_l[i] / |bin i|
 * Returns 0, or -1 on invalid sizes. */
int oracle_backward_head(int N, int d, int gh, int gw, int ph, int pw, int m, int k, int io, int shared,
                         const double* Q, const double* K, const double* V, const double* dOut,
                         double* dQ, double* dK, double* dV) {
    if (N < 1 || d < 1 || gh * gw != N || ph * pw != m || ph > gh || pw > gw || k < 1 || k > N)
        return -1;
    const double scale = 1.0 / sqrt((double)d);
    double* Ql = (double*)malloc(sizeof(double) * (size_t)m * d);
    double* Vl = (double*)malloc(sizeof(double) * (size_t)m * d);
    double* R = (double*)malloc(sizeof(double) * (size_t)m * N);
    double* P = (double*)malloc(sizeof(double) * (size_t)m * N);
    int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)m * k);
    double* dQl = (double*)calloc((size_t)m * d, sizeof(double));
    double* dVl = (double*)calloc((size_t)m * d, sizeof(double));
    double* A = (double*)malloc(sizeof(double) * (size_t)m);
    double* w = (double*)malloc(sizeof(double) * (size_t)(m + k));
    double* dl = (double*)malloc(sizeof(double) * (size_t)(m + k));
    memset(dQ, 0, sizeof(double) * (size_t)N * d);
    memset(dK, 0, sizeof(double) * (size_t)N * d);
    memset(dV, 0, sizeof(double) * (size_t)N * d);

    oracle_pool(gh, gw, ph, pw, d, io, Q, Ql);
    oracle_scores(N, d, m, Ql, K, R);
    oracle_topk(N, m, k, R, idx);
    oracle_landmark_values(N, d, m, io, R, V, Vl);
    for (int i = 0; i < m; ++i) {   /* P = softmax(R / sqrt(d)) per landmark */
        double mx = -INFINITY, den = 0.0;
        for (int j = 0; j < N; ++j) if (R[(size_t)i * N + j] * scale > mx) mx = R[(size_t)i * N + j] * scale;
        for (int j = 0; j < N; ++j) {
            P[(size_t)i * N + j] = exp(R[(size_t)i * N + j] * scale - mx);
            den += P[(size_t)i * N + j];
        }
        for (int j = 0; j < N; ++j) P[(size_t)i * N + j] /= den;
    }
    /* step 6 */
    for (int qi = 0; qi < N; ++qi) {
        const double* q = Q + (size_t)qi * d;
        const double* g = dOut + (size_t)qi * d;
        const int r = oracle_route_one(d, m, q, Ql, A);
        const int32_t* E = idx + (size_t)r * k;
        double mx = -INFINITY;
        for (int i = 0; i < m; ++i) {
            w[i] = shared ? A[i] * scale : -INFINITY;
            if (w[i] > mx) mx = w[i];
        }
        for (int t = 0; t < k; ++t) {
            double s2 = 0.0;
            for (int f = 0; f < d; ++f) s2 += q[f] * K[(size_t)E[t] * d + f];
            w[m + t] = s2 * scale;
            if (w[m + t] > mx) mx = w[m + t];
        }
        double den = 0.0;
        for (int l = 0; l < m + k; ++l) { w[l] = exp(w[l] - mx); den += w[l]; }
        for (int l = 0; l < m + k; ++l) w[l] /= den;
        double wdw = 0.0;
        for (int l = 0; l < m + k; ++l) {
            const double* v = l < m ? Vl + (size_t)l * d : V + (size_t)E[l - m] * d;
            double dw = 0.0;
            for (int f = 0; f < d; ++f) dw += g[f] * v[f];
            dl[l] = dw;
            wdw += w[l] * dw;
        }
        for (int l = 0; l < m + k; ++l) dl[l] = w[l] * (dl[l] - wdw);
        for (int i = 0; i < m; ++i)
            for (int f = 0; f < d; ++f) {
                dVl[(size_t)i * d + f] += w[i] * g[f];
                dQ[(size_t)qi * d + f] += dl[i] * Ql[(size_t)i * d + f] * scale;
                dQl[(size_t)i * d + f] += dl[i] * q[f] * scale;
            }
        for (int t = 0; t < k; ++t) {
            const size_t j = (size_t)E[t];
            for (int f = 0; f < d; ++f) {
                dV[j * d + f] += w[m + t] * g[f];
                dQ[(size_t)qi * d + f] += dl[m + t] * K[j * d + f] * scale;
                dK[j * d + f] += dl[m + t] * q[f] * scale;
            }
        }
    }
    /* step 4, then step 2 */
    for (int i = 0; i < m; ++i) {
        double* dP = (double*)malloc(sizeof(double) * (size_t)N);
        double pdp = 0.0;
        for (int j = 0; j < N; ++j) {
            double s2 = 0.0;
            for (int f = 0; f < d; ++f) s2 += dVl[(size_t)i * d + f] * V[(size_t)j * d + f];
            dP[j] = s2;
            pdp += P[(size_t)i * N + j] * s2;
        }
        for (int j = 0; j < N; ++j) {
            const double pij = P[(size_t)i * N + j];
            const double dR = pij * (dP[j] - pdp) * scale;
            for (int f = 0; f < d; ++f) {
                dV[(size_t)j * d + f] += pij * dVl[(size_t)i * d + f];
                dQl[(size_t)i * d + f] += dR * K[(size_t)j * d + f];
                dK[(size_t)j * d + f] += dR * Ql[(size_t)i * d + f];
            }
        }
        free(dP);
    }
    /* step 1 */
    for (int r = 0; r < ph; ++r) {
        int r0, r1;
        oracle_bin(r, gh, ph, &r0, &r1);
        for (int c = 0; c < pw; ++c) {
            int c0, c1;
            oracle_bin(c, gw, pw, &c0, &c1);
            const double count = (double)((r1 - r0) * (c1 - c0));
            const double* src = dQl + (size_t)(r * pw + c) * d;
            for (int y = r0; y < r1; ++y)
                for (int x = c0; x < c1; ++x)
                    for (int f = 0; f < d; ++f) dQ[(size_t)(y * gw + x) * d + f] += src[f] / count;
        }
    }
    free(Ql); free(Vl); free(R); free(P); free(idx); free(dQl); free(dVl); free(A); free(w); free(dl);
    return 0;
}

/* All heads of a [B*H, N, d] batch, every query. */
int oracle_forward(int BH, int N, int d, int gh, int gw, int ph, int pw, int m, int k, int io, int shared, int s,
                   const double* Q, const double* K, const double* V,
                   double* out, int32_t* idx, int32_t* route) {
    for (int h = 0; h < BH; ++h) {
        size_t o = (size_t)h * N * d;
        int rc = oracle_head(N, d, gh, gw, ph, pw, m, k, io, shared, s, Q + o, K + o, V + o, N, NULL,
                             out + o, idx + (size_t)h * m * k, route + (size_t)h * N,
                             NULL, NULL, NULL, NULL, NULL);
        if (rc) return rc;
    }
    return 0;
}
