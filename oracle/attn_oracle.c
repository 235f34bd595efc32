/*
 * attn_oracle.c -- plain float64 CPU oracle for exact attention (forward and
 * backward).  TEST INFRASTRUCTURE ONLY: it is called by tests/, by the smoke
 * check in __graft_entry__.py and by the cpu_baseline leg of bench.py.  The
 * CUDA library never links, calls or includes anything from here, and this
 * file includes nothing from the CUDA library.
 *
 * What it computes is the definition of scaled dot-product attention, not the
 * tiled algorithm:
 *
 *   O = softmax(scale * Q K^T  [+ causal mask]) V
 *
 * ("FlashAttention and the Kernel Era", section "The Mathematics", the first
 * displayed equation; "FlashAttention 1, 2, and 3 Explained", section 1 "The
 * Standard Attention Memory Wall", the S / P / O equations).  Each query row
 * materialises its full row of scores, takes the row maximum, exponentiates,
 * sums and normalises (the two-pass softmax stated in section 2 of the same
 * page, "The Mathematics of Online Softmax", first paragraph), then multiplies
 * by V.  Nothing is tiled or fused.
 *
 * Readings of points the pages leave open:
 *   - scale multiplies Q K^T before the mask; the pages' default is 1/sqrt(d).
 *   - causal: key j is visible to query i iff j <= i (Nq == Nk, so top-left
 *     and bottom-right alignment coincide).
 *   - lse_i = ln sum_j exp(scale * q_i . k_j) over visible j (natural log of
 *     the scaled scores); it is the row statistic the backward pass keeps.
 *   - GQA / MQA: query head h reads key/value head h / (Hq / Hkv).
 *   - layout: [B, N, H, d] row-major ("Flash Attention" page, "Code Example",
 *     the flash_attn_func reshape); lse is [B, Hq, N].
 *
 * Backward.  The pages give no gradient formulas (they only say that S and P
 * are recomputed rather than stored: "FlashAttention Kernel", the
 * recomputation bullets; "FlashAttention", the recomputation paragraph).  The
 * oracle uses the derivative of the definition above for the loss
 * L = sum(O * dO):
 *   dV = P^T dO
 *   dP = dO V^T
 *   D_i = sum_j P_ij dP_ij                       (softmax Jacobian term)
 *   dS = P o (dP - D)                             (elementwise)
 *   dQ = scale * dS K,   dK = scale * dS^T Q
 * and, for GQA, dK/dV of a key/value head are summed over its query heads.
 * P in the key-major pass is exp(S_ij - lse_i), which is the same softmax
 * entry written through the row's normaliser.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define IDX4(b, n, h, c, N, H, D) ((((size_t)(b) * (N) + (n)) * (H) + (h)) * (D) + (c))

static int check_args(int B, int Hq, int Hkv, int N, int d) {
    if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || d < 1) return 1;
    if (Hq % Hkv != 0) return 1;
    return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static double dot(const double* a, const double* b, int d) {
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += a[c] * b[c];
    return s;
}

/* Softmax row i of head (b, h): p[j] for j < nvis (nvis = i + 1 under the
 * causal mask, N otherwise).  Returns lse_i.  Two passes: max, then
 * exp-and-sum; then normalise. */
static double softmax_row(const double* q, const double* k, int b, int h, int hk, int i,
                          int nvis, int N, int Hq, int Hkv, int d, double scale, double* p) {
    const double* qi = q + IDX4(b, i, h, 0, N, Hq, d);
    double m = -INFINITY;
    for (int j = 0; j < nvis; ++j) {
        p[j] = scale * dot(qi, k + IDX4(b, j, hk, 0, N, Hkv, d), d);
        if (p[j] > m) m = p[j];
    }
    double l = 0.0;
    for (int j = 0; j < nvis; ++j) {
        p[j] = exp(p[j] - m);
        l += p[j];
    }
    for (int j = 0; j < nvis; ++j) p[j] /= l;
    return m + log(l);
}

/* Forward for one query row: o_row (d values), returns lse. */
static double fwd_row(const double* q, const double* k, const double* v, int b, int h, int i,
                      int N, int Hq, int Hkv, int d, int causal, double scale, double* p,
                      double* o_row) {
    int g = Hq / Hkv, hk = h / g;
    int nvis = causal ? i + 1 : N;
    double lse = softmax_row(q, k, b, h, hk, i, nvis, N, Hq, Hkv, d, scale, p);
    for (int c = 0; c < d; ++c) o_row[c] = 0.0;
    for (int j = 0; j < nvis; ++j) {
        const double* vj = v + IDX4(b, j, hk, 0, N, Hkv, d);
        for (int c = 0; c < d; ++c) o_row[c] += p[j] * vj[c];
    }
    return lse;
}

/* Full forward.  q: [B,N,Hq,d]; k, v: [B,N,Hkv,d]; o: [B,N,Hq,d]; lse: [B,Hq,N]. */
int oracle_attn_fwd(const double* q, const double* k, const double* v, double* o, double* lse,
                    int B, int Hq, int Hkv, int N, int d, int causal, double scale) {
    if (check_args(B, Hq, Hkv, N, d)) return 1;
    long long total = (long long)B * Hq * N;
    int fail = 0;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)N);
        if (!p) {
#pragma omp atomic write
            fail = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (long long t = 0; t < total; ++t) {
            if (!p) continue;
            int i = (int)(t % N);
            int h = (int)((t / N) % Hq);
            int b = (int)(t / ((long long)N * Hq));
            lse[((size_t)b * Hq + h) * N + i] =
                fwd_row(q, k, v, b, h, i, N, Hq, Hkv, d, causal, scale, p,
                        o + IDX4(b, i, h, 0, N, Hq, d));
        }
        free(p);
    }
    return fail ? 2 : 0;
}

/* Forward at selected query rows only.  rows: nrows triples (b, h, i).
 * o_rows: [nrows, d]; lse_rows: [nrows].  Each row needs only its own scores,
 * so this equals the full forward at those rows. */
int oracle_attn_fwd_rows(const double* q, const double* k, const double* v, const long long* rows,
                         int nrows, double* o_rows, double* lse_rows, int B, int Hq, int Hkv,
                         int N, int d, int causal, double scale) {
    if (check_args(B, Hq, Hkv, N, d) || nrows < 0) return 1;
    for (int r = 0; r < nrows; ++r) {
        long long b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= N) return 1;
    }
    int fail = 0;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)N);
        if (!p) {
#pragma omp atomic write
            fail = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < nrows; ++r) {
            if (!p) continue;
            lse_rows[r] = fwd_row(q, k, v, (int)rows[3 * r], (int)rows[3 * r + 1],
                                  (int)rows[3 * r + 2], N, Hq, Hkv, d, causal, scale, p,
                                  o_rows + (size_t)r * d);
        }
        free(p);
    }
    return fail ? 2 : 0;
}

/* Forward with separate query and key/value lengths (the split-KV decode
 * entry): q, o [B, Nq, Hq, d]; k, v [B, Nk, Hkv, d]; lse [B, Hq, Nq].  The
 * queries are the last Nq positions of a sequence of Nk, so under the causal
 * mask query i sees keys j <= i + (Nk - Nq) (Nq == Nk gives j <= i, as in
 * oracle_attn_fwd); the causal case needs Nq <= Nk.  Same two-pass softmax of
 * the definition per row. */
int oracle_attn_fwd_kv(const double* q, const double* k, const double* v, double* o,
                       double* lse, int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                       double scale) {
    if (check_args(B, Hq, Hkv, Nq, d) || Nk < 1 || (causal && Nq > Nk)) return 1;
    const int g = Hq / Hkv;
    const long long total = (long long)B * Hq * Nq;
    int fail = 0;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)Nk);
        if (!p) {
#pragma omp atomic write
            fail = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (long long t = 0; t < total; ++t) {
            if (!p) continue;
            const int i = (int)(t % Nq);
            const int h = (int)((t / Nq) % Hq);
            const int b = (int)(t / ((long long)Nq * Hq));
            const int hk = h / g;
            const int nvis = causal ? i + (Nk - Nq) + 1 : Nk;
            const double* qi = q + IDX4(b, i, h, 0, Nq, Hq, d);
            double m = -INFINITY;
            for (int j = 0; j < nvis; ++j) {
                p[j] = scale * dot(qi, k + IDX4(b, j, hk, 0, Nk, Hkv, d), d);
                if (p[j] > m) m = p[j];
            }
            double l = 0.0;
            for (int j = 0; j < nvis; ++j) {
                p[j] = exp(p[j] - m);
                l += p[j];
            }
            double* oi = o + IDX4(b, i, h, 0, Nq, Hq, d);
            for (int c = 0; c < d; ++c) oi[c] = 0.0;
            for (int j = 0; j < nvis; ++j) {
                const double w = p[j] / l;
                const double* vj = v + IDX4(b, j, hk, 0, Nk, Hkv, d);
                for (int c = 0; c < d; ++c) oi[c] += w * vj[c];
            }
            lse[((size_t)b * Hq + h) * Nq + i] = m + log(l);
        }
        free(p);
    }
    return fail ? 2 : 0;
}

/* Forward under a block mask (block-sparse attention): query i of head h may
 * see key j only when mask[h][i / bs][j / bs] != 0 (bs x bs blocks,
 * nb = ceil(N / bs) blocks per side, mask [Hq, nb, nb]), and under the
 * causal mask also only when j <= i.  A row with no visible key has O = 0
 * and lse = -inf (the value that adds nothing when partial results are
 * merged).  Otherwise the same two-pass softmax of the definition. */
int oracle_attn_fwd_blockmask(const double* q, const double* k, const double* v, double* o,
                              double* lse, const unsigned char* mask, int bs, int B, int Hq,
                              int Hkv, int N, int d, int causal, double scale) {
    if (check_args(B, Hq, Hkv, N, d) || bs < 1) return 1;
    const int g = Hq / Hkv;
    const int nb = (N + bs - 1) / bs;
    const long long total = (long long)B * Hq * N;
    int fail = 0;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)N);
        unsigned char* vis = (unsigned char*)malloc((size_t)N);
        if (!p || !vis) {
#pragma omp atomic write
            fail = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (long long t = 0; t < total; ++t) {
            if (!p || !vis) continue;
            const int i = (int)(t % N);
            const int h = (int)((t / N) % Hq);
            const int b = (int)(t / ((long long)N * Hq));
            const int hk = h / g;
            const unsigned char* mrow = mask + ((size_t)h * nb + i / bs) * nb;
            const double* qi = q + IDX4(b, i, h, 0, N, Hq, d);
            double m = -INFINITY;
            int any = 0;
            for (int j = 0; j < N; ++j) {
                vis[j] = (unsigned char)(mrow[j / bs] != 0 && (!causal || j <= i));
                if (!vis[j]) continue;
                any = 1;
                p[j] = scale * dot(qi, k + IDX4(b, j, hk, 0, N, Hkv, d), d);
                if (p[j] > m) m = p[j];
            }
            double* oi = o + IDX4(b, i, h, 0, N, Hq, d);
            for (int c = 0; c < d; ++c) oi[c] = 0.0;
            if (!any) {
                lse[((size_t)b * Hq + h) * N + i] = -INFINITY;
                continue;
            }
            double l = 0.0;
            for (int j = 0; j < N; ++j)
                if (vis[j]) {
                    p[j] = exp(p[j] - m);
                    l += p[j];
                }
            for (int j = 0; j < N; ++j) {
                if (!vis[j]) continue;
                const double w = p[j] / l;
                const double* vj = v + IDX4(b, j, hk, 0, N, Hkv, d);
                for (int c = 0; c < d; ++c) oi[c] += w * vj[c];
            }
            lse[((size_t)b * Hq + h) * N + i] = m + log(l);
        }
        free(p);
        free(vis);
    }
    return fail ? 2 : 0;
}

/* Query-major part of the backward for row (b, h, i): fills dq_row (may be
 * NULL) and returns lse_i; *D_out receives D_i = sum_j P_ij dP_ij. */
static double bwd_query_row(const double* q, const double* k, const double* v, const double* dout,
                            int b, int h, int i, int N, int Hq, int Hkv, int d, int causal,
                            double scale, double* p, double* dq_row, double* D_out) {
    int g = Hq / Hkv, hk = h / g;
    int nvis = causal ? i + 1 : N;
    double lse = softmax_row(q, k, b, h, hk, i, nvis, N, Hq, Hkv, d, scale, p);
    const double* doi = dout + IDX4(b, i, h, 0, N, Hq, d);
    /* dP_ij = dO_i . V_j, kept in a second half of the scratch row. */
    double* dp = p + N;
    double D = 0.0;
    for (int j = 0; j < nvis; ++j) {
        dp[j] = dot(doi, v + IDX4(b, j, hk, 0, N, Hkv, d), d);
        D += p[j] * dp[j];
    }
    if (dq_row) {
        for (int c = 0; c < d; ++c) dq_row[c] = 0.0;
        for (int j = 0; j < nvis; ++j) {
            double ds = p[j] * (dp[j] - D);
            const double* kj = k + IDX4(b, j, hk, 0, N, Hkv, d);
            for (int c = 0; c < d; ++c) dq_row[c] += scale * ds * kj[c];
        }
    }
    *D_out = D;
    return lse;
}

/* Key-major part for key row (b, hk, j): sums over the group's query heads
 * and the query rows that see key j.  lse_all, D_all: [B, Hq, N]. */
static void bwd_key_row(const double* q, const double* k, const double* v, const double* dout,
                        const double* lse_all, const double* D_all, int b, int hk, int j, int N,
                        int Hq, int Hkv, int d, int causal, double scale, double* dk_row,
                        double* dv_row) {
    int g = Hq / Hkv;
    const double* kj = k + IDX4(b, j, hk, 0, N, Hkv, d);
    const double* vj = v + IDX4(b, j, hk, 0, N, Hkv, d);
    for (int c = 0; c < d; ++c) dk_row[c] = dv_row[c] = 0.0;
    for (int h = hk * g; h < (hk + 1) * g; ++h) {
        for (int i = causal ? j : 0; i < N; ++i) {
            const double* qi = q + IDX4(b, i, h, 0, N, Hq, d);
            const double* doi = dout + IDX4(b, i, h, 0, N, Hq, d);
            size_t st = ((size_t)b * Hq + h) * N + i;
            double pij = exp(scale * dot(qi, kj, d) - lse_all[st]);
            double dpij = dot(doi, vj, d);
            double ds = pij * (dpij - D_all[st]);
            for (int c = 0; c < d; ++c) {
                dv_row[c] += pij * doi[c];
                dk_row[c] += scale * ds * qi[c];
            }
        }
    }
}

/* Full backward.  dout, dq: [B,N,Hq,d]; dk, dv: [B,N,Hkv,d]. */
int oracle_attn_bwd(const double* q, const double* k, const double* v, const double* dout,
                    double* dq, double* dk, double* dv, int B, int Hq, int Hkv, int N, int d,
                    int causal, double scale) {
    if (check_args(B, Hq, Hkv, N, d)) return 1;
    size_t nst = (size_t)B * Hq * N;
    double* lse_all = (double*)malloc(sizeof(double) * nst);
    double* D_all = (double*)malloc(sizeof(double) * nst);
    if (!lse_all || !D_all) {
        free(lse_all);
        free(D_all);
        return 2;
    }
    int fail = 0;
    long long total_q = (long long)B * Hq * N;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * 2 * (size_t)N);
        if (!p) {
#pragma omp atomic write
            fail = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (long long t = 0; t < total_q; ++t) {
            if (!p) continue;
            int i = (int)(t % N);
            int h = (int)((t / N) % Hq);
            int b = (int)(t / ((long long)N * Hq));
            size_t st = ((size_t)b * Hq + h) * N + i;
            lse_all[st] = bwd_query_row(q, k, v, dout, b, h, i, N, Hq, Hkv, d, causal, scale, p,
                                        dq + IDX4(b, i, h, 0, N, Hq, d), &D_all[st]);
        }
        free(p);
    }
    if (!fail) {
        long long total_k = (long long)B * Hkv * N;
#pragma omp parallel for schedule(dynamic, 16)
        for (long long t = 0; t < total_k; ++t) {
            int j = (int)(t % N);
            int hk = (int)((t / N) % Hkv);
            int b = (int)(t / ((long long)N * Hkv));
            bwd_key_row(q, k, v, dout, lse_all, D_all, b, hk, j, N, Hq, Hkv, d, causal, scale,
                        dk + IDX4(b, j, hk, 0, N, Hkv, d), dv + IDX4(b, j, hk, 0, N, Hkv, d));
        }
    }
    free(lse_all);
    free(D_all);
    return fail ? 2 : 0;
}

/* Backward at selected rows.  qrows: nq triples (b, h, i) -> dq_rows [nq, d].
 * kvrows: nkv triples (b, hk, j) -> dk_rows, dv_rows [nkv, d].  A key row
 * needs the row statistics (lse_i, D_i) of every query row of its group, so
 * those are computed for each (b, group) that a key row names. */
int oracle_attn_bwd_rows(const double* q, const double* k, const double* v, const double* dout,
                         const long long* qrows, int nq, double* dq_rows, const long long* kvrows,
                         int nkv, double* dk_rows, double* dv_rows, int B, int Hq, int Hkv, int N,
                         int d, int causal, double scale) {
    if (check_args(B, Hq, Hkv, N, d) || nq < 0 || nkv < 0) return 1;
    for (int r = 0; r < nq; ++r) {
        long long b = qrows[3 * r], h = qrows[3 * r + 1], i = qrows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= N) return 1;
    }
    for (int r = 0; r < nkv; ++r) {
        long long b = kvrows[3 * r], h = kvrows[3 * r + 1], j = kvrows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= Hkv || j < 0 || j >= N) return 1;
    }
    int g = Hq / Hkv;
    int fail = 0;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * 2 * (size_t)N);
        if (!p) {
#pragma omp atomic write
            fail = 1;
        }
        double Dtmp;
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < nq; ++r) {
            if (!p) continue;
            bwd_query_row(q, k, v, dout, (int)qrows[3 * r], (int)qrows[3 * r + 1],
                          (int)qrows[3 * r + 2], N, Hq, Hkv, d, causal, scale, p,
                          dq_rows + (size_t)r * d, &Dtmp);
        }
        free(p);
    }
    if (fail || nkv == 0) return fail ? 2 : 0;

    /* mark the (b, hk) groups that key rows need */
    char* need = (char*)calloc((size_t)B * Hkv, 1);
    size_t nst = (size_t)B * Hq * N;
    double* lse_all = (double*)malloc(sizeof(double) * nst);
    double* D_all = (double*)malloc(sizeof(double) * nst);
    if (!need || !lse_all || !D_all) {
        free(need);
        free(lse_all);
        free(D_all);
        return 2;
    }
    for (int r = 0; r < nkv; ++r) need[kvrows[3 * r] * Hkv + kvrows[3 * r + 1]] = 1;
    long long total_q = (long long)B * Hq * N;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * 2 * (size_t)N);
        if (!p) {
#pragma omp atomic write
            fail = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (long long t = 0; t < total_q; ++t) {
            if (!p) continue;
            int i = (int)(t % N);
            int h = (int)((t / N) % Hq);
            int b = (int)(t / ((long long)N * Hq));
            if (!need[(size_t)b * Hkv + h / g]) continue;
            size_t st = ((size_t)b * Hq + h) * N + i;
            lse_all[st] = bwd_query_row(q, k, v, dout, b, h, i, N, Hq, Hkv, d, causal, scale, p,
                                        NULL, &D_all[st]);
        }
        free(p);
    }
    if (!fail) {
#pragma omp parallel for schedule(dynamic, 1)
        for (int r = 0; r < nkv; ++r) {
            bwd_key_row(q, k, v, dout, lse_all, D_all, (int)kvrows[3 * r], (int)kvrows[3 * r + 1],
                        (int)kvrows[3 * r + 2], N, Hq, Hkv, d, causal, scale,
                        dk_rows + (size_t)r * d, dv_rows + (size_t)r * d);
        }
    }
    free(need);
    free(lse_all);
    free(D_all);
    return fail ? 2 : 0;
}
