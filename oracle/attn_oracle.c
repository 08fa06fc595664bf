/*
 * attn_oracle.c -- plain fp64 CPU oracle for masked scaled dot-product
 * attention, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it exists so that tests/, the smoke check and the CPU
 * baseline leg of the benchmark can compare the CUDA kernels against the
 * definition written out.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * Sources (the pages this restates; no code is taken from them):
 *   [A10]  "Appendix A.10 -- Attention matrices and backpropagation"
 *          (glenzli.com, .../a-10-transformer-math), eqs. A.10.1-A.10.9,
 *          section A.10.5 (batch, heads, GQA) and A.10.6 (causality).
 *   [HAND] "Computing attention term by term" (aihero.club,
 *          .../attention-by-hand), worked examples 1 and 2.
 *   [CH15] "Chapter 15 -- matrix formulas" (math.zhuph.uk, .../part-15),
 *          section 15.1 (max subtraction) and 15.3 (bar-notation backward).
 *   [CH31] "Chapter 31 -- attention backprop" (ai-engineering-handbook,
 *          .../chapters/31.html), sections 1-4 (m != n shapes, whole-row
 *          softmax backward, rejection of fully masked rows).
 *
 * What it computes is exactly the definition, in double precision, with no
 * blocking, no online softmax and no reordering beyond the sums the
 * equations write.  Every function below names the equation it follows.
 *
 * Layout (row-major, innermost last):
 *   Q  [B][Hq ][nq][dh]     K [B][Hkv][nk][dh]     V [B][Hkv][nk][dv]
 *   dO [B][Hq ][nq][dv]     O [B][Hq ][nq][dv]     LSE, D, C [B][Hq][nq]
 *   dQ [B][Hq ][nq][dh]     dK[B][Hkv][nk][dh]     dV[B][Hkv][nk][dv]
 * Indices are 0-based; the pages count from 1, which changes no formula.
 *
 * Compile-time negative controls (used only by the oracle's own tests,
 * following [CH31] section 8, which asks for deliberately broken variants):
 *   ORACLE_MUTATION == 1 : the row term c_i is dropped from dS (A.10.7).
 *   ORACLE_MUTATION == 2 : the visible set is ignored (every key in range
 *                          is treated as visible).
 * A normal build defines neither.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif

/* Problem description shared by every entry point (plain C, no CUDA). */
typedef struct {
    int64_t B, Hq, Hkv, nq, nk, dh, dv;
} oracle_shape;

typedef struct {
    int32_t causal;        /* 0: no causal restriction                       */
    int64_t offset;        /* causal: key j visible to query i iff j<=i+offset */
    const int32_t *kv_len; /* NULL or [B]: key j visible only if j < kv_len[b] */
} oracle_mask;

/* ------------------------------------------------------------------------ */
/* Visible set V_i.  [A10] A.10.1 gives each query row a non-empty set of    */
/* visible keys; A.10.6 takes V_i = {j : j <= i} for causal self-attention   */
/* "minus the padding positions".  For n_q != n_k ([CH31] section 1: a new   */
/* chunk of queries over the whole history) the causal bound is shifted by   */
/* an offset: j <= i + offset.  Padding is key padding: j < kv_len[b].       */
/* ------------------------------------------------------------------------ */
static int key_limit(const oracle_shape *sh, const oracle_mask *mk, int64_t b)
{
    int64_t lim = sh->nk;
    if (mk->kv_len) {
        lim = mk->kv_len[b];
    }
    return (int)lim;
}

static int is_visible(const oracle_shape *sh, const oracle_mask *mk,
                      int64_t b, int64_t i, int64_t j)
{
#if ORACLE_MUTATION == 2
    (void)mk; (void)b; (void)i;
    return j >= 0 && j < sh->nk;
#else
    if (j < 0 || j >= key_limit(sh, mk, b)) {
        return 0;
    }
    if (mk->causal && j > i + mk->offset) {
        return 0;
    }
    return 1;
#endif
}

/* The KV head a query head reads: [A10] A.10.5 leaves the map g(r) open;   */
/* here g(r) = floor(r / (Hq / Hkv)), consecutive query heads sharing one.  */
static int64_t kv_head_of(const oracle_shape *sh, int64_t r)
{
    return r / (sh->Hq / sh->Hkv);
}

static const double *q_row(const oracle_shape *sh, const double *Q, int64_t b, int64_t r, int64_t i)
{
    return Q + ((b * sh->Hq + r) * sh->nq + i) * sh->dh;
}
static const double *k_row(const oracle_shape *sh, const double *K, int64_t b, int64_t h, int64_t j)
{
    return K + ((b * sh->Hkv + h) * sh->nk + j) * sh->dh;
}
static const double *v_row(const oracle_shape *sh, const double *V, int64_t b, int64_t h, int64_t j)
{
    return V + ((b * sh->Hkv + h) * sh->nk + j) * sh->dv;
}
static const double *go_row(const oracle_shape *sh, const double *G, int64_t b, int64_t r, int64_t i)
{
    return G + ((b * sh->Hq + r) * sh->nq + i) * sh->dv;
}

static double dot(const double *x, const double *y, int64_t n)
{
    double acc = 0.0;
    for (int64_t a = 0; a < n; ++a) {
        acc += x[a] * y[a];
    }
    return acc;
}

/* ------------------------------------------------------------------------ */
/* One query row of the forward pass.                                        */
/*   S_ij = scale * q_i . k_j            for j in V_i        (A.10.1)        */
/*   m_i  = max_{j in V_i} S_ij                               (A.10.2)        */
/*   A_ij = exp(S_ij - m_i) / sum_{r in V_i} exp(S_ir - m_i), 0 off V_i       */
/* [CH15] 15.1: subtracting the row maximum leaves the softmax unchanged.    */
/* Outputs the dense rows S (NaN off V_i) and A, plus m_i and l_i.  Returns  */
/* the number of visible keys (0 means the row is undefined: A.10.2).        */
/* ------------------------------------------------------------------------ */
static int64_t softmax_row(const oracle_shape *sh, const oracle_mask *mk,
                           const double *Q, const double *K, double scale,
                           int64_t b, int64_t r, int64_t i,
                           double *S, double *A, double *m_out, double *l_out)
{
    const int64_t h = kv_head_of(sh, r);
    const double *q = q_row(sh, Q, b, r, i);
    int64_t count = 0;
    double m = -INFINITY;
    for (int64_t j = 0; j < sh->nk; ++j) {
        if (is_visible(sh, mk, b, i, j)) {
            S[j] = scale * dot(q, k_row(sh, K, b, h, j), sh->dh);
            if (S[j] > m) {
                m = S[j];
            }
            ++count;
        } else {
            S[j] = NAN;
        }
    }
    double l = 0.0;
    for (int64_t j = 0; j < sh->nk; ++j) {
        if (is_visible(sh, mk, b, i, j)) {
            l += exp(S[j] - m);
        }
    }
    for (int64_t j = 0; j < sh->nk; ++j) {
        A[j] = is_visible(sh, mk, b, i, j) ? exp(S[j] - m) / l : 0.0;
    }
    *m_out = m;
    *l_out = l;
    return count;
}

/* O_i = sum_j A_ij v_j   (A.10.3); LSE_i = m_i + ln l_i, the natural log   */
/* of sum_{j in V_i} exp(S_ij), which is what a backward pass needs to      */
/* rebuild A from S.                                                         */
static void output_row(const oracle_shape *sh, const double *V, const double *A,
                       int64_t b, int64_t r, double *o)
{
    const int64_t h = kv_head_of(sh, r);
    for (int64_t l = 0; l < sh->dv; ++l) {
        o[l] = 0.0;
    }
    for (int64_t j = 0; j < sh->nk; ++j) {
        if (A[j] != 0.0) {
            const double *v = v_row(sh, V, b, h, j);
            for (int64_t l = 0; l < sh->dv; ++l) {
                o[l] += A[j] * v[l];
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* One query row of the backward pass, given its A row.                      */
/*   (G_A)_ij = sum_l G_il V_jl                               (A.10.6)       */
/*   c_i      = sum_{r in V_i} A_ir (G_A)_ir                  (A.10.7)       */
/*   (G_S)_ij = A_ij ((G_A)_ij - c_i) on V_i, 0 elsewhere     (A.10.7)       */
/* [CH31] section 3 writes the same row form: p .* (g - sum_j p_j g_j).      */
/* ------------------------------------------------------------------------ */
static double score_grad_row(const oracle_shape *sh, const oracle_mask *mk,
                             const double *V, const double *G, const double *A,
                             int64_t b, int64_t r, int64_t i, double *dA, double *dS)
{
    const int64_t h = kv_head_of(sh, r);
    const double *g = go_row(sh, G, b, r, i);
    double c = 0.0;
    for (int64_t j = 0; j < sh->nk; ++j) {
        if (is_visible(sh, mk, b, i, j)) {
            dA[j] = dot(g, v_row(sh, V, b, h, j), sh->dv);
            c += A[j] * dA[j];
        } else {
            dA[j] = 0.0;
        }
    }
    for (int64_t j = 0; j < sh->nk; ++j) {
        if (is_visible(sh, mk, b, i, j)) {
#if ORACLE_MUTATION == 1
            dS[j] = A[j] * dA[j];
#else
            dS[j] = A[j] * (dA[j] - c);
#endif
        } else {
            dS[j] = 0.0;
        }
    }
    return c;
}

/* ------------------------------------------------------------------------ */
/* Entry points.                                                             */
/* ------------------------------------------------------------------------ */

/* Number of visible (i, j) pairs over every (b, query head), counted one by */
/* one from the visible-set predicate.                                       */
int64_t oracle_visible_pairs(const oracle_shape *sh, const oracle_mask *mk)
{
    int64_t total = 0;
    for (int64_t b = 0; b < sh->B; ++b) {
        int64_t per_head = 0;
        for (int64_t i = 0; i < sh->nq; ++i) {
            for (int64_t j = 0; j < sh->nk; ++j) {
                per_head += is_visible(sh, mk, b, i, j);
            }
        }
        total += per_head * sh->Hq;
    }
    return total;
}

/* Returns the index of the first query row (flattened b, r, i) whose       */
/* visible set is empty, or -1 when every row is defined ([A10] A.10.2;     */
/* [CH31] section 3 rejects fully masked rows).                              */
int64_t oracle_first_empty_row(const oracle_shape *sh, const oracle_mask *mk)
{
    for (int64_t b = 0; b < sh->B; ++b) {
        for (int64_t i = 0; i < sh->nq; ++i) {
            int64_t n = 0;
            for (int64_t j = 0; j < sh->nk; ++j) {
                n += is_visible(sh, mk, b, i, j);
            }
            if (n == 0) {
                return b * sh->Hq * sh->nq + i;
            }
        }
    }
    return -1;
}

/* Dense score, weight and score-gradient matrices for small problems:     */
/* S (NaN off V_i), A, dA (= G_A, 0 off V_i) and dS (= G_S), each           */
/* [B][Hq][nq][nk].  Any output pointer may be NULL.  G may be NULL when    */
/* dA and dS are not requested.  Returns -1 if a row is empty, else 0.      */
int oracle_dense_matrices(const oracle_shape *sh, const oracle_mask *mk, double scale,
                          const double *Q, const double *K, const double *V, const double *G,
                          double *S_out, double *A_out, double *dA_out, double *dS_out)
{
    const int64_t rows = sh->B * sh->Hq * sh->nq;
    int bad = 0;
#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)sh->nk);
        double *A = (double *)malloc(sizeof(double) * (size_t)sh->nk);
        double *dA = (double *)malloc(sizeof(double) * (size_t)sh->nk);
        double *dS = (double *)malloc(sizeof(double) * (size_t)sh->nk);
#pragma omp for schedule(static)
        for (int64_t row = 0; row < rows; ++row) {
            const int64_t i = row % sh->nq;
            const int64_t r = (row / sh->nq) % sh->Hq;
            const int64_t b = row / (sh->nq * sh->Hq);
            double m, l;
            if (softmax_row(sh, mk, Q, K, scale, b, r, i, S, A, &m, &l) == 0) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            if (G && (dA_out || dS_out)) {
                score_grad_row(sh, mk, V, G, A, b, r, i, dA, dS);
            }
            for (int64_t j = 0; j < sh->nk; ++j) {
                if (S_out) S_out[row * sh->nk + j] = S[j];
                if (A_out) A_out[row * sh->nk + j] = A[j];
                if (dA_out) dA_out[row * sh->nk + j] = G ? dA[j] : 0.0;
                if (dS_out) dS_out[row * sh->nk + j] = G ? dS[j] : 0.0;
            }
        }
        free(S); free(A); free(dA); free(dS);
    }
    return bad ? -1 : 0;
}

/* Forward pass on selected query rows.  rows == NULL means every row       */
/* (b, r, i) in flattened order; otherwise rows[t] is a flattened index and */
/* the t-th output row goes to O[t], LSE[t].  Returns -1 on an empty row.   */
int oracle_forward(const oracle_shape *sh, const oracle_mask *mk, double scale,
                   const double *Q, const double *K, const double *V,
                   const int64_t *rows, int64_t n_rows, double *O, double *LSE)
{
    const int64_t total = rows ? n_rows : sh->B * sh->Hq * sh->nq;
    int bad = 0;
#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)sh->nk);
        double *A = (double *)malloc(sizeof(double) * (size_t)sh->nk);
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < total; ++t) {
            const int64_t row = rows ? rows[t] : t;
            const int64_t i = row % sh->nq;
            const int64_t r = (row / sh->nq) % sh->Hq;
            const int64_t b = row / (sh->nq * sh->Hq);
            double m, l;
            if (softmax_row(sh, mk, Q, K, scale, b, r, i, S, A, &m, &l) == 0) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            output_row(sh, V, A, b, r, O + t * sh->dv);
            LSE[t] = m + log(l);
        }
        free(S); free(A);
    }
    return bad ? -1 : 0;
}

/* Backward pass.                                                             */
/*                                                                            */
/* Part 1, per query row (b, r, i): A row (A.10.2), O row (A.10.3), dA and   */
/* dS rows (A.10.6-A.10.7), then                                              */
/*   dQ_i = scale * sum_j dS_ij k_j                           (A.10.8)        */
/*   D_i  = sum_l G_il O_il   and   C_i = c_i                                 */
/* D is the row-sum of G .* O; since O_i = sum_j A_ij v_j it equals c_i       */
/* exactly in real arithmetic, and both are returned so a test can check it. */
/*                                                                            */
/* Part 2, per key row (b, h, j) of KV head h:                               */
/*   dV_j = sum over query heads r with g(r) = h, rows i:  A_ij G_i  (A.10.5) */
/*   dK_j = scale * sum over the same (r, i):            dS_ij q_i  (A.10.9) */
/* [A10] A.10.5: query heads sharing a KV head add their contributions.      */
/* Part 2 rebuilds A_ij and dS_ij with the same formulas as part 1 from the  */
/* row's m_i, l_i and c_i, so every term is the one part 1 used.             */
/*                                                                            */
/* q_rows / k_rows select outputs like oracle_forward's rows (NULL = all).  */
/* Per-row statistics are computed for every query row whenever dK or dV is */
/* requested, because a key's gradient sums over all rows that see it;      */
/* with neither requested only the selected rows are visited.  Outputs:     */
/*   dQ[t] for q_rows[t]; D[t], C[t] likewise;                                */
/*   dK[t], dV[t] for k_rows[t] (flattened (b, h, j)).                        */
/* Any output pointer may be NULL.  Returns -1 on an empty row.              */
int oracle_backward(const oracle_shape *sh, const oracle_mask *mk, double scale,
                    const double *Q, const double *K, const double *V, const double *G,
                    const int64_t *q_rows, int64_t n_q_rows,
                    const int64_t *k_rows, int64_t n_k_rows,
                    double *dQ, double *D, double *C, double *dK, double *dV)
{
    const int64_t all_rows = sh->B * sh->Hq * sh->nq;
    double *row_m = (double *)malloc(sizeof(double) * (size_t)all_rows);
    double *row_l = (double *)malloc(sizeof(double) * (size_t)all_rows);
    double *row_c = (double *)malloc(sizeof(double) * (size_t)all_rows);
    int64_t *slot = (int64_t *)malloc(sizeof(int64_t) * (size_t)all_rows);
    if (!row_m || !row_l || !row_c || !slot) {
        free(row_m); free(row_l); free(row_c); free(slot);
        return -2;
    }
    for (int64_t t = 0; t < all_rows; ++t) {
        slot[t] = q_rows ? -1 : t;
    }
    if (q_rows) {
        for (int64_t t = 0; t < n_q_rows; ++t) {
            slot[q_rows[t]] = t;
        }
    }
    int bad = 0;

    /* Part 1. */
#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)sh->nk);
        double *A = (double *)malloc(sizeof(double) * (size_t)sh->nk);
        double *dA = (double *)malloc(sizeof(double) * (size_t)sh->nk);
        double *dS = (double *)malloc(sizeof(double) * (size_t)sh->nk);
        double *o = (double *)malloc(sizeof(double) * (size_t)sh->dv);
#pragma omp for schedule(dynamic, 4)
        for (int64_t row = 0; row < all_rows; ++row) {
            if (!dK && !dV && slot[row] < 0) {
                continue;
            }
            const int64_t i = row % sh->nq;
            const int64_t r = (row / sh->nq) % sh->Hq;
            const int64_t b = row / (sh->nq * sh->Hq);
            const int64_t h = kv_head_of(sh, r);
            double m, l;
            if (softmax_row(sh, mk, Q, K, scale, b, r, i, S, A, &m, &l) == 0) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            const double c = score_grad_row(sh, mk, V, G, A, b, r, i, dA, dS);
            row_m[row] = m;
            row_l[row] = l;
            row_c[row] = c;
            const int64_t t = slot[row];
            if (t < 0) {
                continue;
            }
            if (dQ) {
                double *dq = dQ + t * sh->dh;
                for (int64_t a = 0; a < sh->dh; ++a) {
                    dq[a] = 0.0;
                }
                for (int64_t j = 0; j < sh->nk; ++j) {
                    if (dS[j] != 0.0) {
                        const double *k = k_row(sh, K, b, h, j);
                        for (int64_t a = 0; a < sh->dh; ++a) {
                            dq[a] += dS[j] * k[a];
                        }
                    }
                }
                for (int64_t a = 0; a < sh->dh; ++a) {
                    dq[a] *= scale;
                }
            }
            if (D) {
                output_row(sh, V, A, b, r, o);
                D[t] = dot(go_row(sh, G, b, r, i), o, sh->dv);
            }
            if (C) {
                C[t] = c;
            }
        }
        free(S); free(A); free(dA); free(dS); free(o);
    }
    if (bad) {
        free(row_m); free(row_l); free(row_c); free(slot);
        return -1;
    }

    /* Part 2. */
    const int64_t all_keys = sh->B * sh->Hkv * sh->nk;
    const int64_t total_k = k_rows ? n_k_rows : all_keys;
    const int64_t group = sh->Hq / sh->Hkv;
    if (dK || dV) {
#pragma omp parallel for schedule(dynamic, 4)
        for (int64_t t = 0; t < total_k; ++t) {
            const int64_t key = k_rows ? k_rows[t] : t;
            const int64_t j = key % sh->nk;
            const int64_t h = (key / sh->nk) % sh->Hkv;
            const int64_t b = key / (sh->nk * sh->Hkv);
            const double *k = k_row(sh, K, b, h, j);
            const double *v = v_row(sh, V, b, h, j);
            double *dk = dK ? dK + t * sh->dh : NULL;
            double *dv = dV ? dV + t * sh->dv : NULL;
            if (dk) for (int64_t a = 0; a < sh->dh; ++a) dk[a] = 0.0;
            if (dv) for (int64_t l = 0; l < sh->dv; ++l) dv[l] = 0.0;
            for (int64_t r = h * group; r < (h + 1) * group; ++r) {
                for (int64_t i = 0; i < sh->nq; ++i) {
                    if (!is_visible(sh, mk, b, i, j)) {
                        continue;
                    }
                    const int64_t row = (b * sh->Hq + r) * sh->nq + i;
                    const double *q = q_row(sh, Q, b, r, i);
                    const double *g = go_row(sh, G, b, r, i);
                    const double s_ij = scale * dot(q, k, sh->dh);
                    const double a_ij = exp(s_ij - row_m[row]) / row_l[row];
                    if (dv) {
                        for (int64_t l = 0; l < sh->dv; ++l) {
                            dv[l] += a_ij * g[l];
                        }
                    }
                    if (dk) {
                        const double da_ij = dot(g, v, sh->dv);
#if ORACLE_MUTATION == 1
                        const double ds_ij = a_ij * da_ij;
#else
                        const double ds_ij = a_ij * (da_ij - row_c[row]);
#endif
                        for (int64_t a = 0; a < sh->dh; ++a) {
                            dk[a] += ds_ij * q[a];
                        }
                    }
                }
            }
            if (dk) for (int64_t a = 0; a < sh->dh; ++a) dk[a] *= scale;
        }
    }
    free(row_m); free(row_l); free(row_c); free(slot);
    return 0;
}

/* Threads the OpenMP runtime will use (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) {
        omp_set_num_threads(n);
    }
#else
    (void)n;
#endif
}
