/*
 * CPU oracle for the forward pass of one Mixture-of-Experts layer, and for its
 * backward pass with the top-K choice held fixed.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the test suite, the smoke check and the
 * benchmark's CPU-baseline leg, never by the CUDA library. It is deliberately
 * slow and plain: each function is the definition written out, in the order the
 * pages state it, with no blocking, fusion or reordering beyond what the
 * definition itself fixes (the router logits' 1024-step blocks). The sources and
 * the readings taken where the pages are silent are listed in moe_oracle.h.
 *
 * Build: plain C11, -ffp-contract=off (no implicit fused multiply-adds; the one
 * fma that belongs to the definition is written as fmaf), no fast-math. OpenMP
 * splits independent tokens or rows across threads; no result depends on the
 * thread count.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- bf16 -- */

double oracle_bf16_to_double(uint16_t b) {
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static float bf16_to_float(uint16_t b) {
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* Nearest bf16 (8 significant bits, fp32 exponent range), ties to even, by
 * scaling the magnitude so that one bf16 ulp becomes 1, rounding to an integer
 * with nearbyint (round-half-even in the default rounding mode) and scaling
 * back. Both scalings are by powers of two and therefore exact. */
uint16_t oracle_bf16_from_double(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0x0000;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7F80;
    int ex;
    frexp(a, &ex);             /* a in [2^(ex-1), 2^ex) */
    int e_ulp = ex - 8;        /* ulp of an 8-significant-bit number there */
    if (e_ulp < -133) e_ulp = -133; /* subnormal range: fixed ulp 2^-133 */
    double r = nearbyint(ldexp(a, -e_ulp));
    double res = ldexp(r, e_ulp);
    if (res >= 0x1p128) return sign | 0x7F80; /* rounds past the largest bf16 */
    float f = (float)res;      /* exact: res has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return sign | (uint16_t)(bits >> 16);
}

/* ------------------------------------------------------------- router -- */

/* Logits of one token row. With E <= LOGIT_FEW_EXPERTS the sum over j runs in
 * blocks of LOGIT_BLOCK reduction steps; with more experts the whole of j is
 * one block. For block b and expert e, s = +0.0f, then for j in the block in
 * ascending order s = fmaf(x_j, Wr[j,e], s). The block sums are then added in
 * ascending block order (acc = s_0, then acc = acc + s_b for b = 1, 2, ...),
 * and finally acc + bias[e]. With one block this is the single fused
 * multiply-add chain over j = 0..d-1. */
#define LOGIT_BLOCK 1024
#define LOGIT_FEW_EXPERTS 32
static void logits_row(const uint16_t *x, const float *Wr, const float *bias,
                       int d, int E, float *acc, float *blk) {
    const int len = E <= LOGIT_FEW_EXPERTS ? LOGIT_BLOCK : d;
    for (int j0 = 0; j0 < d; j0 += len) {
        const int j1 = j0 + len < d ? j0 + len : d;
        for (int e = 0; e < E; ++e) blk[e] = 0.0f;
        for (int j = j0; j < j1; ++j) {
            float xj = bf16_to_float(x[j]);
            const float *w = Wr + (int64_t)j * E;
            for (int e = 0; e < E; ++e) blk[e] = fmaf(xj, w[e], blk[e]);
        }
        for (int e = 0; e < E; ++e) acc[e] = j0 == 0 ? blk[e] : acc[e] + blk[e];
    }
    if (d == 0)
        for (int e = 0; e < E; ++e) acc[e] = 0.0f;
    if (bias)
        for (int e = 0; e < E; ++e) acc[e] = acc[e] + bias[e];
}

void oracle_router_logits(const uint16_t *X, const float *Wr, const float *bias,
                          int64_t T, int d, int E, float *L) {
#pragma omp parallel
    {
        float *blk = (float *)malloc(sizeof(float) * (size_t)(E > 0 ? E : 1));
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t)
            logits_row(X + t * d, Wr, bias, d, E, L + t * E, blk);
        free(blk);
    }
}

typedef struct {
    float v;
    int e;
} scored;

/* Higher score first; equal scores: lower expert index first. */
static int by_score_then_index(const void *pa, const void *pb) {
    const scored *a = (const scored *)pa, *b = (const scored *)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->e > b->e) - (a->e < b->e);
}

/* One row: sort all E experts by (score desc, index asc), keep the first K.
 * p = softmax(L) in double with the maximum subtracted; w_k = p_k, divided by
 * the sum of the kept p when renormalising. */
static void route_row(const float *L, int E, int K, int renorm, int32_t *idx, float *w) {
    scored *s = (scored *)malloc(sizeof(scored) * (size_t)E);
    for (int e = 0; e < E; ++e) {
        s[e].v = L[e];
        s[e].e = e;
    }
    qsort(s, (size_t)E, sizeof(scored), by_score_then_index);
    double m = (double)s[0].v;
    double denom = 0.0;
    for (int e = 0; e < E; ++e) denom += exp((double)L[e] - m);
    double kept = 0.0;
    for (int k = 0; k < K; ++k) kept += exp((double)s[k].v - m) / denom;
    for (int k = 0; k < K; ++k) {
        double p = exp((double)s[k].v - m) / denom;
        idx[k] = s[k].e;
        w[k] = (float)(renorm ? p / kept : p);
    }
    free(s);
}

void oracle_topk_softmax(const float *L, int64_t T, int E, int K, int renorm,
                         int32_t *idx, float *w) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        route_row(L + t * E, E, K, renorm, idx + t * K, w + t * K);
}

/* ------------------------------------------------- counts / permutation -- */

void oracle_expert_counts(const int32_t *idx, int64_t T, int K, int E, int32_t *counts) {
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) counts[idx[t * K + k]] += 1;
}

void oracle_permute(const int32_t *idx, int64_t T, int E, int K,
                    int32_t *offsets, int32_t *perm_token, int32_t *perm_slot,
                    int32_t *row_of_slot) {
    int32_t *counts = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    oracle_expert_counts(idx, T, K, E, counts);
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    /* stable counting sort of the slots (t,k) by expert: visiting slots in
     * ascending t puts each expert's rows in ascending token order */
    int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    for (int e = 0; e < E; ++e) cursor[e] = offsets[e];
    for (int64_t t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            int32_t slot = (int32_t)(t * K + k);
            int32_t p = cursor[idx[slot]]++;
            perm_token[p] = (int32_t)t;
            perm_slot[p] = slot;
            row_of_slot[slot] = p;
        }
    free(cursor);
    free(counts);
}

int oracle_tile_schedule(const int32_t *offsets, int E, int M, int32_t *tiles, int max_tiles) {
    int nt = 0;
    for (int e = 0; e < E; ++e) {
        int32_t c = offsets[e + 1] - offsets[e];
        for (int32_t r = 0; r < c; r += M) {
            if (nt < max_tiles) {
                tiles[4 * nt + 0] = e;
                tiles[4 * nt + 1] = offsets[e] + r;
                tiles[4 * nt + 2] = (c - r < M) ? (c - r) : M;
                tiles[4 * nt + 3] = 0;
            }
            ++nt;
        }
    }
    return nt;
}

/* ---------------------------------------------------------- expert MLP -- */

static double silu(double a) { return a / (1.0 + exp(-a)); }

/* h = bf16( SiLU(x W1e) * (x W3e) ), sums over i = 0..d-1 ascending in double.
 * a1, a3: caller scratch of n doubles. */
static void gate_up_row(const uint16_t *x, const uint16_t *W1e, const uint16_t *W3e,
                        int d, int n, double *a1, double *a3, uint16_t *h) {
    for (int j = 0; j < n; ++j) a1[j] = a3[j] = 0.0;
    for (int i = 0; i < d; ++i) {
        double xi = oracle_bf16_to_double(x[i]);
        const uint16_t *w1 = W1e + (int64_t)i * n;
        const uint16_t *w3 = W3e + (int64_t)i * n;
        for (int j = 0; j < n; ++j) {
            a1[j] = a1[j] + xi * oracle_bf16_to_double(w1[j]);
            a3[j] = a3[j] + xi * oracle_bf16_to_double(w3[j]);
        }
    }
    for (int j = 0; j < n; ++j) h[j] = oracle_bf16_from_double(silu(a1[j]) * a3[j]);
}

/* z = w * (h W2e), sums over j = 0..n-1 ascending in double. */
static void down_row(const uint16_t *h, const uint16_t *W2e, double w, int n, int d,
                     double *z) {
    for (int c = 0; c < d; ++c) z[c] = 0.0;
    for (int j = 0; j < n; ++j) {
        double hj = oracle_bf16_to_double(h[j]);
        const uint16_t *w2 = W2e + (int64_t)j * d;
        for (int c = 0; c < d; ++c) z[c] = z[c] + hj * oracle_bf16_to_double(w2[c]);
    }
    for (int c = 0; c < d; ++c) z[c] = w * z[c];
}

/* expert owning grouped row p, from the offsets */
static int expert_of_row(const int32_t *offsets, int E, int32_t p) {
    int e = 0;
    while (e + 1 < E && offsets[e + 1] <= p) ++e;
    return e;
}

void oracle_gate_up(const uint16_t *X, const uint16_t *W1, const uint16_t *W3,
                    const int32_t *perm_token, const int32_t *offsets,
                    int E, int d, int n, uint16_t *H) {
    int32_t R = offsets[E];
#pragma omp parallel
    {
        double *a1 = (double *)malloc(sizeof(double) * (size_t)n);
        double *a3 = (double *)malloc(sizeof(double) * (size_t)n);
#pragma omp for schedule(dynamic, 1)
        for (int32_t p = 0; p < R; ++p) {
            int e = expert_of_row(offsets, E, p);
            const uint16_t *x = X + (int64_t)perm_token[p] * d;
            gate_up_row(x, W1 + (int64_t)e * d * n, W3 + (int64_t)e * d * n, d, n, a1, a3,
                        H + (int64_t)p * n);
        }
        free(a1);
        free(a3);
    }
}

void oracle_gate_up_pre(const uint16_t *X, const uint16_t *W1, const uint16_t *W3,
                        const int32_t *perm_token, const int32_t *offsets, int E, int d, int n,
                        double *A1, double *A3) {
    int32_t R = offsets[E];
#pragma omp parallel
    {
        uint16_t *h = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)n);
#pragma omp for schedule(dynamic, 1)
        for (int32_t p = 0; p < R; ++p) {
            int e = expert_of_row(offsets, E, p);
            const uint16_t *x = X + (int64_t)perm_token[p] * d;
            gate_up_row(x, W1 + (int64_t)e * d * n, W3 + (int64_t)e * d * n, d, n,
                        A1 + (int64_t)p * n, A3 + (int64_t)p * n, h);
        }
        free(h);
    }
}

void oracle_down(const uint16_t *H, const uint16_t *W2, const float *topk_w,
                 const int32_t *perm_slot, const int32_t *offsets,
                 int E, int n, int d, double *Z) {
    int32_t R = offsets[E];
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t p = 0; p < R; ++p) {
        int e = expert_of_row(offsets, E, p);
        down_row(H + (int64_t)p * n, W2 + (int64_t)e * n * d, (double)topk_w[perm_slot[p]],
                 n, d, Z + (int64_t)p * d);
    }
}

/* ------------------------------------------------------------- combine -- */

void oracle_combine(const double *Z, const int32_t *row_of_slot, int64_t T, int K,
                    int d, uint16_t *Y) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int c = 0; c < d; ++c) {
            double y = 0.0;
            for (int k = 0; k < K; ++k) y = y + Z[(int64_t)row_of_slot[t * K + k] * d + c];
            Y[t * d + c] = oracle_bf16_from_double(y);
        }
}

void oracle_combine_bf16(const uint16_t *Z, const int32_t *row_of_slot, int64_t T,
                         int K, int d, uint16_t *Y) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int c = 0; c < d; ++c) {
            double y = 0.0;
            for (int k = 0; k < K; ++k)
                y = y + oracle_bf16_to_double(Z[(int64_t)row_of_slot[t * K + k] * d + c]);
            Y[t * d + c] = oracle_bf16_from_double(y);
        }
}

/* ------------------------------------------------------ whole layer -- */

void oracle_forward_tokens(const uint16_t *X, const float *Wr, const float *bias,
                           const uint16_t *W1, const uint16_t *W3, const uint16_t *W2,
                           int64_t T, int d, int E, int K, int n, int renorm,
                           const int64_t *tokens, int64_t n_tok,
                           uint16_t *Y_rows, int32_t *idx_rows, float *w_rows) {
    (void)T;
#pragma omp parallel
    {
        float *L = (float *)malloc(sizeof(float) * (size_t)E);
        float *blk = (float *)malloc(sizeof(float) * (size_t)E);
        double *a1 = (double *)malloc(sizeof(double) * (size_t)n);
        double *a3 = (double *)malloc(sizeof(double) * (size_t)n);
        uint16_t *h = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)n);
        double *z = (double *)malloc(sizeof(double) * (size_t)d);
        double *y = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_tok; ++i) {
            int64_t t = tokens[i];
            const uint16_t *x = X + t * d;
            int32_t *idx = idx_rows + i * K;
            float *w = w_rows + i * K;
            logits_row(x, Wr, bias, d, E, L, blk);
            route_row(L, E, K, renorm, idx, w);
            for (int c = 0; c < d; ++c) y[c] = 0.0;
            for (int k = 0; k < K; ++k) {
                int e = idx[k];
                gate_up_row(x, W1 + (int64_t)e * d * n, W3 + (int64_t)e * d * n, d, n, a1, a3, h);
                down_row(h, W2 + (int64_t)e * n * d, (double)w[k], n, d, z);
                for (int c = 0; c < d; ++c) y[c] = y[c] + z[c];
            }
            for (int c = 0; c < d; ++c) Y_rows[i * d + c] = oracle_bf16_from_double(y[c]);
        }
        free(L);
        free(blk);
        free(a1);
        free(a3);
        free(h);
        free(z);
        free(y);
    }
}

/* ------------------------------------------------------ token rounding -- */

typedef struct {
    int member;  /* 1 when the token chose this expert in its top-K */
    float v;     /* L[t,e] */
    int64_t t;
} candidate;

/* chosen first; then higher score; then lower token index */
static int by_member_score_token(const void *pa, const void *pb) {
    const candidate *a = (const candidate *)pa, *b = (const candidate *)pb;
    if (a->member != b->member) return a->member ? -1 : 1;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->t > b->t) - (a->t < b->t);
}

int64_t oracle_token_rounding(const float *L, const int32_t *idx, int64_t T, int E, int K,
                              int M, int renorm, int64_t cap, int32_t *counts_out,
                              int32_t *offsets, int32_t *perm_token, int32_t *row_map,
                              float *row_w) {
    /* 1. expert frequencies */
    int32_t *f = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    oracle_expert_counts(idx, T, K, E, f);
    /* 2. rounded targets */
    for (int e = 0; e < E; ++e) {
        int64_t c = (int64_t)M * ((f[e] + M / 2) / M);
        if (c > T) c = (int64_t)M * (f[e] / M);
        counts_out[e] = (int32_t)c;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts_out[e];
    if (offsets[E] > cap) {
        free(f);
        return -1;
    }
    /* 3. the second sort, one expert at a time; keep[t*E+e] marks the kept pairs */
    unsigned char *member = (unsigned char *)calloc((size_t)(T * E), 1);
    unsigned char *keep = (unsigned char *)calloc((size_t)(T * E), 1);
    for (int64_t t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) member[t * E + idx[t * K + k]] = 1;
    candidate *cand = (candidate *)malloc(sizeof(candidate) * (size_t)T);
    for (int e = 0; e < E; ++e) {
        for (int64_t t = 0; t < T; ++t) {
            cand[t].member = member[t * E + e];
            cand[t].v = L[t * E + e];
            cand[t].t = t;
        }
        qsort(cand, (size_t)T, sizeof(candidate), by_member_score_token);
        for (int32_t i = 0; i < counts_out[e]; ++i) keep[cand[i].t * E + e] = 1;
    }
    /* 4. rows grouped by expert, ascending t */
    int32_t p = 0;
    for (int e = 0; e < E; ++e)
        for (int64_t t = 0; t < T; ++t) {
            if (keep[t * E + e]) {
                row_map[t * E + e] = p;
                perm_token[p] = (int32_t)t;
                ++p;
            } else {
                row_map[t * E + e] = -1;
            }
        }
    /* 5. softmax weights of the kept pairs */
    for (int64_t t = 0; t < T; ++t) {
        const float *l = L + t * E;
        double m = (double)l[0];
        for (int e = 1; e < E; ++e)
            if ((double)l[e] > m) m = (double)l[e];
        double denom = 0.0;
        for (int e = 0; e < E; ++e) denom += exp((double)l[e] - m);
        double kept = 0.0;
        for (int e = 0; e < E; ++e)
            if (keep[t * E + e]) kept += exp((double)l[e] - m) / denom;
        for (int e = 0; e < E; ++e)
            if (keep[t * E + e]) {
                double pe = exp((double)l[e] - m) / denom;
                row_w[row_map[t * E + e]] = (float)(renorm ? pe / kept : pe);
            }
    }
    free(cand);
    free(keep);
    free(member);
    free(f);
    return offsets[E];
}

void oracle_combine_rows(const double *Z, const int32_t *row_map, int64_t T, int E, int d,
                         uint16_t *Y) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int c = 0; c < d; ++c) {
            double y = 0.0;
            for (int e = 0; e < E; ++e) {
                int32_t r = row_map[t * E + e];
                if (r >= 0) y = y + Z[(int64_t)r * d + c];
            }
            Y[t * d + c] = oracle_bf16_from_double(y);
        }
}

void oracle_combine_rows_bf16(const uint16_t *Z, const int32_t *row_map, int64_t T, int E,
                              int d, uint16_t *Y) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int c = 0; c < d; ++c) {
            double y = 0.0;
            for (int e = 0; e < E; ++e) {
                int32_t r = row_map[t * E + e];
                if (r >= 0) y = y + oracle_bf16_to_double(Z[(int64_t)r * d + c]);
            }
            Y[t * d + c] = oracle_bf16_from_double(y);
        }
}

void oracle_forward_assigned(const uint16_t *X, const uint16_t *W1, const uint16_t *W3,
                             const uint16_t *W2, int64_t T, int d, int E, int n,
                             const int32_t *row_map, const float *row_w,
                             const int64_t *tokens, int64_t n_tok, uint16_t *Y_rows) {
    (void)T;
#pragma omp parallel
    {
        double *a1 = (double *)malloc(sizeof(double) * (size_t)n);
        double *a3 = (double *)malloc(sizeof(double) * (size_t)n);
        uint16_t *h = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)n);
        double *z = (double *)malloc(sizeof(double) * (size_t)d);
        double *y = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_tok; ++i) {
            int64_t t = tokens[i];
            const uint16_t *x = X + t * d;
            for (int c = 0; c < d; ++c) y[c] = 0.0;
            for (int e = 0; e < E; ++e) {
                int32_t r = row_map[t * E + e];
                if (r < 0) continue;
                gate_up_row(x, W1 + (int64_t)e * d * n, W3 + (int64_t)e * d * n, d, n, a1, a3, h);
                down_row(h, W2 + (int64_t)e * n * d, (double)row_w[r], n, d, z);
                for (int c = 0; c < d; ++c) y[c] = y[c] + z[c];
            }
            for (int c = 0; c < d; ++c) Y_rows[i * d + c] = oracle_bf16_from_double(y[c]);
        }
        free(a1);
        free(a3);
        free(h);
        free(z);
        free(y);
    }
}

/* ------------------------------------------------------------ backward -- */

/* The layer in double with the top-K choice held fixed (idx [T,K]): the
 * function whose gradient oracle_backward returns. Every input is double (bf16
 * and fp32 tensors widen exactly). For token t:
 *   L[e] = sum_j x_j Wr[j,e] (+ bias[e]); p = softmax(L) over all E;
 *   w_k = p[idx_k] / sum_k' p[idx_k'] (renorm) or p[idx_k];
 *   a1 = x W1[e], a3 = x W3[e], h = silu(a1) * a3, o = h W2[e] for e = idx_k;
 *   Y[t] = sum_k w_k o_k.
 * No bf16 rounding of h or Y and no fp32 logits: the forward pass's roundings
 * pass gradients through unchanged, so this is the function they differentiate. */
static void fixed_token(const double *x, const double *Wr, const double *bias,
                        const int32_t *idx, int d, int E, int K, int renorm, double *p,
                        double *w) {
    double m = -INFINITY;
    for (int e = 0; e < E; ++e) {
        double l = 0.0;
        for (int j = 0; j < d; ++j) l += x[j] * Wr[(int64_t)j * E + e];
        if (bias) l += bias[e];
        p[e] = l;
        if (l > m) m = l;
    }
    double s = 0.0;
    for (int e = 0; e < E; ++e) {
        p[e] = exp(p[e] - m);
        s += p[e];
    }
    for (int e = 0; e < E; ++e) p[e] /= s;
    double kept = 0.0;
    for (int k = 0; k < K; ++k) kept += p[idx[k]];
    for (int k = 0; k < K; ++k) w[k] = renorm ? p[idx[k]] / kept : p[idx[k]];
}

static void expert_acts(const double *x, const double *W1e, const double *W3e, int d, int n,
                        double *a1, double *a3) {
    for (int i = 0; i < n; ++i) a1[i] = a3[i] = 0.0;
    for (int j = 0; j < d; ++j) {
        const double *w1 = W1e + (int64_t)j * n, *w3 = W3e + (int64_t)j * n;
        for (int i = 0; i < n; ++i) {
            a1[i] += x[j] * w1[i];
            a3[i] += x[j] * w3[i];
        }
    }
}

void oracle_forward_fixed(const double *X, const double *Wr, const double *bias,
                          const double *W1, const double *W3, const double *W2,
                          const int32_t *idx, int64_t T, int d, int E, int K, int n, int renorm,
                          double *Y) {
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    double *w = (double *)malloc(sizeof(double) * (size_t)K);
    double *a1 = (double *)malloc(sizeof(double) * (size_t)n);
    double *a3 = (double *)malloc(sizeof(double) * (size_t)n);
    for (int64_t t = 0; t < T; ++t) {
        const double *x = X + t * d;
        const int32_t *it = idx + t * K;
        fixed_token(x, Wr, bias, it, d, E, K, renorm, p, w);
        double *y = Y + t * d;
        for (int c = 0; c < d; ++c) y[c] = 0.0;
        for (int k = 0; k < K; ++k) {
            const int e = it[k];
            expert_acts(x, W1 + (int64_t)e * d * n, W3 + (int64_t)e * d * n, d, n, a1, a3);
            const double *W2e = W2 + (int64_t)e * n * d;
            for (int i = 0; i < n; ++i) {
                const double h = silu(a1[i]) * a3[i];
                for (int c = 0; c < d; ++c) y[c] += w[k] * h * W2e[(int64_t)i * d + c];
            }
        }
    }
    free(p);
    free(w);
    free(a1);
    free(a3);
}

/* Gradient of sum(Y * dY) for Y = oracle_forward_fixed(...), by the chain rule
 * written out per token and routed pair (single-threaded: the weight gradients
 * accumulate over tokens). With s = sigmoid(a1), silu(a1) = a1 s and
 * silu'(a1) = s (1 + a1 (1 - s)):
 *   o = h W2[e];  dw_k = dY[t] . o;  dh = w_k (dY[t] W2[e]^T);
 *   dW2[e] += h^T (w_k dY[t]);  da1 = dh * a3 * silu'(a1);  da3 = dh * silu(a1);
 *   dX[t] += da1 W1[e]^T + da3 W3[e]^T;  dW1[e] += x^T da1;  dW3[e] += x^T da3.
 * Router: dp[idx_k] = (dw_k - sum_k' w_k' dw_k') / kept (renorm) or dw_k, 0 for
 * the other experts; dL = p * (dp - sum_e p_e dp_e) (softmax); dbias += dL;
 * dWr += x^T dL;  dX[t] += dL Wr^T.
 * Outputs are overwritten; bias and dbias may be NULL. */
void oracle_backward(const double *X, const double *Wr, const double *bias,
                     const double *W1, const double *W3, const double *W2,
                     const int32_t *idx, const double *dY, int64_t T, int d, int E, int K, int n,
                     int renorm, double *dX, double *dWr, double *dbias, double *dW1,
                     double *dW3, double *dW2) {
    memset(dX, 0, sizeof(double) * (size_t)(T * d));
    memset(dWr, 0, sizeof(double) * (size_t)d * E);
    if (dbias) memset(dbias, 0, sizeof(double) * (size_t)E);
    memset(dW1, 0, sizeof(double) * (size_t)E * d * n);
    memset(dW3, 0, sizeof(double) * (size_t)E * d * n);
    memset(dW2, 0, sizeof(double) * (size_t)E * n * d);
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    double *dp = (double *)malloc(sizeof(double) * (size_t)E);
    double *w = (double *)malloc(sizeof(double) * (size_t)K);
    double *dw = (double *)malloc(sizeof(double) * (size_t)K);
    double *a1 = (double *)malloc(sizeof(double) * (size_t)n);
    double *a3 = (double *)malloc(sizeof(double) * (size_t)n);
    double *dh = (double *)malloc(sizeof(double) * (size_t)n);
    for (int64_t t = 0; t < T; ++t) {
        const double *x = X + t * d;
        const int32_t *it = idx + t * K;
        const double *g = dY + t * d;
        double *dx = dX + t * d;
        fixed_token(x, Wr, bias, it, d, E, K, renorm, p, w);
        for (int k = 0; k < K; ++k) {
            const int e = it[k];
            const double *W1e = W1 + (int64_t)e * d * n, *W3e = W3 + (int64_t)e * d * n;
            const double *W2e = W2 + (int64_t)e * n * d;
            expert_acts(x, W1e, W3e, d, n, a1, a3);
            dw[k] = 0.0;
            for (int i = 0; i < n; ++i) {
                const double h = silu(a1[i]) * a3[i];
                const double *w2 = W2e + (int64_t)i * d;
                double gw = 0.0;  /* dY[t] . W2[e][i,:] */
                for (int c = 0; c < d; ++c) {
                    gw += g[c] * w2[c];
                    dW2[((int64_t)e * n + i) * d + c] += h * w[k] * g[c];
                }
                dw[k] += h * gw;  /* dY[t] . o = sum_i h_i (dY[t] . W2[e][i,:]) */
                dh[i] = w[k] * gw;
            }
            for (int i = 0; i < n; ++i) {
                const double s = 1.0 / (1.0 + exp(-a1[i]));
                const double da1 = dh[i] * a3[i] * s * (1.0 + a1[i] * (1.0 - s));
                const double da3 = dh[i] * a1[i] * s;
                for (int j = 0; j < d; ++j) {
                    dx[j] += da1 * W1e[(int64_t)j * n + i] + da3 * W3e[(int64_t)j * n + i];
                    dW1[((int64_t)e * d + j) * n + i] += x[j] * da1;
                    dW3[((int64_t)e * d + j) * n + i] += x[j] * da3;
                }
            }
        }
        /* router */
        double kept = 0.0, wdw = 0.0;
        for (int k = 0; k < K; ++k) {
            kept += p[it[k]];
            wdw += w[k] * dw[k];
        }
        for (int e = 0; e < E; ++e) dp[e] = 0.0;
        for (int k = 0; k < K; ++k) dp[it[k]] += renorm ? (dw[k] - wdw) / kept : dw[k];
        double pdp = 0.0;
        for (int e = 0; e < E; ++e) pdp += p[e] * dp[e];
        for (int e = 0; e < E; ++e) {
            const double dl = p[e] * (dp[e] - pdp);
            if (dbias) dbias[e] += dl;
            for (int j = 0; j < d; ++j) {
                dWr[(int64_t)j * E + e] += x[j] * dl;
                dx[j] += dl * Wr[(int64_t)j * E + e];
            }
        }
    }
    free(p);
    free(dp);
    free(w);
    free(dw);
    free(a1);
    free(a3);
    free(dh);
}

/* The backward's per-row quantities in grouped row order, for checking a
 * backward that runs expert by expert. Row p holds slot perm_slot[p] = t*K + k
 * (expert e = idx[t,k]); with a1 = x W1[e], a3 = x W3[e], h = silu(a1) a3 and
 * g = dY[t] W2[e]^T (the gradient of h W2[e] taken through W2):
 *   dS[p]    = h . g, the gradient of the routing weight w_k (dY[t] . h W2[e]);
 *   dA1[p,:] = w_k g a3 silu'(a1) and dA3[p,:] = w_k g silu(a1);
 *   dXg[p,:] = dA1 W1[e]^T + dA3 W3[e]^T, row p's share of dX[t];
 * and per token dL[t,:], the gradient of the logits (the routing weights'
 * softmax and renormalisation taken backwards from the K values dS).
 * Then dX[t] = sum over t's rows of dXg + dL[t] Wr^T, dW1[e] = sum over e's
 * rows of x^T dA1 (dW3 likewise) and dWr = sum_t x^T dL[t]: the outputs of
 * oracle_backward, computed there token by token. */
void oracle_backward_rows(const double *X, const double *Wr, const double *bias,
                          const double *W1, const double *W3, const double *W2,
                          const int32_t *idx, const int32_t *perm_slot, const double *dY,
                          int64_t T, int d, int E, int K, int n, int renorm, double *dS,
                          double *dA1, double *dA3, double *dXg, double *dL) {
    const int64_t R = T * K;
    double *P = (double *)malloc(sizeof(double) * (size_t)(T * E));  /* softmax per token */
    double *g = (double *)malloc(sizeof(double) * (size_t)n);
    double *a1 = (double *)malloc(sizeof(double) * (size_t)n);
    double *a3 = (double *)malloc(sizeof(double) * (size_t)n);
    int64_t *row_of = (int64_t *)malloc(sizeof(int64_t) * (size_t)R);
    /* routing probabilities of every token */
    for (int64_t t = 0; t < T; ++t) {
        double *pt = P + t * E, mx = -INFINITY, z = 0.0;
        for (int e = 0; e < E; ++e) {
            double l = bias ? bias[e] : 0.0;
            for (int j = 0; j < d; ++j) l += X[t * d + j] * Wr[(int64_t)j * E + e];
            pt[e] = l;
            mx = l > mx ? l : mx;
        }
        for (int e = 0; e < E; ++e) z += (pt[e] = exp(pt[e] - mx));
        for (int e = 0; e < E; ++e) pt[e] /= z;
    }
    for (int64_t p = 0; p < R; ++p) {
        const int64_t slot = perm_slot[p], t = slot / K;
        const int e = idx[slot];
        row_of[slot] = p;
        const double *x = X + t * d, *gy = dY + t * d, *pt = P + t * E;
        double kept = 0.0;
        for (int k = 0; k < K; ++k) kept += pt[idx[t * K + k]];
        const double wk = renorm ? pt[e] / kept : pt[e];
        const double *W1e = W1 + (int64_t)e * d * n, *W3e = W3 + (int64_t)e * d * n;
        const double *W2e = W2 + (int64_t)e * n * d;
        double ds = 0.0;
        for (int i = 0; i < n; ++i) {
            double u = 0.0, v = 0.0, q = 0.0;
            for (int j = 0; j < d; ++j) {
                u += x[j] * W1e[(int64_t)j * n + i];
                v += x[j] * W3e[(int64_t)j * n + i];
            }
            for (int c = 0; c < d; ++c) q += gy[c] * W2e[(int64_t)i * d + c];
            a1[i] = u;
            a3[i] = v;
            g[i] = q;
            ds += silu(u) * v * q;
        }
        dS[p] = ds;
        double *r1 = dA1 + p * n, *r3 = dA3 + p * n, *rx = dXg + p * d;
        for (int i = 0; i < n; ++i) {
            const double sg = 1.0 / (1.0 + exp(-a1[i]));
            r1[i] = wk * g[i] * a3[i] * (sg + a1[i] * sg * (1.0 - sg));
            r3[i] = wk * g[i] * a1[i] * sg;
        }
        for (int j = 0; j < d; ++j) {
            double acc = 0.0;
            for (int i = 0; i < n; ++i)
                acc += r1[i] * W1e[(int64_t)j * n + i] + r3[i] * W3e[(int64_t)j * n + i];
            rx[j] = acc;
        }
    }
    /* logits: w_k = p_k / kept (renorm) or p_k; p = softmax(L) */
    for (int64_t t = 0; t < T; ++t) {
        const double *pt = P + t * E;
        double *dl = dL + t * E;
        double kept = 0.0, sw = 0.0;
        for (int k = 0; k < K; ++k) kept += pt[idx[t * K + k]];
        for (int e = 0; e < E; ++e) dl[e] = 0.0;  /* first dp, then dL in place */
        for (int k = 0; k < K; ++k) {
            const int e = idx[t * K + k];
            const double wk = renorm ? pt[e] / kept : pt[e];
            sw += wk * dS[row_of[t * K + k]];
        }
        for (int k = 0; k < K; ++k) {
            const int e = idx[t * K + k];
            const double s = dS[row_of[t * K + k]];
            dl[e] += renorm ? (s - sw) / kept : s;
        }
        double mean = 0.0;
        for (int e = 0; e < E; ++e) mean += pt[e] * dl[e];
        for (int e = 0; e < E; ++e) dl[e] = pt[e] * (dl[e] - mean);
    }
    free(P);
    free(g);
    free(a1);
    free(a3);
    free(row_of);
}
