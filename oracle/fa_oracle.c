/*
 * fa_oracle.c -- float64 CPU oracle for exact attention with sinks, masks,
 * causal / sliding-window visibility and GQA.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  The CUDA path never
 * links, includes or calls it, and it shares no code with the CUDA path.
 *
 * What it computes is the plain definition, written out one query row at a
 * time with no tiling and no online softmax:
 *
 *   "FlashAttention forward in C", section 2.1 ("What is computed"):
 *     o_i   = sum_{j in V_i} e^{s_ij} v_j / ( sum_{j in V_i} e^{s_ij} + e^{z_h} )
 *     V_i   = { j < Tk : (causal == 0 or j <= p_i) and (w <= 0 or j > p_i - w) }
 *     p_i   = q_offset + i,   KV head of query head h = floor(h / (H / Hkv))
 *     lse_i = log( sum_{j in V_i} e^{s_ij} + e^{z_h} )   (section 2, symbol table)
 *     the e^{z_h} term only with sinks; a row with no visible key and no sink
 *     gives o_i = 0 and lse_i = -inf.
 *   "Fused attention and softmax: fast and exact", "What is computed":
 *     s_ij = scale * q_i . k_j + mask[i, j], the mask additive with free
 *     element strides (stride 0 broadcasts).
 *
 * Readings where the pages leave a step open (each is listed with the design
 * notes of the repository):
 *   - the sink logit z_h is a raw logit: not scaled, not masked, not windowed;
 *   - a visible key whose masked score is -inf contributes e^{-inf} = 0, so a
 *     row whose every score is -inf and has no sink is an empty row
 *     (o = 0, lse = -inf), as the C page's contract says for empty rows;
 *   - lse is the natural logarithm, computed from the scaled, masked scores.
 *
 * The maximum M over the row's scores (and the sink) is subtracted before
 * exponentiating; this only keeps exp() in range and is part of the plain
 * softmax definition, not the tiled method.
 *
 * Parity: pinned by tests/test_oracle_pins.py (worked example of the C page,
 * section 3; sink identity of its test catalogue; empty-row contract; closed
 * forms; a float64 library cross-check) and tests/test_oracle_mutants.py.
 *
 * ORACLE_MUTANT (compile-time, default 0) plants one known mistake for the
 * mutant tests; a normal build never defines it.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ESHAPE 2
#define ORACLE_ENOMEM 3

typedef struct {
    const double *q, *k, *v;
    double *o, *lse;
    int64_t B, Hq, Hkv, Tq, Tk, D;
    double scale;
    int64_t q_offset;
    int causal;
    int64_t window;
    const double *sinks;
    const double *mask;
    int64_t msb, msh, msq, msk;
    const int64_t *rows; /* query indices to compute, or NULL for all Tq */
    int64_t nrows;
} oracle_problem;

/* KV head read by query head h ("FlashAttention forward in C", section 2.1). */
static int64_t kv_head_of(int64_t h, int64_t Hq, int64_t Hkv) {
#if ORACLE_MUTANT == 3
    (void)Hq;
    return h % Hkv; /* planted: round-robin head map */
#else
    return h / (Hq / Hkv);
#endif
}

/* Absolute position of query row i (section 2, symbol table: p_i). */
static int64_t position_of(int64_t i, int64_t q_offset) {
#if ORACLE_MUTANT == 6
    (void)q_offset;
    return i; /* planted: q_offset ignored */
#else
    return q_offset + i;
#endif
}

/* Membership of key j in V_i (section 2.1). */
static int key_visible(int64_t j, int64_t p, int64_t Tk, int causal, int64_t w) {
    if (j >= Tk) return 0;
#if ORACLE_MUTANT == 4
    if (causal && !(j < p)) return 0; /* planted: a token cannot see itself */
#else
    if (causal && !(j <= p)) return 0;
#endif
#if ORACLE_MUTANT == 5
    if (w > 0 && !(j > p - w - 1)) return 0; /* planted: w + 1 keys */
#else
    if (w > 0 && !(j > p - w)) return 0;
#endif
    return 1;
}

/* Additive mask entry for (b, h, i, j), 0 without a mask ("Fused attention
 * and softmax", "What is computed": free strides, stride 0 broadcasts). */
static double mask_at(const oracle_problem *P, int64_t b, int64_t h, int64_t i, int64_t j) {
    if (!P->mask) return 0.0;
#if ORACLE_MUTANT == 24
    return P->mask[b * P->msb + h * P->msh + i * P->msk + j * P->msq]; /* planted: strides swapped */
#else
    return P->mask[b * P->msb + h * P->msh + i * P->msq + j * P->msk];
#endif
}

/* One query row (b, h, i): scores, softmax with the sink in the denominator,
 * weighted sum of values, lse.  `s` is Tk doubles of scratch. */
static void oracle_row(const oracle_problem *P, int64_t b, int64_t h, int64_t i,
                       double *out_o, double *out_lse, double *s, unsigned char *vis) {
    const int64_t D = P->D;
    const int64_t g = kv_head_of(h, P->Hq, P->Hkv);
    const int64_t p = position_of(i, P->q_offset);
    const double *qi = P->q + ((b * P->Hq + h) * P->Tq + i) * D;
    const double *kb = P->k + (b * P->Hkv + g) * P->Tk * D;
    const double *vb = P->v + (b * P->Hkv + g) * P->Tk * D;
    const int has_sink = P->sinks != NULL;
    double z = has_sink ? P->sinks[h] : 0.0;
#if ORACLE_MUTANT == 25
    z *= P->scale; /* planted: sink logit scaled like a score */
#endif

    /* Scores s_ij = scale * q_i . k_j + mask_ij for j in V_i, and their max. */
    double M = -INFINITY;
    for (int64_t j = 0; j < P->Tk; ++j) {
        vis[j] = (unsigned char)key_visible(j, p, P->Tk, P->causal, P->window);
        if (!vis[j]) continue;
        const double *kj = kb + j * D;
        double dot = 0.0;
        for (int64_t x = 0; x < D; ++x) dot += qi[x] * kj[x];
#if ORACLE_MUTANT == 20
        s[j] = dot + mask_at(P, b, h, i, j); /* planted: scale dropped */
#elif ORACLE_MUTANT == 21
        s[j] = P->scale * (dot + mask_at(P, b, h, i, j)); /* planted: mask scaled */
#else
        s[j] = P->scale * dot + mask_at(P, b, h, i, j);
#endif
        if (s[j] > M) M = s[j];
    }
    if (has_sink && z > M) M = z;

    for (int64_t x = 0; x < D; ++x) out_o[x] = 0.0;
#if ORACLE_MUTANT != 9
    if (M == -INFINITY) { /* no visible key with a finite score, no sink */
        *out_lse = -INFINITY;
        return;
    }
#endif
#if ORACLE_MUTANT == 26
    M = 0.0; /* planted: no max subtraction (overflows on large logits) */
#endif

    /* Denominator Z and numerator sum_j e^{s_j - M} v_j. */
    double Z = 0.0;
    for (int64_t j = 0; j < P->Tk; ++j) {
        if (!vis[j]) continue;
#if ORACLE_MUTANT == 23
        const double e = exp(M - s[j]); /* planted: sign flipped */
#else
        const double e = exp(s[j] - M);
#endif
        Z += e;
#if ORACLE_MUTANT == 22
        const double *vj = kb + j * D; /* planted: keys used as values */
#else
        const double *vj = vb + j * D;
#endif
        for (int64_t x = 0; x < D; ++x) out_o[x] += e * vj[x];
    }
#if ORACLE_MUTANT != 7
    if (has_sink) Z += exp(z - M); /* the sink joins the denominator only */
#endif
    for (int64_t x = 0; x < D; ++x) out_o[x] /= Z;
#if ORACLE_MUTANT == 8
    *out_lse = log(Z); /* planted: lse without the maximum */
#else
    *out_lse = M + log(Z);
#endif
}

typedef struct {
    const oracle_problem *P;
    int64_t begin, end; /* range over flattened (b, h, row) work */
    int status;
} oracle_slice;

static void *oracle_worker(void *arg) {
    oracle_slice *W = (oracle_slice *)arg;
    const oracle_problem *P = W->P;
    double *s = (double *)malloc((size_t)(P->Tk > 0 ? P->Tk : 1) * sizeof(double));
    unsigned char *vis = (unsigned char *)malloc((size_t)(P->Tk > 0 ? P->Tk : 1));
    if (!s || !vis) {
        free(s);
        free(vis);
        W->status = ORACLE_ENOMEM;
        return NULL;
    }
    for (int64_t u = W->begin; u < W->end; ++u) {
        const int64_t r = u % P->nrows;   /* output row slot */
        const int64_t bh = u / P->nrows;  /* b * Hq + h */
        const int64_t b = bh / P->Hq, h = bh % P->Hq;
        const int64_t i = P->rows ? P->rows[r] : r;
        oracle_row(P, b, h, i, P->o + u * P->D, P->lse + u, s, vis);
    }
    free(s);
    free(vis);
    W->status = ORACLE_OK;
    return NULL;
}

static int oracle_check_args(const oracle_problem *P) {
    if (P->B < 0 || P->Hq < 0 || P->Hkv < 0 || P->Tq < 0 || P->Tk < 0 || P->D < 0 ||
        P->q_offset < 0 || P->nrows < 0)
        return ORACLE_EINVAL;
    if (P->Hkv == 0 ? P->Hq > 0 : P->Hkv > P->Hq) return ORACLE_ESHAPE;
#if ORACLE_MUTANT != 15 /* the mutant accepts H % Hkv != 0 */
    if (P->Hkv > 0 && P->Hq % P->Hkv != 0) return ORACLE_ESHAPE;
#endif
    if (P->rows)
        for (int64_t r = 0; r < P->nrows; ++r)
            if (P->rows[r] < 0 || P->rows[r] >= P->Tq) return ORACLE_EINVAL;
    return ORACLE_OK;
}

/*
 * fa_oracle_f64: o [B, Hq, R, D] and lse [B, Hq, R] for the query rows listed
 * in rows[0..nrows) (R = nrows), or for every row 0..Tq-1 when rows == NULL
 * (R = Tq, nrows ignored).  q [B, Hq, Tq, D], k and v [B, Hkv, Tk, D], all
 * contiguous float64.  sinks [Hq] or NULL; mask indexed
 * b*msb + h*msh + i*msq + j*msk (elements) or NULL.  nthreads <= 0 uses one
 * thread.  Returns 0, or an error code before writing anything.
 */
int fa_oracle_f64(const double *q, const double *k, const double *v, double *o, double *lse,
                  int64_t B, int64_t Hq, int64_t Hkv, int64_t Tq, int64_t Tk, int64_t D,
                  double scale, int64_t q_offset, int causal, int64_t window,
                  const double *sinks, const double *mask, int64_t msb, int64_t msh,
                  int64_t msq, int64_t msk, const int64_t *rows, int64_t nrows, int nthreads) {
    oracle_problem P;
    memset(&P, 0, sizeof P);
    P.q = q; P.k = k; P.v = v; P.o = o; P.lse = lse;
    P.B = B; P.Hq = Hq; P.Hkv = Hkv; P.Tq = Tq; P.Tk = Tk; P.D = D;
    P.scale = scale; P.q_offset = q_offset; P.causal = causal; P.window = window;
    P.sinks = sinks; P.mask = mask; P.msb = msb; P.msh = msh; P.msq = msq; P.msk = msk;
    P.rows = rows;
    P.nrows = rows ? nrows : Tq;
    const int st = oracle_check_args(&P);
    if (st != ORACLE_OK) return st;
    const int64_t total = B * Hq * P.nrows;
    if (total == 0) return ORACLE_OK;
    if (!o || !lse || !q) return ORACLE_EINVAL;
    if (Tk > 0 && (!k || !v)) return ORACLE_EINVAL;

    int nt = nthreads > 0 ? nthreads : 1;
    if ((int64_t)nt > total) nt = (int)total;
    pthread_t *th = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    oracle_slice *ws = (oracle_slice *)calloc((size_t)nt, sizeof(oracle_slice));
    if (!th || !ws) {
        free(th);
        free(ws);
        return ORACLE_ENOMEM;
    }
    for (int t = 0; t < nt; ++t) {
        ws[t].P = &P;
        ws[t].begin = total * t / nt;
        ws[t].end = total * (t + 1) / nt;
        ws[t].status = ORACLE_OK;
    }
    int started = 0;
    for (int t = 1; t < nt; ++t) {
        if (pthread_create(&th[t], NULL, oracle_worker, &ws[t]) != 0) break;
        started = t;
    }
    oracle_worker(&ws[0]);
    /* any slice whose thread failed to start runs here, serially */
    for (int t = started + 1; t < nt; ++t) oracle_worker(&ws[t]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    int rc = ORACLE_OK;
    for (int t = 0; t < nt; ++t)
        if (ws[t].status != ORACLE_OK) rc = ws[t].status;
    free(th);
    free(ws);
    return rc;
}
