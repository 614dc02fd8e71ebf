/*
 * spec_oracle.c -- plain, slow, fp64 CPU oracle of the speculative-decoding
 * verification pass.
 *
 * TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference arm load this file's library. The CUDA library
 * shares no code with it and never calls it.
 *
 * Every floating-point step is done in double precision from the exact input
 * values (fp32, or bf16 widened by appending 16 zero bits). Every loop runs in
 * ascending index order, with no blocking, fusion or reordering, so that each
 * function reads against the passage it cites.
 *
 * Sources, cited by page title and section:
 *  [SD]  "Speculative Decoding: как черновая модель ускоряет генерацию LLM без
 *        потери качества", sections "Алгоритм на каждом шаге" (steps 1-4) and
 *        "Математика верификации".
 *  [AV]  "Verificación Adaptativa sin una cabeza de confianza", sections
 *        "Solución: Estimador de aceptación ajustado en línea",
 *        "Puntuar la Distribución", "Ajuste de los Coeficientes", footnote 1.
 *  [FLy] "Training-Free Loosely Speculative Decoding: Accepting Semantically
 *        Correct Drafts Beyond Exact Match", section 2.A ("Mecanismo de
 *        Verificação de Dois Níveis"): 2.A.1 entropy gate, 2.A.2 deferral window.
 *
 * Readings where the pages are silent are listed beside the code that takes
 * them; each is also recorded in the repository's design notes.
 *
 * Pins: every function here is pinned by tests/test_oracle_pins.py against
 * closed forms, the worked example of [AV] footnote 1, brute force on tiny
 * vocabularies and a Monte Carlo chi-square test of losslessness ([SD]); the
 * IRLS refit against finite differences, a library linear solve and the
 * maximum-likelihood fit of a general-purpose minimiser.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F32 0
#define OR_BF16 1

#define OR_STOCHASTIC 0
#define OR_GREEDY 1
#define OR_FLY 2

/* degenerate-case bits written to flags[b] */
#define OR_FLAG_Q_ZERO 1     /* q(x_i) == 0 at a tested position            */
#define OR_FLAG_Z_ZERO 2     /* residual mass 0 after a reject: fell back to p */
#define OR_FLAG_CDF_FALLBACK 4 /* no cumulative value exceeded u*Z           */
#define OR_FLAG_REST_ZERO 8  /* logit(q_max) capped at 30 (q_max ~ 1)          */
#define OR_FLAG_NUCLEUS 32   /* a nucleus boundary (top-p) is in doubt         */
#define OR_FLAG_BAD_ROW 16   /* a row with no finite logit                    */

/* logit(q_max) when the complement mass is exactly zero */
#define OR_F_CLAMP 30.0

static double dmin(double a, double b) { return a < b ? a : b; }

static double logit_at(const void *row, int dtype, int64_t v) {
    if (dtype == OR_F32) return (double)((const float *)row)[v];
    uint32_t bits = ((uint32_t)((const uint16_t *)row)[v]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Softmax of one vocabulary row: p_v = exp(z_v - m) / sum_w exp(z_w - m),
 * m = max_v z_v ([SD] "Математика верификации": p(x) and q(x) are the
 * target's and the draft's next-token distributions). Writes p[0..V) and
 * returns lse = m + log(sum). Returns 0 and sets *ok = 0 when no logit is
 * finite. */
static double softmax_row(const void *row, int dtype, int32_t V, double sc, double *p, int *ok) {
    /* softmax of sc * z (sc: the inverse sampling temperature, 1 by default) */
    double m = -INFINITY;
    for (int32_t v = 0; v < V; ++v) {
        double z = sc * logit_at(row, dtype, v);
        if (z > m) m = z;
    }
    if (!(m > -INFINITY) || isinf(m)) {
        *ok = 0;
        for (int32_t v = 0; v < V; ++v) p[v] = 0.0;
        return 0.0;
    }
    double s = 0.0;
    for (int32_t v = 0; v < V; ++v) {
        p[v] = exp(sc * logit_at(row, dtype, v) - m);
        s += p[v];
    }
    for (int32_t v = 0; v < V; ++v) p[v] /= s;
    *ok = 1;
    return m + log(s);
}

/* Top-p (nucleus) truncation of a normalised row p ([AV] "Benchmarks": the
 * serving setting samples with top-p 0.95; [SD] "Математика верификации":
 * the rule is lossless for whatever distributions the models sample from).
 * Reading: the nucleus is every token whose logit is at least z*, the
 * largest logit value t for which the tokens with logit >= t hold at least
 * top_p of the mass. Tokens tied at z* are all kept, so the set does not
 * depend on an order among equal logits. p is zeroed outside the nucleus and
 * renormalised; the nucleus mass P (before renormalising) is returned and z*
 * in *zstar. keys: V entries of scratch.
 *
 * Decision margin. A computation whose cumulative masses carry a relative
 * error e can place the boundary one tie group off: it can drop the group at
 * z* when (top_p - above) < e above, or add the next group down when
 * (P - top_p) < e P ("above" = the mass strictly above z*). Such a
 * difference is harmless when the group in doubt holds at most
 * OR_NUC_BENIGN of P (it moves every probability by less than that), unless
 * a draft token is in it. Reading of the flag (the pages fix no precision):
 * with e = OR_NUC_REL, *margin is the smaller relative distance when a group
 * in doubt is above OR_NUC_BENIGN, else +inf; *zamb_hi / *zamb_lo are the
 * logits of the groups in doubt (NaN: none), for the caller to flag a draft
 * token there. */
#define OR_NUC_REL 1e-5
#define OR_NUC_BENIGN 1e-6
typedef struct {
    double z;
    int32_t v;
} OrKey;

static int key_desc(const void *a, const void *b) {
    const OrKey *x = (const OrKey *)a, *y = (const OrKey *)b;
    if (x->z != y->z) return x->z > y->z ? -1 : 1;
    return x->v < y->v ? -1 : (x->v > y->v ? 1 : 0);
}

static double nucleus(const void *row, int dtype, int32_t V, double top_p, int shift, double *p, OrKey *keys,
                      double *zstar, double *margin_hi, double *margin_lo, double *zamb_hi, double *zamb_lo) {
    for (int32_t v = 0; v < V; ++v) {
        keys[v].z = logit_at(row, dtype, v);
        keys[v].v = v;
    }
    qsort(keys, (size_t)V, sizeof(OrKey), key_desc);
    double above = 0.0;   /* mass of logits strictly above the current value */
    int32_t i = 0;
    *zstar = keys[0].z;
    *margin_hi = *margin_lo = INFINITY;
    *zamb_hi = *zamb_lo = NAN;
    while (i < V) {
        int32_t j = i;
        double g = 0.0;   /* mass of the tokens tied at keys[i].z */
        while (j < V && keys[j].z == keys[i].z) g += p[keys[j++].v];
        if (above + g >= top_p || j == V) {
            const double P = above + g;
            *zstar = keys[i].z;
            /* the group at z* may be dropped */
            if (above > 0.0 && top_p - above < OR_NUC_REL * above) {
                if (g > OR_NUC_BENIGN * P) *margin_hi = (top_p - above) / above;
                *zamb_hi = keys[i].z;
            }
            /* the next group down may be added */
            if (j < V && P - top_p < OR_NUC_REL * P) {
                double gn = 0.0;
                for (int32_t k = j; k < V && keys[k].z == keys[j].z; ++k) gn += p[keys[k].v];
                if (gn > OR_NUC_BENIGN * P) *margin_lo = (P - top_p) / P;
                *zamb_lo = keys[j].z;
            }
            /* a caller-chosen boundary one tie group off (parity checks of a
             * computation that placed a boundary in doubt the other way):
             * -1 drops the group at z*, +1 adds the next group down */
            if (shift < 0 && i > 0) *zstar = keys[i - 1].z;
            if (shift > 0 && j < V) *zstar = keys[j].z;
            break;
        }
        above += g;
        i = j;
    }
    double P = 0.0;
    for (int32_t v = 0; v < V; ++v) {
        if (logit_at(row, dtype, v) >= *zstar) P += p[v];
        else p[v] = 0.0;
    }
    for (int32_t v = 0; v < V; ++v) p[v] /= P;
    return P;
}

/* The distribution a model samples from for one row: softmax of sc*z, then,
 * with top_p < 1, its nucleus renormalised. Returns the log of its
 * normaliser (lse of the processed row: lse of sc*z plus ln P) and sets
 * *zstar (-inf without truncation); *margin takes the smaller of itself and
 * the nucleus boundary's margin, which is 0 when the logit of token `xtok`
 * (-1: none) lies in a tie group whose membership is in doubt. */
static double processed_row(const void *row, int dtype, int32_t V, double sc, double top_p, int shift,
                            double *p, OrKey *keys, int *ok, double *zstar, double *margin, int32_t xtok,
                            int *doubt) {
    double lse = softmax_row(row, dtype, V, sc, p, ok);
    *zstar = -INFINITY;
    if (doubt) *doubt = 0;
    if (*ok && top_p < 1.0) {
        double mh, ml, zh, zl;
        lse += log(nucleus(row, dtype, V, top_p, shift, p, keys, zstar, &mh, &ml, &zh, &zl));
        int tok_hi = 0, tok_lo = 0;
        if (xtok >= 0 && xtok < V) {
            const double zx = logit_at(row, dtype, xtok);
            tok_hi = zx == zh;
            tok_lo = zx == zl;
        }
        *margin = dmin(*margin, dmin(mh, ml));
        if (tok_hi || tok_lo) *margin = 0.0;
        /* which way the boundary is in doubt: bit 1 the group at z* may be
         * dropped, bit 2 the next group down may be added */
        if (doubt) *doubt = ((mh < INFINITY || tok_hi) ? 1 : 0) | ((ml < INFINITY || tok_lo) ? 2 : 0);
    }
    return lse;
}

/* Index of the largest logit; ties go to the lowest index (reading: the pages
 * do not say how ties break). */
static int32_t argmax_row(const void *row, int dtype, int32_t V) {
    int32_t best = 0;
    double bz = logit_at(row, dtype, 0);
    for (int32_t v = 1; v < V; ++v) {
        double z = logit_at(row, dtype, v);
        if (z > bz) { bz = z; best = v; }
    }
    return best;
}

/* Normalised entropy h = -sum_{p_v>0} p_v ln p_v / ln V ([FLy] 2.A.1: the
 * gate reads the normalised entropy of the target's prediction; reading:
 * natural logarithm divided by ln V, so a uniform row gives 1). */
static double norm_entropy(const double *p, int32_t V) {
    double h = 0.0;
    for (int32_t v = 0; v < V; ++v)
        if (p[v] > 0.0) h -= p[v] * log(p[v]);
    return h / log((double)V);
}

/* logit(q_max) = ln q_max - ln(sum_{v != argmax} q_v) ([AV] "Puntuar la
 * Distribución": the feature is the log-odds of the draft's most likely
 * token). The complement is summed directly rather than formed as 1 - q_max.
 * Reading: the feature is capped at OR_F_CLAMP (30, q_max within 1e-13 of 1);
 * the pages give no value for that regime, and the cap keeps the feature
 * continuous where the complement underflows (fp64 beyond 708, fp32 beyond
 * 87). Capped values are flagged. */
static double logit_qmax(const double *q, int32_t V, int32_t amax, int *flags) {
    double rest = 0.0;
    for (int32_t v = 0; v < V; ++v)
        if (v != amax) rest += q[v];
    const double f = rest > 0.0 ? log(q[amax]) - log(rest) : INFINITY;
    if (f >= OR_F_CLAMP) {
        *flags |= OR_FLAG_REST_ZERO;
        return OR_F_CLAMP;
    }
    return f;
}

/* Inverse-CDF draw from the unnormalised weights r[0..V) with total Z: the
 * smallest v whose running sum (ascending v) exceeds u*Z. Writes the distance
 * of u to the nearer boundary of v's interval, in units of Z, to *margin. */
static int32_t inverse_cdf(const double *r, int32_t V, double Z, double u,
                           double *margin, int *flags) {
    double target = u * Z;
    double c = 0.0;
    for (int32_t v = 0; v < V; ++v) {
        double prev = c;
        c += r[v];
        if (c > target) {
            double a = (target - prev) / Z, b = (c - target) / Z;
            *margin = a < b ? a : b;
            return v;
        }
    }
    /* rounding left u*Z at or above the total: largest v with mass */
    *flags |= OR_FLAG_CDF_FALLBACK;
    *margin = 0.0;
    for (int32_t v = V - 1; v >= 0; --v)
        if (r[v] > 0.0) return v;
    return V - 1;
}

/* Normalised running sum of the draw's weights, c[v] = (r_0 + .. + r_v) / Z,
 * summed in the same ascending order as inverse_cdf (for validity checks of
 * draws that land within the flag margin of a boundary). */
static void cumulative(const double *r, int32_t V, double Z, double *c) {
    double s = 0.0;
    for (int32_t v = 0; v < V; ++v) {
        s += r[v];
        c[v] = s / Z;
    }
}

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }


/* One sequence of the verification pass.
 *  zt: K+1 target rows, row j at zt + j*t_stride elements.
 *  zd: K draft rows (NULL allowed in greedy / FLy mode).
 *  x:  K draft tokens.  u: K+1 uniforms (NULL allowed in greedy / FLy mode).
 * Scratch: p, q, r of V doubles each. */
static void verify_one(int32_t K, int32_t Kb, double sc, double top_p, int32_t V, int dtype, int mode,
                       const void *zt, int64_t t_stride, const void *zd, int64_t d_stride,
                       const int32_t *x, const float *u, double fly_theta, int32_t fly_window,
                       const double *est, int32_t *out_tokens, int32_t *acc_len,
                       double *pos_stats, double *conf, double *feature,
                       double *margin_acc, double *margin_cdf, double *cdf_out, int *flags,
                       const int32_t *force, const int32_t *nshift, double *margin_pos, int32_t *natural_pos,
                       int32_t *nuc_doubt, double *p, double *q, double *r, OrKey *keys) {
    const size_t es = dtype == OR_F32 ? 4 : 2;
    const char *tbase = (const char *)zt;
    const char *dbase = (const char *)zd;
    double mg = INFINITY;      /* acceptance (and FLy gate) margin */
    double mn = INFINITY;      /* nucleus boundary margin (top-p), folded into mg at the end */
    double mc = INFINITY;      /* margin of the final inverse-CDF draw */
    int fl = 0;
    /* boundary override of row (target j: j; draft j: K+1+j), 0 = natural */
#define OR_SHIFT_T(j) (nshift ? nshift[(j)] : 0)
#define OR_SHIFT_D(j) (nshift ? nshift[K + 1 + (j)] : 0)
    for (int32_t j = 0; j < K; ++j) {
        if (margin_pos) margin_pos[j] = INFINITY;
        if (natural_pos) natural_pos[j] = -1;
    }
    if (nuc_doubt)
        for (int32_t j = 0; j < 2 * K + 1; ++j) nuc_doubt[j] = 0;

    /* Per-position statistics (written whether or not the position is reached).
     * Only the first Kb drafts were submitted for verification (Kb = K unless
     * the batch was pruned, [AV] "Antecedentes": a subset of the drafts is
     * verified); target rows after Kb and draft rows from Kb on were never
     * computed and stay NaN. */
    if (pos_stats)
        for (int32_t j = 0; j < 4 * (K + 1); ++j) pos_stats[j] = NAN;
    for (int32_t j = 0; j < K; ++j) {
        if (feature) feature[j] = NAN;
        if (conf) conf[j] = NAN;
    }
    for (int32_t j = 0; j <= Kb; ++j) {
        const void *trow = tbase + (size_t)j * (size_t)t_stride * es;
        int ok;
        double zs_t, zs_d;
        int dbt = 0;
        double lse_t = processed_row(trow, dtype, V, sc, top_p, OR_SHIFT_T(j), p, keys, &ok, &zs_t, &mn,
                                     j < Kb ? x[j] : -1, &dbt);
        if (nuc_doubt) nuc_doubt[j] = dbt;
        if (!ok) fl |= OR_FLAG_BAD_ROW;
        double h = norm_entropy(p, V);
        double lr = NAN, f = NAN;
        if (j < Kb && zd) {
            const void *drow = dbase + (size_t)j * (size_t)d_stride * es;
            int okd;
            double lse_d = processed_row(drow, dtype, V, sc, top_p, OR_SHIFT_D(j), q, keys, &okd, &zs_d, &mn,
                                         x[j], &dbt);
            if (nuc_doubt) nuc_doubt[K + 1 + j] = dbt;
            if (!okd) fl |= OR_FLAG_BAD_ROW;
            int32_t amax_d = argmax_row(drow, dtype, V);
            f = logit_qmax(q, V, amax_d, &fl);
            /* ln p(x) - ln q(x); a token outside a nucleus has probability 0 */
            const double zx = logit_at(trow, dtype, x[j]), qx = logit_at(drow, dtype, x[j]);
            lr = (zx >= zs_t ? sc * zx - lse_t : -INFINITY) - (qx >= zs_d ? sc * qx - lse_d : -INFINITY);
            if (feature) feature[j] = f;
            /* [AV] "Puntuar la Distribución": confidence = sigmoid of the
             * shared slope times logit(q_max) plus the position's intercept;
             * params = [omega, beta_1 .. beta_K], draft position j uses
             * beta_{j+1}. */
            if (conf && est) conf[j] = sigmoid(est[0] * f + est[1 + j]);
        }
        if (pos_stats) {
            pos_stats[4 * j + 0] = lse_t;
            pos_stats[4 * j + 1] = h;
            pos_stats[4 * j + 2] = lr;
            pos_stats[4 * j + 3] = f;
        }
    }

    int32_t n = 0, token = -1;
    if (mode == OR_STOCHASTIC) {
        /* [SD] "Математика верификации": accept x_i with probability 1 when
         * p(x_i) >= q(x_i), else with probability p(x_i)/q(x_i); i.e. accept
         * iff u_i < min(1, p(x_i)/q(x_i)). [SD] step 4: stop at the first
         * rejection and draw the correction from norm(max(0, p - q)). */
        int rejected = 0;
        for (int32_t i = 0; i < Kb; ++i) {
            const void *trow = tbase + (size_t)i * (size_t)t_stride * es;
            const void *drow = dbase + (size_t)i * (size_t)d_stride * es;
            int ok;
            double zs;
            double mni = INFINITY;   /* nucleus margins of this position's two rows */
            processed_row(trow, dtype, V, sc, top_p, OR_SHIFT_T(i), p, keys, &ok, &zs, &mni, x[i], NULL);
            processed_row(drow, dtype, V, sc, top_p, OR_SHIFT_D(i), q, keys, &ok, &zs, &mni, x[i], NULL);
            mn = dmin(mn, mni);
            double px = p[x[i]], qx = q[x[i]];
            double acc;
            if (qx > 0.0) {
                acc = dmin(1.0, px / qx);
            } else {
                /* q(x) = 0: the ratio is +inf if p(x) > 0, else the draft is
                 * rejected (reading; the pages assume x ~ q). */
                fl |= OR_FLAG_Q_ZERO;
                acc = px > 0.0 ? 1.0 : 0.0;
            }
            mg = dmin(mg, fabs((double)u[i] - acc));
            int take = (double)u[i] < acc;
            /* per-position report: the margin of this decision (with its
             * rows' nucleus margins) and the decision the rule takes */
            if (margin_pos) margin_pos[i] = dmin(fabs((double)u[i] - acc), mni);
            if (natural_pos) natural_pos[i] = take;
            /* a caller-imposed decision (parity checks of a computation that
             * decided a position in doubt the other way) */
            if (force && force[i] >= 0) take = force[i] != 0;
            if (take) { ++n; continue; }
            double Z = 0.0;
            for (int32_t v = 0; v < V; ++v) {
                r[v] = p[v] > q[v] ? p[v] - q[v] : 0.0;
                Z += r[v];
            }
            if (!(Z > 0.0)) {
                /* only reachable through rounding: draw from p itself */
                fl |= OR_FLAG_Z_ZERO;
                Z = 0.0;
                for (int32_t v = 0; v < V; ++v) { r[v] = p[v]; Z += r[v]; }
            }
            token = inverse_cdf(r, V, Z, (double)u[K], &mc, &fl);
            if (cdf_out) cumulative(r, V, Z, cdf_out);
            rejected = 1;
            break;
        }
        if (!rejected) {
            /* Bonus token after Kb acceptances (reading: a draw from the target's
             * row Kb, standard for rejection-sampling verification; the final
             * draw always uses u[K]). */
            const void *trow = tbase + (size_t)Kb * (size_t)t_stride * es;
            int ok;
            double zs;
            processed_row(trow, dtype, V, sc, top_p, OR_SHIFT_T(Kb), p, keys, &ok, &zs, &mn, -1, NULL);
            double Z = 0.0;
            for (int32_t v = 0; v < V; ++v) Z += p[v];
            token = inverse_cdf(p, V, Z, (double)u[K], &mc, &fl);
            if (cdf_out) cumulative(p, V, Z, cdf_out);
        }
    } else if (mode == OR_GREEDY) {
        /* Exact match: accept x_i iff it is the target's top prediction
         * ([FLy] section 1; [SD] "Проверка результата", greedy output is
         * reproducible). The correction is the target's argmax at the stop. */
        n = Kb;
        for (int32_t i = 0; i < Kb; ++i) {
            const void *trow = tbase + (size_t)i * (size_t)t_stride * es;
            int32_t a = argmax_row(trow, dtype, V);
            if (x[i] != a) { n = i; token = a; break; }
        }
        if (n == Kb) token = argmax_row(tbase + (size_t)Kb * (size_t)t_stride * es, dtype, V);
    } else {
        /* [FLy] 2.A: a deviation at j (x_j differs from the target's argmax)
         * is rejected at once when the target's normalised entropy h_j < theta;
         * when h_j >= theta it is deferred: accepted if none of the next W draft
         * positions deviates, rejected retroactively if one does, and rejected
         * conservatively if the window does not fit inside the draft. */
        n = Kb;
        for (int32_t j = 0; j < Kb; ++j) {
            const void *trow = tbase + (size_t)j * (size_t)t_stride * es;
            int32_t a = argmax_row(trow, dtype, V);
            if (x[j] == a) continue;               /* no deviation: accept j */
            int ok;
            double zs;
            double mnj = INFINITY;
            processed_row(trow, dtype, V, sc, top_p, OR_SHIFT_T(j), p, keys, &ok, &zs, &mnj, -1, NULL);
            mn = dmin(mn, mnj);
            double h = norm_entropy(p, V);
            mg = dmin(mg, fabs(h - fly_theta));
            int open = h >= fly_theta;
            if (margin_pos) margin_pos[j] = dmin(fabs(h - fly_theta), mnj);
            if (natural_pos) natural_pos[j] = open;
            if (force && force[j] >= 0) open = force[j] != 0;   /* caller-imposed gate */
            int reject;
            if (!open) {
                reject = 1;                        /* confident target */
            } else if (j + fly_window > Kb - 1) {
                reject = 1;                        /* window past the draft end */
            } else {
                reject = 0;
                for (int32_t k = j + 1; k <= j + fly_window; ++k) {
                    const void *krow = tbase + (size_t)k * (size_t)t_stride * es;
                    if (x[k] != argmax_row(krow, dtype, V)) { reject = 1; break; }
                }
            }
            if (reject) { n = j; token = a; break; }
        }
        if (n == Kb) token = argmax_row(tbase + (size_t)Kb * (size_t)t_stride * es, dtype, V);
    }

    /* Writeback ([SD] step 4): the accepted prefix, then the correction or
     * bonus token; unused slots are -1. */
    for (int32_t j = 0; j <= K; ++j) out_tokens[j] = -1;
    for (int32_t j = 0; j < n; ++j) out_tokens[j] = x[j];
    out_tokens[n] = token;
    *acc_len = n;
    if (mn < INFINITY) fl |= OR_FLAG_NUCLEUS;
    mg = dmin(mg, mn);
    if (margin_acc) *margin_acc = mg;
    if (margin_cdf) *margin_cdf = mc;
    if (flags) *flags = fl;
#undef OR_SHIFT_T
#undef OR_SHIFT_D
}

/* Full verification over B sequences. Layouts (row-major, elements):
 *  zt [B][K+1][t_stride] (first V used), zd [B][K][d_stride], x [B][K],
 *  u [B][K+1], out_tokens [B][K+1], accepted_len [B],
 *  pos_stats [B][K+1][4] = (lse_t, h_t, log_ratio, f) or NULL,
 *  est [K+1] or NULL, conf [B][K] or NULL, feature [B][K] or NULL,
 *  margin_acc [B] or NULL: smallest acceptance margin |u_i - min(1, p/q)| over
 *    the tested positions (FLy: |h_j - theta| over the gates evaluated),
 *  margin_cdf [B] or NULL: distance of u to the nearer boundary of the drawn
 *    token's interval, in units of Z (stochastic mode; +inf otherwise),
 *  cdf [B][V] or NULL: normalised running sum of the final draw's weights
 *    (stochastic mode; untouched otherwise),
 *  flags [B] or NULL (OR_FLAG_* bits),
 *  draft_len [B] or NULL: drafts submitted for verification per sequence,
 *    in [0, K] (NULL: all K). Sequence b verifies drafts 0..draft_len[b]-1
 *    against target rows 0..draft_len[b]; the rest of its outputs are NaN/-1,
 *  inv_temp [B] or NULL: per-sequence inverse sampling temperature (> 0).
 *    Verification then runs on the temperature-processed distributions
 *    p = softmax(z / T) and q = softmax(y / T) of sequence b ([AV]
 *    "Benchmarks": the pages serve at a sampling temperature; speculative
 *    sampling is lossless for whatever p and q it is given). Argmax is
 *    unchanged; lse, entropy, the log-ratio and logit(q_max) are those of
 *    the processed distributions. NULL: temperature 1.
 *  top_p in (0, 1]: with top_p < 1 every row's processed distribution is
 *    further truncated to its nucleus (see nucleus()) and renormalised,
 *    before every use; the nucleus boundary's margin (see nucleus()) joins
 *    margin_acc.
 * Per-position report and overrides, for parity checks of a computation
 * that decided a position in doubt the other way (all may be NULL):
 *  margin_pos [B][K]: the margin of each decision the scan takes
 *    (stochastic: |u_i - min(1, p/q)|; FLy: |h_j - theta| at each gate
 *    evaluated), with the nucleus margins of the position's rows under
 *    top-p; +inf at positions not decided,
 *  natural_pos [B][K]: the decision the rule takes there (1 accept / gate
 *    open, 0 reject / gate closed), -1 at positions not decided,
 *  force [B][K]: -1 follows the rule; 0 or 1 imposes that decision at the
 *    position if the scan reaches it (margin_pos and natural_pos still
 *    report the rule's own),
 *  nshift [B][2K+1] (rows: target 0..K, then draft 0..K-1): 0 the natural
 *    nucleus boundary, -1 the group at z* dropped, +1 the next group down
 *    added (top-p only),
 *  nuc_doubt [B][2K+1]: which way each verified row's nucleus boundary is in
 *    doubt (bit 1: the group at z* may be dropped; bit 2: the next group
 *    down may be added).
 * nthreads > 0 sets the OpenMP thread count. Returns 0, or -1 on bad args. */
int oracle_verify(int32_t B, int32_t K, int32_t V, int dtype, int mode,
                  const void *zt, int64_t t_stride, const void *zd, int64_t d_stride,
                  const int32_t *x, const float *u, double fly_theta, int32_t fly_window,
                  const double *est, int32_t *out_tokens, int32_t *accepted_len,
                  double *pos_stats, double *conf, double *feature,
                  double *margin_acc, double *margin_cdf, double *cdf, int32_t *flags,
                  const int32_t *draft_len, const float *inv_temp, double top_p,
                  const int32_t *force, const int32_t *nshift, double *margin_pos, int32_t *natural_pos,
                  int32_t *nuc_doubt, int nthreads) {
    if (B < 0 || K < 1 || V < 2 || !zt || !x || !out_tokens || !accepted_len) return -1;
    if (!(top_p > 0.0 && top_p <= 1.0)) return -1;
    if (inv_temp)
        for (int32_t b = 0; b < B; ++b)
            if (!(inv_temp[b] > 0.0f) || isinf(inv_temp[b])) return -1;
    if (draft_len)
        for (int32_t b = 0; b < B; ++b)
            if (draft_len[b] < 0 || draft_len[b] > K) return -1;
    if (mode == OR_STOCHASTIC && (!zd || !u)) return -1;
    if (t_stride <= 0) t_stride = V;
    if (d_stride <= 0) d_stride = V;
    const size_t es = dtype == OR_F32 ? 4 : 2;
    int bad = 0;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : 1)
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)V);
        double *q = (double *)malloc(sizeof(double) * (size_t)V);
        double *r = (double *)malloc(sizeof(double) * (size_t)V);
        OrKey *keys = top_p < 1.0 ? (OrKey *)malloc(sizeof(OrKey) * (size_t)V) : NULL;
        if (!p || !q || !r || (top_p < 1.0 && !keys)) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(static)
            for (int32_t b = 0; b < B; ++b) {
                int fl = 0;
                verify_one(K, draft_len ? draft_len[b] : K, inv_temp ? (double)inv_temp[b] : 1.0, top_p, V, dtype,
                           mode,
                           (const char *)zt + (size_t)b * (size_t)(K + 1) * (size_t)t_stride * es, t_stride,
                           zd ? (const char *)zd + (size_t)b * (size_t)K * (size_t)d_stride * es : NULL, d_stride,
                           x + (size_t)b * K, u ? u + (size_t)b * (K + 1) : NULL, fly_theta, fly_window,
                           est, out_tokens + (size_t)b * (K + 1), accepted_len + b,
                           pos_stats ? pos_stats + (size_t)b * (K + 1) * 4 : NULL,
                           conf ? conf + (size_t)b * K : NULL,
                           feature ? feature + (size_t)b * K : NULL,
                           margin_acc ? margin_acc + b : NULL, margin_cdf ? margin_cdf + b : NULL,
                           cdf ? cdf + (size_t)b * (size_t)V : NULL, &fl,
                           force ? force + (size_t)b * K : NULL,
                           nshift ? nshift + (size_t)b * (2 * K + 1) : NULL,
                           margin_pos ? margin_pos + (size_t)b * K : NULL,
                           natural_pos ? natural_pos + (size_t)b * K : NULL,
                           nuc_doubt ? nuc_doubt + (size_t)b * (2 * K + 1) : NULL, p, q, r, keys);
                if (flags) flags[b] = fl;
            }
        }
        free(p);
        free(q);
        free(r);
        free(keys);
    }
    return bad ? -1 : 0;
}

/* Confidence features of draft rows only: feature[b][i] = logit(q_max) of
 * draft row (b, i) and conf[b][i] = sigmoid(omega * feature + beta_{i+1})
 * ([AV] "Puntuar la Distribución"). conf may be NULL; est is needed for conf. */
int oracle_confidence(int32_t B, int32_t K, int32_t V, int dtype, const void *zd, int64_t d_stride,
                      const double *est, double *feature, double *conf, int32_t *flags,
                      int nthreads) {
    if (B < 0 || K < 1 || V < 2 || !zd || !feature) return -1;
    if (conf && !est) return -1;
    if (d_stride <= 0) d_stride = V;
    const size_t es = dtype == OR_F32 ? 4 : 2;
    int bad = 0;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : 1)
    {
        double *q = (double *)malloc(sizeof(double) * (size_t)V);
        if (!q) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(static)
            for (int32_t b = 0; b < B; ++b) {
                int fl = 0;
                for (int32_t i = 0; i < K; ++i) {
                    const void *drow = (const char *)zd + ((size_t)b * K + i) * (size_t)d_stride * es;
                    int ok;
                    softmax_row(drow, dtype, V, 1.0, q, &ok);
                    if (!ok) fl |= OR_FLAG_BAD_ROW;
                    double f = logit_qmax(q, V, argmax_row(drow, dtype, V), &fl);
                    feature[(size_t)b * K + i] = f;
                    if (conf) conf[(size_t)b * K + i] = sigmoid(est[0] * f + est[1 + i]);
                }
                if (flags) flags[b] = fl;
            }
        }
        free(q);
    }
    return bad ? -1 : 0;
}

/* One online update of the acceptance estimator ([AV] "Ajuste de los
 * Coeficientes").
 * Labels: only drafts up to and including the first rejection are eligible;
 * y_i = 1 for i < n_acc, y_{n_acc} = 0 when n_acc < K, later positions carry
 * no label. With pruned verification (draft_len, NULL = K for all) only the
 * K_b verified drafts of sequence b can carry a label: y_{n_acc} = 0 only
 * when n_acc < K_b.
 * Step (reading: the pages solve an IRLS Newton system over N steps; this
 * entry point takes one plain gradient step of size lr on the mean log-loss
 * over the batch's eligible labels):
 *   z = omega * f_i + beta_{i+1},  e = sigmoid(z) - y,
 *   g_omega = (1/N) sum e * f_i,   g_beta_k = (1/N) sum_{i = k-1} e,
 *   params -= lr * g.
 * N = 0 leaves params unchanged. grad_out [K+1] and count_out [K+1]
 * (count_out[0] = N, count_out[k] = labels at draft position k-1) may be NULL.
 * The loss is accumulated in ascending (b, i) order. */
int oracle_estimator_update(int32_t B, int32_t K, const double *feature, const int32_t *accepted_len,
                            const int32_t *draft_len, double *params, double lr, double *grad_out,
                            int64_t *count_out) {
    if (B < 0 || K < 1 || !feature || !accepted_len || !params) return -1;
    double *g = (double *)calloc((size_t)K + 1, sizeof(double));
    int64_t *cnt = (int64_t *)calloc((size_t)K + 1, sizeof(int64_t));
    if (!g || !cnt) { free(g); free(cnt); return -1; }
    for (int32_t b = 0; b < B; ++b) {
        int32_t n = accepted_len[b];
        int32_t kb = draft_len ? draft_len[b] : K;
        if (kb < 0 || kb > K || n < 0 || n > kb) { free(g); free(cnt); return -1; }
        int32_t last = n < kb ? n : kb - 1;  /* last eligible (verified) position */
        for (int32_t i = 0; i <= last; ++i) {
            double y = i < n ? 1.0 : 0.0;
            double f = feature[(size_t)b * K + i];
            double e = sigmoid(params[0] * f + params[1 + i]) - y;
            g[0] += e * f;
            g[1 + i] += e;
            cnt[0] += 1;
            cnt[1 + i] += 1;
        }
    }
    int64_t N = cnt[0];
    for (int32_t k = 0; k <= K; ++k) {
        double gk = N > 0 ? g[k] / (double)N : 0.0;
        if (grad_out) grad_out[k] = gk;
        if (count_out) count_out[k] = cnt[k];
    }
    if (N > 0)
        for (int32_t k = 0; k <= K; ++k) params[k] -= lr * (g[k] / (double)N);
    free(g);
    free(cnt);
    return 0;
}

/* Mean log-loss of the same eligible labels, for finite-difference checks of
 * the update ([AV] "Otras Características Consideradas": log-loss is the mean
 * negative log-likelihood of the predicted acceptance probability). */
double oracle_estimator_loss(int32_t B, int32_t K, const double *feature, const int32_t *accepted_len,
                             const int32_t *draft_len, const double *params) {
    double L = 0.0;
    int64_t N = 0;
    for (int32_t b = 0; b < B; ++b) {
        int32_t n = accepted_len[b];
        int32_t kb = draft_len ? draft_len[b] : K;
        int32_t last = n < kb ? n : kb - 1;
        for (int32_t i = 0; i <= last; ++i) {
            double s = sigmoid(params[0] * feature[(size_t)b * K + i] + params[1 + i]);
            L += i < n ? -log(s) : -log(1.0 - s);
            ++N;
        }
    }
    return N > 0 ? L / (double)N : 0.0;
}

/* IRLS refit of the acceptance estimator ([AV] "Ajuste de los Coeficientes").
 * The coefficients stay fixed during a round of decoding steps; each step
 * adds the gradient and Hessian of the summed log-loss of its eligible labels
 * (the labelling of oracle_estimator_update) to the round's totals, and the
 * refit at the end of the round solves H d = g and moves every coefficient by
 * its step scaled by n / (n + c), n being the labels behind that coefficient.
 * With x = (f_i, one-hot of position i) the regressors of a label, s =
 * sigmoid(theta . x), e = s - y and w = s (1 - s):
 *   g += e x,   H += w x x^T,   n_0 += 1,   n_{1+i} += 1.
 * g [K+1], H [(K+1)*(K+1)] row-major and n [K+1] are added to (the caller
 * zeroes them at the start of a round). Labels are visited in ascending
 * (b, i) order. */
int oracle_irls_accumulate(int32_t B, int32_t K, const double *feature, const int32_t *accepted_len,
                           const int32_t *draft_len, const double *params, double *g, double *H, int64_t *n) {
    if (B < 0 || K < 1 || !feature || !accepted_len || !params || !g || !H || !n) return -1;
    const int32_t D = K + 1;
    double *x = (double *)calloc((size_t)D, sizeof(double));
    if (!x) return -1;
    for (int32_t b = 0; b < B; ++b) {
        int32_t na = accepted_len[b];
        int32_t kb = draft_len ? draft_len[b] : K;
        if (kb < 0 || kb > K || na < 0 || na > kb) { free(x); return -1; }
        int32_t last = na < kb ? na : kb - 1;
        for (int32_t i = 0; i <= last; ++i) {
            double y = i < na ? 1.0 : 0.0;
            for (int32_t j = 0; j < D; ++j) x[j] = 0.0;
            x[0] = feature[(size_t)b * K + i];
            x[1 + i] = 1.0;
            double z = 0.0;
            for (int32_t j = 0; j < D; ++j) z += params[j] * x[j];
            double sg = sigmoid(z);
            double e = sg - y, w = sg * (1.0 - sg);
            for (int32_t r = 0; r < D; ++r) {
                g[r] += e * x[r];
                for (int32_t c = 0; c < D; ++c) H[(size_t)r * D + c] += w * x[r] * x[c];
            }
            n[0] += 1;
            n[1 + i] += 1;
        }
    }
    free(x);
    return 0;
}

/* The refit at the end of a round. Coefficients without labels (n == 0) keep
 * their value and leave the system. The rest solve H d = g by Gaussian
 * elimination without pivoting (H is symmetric positive semi-definite),
 * eliminating the intercepts first and the slope last. Reading where the
 * pages are silent: if the slope's final pivot is not positive (below 1e-12 of
 * its diagonal entry, i.e. the slope is not determined by this round's data,
 * as when every feature is equal within each position) the slope is held
 * (d_0 = 0) and the intercepts are solved with it fixed. Then every step is
 * damped, d_k *= n_k / (n_k + c), and params -= d. A round without labels
 * changes nothing. step_out [K+1] (may be NULL) receives the applied step. */
int oracle_irls_refit(int32_t K, const double *g, const double *H, const int64_t *n, double damping,
                      double *params, double *step_out) {
    if (K < 1 || !g || !H || !n || !params || !(damping >= 0.0)) return -1;
    const int32_t D = K + 1;
    double *d = (double *)calloc((size_t)D, sizeof(double));
    int32_t *ord = (int32_t *)malloc(sizeof(int32_t) * (size_t)D);
    double *A = (double *)malloc(sizeof(double) * (size_t)D * (size_t)D);
    double *rhs = (double *)malloc(sizeof(double) * (size_t)D);
    if (!d || !ord || !A || !rhs) { free(d); free(ord); free(A); free(rhs); return -1; }
    int32_t m = 0;                                 /* unknowns: labelled intercepts, then the slope */
    for (int32_t k = 1; k < D; ++k)                /* (an intercept whose labels all saturated, */
        if (n[k] > 0 && H[(size_t)k * D + k] > 0.0) ord[m++] = k;   /* w = 0, is held too) */
    if (n[0] > 0) ord[m++] = 0;
    for (int32_t r = 0; r < m; ++r) {
        rhs[r] = g[ord[r]];
        for (int32_t c = 0; c < m; ++c) A[(size_t)r * m + c] = H[(size_t)ord[r] * D + ord[c]];
    }
    int32_t msolve = m;
    for (int32_t p = 0; p < m; ++p) {                /* forward elimination */
        double piv = A[(size_t)p * m + p];
        if (ord[p] == 0 && !(piv > 1e-12 * H[0])) { msolve = p; break; }   /* slope held */
        if (!(piv > 0.0)) { free(d); free(ord); free(A); free(rhs); return -2; }
        for (int32_t r = p + 1; r < m; ++r) {
            double f = A[(size_t)r * m + p] / piv;
            for (int32_t c = p; c < m; ++c) A[(size_t)r * m + c] -= f * A[(size_t)p * m + c];
            rhs[r] -= f * rhs[p];
        }
    }
    for (int32_t p = msolve - 1; p >= 0; --p) {      /* back substitution */
        double acc = rhs[p];
        for (int32_t c = p + 1; c < msolve; ++c) acc -= A[(size_t)p * m + c] * d[ord[c]];
        d[ord[p]] = acc / A[(size_t)p * m + p];
    }
    for (int32_t k = 0; k < D; ++k) {
        double nk = (double)n[k];
        double step = nk > 0.0 ? d[k] * (nk / (nk + damping)) : 0.0;
        params[k] -= step;
        if (step_out) step_out[k] = step;
    }
    free(d); free(ord); free(A); free(rhs);
    return 0;
}

/* Adaptive-verification pruning and budget ([AV] "Otras Características
 * Consideradas": survival is the running product of the confidences along
 * each sequence's drafts; the drafts are ranked by survival over the whole
 * batch; the budget maximises the expected emitted tokens, the number of
 * requests plus the sum of the top-k survivals, divided by the measured cost
 * of drafting and verifying k tokens; the top `budget` drafts are verified).
 * Readings: survival is an fp32 running product in ascending position (the
 * precision that decides the ranking on the GPU too); ties in survival rank
 * by ascending flat index b*K + i, so each sequence's winners are a prefix
 * of its drafts; NaN survival ranks last. The top-k sum is kept in fixed
 * point: each positive survival is rounded to the nearest multiple of 2^-32
 * and the multiples are added as integers, so S_k is exact and the same in
 * any order. The decision is taken in fp32 (the pages fix no precision; the
 * GPU's): num_k = (float)(B * 2^32 + S_k), cost_k = draft_cost[k] +
 * verify_cost[k] in fp32, objective_k = num_k / cost_k (each step correctly
 * rounded), reported times 2^-32; a cost that is not positive makes its k
 * ineligible; the first k of the maximum wins (k = 0 if none is eligible).
 * Every quantity the decision reads is computed identically on any machine,
 * so the budget needs no knife-edge allowance.
 * conf [B][K] f32, draft_cost and verify_cost [B*K+1] f32 (k = 0..B*K).
 * Outputs: draft_len [B], *budget, survival [B][K] f32 (may be NULL),
 * objective [B*K+1] f32 (may be NULL; -inf where ineligible), *gap (may be
 * NULL): the relative gap between the best and the second-best objective. */
typedef struct {
    float key;     /* survival (NaN replaced by -1) */
    int32_t idx;   /* flat index b*K + i */
} AvRank;

static int av_cmp(const void *pa, const void *pb) {
    const AvRank *a = (const AvRank *)pa, *b = (const AvRank *)pb;
    if (a->key > b->key) return -1;
    if (a->key < b->key) return 1;
    return a->idx < b->idx ? -1 : (a->idx > b->idx ? 1 : 0);
}

int oracle_av_budget(int32_t B, int32_t K, const float *conf, const float *draft_cost, const float *verify_cost,
                     int32_t *draft_len, int32_t *budget, float *survival, float *objective, double *gap) {
    if (B < 0 || K < 1 || (B > 0 && !conf) || !draft_cost || !verify_cost || !draft_len || !budget) return -1;
    const int64_t N = (int64_t)B * K;
    AvRank *rk = (AvRank *)malloc(sizeof(AvRank) * (size_t)(N > 0 ? N : 1));
    float *obj = (float *)malloc(sizeof(float) * (size_t)(N + 1));
    if (!rk || !obj) { free(rk); free(obj); return -1; }
    for (int32_t b = 0; b < B; ++b) {
        float sv = 1.0f;
        for (int32_t i = 0; i < K; ++i) {
            sv = sv * conf[(size_t)b * K + i];
            if (survival) survival[(size_t)b * K + i] = sv;
            rk[(size_t)b * K + i].key = sv == sv ? sv : -1.0f;   /* NaN ranks last */
            rk[(size_t)b * K + i].idx = b * K + i;
        }
    }
    qsort(rk, (size_t)N, sizeof(AvRank), av_cmp);
    uint64_t S = 0;                            /* sum of the top k, in units of 2^-32 */
    float best = -INFINITY, second = -INFINITY;
    int64_t kbest = 0;
    for (int64_t k = 0; k <= N; ++k) {
        if (k > 0 && rk[k - 1].key > 0.0f) S += (uint64_t)llrint((double)rk[k - 1].key * 4294967296.0);
        volatile float c = draft_cost[k] + verify_cost[k];          /* fp32 add, no contraction */
        volatile float num = (float)((uint64_t)B * 4294967296ull + S);
        volatile float q = num / c;
        float o = c > 0.0f ? q * (1.0f / 4294967296.0f) : -INFINITY;
        obj[k] = o;
        if (o > best) { second = best; best = o; kbest = k; }
        else if (o > second) second = o;
    }
    for (int32_t b = 0; b < B; ++b) draft_len[b] = 0;
    if (best == -INFINITY) kbest = 0;
    for (int64_t j = 0; j < kbest; ++j) draft_len[rk[j].idx / K] += 1;
    *budget = (int32_t)kbest;
    if (objective) for (int64_t k = 0; k <= N; ++k) objective[k] = obj[k];
    if (gap) *gap = (best > -INFINITY && second > -INFINITY) ? ((double)best - second) / fabs((double)best) : INFINITY;
    free(rk); free(obj);
    return 0;
}

/* N-gram (prompt-lookup) drafting ("Speculative Decoding: как черновая модель
 * ускоряет генерацию LLM без потери качества", section "N-gram (prompt
 * lookup)"; the FLy page's "Aceleração Multinível" drafts this way): the
 * drafts are read from the context itself, the tokens that followed an
 * earlier occurrence of the context's last n tokens. Readings (the pages do
 * not say): n runs from n_max down to n_min and the first n with a match
 * wins (the longest match); among its matches the most recent occurrence is
 * taken (the one that ends last, before the context's end); up to K tokens
 * that follow it are proposed (fewer if the context ends first); no match
 * proposes nothing.
 * ctx [B][ld] int32 (sequence b's context is ctx[b][0 .. len[b]-1]),
 * draft_tokens [B][K] out (-1 past draft_len), draft_len [B] out.
 * 1 <= n_min <= n_max; 0 <= len[b] <= ld. */
int oracle_ngram_draft(int32_t B, int32_t ld, const int32_t *ctx, const int32_t *len, int32_t n_min,
                       int32_t n_max, int32_t K, int32_t *draft_tokens, int32_t *draft_len) {
    if (B < 0 || ld < 0 || K < 1 || n_min < 1 || n_max < n_min || !draft_tokens || !draft_len) return -1;
    if (B > 0 && (!ctx || !len)) return -1;
    for (int32_t b = 0; b < B; ++b) {
        const int32_t *c = ctx + (size_t)b * ld;
        const int32_t L = len[b];
        if (L < 0 || L > ld) return -1;
        int32_t start = -1;                   /* first proposed token's index */
        for (int32_t n = n_max; n >= n_min && start < 0; --n) {
            if (n > L - 1) continue;          /* the query and an earlier copy must fit */
            for (int32_t e = L - 1; e >= n; --e) {        /* occurrence c[e-n .. e-1], follow-up from e */
                int32_t t = 0;
                while (t < n && c[e - n + t] == c[L - n + t]) ++t;
                if (t == n) { start = e; break; }
            }
        }
        int32_t m = 0;
        for (int32_t k = 0; k < K; ++k) {
            int32_t tok = -1;
            if (start >= 0 && start + k < L) { tok = c[start + k]; ++m; }
            draft_tokens[(size_t)b * K + k] = tok;
        }
        draft_len[b] = m;
    }
    return 0;
}

/* Row statistics of `rows` rows of V logits each (row r at z + r*stride):
 * lse, normalised entropy, argmax, logit(q_max). Any output may be NULL. */
int oracle_row_stats(int64_t rows, int32_t V, int dtype, const void *z, int64_t stride,
                     double *lse, double *entropy, int32_t *argmax, double *fq, int nthreads) {
    if (rows < 0 || V < 2 || !z) return -1;
    if (stride <= 0) stride = V;
    const size_t es = dtype == OR_F32 ? 4 : 2;
    int bad = 0;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : 1)
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)V);
        if (!p) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t r = 0; r < rows; ++r) {
                const void *row = (const char *)z + (size_t)r * (size_t)stride * es;
                int ok, fl = 0;
                double l = softmax_row(row, dtype, V, 1.0, p, &ok);
                int32_t a = argmax_row(row, dtype, V);
                if (lse) lse[r] = ok ? l : NAN;
                if (entropy) entropy[r] = ok ? norm_entropy(p, V) : NAN;
                if (argmax) argmax[r] = a;
                if (fq) fq[r] = ok ? logit_qmax(p, V, a, &fl) : NAN;
            }
        }
        free(p);
    }
    return bad ? -1 : 0;
}
