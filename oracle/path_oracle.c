/*
 * fp64 CPU oracle for PaTH causal attention — TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
 * leg may load this library.  It shares no code, header, table or constant with
 * the CUDA library in attention_causal_attn_fwd_gb300/csrc; neither side
 * includes or links the other.
 *
 * Source of the definitions: "Resumo Técnico: Atenção PaTH"
 * (gist.science/pt/paper/2505.16381):
 *   - §2 "Mecanismo Central", attention-logit equation:
 *         A_ij ∝ exp( k_j^T (prod_{s=j+1}^{i} H_s) q_i ),  j <= i,
 *   - §2 "Mecanismo Central", transition equation:  H_s = I - beta_s w_s w_s^T,
 *   - §2 "Extensões: PaTH-FoX": FoX's additive, data-dependent forget gates on
 *     top of the PaTH logits,
 *   - §3 "Treinamento e Inferência Eficientes", "Inferência" bullet: at decode
 *     time the historical keys are updated in place with the current step's
 *     transition.
 *
 * Readings taken where the page is silent:
 *   - the product is ascending, H_{j+1} H_{j+2} ... H_i (the only order under
 *     which the in-place key update of the "Inferência" bullet is exact);
 *   - the product is empty (= I) at j = i, and j = i takes part in the softmax;
 *   - logits are multiplied by `scale` after transport; the FoX bias
 *     sum_{s=j+1..i} log f_s is added unscaled to the scaled logit;
 *   - decode step t first applies H_t to every cached key, then appends the
 *     new key k_t untransported, then attends over all keys.
 *
 * The walk: s_ij = k_j^T H_{j+1} ... H_i q_i is evaluated by walking the query
 * backwards: u <- q_i; for j = i, i-1, ..., 0 { s_ij = k_j . u; u <- H_j u }.
 * No blocking, no UT transform, no fusion: one row at a time, in fp64.
 *
 * parity pins: see tests/test_oracle.py (dense product, beta = 0 library
 * attention, closed forms, orthogonality, decode = prefill, hand-derived
 * golden values).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int path_oracle_threads(void) {
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

/* u <- (I - beta w w^T) u  (one Householder-like transition, §2 Mecanismo Central) */
static void apply_transition(double* u, const double* w, double beta, int d) {
    double t = beta * dot(w, u, d);
    for (int c = 0; c < d; ++c) u[c] -= t * w[c];
}

/*
 * Logits of one query row i of one head, written to s[0..i].
 * q_i: [d]; k, w: [L, d] of this head; beta, log_f: [L] of this head
 * (log_f may be NULL); rel: [L] relative-position bias of this head, rel[i - j]
 * added to s_ij (may be NULL).  u is a scratch vector of length d.
 */
static void row_logits(const double* qi, const double* k, const double* w,
                       const double* beta, const double* log_f, const double* rel, int i, int d,
                       double scale, double* s, double* u) {
    memcpy(u, qi, sizeof(double) * (size_t)d);
    double bias = 0.0; /* sum_{s=j+1..i} log f_s, empty (0) at j = i */
    for (int j = i; j >= 0; --j) {
        s[j] = scale * dot(k + (size_t)j * d, u, d) + bias;
        if (rel) s[j] += rel[i - j];
        /* next key j-1 sees H_j ... H_i q_i */
        apply_transition(u, w + (size_t)j * d, beta[j], d);
        if (log_f) bias += log_f[j];
    }
}

/* softmax over s[0..n-1] (max-subtracted), o = sum_j p_j v_j, returns lse */
static double softmax_combine(const double* s, const double* v, int n, int d, double* o) {
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) m = s[j] > m ? s[j] : m;
    double l = 0.0;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int j = 0; j < n; ++j) {
        double p = exp(s[j] - m);
        l += p;
        const double* vj = v + (size_t)j * d;
        for (int c = 0; c < d; ++c) o[c] += p * vj[c];
    }
    for (int c = 0; c < d; ++c) o[c] /= l;
    return m + log(l);
}

/*
 * PaTH (or PaTH-FoX when log_f != NULL) causal attention forward for a list of
 * rows.  Tensors are [B*H, L, d] row-major fp64 (beta, log_f: [B*H, L]).
 * rows[r] = bh * L + i selects query i of head bh; n_rows rows are computed
 * and o_rows[r*d ...], lse_rows[r] receive the results.  rows == NULL means
 * every row of every head in natural order (n_rows must be BH*L).
 */
static void fwd_rows(const double* q, const double* k, const double* v, const double* w,
                     const double* beta, const double* log_f, const double* rel, int L, int d,
                     double scale, const int64_t* rows, int64_t n_rows, double* o_rows, double* lse_rows) {
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)L);
        double* u = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < n_rows; ++r) {
            int64_t gi = rows ? rows[r] : r;
            int64_t bh = gi / L;
            int i = (int)(gi % L);
            size_t hoff = (size_t)bh * (size_t)L;
            row_logits(q + (size_t)gi * d, k + hoff * d, w + hoff * d, beta + hoff,
                       log_f ? log_f + hoff : NULL, rel ? rel + hoff : NULL, i, d, scale, s, u);
            double lse = softmax_combine(s, v + hoff * d, i + 1, d, o_rows + (size_t)r * d);
            if (lse_rows) lse_rows[r] = lse;
        }
        free(s);
        free(u);
    }
}

void path_oracle_fwd_rows(const double* q, const double* k, const double* v,
                          const double* w, const double* beta, const double* log_f,
                          int BH, int L, int d, double scale,
                          const int64_t* rows, int64_t n_rows,
                          double* o_rows, double* lse_rows) {
    (void)BH;
    fwd_rows(q, k, v, w, beta, log_f, NULL, L, d, scale, rows, n_rows, o_rows, lse_rows);
}

/*
 * As path_oracle_fwd_rows, with a relative-position bias instead of forget
 * gates: rel [B*H, L], rel[bh*L + (i - j)] added unscaled to s_ij — the additive
 * positional prior of "Resumo Técnico: Mecanismo de Atenção Bayesiana (BAM)",
 * §"Solução Proposta: GGD-BAM" (bias matrix b_ij depending on i - j only),
 * on top of the PaTH logits.
 */
void path_oracle_fwd_rows_relbias(const double* q, const double* k, const double* v,
                                  const double* w, const double* beta, const double* rel,
                                  int BH, int L, int d, double scale,
                                  const int64_t* rows, int64_t n_rows,
                                  double* o_rows, double* lse_rows) {
    (void)BH;
    fwd_rows(q, k, v, w, beta, NULL, rel, L, d, scale, rows, n_rows, o_rows, lse_rows);
}

/*
 * Full L x L logit matrix of one head (tiny inputs; for pins).  Entries above
 * the diagonal (j > i) are set to -INFINITY.
 */
void path_oracle_logits(const double* q, const double* k, const double* w,
                        const double* beta, const double* log_f, int L, int d,
                        double scale, double* S) {
    double* u = (double*)malloc(sizeof(double) * (size_t)d);
    for (int i = 0; i < L; ++i) {
        double* row = S + (size_t)i * L;
        for (int j = i + 1; j < L; ++j) row[j] = -INFINITY;
        row_logits(q + (size_t)i * d, k, w, beta, log_f, NULL, i, d, scale, row, u);
    }
    free(u);
}

/*
 * Decode for ONE head, following the "Inferência" bullet of §3: the cache holds
 * transported keys  k~_j = H_{t-1} ... H_{j+1} k_j  (rows 0..n0-1 on entry).
 * For each step t = 0..T-1 (token position p = n0 + t):
 *     k~_j <- H_p k~_j for every cached j < p         (in-place key update)
 *     append k_p (untransported) and v_p at slot p
 *     o_t = softmax_j(scale * q_p . k~_j) v_j over j = 0..p
 * kc, vc: [n_max, d] fp64, updated in place; q, k, v, w: [T, d]; beta: [T];
 * o: [T, d]; lse: [T] (nullable).  n_max >= n0 + T.
 */
void path_oracle_decode(double* kc, double* vc, int n0, int n_max, int d,
                        const double* q, const double* k, const double* v,
                        const double* w, const double* beta, int T, double scale,
                        double* o, double* lse) {
    (void)n_max;
    double* s = (double*)malloc(sizeof(double) * (size_t)(n0 + T));
    for (int t = 0; t < T; ++t) {
        int p = n0 + t;
        const double* wt = w + (size_t)t * d;
#pragma omp parallel for schedule(static)
        for (int j = 0; j < p; ++j) apply_transition(kc + (size_t)j * d, wt, beta[t], d);
        memcpy(kc + (size_t)p * d, k + (size_t)t * d, sizeof(double) * (size_t)d);
        memcpy(vc + (size_t)p * d, v + (size_t)t * d, sizeof(double) * (size_t)d);
        const double* qt = q + (size_t)t * d;
#pragma omp parallel for schedule(static)
        for (int j = 0; j <= p; ++j) s[j] = scale * dot(kc + (size_t)j * d, qt, d);
        double l = softmax_combine(s, vc, p + 1, d, o + (size_t)t * d);
        if (lse) lse[t] = l;
    }
    free(s);
}

/*
 * Value-side transport ("Resumo Técnico: Por que Transformações Acumuladas
 * Extrapolam?", §"Metodologia" 1: the route transport P_{j->i} is the product of
 * the per-token steps from source j to query i; §"Principais Contribuições" 3
 * "Proteção do Lado de Valor": the same accumulated route transport applied to
 * the values).  With PaTH's steps the route operator that carries key j to
 * query i in the logit is P_{j->i} = H_i ... H_{j+1} (s_ij = q_i . P_{j->i} k_j,
 * since every H_s is symmetric), so
 *     o_i = sum_j alpha_ij P_{j->i} v_j,   alpha_ij = softmax_j(s_i.)
 * with the logits (and FoX bias) of the plain forward.  Evaluated left to right:
 *     acc <- alpha_i0 v_0;  for j = 1..i: acc <- H_j acc + alpha_ij v_j;  o_i = acc
 * (after step j, acc holds sum_{j' <= j} alpha_ij' H_j ... H_{j'+1} v_j').
 */
static double vt_combine(const double* s, const double* v, const double* w, const double* beta, int n, int d,
                         double* o) {
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) m = s[j] > m ? s[j] : m;
    double l = 0.0;
    for (int j = 0; j < n; ++j) l += exp(s[j] - m);
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int j = 0; j < n; ++j) {
        if (j > 0) apply_transition(o, w + (size_t)j * d, beta[j], d);
        const double a = exp(s[j] - m) / l;
        const double* vj = v + (size_t)j * d;
        for (int c = 0; c < d; ++c) o[c] += a * vj[c];
    }
    return m + log(l);
}

/* As path_oracle_fwd_rows, with value-side transport (log_f may be NULL). */
void path_oracle_fwd_rows_vt(const double* q, const double* k, const double* v,
                             const double* w, const double* beta, const double* log_f,
                             int BH, int L, int d, double scale,
                             const int64_t* rows, int64_t n_rows,
                             double* o_rows, double* lse_rows) {
    (void)BH;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)L);
        double* u = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < n_rows; ++r) {
            int64_t gi = rows ? rows[r] : r;
            int64_t bh = gi / L;
            int i = (int)(gi % L);
            size_t hoff = (size_t)bh * (size_t)L;
            row_logits(q + (size_t)gi * d, k + hoff * d, w + hoff * d, beta + hoff,
                       log_f ? log_f + hoff : NULL, NULL, i, d, scale, s, u);
            double lse = vt_combine(s, v + hoff * d, w + hoff * d, beta + hoff, i + 1, d,
                                    o_rows + (size_t)r * d);
            if (lse_rows) lse_rows[r] = lse;
        }
        free(s);
        free(u);
    }
}

/*
 * Decode for ONE head with value-side transport: as path_oracle_decode, and the
 * value cache is transported in place with the keys (v~_j = H_{t-1} ... H_{j+1} v_j,
 * the values carried to the current position along the same route), so
 * o_t = softmax_j(scale q_p . k~_j) v~_j over j = 0..p.
 */
void path_oracle_decode_vt(double* kc, double* vc, int n0, int n_max, int d,
                           const double* q, const double* k, const double* v,
                           const double* w, const double* beta, int T, double scale,
                           double* o, double* lse) {
    (void)n_max;
    double* s = (double*)malloc(sizeof(double) * (size_t)(n0 + T));
    for (int t = 0; t < T; ++t) {
        int p = n0 + t;
        const double* wt = w + (size_t)t * d;
#pragma omp parallel for schedule(static)
        for (int j = 0; j < p; ++j) {
            apply_transition(kc + (size_t)j * d, wt, beta[t], d);
            apply_transition(vc + (size_t)j * d, wt, beta[t], d);
        }
        memcpy(kc + (size_t)p * d, k + (size_t)t * d, sizeof(double) * (size_t)d);
        memcpy(vc + (size_t)p * d, v + (size_t)t * d, sizeof(double) * (size_t)d);
        const double* qt = q + (size_t)t * d;
#pragma omp parallel for schedule(static)
        for (int j = 0; j <= p; ++j) s[j] = scale * dot(kc + (size_t)j * d, qt, d);
        double l = softmax_combine(s, vc, p + 1, d, o + (size_t)t * d);
        if (lse) lse[t] = l;
    }
    free(s);
}

/* The in-place key update alone: k~_j <- (I - beta w w^T) k~_j for j < n. */
void path_oracle_kcache_update(double* kc, int n, int d, const double* w, double beta) {
#pragma omp parallel for schedule(static)
    for (int j = 0; j < n; ++j) apply_transition(kc + (size_t)j * d, w, beta, d);
}

/*
 * Gradients of PaTH (or PaTH-FoX) causal attention for whole heads — the
 * reverse mode of the walk above, written out by the chain rule.  The pages
 * give the forward only; the gradient is fixed by it (§3 "Treinamento e
 * Inferência Eficientes" trains the forward by backpropagation).
 *
 * Loss convention: the caller's scalar loss has gradient dO = dL/do.  Per row
 * i the forward walk gives u_j = H_{j+1} ... H_i q_i (u_i = q_i) and
 * s_ij = scale k_j . u_j + bias_ij, p_ij = softmax_j, o_i = sum_j p_ij v_j.  Then
 *     dv_j  += p_ij dO_i
 *     ds_ij  = p_ij (dO_i . v_j - dO_i . o_i)              (softmax gradient)
 *     dk_j  += scale ds_ij u_j
 * and walking back up the row (u_{j-1} = H_j u_j), with g the gradient with
 * respect to the walk's current vector:
 *     g <- scale ds_i0 k_0;  for j = 1..i:
 *         dH_j  = g u_j^T    (g is dL/du_{j-1})
 *         dbeta_j += -(w_j . g)(w_j . u_j)
 *         dw_j    += -beta_j ((w_j . u_j) g + (w_j . g) u_j)
 *         g <- H_j g + scale ds_ij k_j
 *     dq_i = g.
 * FoX: bias_ij = sum_{s=j+1..i} log f_s, so dlog_f_s += sum_{j<s} ds_ij for
 * every s <= i of the row.
 *
 * Tensors as in path_oracle_fwd_rows ([BH, L, d] fp64; beta, log_f [BH, L]);
 * dO [BH, L, d].  Outputs (overwritten): dq, dk, dv, dw [BH, L, d];
 * dbeta [BH, L]; dlog_f [BH, L] (ignored when log_f is NULL).  The rows of a
 * head run in parallel (OpenMP), each thread summing its rows' contributions
 * into its own buffers, which are then added in thread order.
 */
static void bwd_row(const double* qh, const double* kh, const double* vh, const double* wh,
                    const double* bh_beta, const double* lf, const double* dOh, int i, int d, double scale,
                    double* U, double* s, double* ds, double* o, double* g,
                    double* dqh, double* dk, double* dv, double* dw, double* db, double* dlf) {
    /* forward walk of row i, keeping every u_j */
    double* u = U + (size_t)i * d;
    memcpy(u, qh + (size_t)i * d, sizeof(double) * (size_t)d);
    double bias = 0.0;
    for (int j = i; j >= 0; --j) {
        double* uj = U + (size_t)j * d;
        if (j < i) {
            memcpy(uj, uj + d, sizeof(double) * (size_t)d);
            apply_transition(uj, wh + (size_t)(j + 1) * d, bh_beta[j + 1], d);
        }
        s[j] = scale * dot(kh + (size_t)j * d, uj, d) + bias;
        if (lf) bias += lf[j];
    }
    softmax_combine(s, vh, i + 1, d, o);
    double m = -INFINITY, l = 0.0;
    for (int j = 0; j <= i; ++j) m = s[j] > m ? s[j] : m;
    for (int j = 0; j <= i; ++j) l += exp(s[j] - m);
    const double* dOi = dOh + (size_t)i * d;
    double delta = dot(dOi, o, d);
    for (int j = 0; j <= i; ++j) {
        double p = exp(s[j] - m) / l;
        ds[j] = p * (dot(dOi, vh + (size_t)j * d, d) - delta);
        double* dvj = dv + (size_t)j * d;
        double* dkj = dk + (size_t)j * d;
        const double* uj = U + (size_t)j * d;
        for (int c = 0; c < d; ++c) {
            dvj[c] += p * dOi[c];
            dkj[c] += scale * ds[j] * uj[c];
        }
    }
    /* back up the walk */
    for (int c = 0; c < d; ++c) g[c] = scale * ds[0] * kh[c];
    for (int j = 1; j <= i; ++j) {
        const double* wj = wh + (size_t)j * d;
        const double* uj = U + (size_t)j * d;
        double wu = dot(wj, uj, d), wg = dot(wj, g, d);
        db[j] += -wg * wu;
        double* dwj = dw + (size_t)j * d;
        for (int c = 0; c < d; ++c) dwj[c] += -bh_beta[j] * (wu * g[c] + wg * uj[c]);
        for (int c = 0; c < d; ++c) g[c] += -bh_beta[j] * wg * wj[c] + scale * ds[j] * kh[(size_t)j * d + c];
    }
    memcpy(dqh + (size_t)i * d, g, sizeof(double) * (size_t)d);
    if (dlf) {
        double pre = 0.0; /* sum_{j<s} ds_ij */
        for (int sp = 1; sp <= i; ++sp) {
            pre += ds[sp - 1];
            dlf[sp] += pre;
        }
    }
}

void path_oracle_bwd(const double* q, const double* k, const double* v, const double* w,
                     const double* beta, const double* log_f, const double* dO,
                     int BH, int L, int d, double scale,
                     double* dq, double* dk, double* dv, double* dw, double* dbeta, double* dlog_f) {
    const size_t Ld = (size_t)L * d;
    for (int bh = 0; bh < BH; ++bh) {
        size_t ho = (size_t)bh * L;
        const double *qh = q + ho * d, *kh = k + ho * d, *vh = v + ho * d, *wh = w + ho * d;
        const double *bb = beta + ho, *lf = log_f ? log_f + ho : NULL, *dOh = dO + ho * d;
        double *dkh = dk + ho * d, *dvh = dv + ho * d, *dwh = dw + ho * d;
        double *dbh = dbeta + ho, *dlfh = log_f ? dlog_f + ho : NULL;
        memset(dkh, 0, sizeof(double) * Ld);
        memset(dvh, 0, sizeof(double) * Ld);
        memset(dwh, 0, sizeof(double) * Ld);
        memset(dbh, 0, sizeof(double) * (size_t)L);
        if (dlfh) memset(dlfh, 0, sizeof(double) * (size_t)L);
#pragma omp parallel
        {
            double* U = (double*)malloc(sizeof(double) * Ld); /* u_j of the current row */
            double* s = (double*)malloc(sizeof(double) * (size_t)L);
            double* ds = (double*)malloc(sizeof(double) * (size_t)L);
            double* o = (double*)malloc(sizeof(double) * (size_t)d);
            double* g = (double*)malloc(sizeof(double) * (size_t)d);
            /* this thread's share of the per-key sums: dk, dv, dw, dbeta, dlog_f */
            double* acc = (double*)calloc(3 * Ld + 2 * (size_t)L, sizeof(double));
            double *tk = acc, *tv = acc + Ld, *tw = acc + 2 * Ld, *tb = acc + 3 * Ld, *tf = tb + L;
#pragma omp for schedule(dynamic, 4)
            for (int i = 0; i < L; ++i)
                bwd_row(qh, kh, vh, wh, bb, lf, dOh, i, d, scale, U, s, ds, o, g, dq + ho * d, tk, tv, tw, tb,
                        lf ? tf : NULL);
#ifdef _OPENMP
            const int nt = omp_get_num_threads(), me = omp_get_thread_num();
#else
            const int nt = 1, me = 0;
#endif
            for (int t = 0; t < nt; ++t) {
#pragma omp barrier
                if (t == me) {
                    for (size_t x = 0; x < Ld; ++x) {
                        dkh[x] += tk[x];
                        dvh[x] += tv[x];
                        dwh[x] += tw[x];
                    }
                    for (int x = 0; x < L; ++x) {
                        dbh[x] += tb[x];
                        if (dlfh) dlfh[x] += tf[x];
                    }
                }
            }
            free(acc);
            free(U);
            free(s);
            free(ds);
            free(o);
            free(g);
        }
    }
}
