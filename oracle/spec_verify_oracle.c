/*
 * Float64 CPU oracle for the speculative-decoding verification step.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  It shares no code, header, table or
 * helper with the CUDA path; it is a plain sequential restatement of the method
 * written for a reader to check against the pages by eye.  Status: pinned (see
 * tests/test_oracle_pins.py and tests/test_oracle_law.py).
 *
 * Sources (page title, section):
 *   [P1] "Speculative Decoding" (atonlee.tistory.com/330): ch.2 (one
 *        propose/verify round, cut at the first rejection, k accepted + 1),
 *        ch.3 (the acceptance rule r < min(1, p/q), residual
 *        norm(max(0, p - q)), greedy rule at temperature 0).
 *   [P2] "Speculative Decoding으로 LLM 추론 속도 높이기" (donmain.dev), section
 *        "품질은 rejection sampling이 지킨다" (worked example and the rule).
 *   [P3] "Fast Inference from Transformers via Speculative Decoding" notes
 *        (obsidian-dorae222.pages.dev), method details, steps 2 and 3 (gamma+1
 *        target distributions, accept probability, residual, bonus token).
 *   [P4] "투기적 디코딩 — 초안 모델을 무엇으로 세울 것인가" (ailab.paldyn.com),
 *        section on why the output does not change (rule, greedy argmax).
 *
 * Readings where the pages leave a step open:
 *   - p and q are softmax(logits / T) with the sequence's own T; "/T" is a
 *     true float64 division (the pages only say that a low T sharpens both).
 *   - The accept test is evaluated as  r * q(x) < p(x), which equals the
 *     printed strict test r < min(1, p(x)/q(x)) for r in [0,1) and q(x) > 0,
 *     and accepts a zero-q draft exactly when p(x) > 0.
 *   - T == 0 is greedy: accept iff the draft equals argmax of the raw target
 *     logits, the lowest id winning ties; on rejection emit that argmax; when
 *     every draft matches, emit the argmax of the bonus row.  No draft row and
 *     no uniform is read.
 *   - The final sample uses the fixed last uniform column uniforms[b, gmax],
 *     also for sequences with fewer drafts.  Inverse CDF: the smallest j with
 *     u*S < C_j, C_j the inclusive running sum of the weights in index order,
 *     S their total; if rounding leaves no such j, the last j with weight > 0.
 *   - A rejected row whose residual mass is not above 1e-300 (unreachable in
 *     exact arithmetic) samples from p of that row instead.
 *   - A NULL draft-logit array means deterministic proposals: q_i is the
 *     point mass at the drafted id x_i (a prompt-lookup / n-gram proposer,
 *     [P1] ch.5 and [P4]'s table of draft methods, copies tokens from the
 *     context).  Then the test is r < p(x_i) and the residual is p with x_i
 *     removed: max(0, p - q) for that q.
 *   - A sequence with num_draft outside [0, gmax], a temperature that is
 *     negative, NaN, infinite or positive-but-below FLT_MIN, a drafted id
 *     outside [0, V) at a position it uses, or a sampled row it uses whose
 *     logits have no finite softmax normaliser (all -inf, any +inf or NaN) is
 *     invalid: it emits -1 everywhere, 0 accepted, and sets a status bit.
 */
#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1

#define ORACLE_BAD_TOKEN 1
#define ORACLE_BAD_TEMPERATURE 2
#define ORACLE_BAD_NUM_DRAFT 4
#define ORACLE_BAD_LOGITS 8

/* One stored logit widened exactly to float64.  bfloat16 is the upper half
 * of a float32, so the widening shifts the 16 stored bits up. */
static double logit_at(const void *base, int dtype, size_t idx)
{
    if (dtype == ORACLE_F32)
        return (double)((const float *)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Normaliser of softmax(l / T) over one row:  m = max_j l_j / T and
 * z = sum_j exp(l_j / T - m), so that p_j = exp(l_j / T - m) / z. */
typedef struct {
    double m;
    double z;
} softmax_norm;

static softmax_norm row_softmax_norm(const void *base, int dtype, size_t row_off, int V, double T)
{
    softmax_norm s;
    s.m = -INFINITY;
    for (int j = 0; j < V; ++j) {
        double zj = logit_at(base, dtype, row_off + (size_t)j) / T;
        if (zj > s.m)
            s.m = zj;
    }
    s.z = 0.0;
    if (!isfinite(s.m)) {
        s.z = NAN; /* no finite maximum: the row defines no distribution */
        return s;
    }
    for (int j = 0; j < V; ++j)
        s.z += exp(logit_at(base, dtype, row_off + (size_t)j) / T - s.m);
    return s;
}

static int norm_is_valid(softmax_norm s)
{
    return isfinite(s.m) && isfinite(s.z) && s.z > 0.0;
}

/* p_j of one row, given its normaliser. */
static double row_prob(const void *base, int dtype, size_t row_off, int j, double T, softmax_norm s)
{
    return exp(logit_at(base, dtype, row_off + (size_t)j) / T - s.m) / s.z;
}

/* Greedy decision value: index of the largest raw logit, lowest index on ties. */
static int row_argmax(const void *base, int dtype, size_t row_off, int V)
{
    int best = 0;
    double bv = logit_at(base, dtype, row_off);
    for (int j = 1; j < V; ++j) {
        double v = logit_at(base, dtype, row_off + (size_t)j);
        if (v > bv) {
            bv = v;
            best = j;
        }
    }
    return best;
}

typedef struct {
    const void *target;
    const void *draft;
    int dtype;
    const int32_t *tokens;
    const int32_t *num_draft;
    const float *uniforms;
    const float *temperature;
    int B, gmax, V;
    int32_t *out_tokens;
    int32_t *out_num_accepted;
    /* optional diagnostics (may be NULL) */
    double *p_hat;       /* [B, gmax]  p_i(x_i) for every i < g (sampled seqs) */
    double *q_hat;       /* [B, gmax]  q_i(x_i) */
    double *logz_t;      /* [B, gmax+1] m + log z of target rows i <= g */
    double *logz_d;      /* [B, gmax]   of draft rows i < g */
    double *resid_mass;  /* [B] S of the decided row */
    double *acc_margin;  /* [B, gmax]   |r_i - p_i(x)/q_i(x)| at evaluated positions */
    double *samp_margin; /* [B] distance of u to the nearest CDF boundary of the pick */
    int32_t *seq_status; /* [B] status bits of each sequence */
} oracle_args;

static void write_invalid(const oracle_args *a, int b, int bits)
{
    for (int i = 0; i <= a->gmax; ++i)
        a->out_tokens[(size_t)b * (a->gmax + 1) + i] = -1;
    a->out_num_accepted[b] = 0;
    if (a->seq_status)
        a->seq_status[b] = bits;
}

static int temperature_is_valid(float T)
{
    if (isnan(T) || isinf(T) || T < 0.0f)
        return 0;
    if (T > 0.0f && T < FLT_MIN)
        return 0;
    return 1;
}

/* Diagnostics only: softmax values at every position of a sampled sequence,
 * independent of where the round stops.  Not part of the decision path. */
static void fill_diagnostics(const oracle_args *a, int b, int g, double T)
{
    const int gmax = a->gmax, V = a->V;
    for (int i = 0; i <= g; ++i) {
        size_t toff = ((size_t)b * (gmax + 1) + i) * (size_t)V;
        softmax_norm st = row_softmax_norm(a->target, a->dtype, toff, V, T);
        if (a->logz_t)
            a->logz_t[(size_t)b * (gmax + 1) + i] = st.m + log(st.z);
        if (i == g)
            break;
        int x = a->tokens[(size_t)b * gmax + i];
        if (a->p_hat)
            a->p_hat[(size_t)b * gmax + i] = row_prob(a->target, a->dtype, toff, x, T, st);
        if (!a->draft) { /* point-mass draft: q(x) = 1, no draft row */
            if (a->q_hat)
                a->q_hat[(size_t)b * gmax + i] = 1.0;
            continue;
        }
        size_t doff = ((size_t)b * gmax + i) * (size_t)V;
        softmax_norm sd = row_softmax_norm(a->draft, a->dtype, doff, V, T);
        if (a->logz_d)
            a->logz_d[(size_t)b * gmax + i] = sd.m + log(sd.z);
        if (a->q_hat)
            a->q_hat[(size_t)b * gmax + i] = row_prob(a->draft, a->dtype, doff, x, T, sd);
    }
}

/* Weights w_j of one decided row ([P1] ch.3 step 3, [P3] step 3): with
 * 'rejected', the residual max(0, p - q) of the row (q from the draft row at
 * doff, or the point mass at xn when there is no draft array); otherwise p of
 * the target row (the bonus row when every draft was accepted).  A residual
 * whose total is not above 1e-300 (unreachable in exact arithmetic) falls back
 * to p of the same row.  Returns the total S, summed in index order. */
static double decided_row_weights(const void *target, const void *draft, int dtype, size_t toff, size_t doff, int V,
                                  double T, softmax_norm st, softmax_norm sd, int rejected, int xn, double *w)
{
    double S = 0.0;
    for (int j = 0; j < V; ++j) {
        double pj = row_prob(target, dtype, toff, j, T, st);
        double wj = pj;
        if (rejected) {
            double qj = draft ? row_prob(draft, dtype, doff, j, T, sd) : (j == xn ? 1.0 : 0.0);
            wj = pj - qj > 0.0 ? pj - qj : 0.0;
        }
        w[j] = wj;
        S += wj;
    }
    if (!(S > 1e-300)) {
        S = 0.0;
        for (int j = 0; j < V; ++j) {
            w[j] = row_prob(target, dtype, toff, j, T, st);
            S += w[j];
        }
    }
    return S;
}

/* Inverse CDF with uniform u: the smallest j with u*S < C_j, C_j the running
 * sum of w in index order (C[j] when the caller has them, else summed here);
 * if rounding leaves no such j, the last j with w_j > 0.  margin: the distance
 * of u to the nearer boundary C_{j-1}/S, C_j/S of the pick (0 in the fallback). */
static int pick_by_cdf(const double *w, const double *C, int V, double S, double u, double *margin)
{
    double thr = u * S;
    int pick = -1;
    double lo_c = 0.0, hi_c = 0.0;
    if (C) {
        /* C is nondecreasing: bisect for the smallest j with thr < C[j] */
        int lo = 0, hi = V;
        while (lo < hi) {
            int mid = lo + (hi - lo) / 2;
            if (thr < C[mid])
                hi = mid;
            else
                lo = mid + 1;
        }
        if (lo < V) {
            pick = lo;
            lo_c = lo > 0 ? C[lo - 1] : 0.0;
            hi_c = C[lo];
        }
    } else {
        double acc = 0.0;
        for (int j = 0; j < V; ++j) {
            double prev = acc;
            acc += w[j];
            if (thr < acc) {
                pick = j;
                lo_c = prev;
                hi_c = acc;
                break;
            }
        }
    }
    if (pick < 0) {
        for (int j = V - 1; j >= 0; --j)
            if (w[j] > 0.0) {
                pick = j;
                break;
            }
        *margin = 0.0;
        return pick;
    }
    double m0 = u - lo_c / S, m1 = hi_c / S - u;
    *margin = m0 < m1 ? m0 : m1;
    return pick;
}

/* Sample one decided row of sequence b: its weights, then the inverse CDF. */
static int sample_decided_row(const oracle_args *a, int b, int n, int rejected, double T, double u,
                              softmax_norm st, softmax_norm sd, int xn, double *mass_out, double *margin_out)
{
    const int gmax = a->gmax, V = a->V;
    size_t toff = ((size_t)b * (gmax + 1) + n) * (size_t)V;
    size_t doff = ((size_t)b * gmax + n) * (size_t)V;
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    if (!w)
        return -1;
    double S = decided_row_weights(a->target, a->draft, a->dtype, toff, doff, V, T, st, sd, rejected, xn, w);
    *mass_out = S;
    int pick = pick_by_cdf(w, NULL, V, S, u, margin_out);
    free(w);
    return pick;
}

/* One sequence of the round, in the pages' order. */
static void verify_one(const oracle_args *a, int b)
{
    const int gmax = a->gmax, V = a->V;
    int32_t *out = a->out_tokens + (size_t)b * (gmax + 1);
    const int32_t *x = a->tokens + (size_t)b * gmax;
    const float *r = a->uniforms + (size_t)b * (gmax + 1);
    int g = a->num_draft[b];
    float Tf = a->temperature[b];

    for (int i = 0; i < gmax; ++i) {
        if (a->acc_margin)
            a->acc_margin[(size_t)b * gmax + i] = NAN;
        if (a->p_hat)
            a->p_hat[(size_t)b * gmax + i] = NAN;
        if (a->q_hat)
            a->q_hat[(size_t)b * gmax + i] = NAN;
        if (a->logz_d)
            a->logz_d[(size_t)b * gmax + i] = NAN;
    }
    for (int i = 0; i <= gmax; ++i)
        if (a->logz_t)
            a->logz_t[(size_t)b * (gmax + 1) + i] = NAN;
    if (a->resid_mass)
        a->resid_mass[b] = NAN;
    if (a->samp_margin)
        a->samp_margin[b] = NAN;
    if (a->seq_status)
        a->seq_status[b] = 0;

    if (g < 0 || g > gmax) {
        write_invalid(a, b, ORACLE_BAD_NUM_DRAFT);
        return;
    }
    int bits = 0;
    if (!temperature_is_valid(Tf))
        bits |= ORACLE_BAD_TEMPERATURE;
    for (int i = 0; i < g; ++i)
        if (x[i] < 0 || x[i] >= V)
            bits |= ORACLE_BAD_TOKEN;
    if (bits) {
        write_invalid(a, b, bits);
        return;
    }

    int n = g;
    if (Tf == 0.0f) {
        /* Greedy ([P1] ch.3, [P2], [P4]): accept while the draft equals the
         * target argmax; the first mismatch is replaced by that argmax. */
        int emit = -1;
        for (int i = 0; i < g; ++i) {
            int am = row_argmax(a->target, a->dtype, ((size_t)b * (gmax + 1) + i) * (size_t)V, V);
            if (x[i] != am) {
                n = i;
                emit = am;
                break;
            }
        }
        if (emit < 0)
            emit = row_argmax(a->target, a->dtype, ((size_t)b * (gmax + 1) + g) * (size_t)V, V);
        for (int i = 0; i < n; ++i)
            out[i] = x[i];
        out[n] = emit;
        for (int i = n + 1; i <= gmax; ++i)
            out[i] = -1;
        a->out_num_accepted[b] = n;
        return;
    }

    const double T = (double)Tf;
    if (a->p_hat || a->q_hat || a->logz_t || a->logz_d)
        fill_diagnostics(a, b, g, T);

    /* Sampled: test drafts in order; stop at the first rejection
     * ([P1] ch.2-3, [P3] step 3). */
    int rejected = 0;
    softmax_norm st_dec, sd_dec;
    sd_dec.m = NAN;
    sd_dec.z = NAN;
    for (int i = 0; i < g; ++i) {
        size_t toff = ((size_t)b * (gmax + 1) + i) * (size_t)V;
        size_t doff = ((size_t)b * gmax + i) * (size_t)V;
        softmax_norm st = row_softmax_norm(a->target, a->dtype, toff, V, T);
        softmax_norm sd = {0.0, 1.0};
        if (a->draft)
            sd = row_softmax_norm(a->draft, a->dtype, doff, V, T);
        if (!norm_is_valid(st) || !norm_is_valid(sd)) {
            write_invalid(a, b, ORACLE_BAD_LOGITS);
            return;
        }
        double p = row_prob(a->target, a->dtype, toff, x[i], T, st);
        double q = a->draft ? row_prob(a->draft, a->dtype, doff, x[i], T, sd) : 1.0;
        double ri = (double)r[i];
        if (a->acc_margin)
            a->acc_margin[(size_t)b * gmax + i] = q > 0.0 ? fabs(ri - p / q) : INFINITY;
        if (!(ri * q < p)) {
            n = i;
            rejected = 1;
            st_dec = st;
            sd_dec = sd;
            break;
        }
    }
    if (!rejected) {
        size_t toff = ((size_t)b * (gmax + 1) + g) * (size_t)V;
        st_dec = row_softmax_norm(a->target, a->dtype, toff, V, T);
        if (!norm_is_valid(st_dec)) {
            write_invalid(a, b, ORACLE_BAD_LOGITS);
            return;
        }
    }
    double mass = NAN, margin = NAN;
    int y = sample_decided_row(a, b, n, rejected, T, (double)r[gmax], st_dec, sd_dec, rejected ? x[n] : -1,
                               &mass, &margin);
    if (a->resid_mass)
        a->resid_mass[b] = mass;
    if (a->samp_margin)
        a->samp_margin[b] = margin;
    for (int i = 0; i < n; ++i)
        out[i] = x[i];
    out[n] = y;
    for (int i = n + 1; i <= gmax; ++i)
        out[i] = -1;
    a->out_num_accepted[b] = n;
}

typedef struct {
    const oracle_args *a;
    int b0, b1;
} oracle_slice;

static void *run_slice(void *p)
{
    const oracle_slice *s = (const oracle_slice *)p;
    for (int b = s->b0; b < s->b1; ++b)
        verify_one(s->a, b);
    return NULL;
}

/* Entry point.  All pointers are host memory.  Returns 0, or -1 on a bad
 * argument.  Sequences are independent; nthreads > 1 splits them over POSIX
 * threads in contiguous ranges (results do not depend on nthreads). */
int oracle_verify(const void *target, const void *draft, int dtype, const int32_t *tokens,
                  const int32_t *num_draft, const float *uniforms, const float *temperature, int B,
                  int gmax, int V, int32_t *out_tokens, int32_t *out_num_accepted, double *p_hat,
                  double *q_hat, double *logz_t, double *logz_d, double *resid_mass,
                  double *acc_margin, double *samp_margin, int32_t *seq_status, int nthreads)
{
    if (B < 0 || gmax < 0 || V < 1 || (dtype != ORACLE_F32 && dtype != ORACLE_BF16))
        return -1;
    if (B == 0)
        return 0;
    if (!target || !tokens || !num_draft || !uniforms || !temperature || !out_tokens || !out_num_accepted)
        return -1; /* draft may be NULL: point-mass proposals */
    oracle_args a = {target, draft, dtype, tokens, num_draft, uniforms, temperature, B, gmax, V,
                     out_tokens, out_num_accepted, p_hat, q_hat, logz_t, logz_d, resid_mass,
                     acc_margin, samp_margin, seq_status};
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > B)
        nthreads = B;
    if (nthreads == 1) {
        for (int b = 0; b < B; ++b)
            verify_one(&a, b);
        return 0;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    oracle_slice *sl = (oracle_slice *)malloc(sizeof(oracle_slice) * (size_t)nthreads);
    if (!th || !sl) {
        free(th);
        free(sl);
        return -1;
    }
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        sl[t].a = &a;
        sl[t].b0 = (int)((long long)B * t / nthreads);
        sl[t].b1 = (int)((long long)B * (t + 1) / nthreads);
        if (pthread_create(&th[started], NULL, run_slice, &sl[t]) == 0)
            ++started;
        else
            run_slice(&sl[t]); /* could not start a thread: do the slice here */
    }
    for (int t = 0; t < started; ++t)
        pthread_join(th[t], NULL);
    free(th);
    free(sl);
    return 0;
}

/* ------------------------------------------------------------------------
 * Tree verification (several candidate paths checked in one round).
 *
 * Sources: [P1] ch.5 (Medusa heads each propose their top few candidates; the
 * combinations form a tree that one target forward checks through a tree
 * attention mask) and its glossary entry on tree attention; [P2]'s EAGLE
 * paragraph (EAGLE-2 draws the candidates as a tree and checks it in one
 * forward).  The pages state the acceptance rule for one candidate per
 * position only ([P1] ch.3).  Readings used here:
 *   - Node 0 is the root (the last emitted token); node k >= 1 carries the
 *     candidate token tokens[b][k] and hangs under parent[b][k] < k.  Row k of
 *     the target logits is the target's next-token distribution after the
 *     path root..k.
 *   - Candidates are deterministic (a proposer's top tokens), so each one is
 *     a point mass, as for prompt lookup.  The children of the current node
 *     are tried in index order with the page's rule applied to what is left:
 *     with R the ids of the children already rejected, child c is accepted
 *     iff  u_c * (1 - p(R)) < p(tok_c)  (u_c = uniforms[b][c]); a child whose
 *     id is already in R has no mass left and is rejected.  This is the
 *     single-candidate rule r < p'(x) for the residual p' = p without R,
 *     renormalised, so each step keeps the target's law, and with one child
 *     per node it is the chain rule for point-mass drafts exactly.
 *   - When no child is accepted (or the node is a leaf) the walk stops and
 *     one token is sampled from p without R (renormalised) by inverse CDF
 *     with uniforms[b][0] (node 0 is never tested, so its column is free);
 *     a residual with mass not above 1e-300 samples p instead.
 *   - T == 0: the accepted child is the first whose id equals the argmax of
 *     the node's raw logits (lowest id on ties); the walk stops at a node
 *     with no such child and emits that argmax.
 *   - Invalid sequences (num_nodes outside [1, N], a parent outside [0, k),
 *     a candidate id outside [0, V), a bad temperature, or a sampled row on
 *     the walk with no finite normaliser) emit -1 everywhere and 0 accepted.
 * Outputs: out_tokens[b] = accepted tokens then the sampled one, -1 after;
 * out_path[b] = the accepted node indices, -1 after; out_num[b] = accepted.
 * ---------------------------------------------------------------------- */
#define ORACLE_BAD_TREE 32

typedef struct {
    const void *target;
    int dtype;
    const int32_t *parent, *tokens, *num_nodes;
    const float *uniforms, *temperature;
    int B, N, V;
    int32_t *out_tokens, *out_num, *out_path;
    double *acc_margin;  /* [B, N] |u_c - p(tok_c)/(1 - p(R))| at tested nodes, NaN elsewhere */
    double *samp_margin; /* [B] distance of u_0 to the nearest CDF boundary of the final pick */
    int32_t *seq_status; /* [B] */
} tree_args;

static void tree_write_invalid(const tree_args *a, int b, int bits)
{
    for (int k = 0; k < a->N; ++k) {
        a->out_tokens[(size_t)b * a->N + k] = -1;
        if (a->out_path)
            a->out_path[(size_t)b * a->N + k] = -1;
    }
    a->out_num[b] = 0;
    if (a->seq_status)
        a->seq_status[b] = bits;
}

static void tree_one(const tree_args *a, int b)
{
    const int N = a->N, V = a->V;
    const int32_t *par = a->parent + (size_t)b * N;
    const int32_t *tok = a->tokens + (size_t)b * N;
    const float *u = a->uniforms + (size_t)b * N;
    const int nn = a->num_nodes[b];
    const float Tf = a->temperature[b];
    if (a->acc_margin)
        for (int k = 0; k < N; ++k)
            a->acc_margin[(size_t)b * N + k] = NAN;
    if (a->samp_margin)
        a->samp_margin[b] = NAN;
    if (a->seq_status)
        a->seq_status[b] = 0;
    if (nn < 1 || nn > N) {
        tree_write_invalid(a, b, ORACLE_BAD_NUM_DRAFT);
        return;
    }
    int bits = 0;
    if (!temperature_is_valid(Tf))
        bits |= ORACLE_BAD_TEMPERATURE;
    for (int k = 1; k < nn; ++k) {
        if (par[k] < 0 || par[k] >= k)
            bits |= ORACLE_BAD_TREE;
        if (tok[k] < 0 || tok[k] >= V)
            bits |= ORACLE_BAD_TOKEN;
    }
    if (bits) {
        tree_write_invalid(a, b, bits);
        return;
    }
    int32_t *out = a->out_tokens + (size_t)b * N;
    int32_t *path = a->out_path ? a->out_path + (size_t)b * N : NULL;
    int *rej = (int *)malloc(sizeof(int) * (size_t)(nn > 1 ? nn : 1));
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    if (!rej || !w) {
        free(rej);
        free(w);
        tree_write_invalid(a, b, ORACLE_BAD_NUM_DRAFT);
        return;
    }
    const double T = (double)Tf;
    int node = 0, n = 0, emit = -1;
    for (;;) {
        const size_t off = ((size_t)b * N + node) * (size_t)V;
        int next = -1;
        if (Tf == 0.0f) {
            const int am = row_argmax(a->target, a->dtype, off, V);
            for (int c = node + 1; c < nn; ++c)
                if (par[c] == node && tok[c] == am) {
                    next = c;
                    break;
                }
            if (next < 0)
                emit = am;
        } else {
            const softmax_norm st = row_softmax_norm(a->target, a->dtype, off, V, T);
            if (!norm_is_valid(st)) {
                free(rej);
                free(w);
                tree_write_invalid(a, b, ORACLE_BAD_LOGITS);
                return;
            }
            double pR = 0.0;
            int nrej = 0;
            for (int c = node + 1; c < nn; ++c) {
                if (par[c] != node)
                    continue;
                int dup = 0;
                for (int r = 0; r < nrej; ++r)
                    dup |= rej[r] == tok[c];
                const double pc = dup ? 0.0 : row_prob(a->target, a->dtype, off, tok[c], T, st);
                const double left = 1.0 - pR;
                if (a->acc_margin)
                    a->acc_margin[(size_t)b * N + c] = left > 0.0 ? fabs((double)u[c] - pc / left) : INFINITY;
                if ((double)u[c] * left < pc) {
                    next = c;
                    break;
                }
                if (!dup) {
                    pR += pc;
                    rej[nrej++] = tok[c];
                }
            }
            if (next < 0) {
                /* p without the rejected ids, by inverse CDF with u_0 */
                double S = 0.0;
                for (int j = 0; j < V; ++j) {
                    int out_of = 0;
                    for (int r = 0; r < nrej; ++r)
                        out_of |= rej[r] == j;
                    w[j] = out_of ? 0.0 : row_prob(a->target, a->dtype, off, j, T, st);
                    S += w[j];
                }
                if (!(S > 1e-300)) {
                    S = 0.0;
                    for (int j = 0; j < V; ++j) {
                        w[j] = row_prob(a->target, a->dtype, off, j, T, st);
                        S += w[j];
                    }
                }
                const double u0 = (double)u[0], thr = u0 * S;
                double C = 0.0, Cprev = 0.0;
                for (int j = 0; j < V; ++j) {
                    Cprev = C;
                    C += w[j];
                    if (thr < C) {
                        emit = j;
                        break;
                    }
                }
                if (emit < 0) {
                    for (int j = V - 1; j >= 0; --j)
                        if (w[j] > 0.0) {
                            emit = j;
                            break;
                        }
                    if (a->samp_margin)
                        a->samp_margin[b] = 0.0;
                } else if (a->samp_margin) {
                    const double lo = u0 - Cprev / S, hi = C / S - u0;
                    a->samp_margin[b] = lo < hi ? lo : hi;
                }
            }
        }
        if (next < 0)
            break;
        out[n] = tok[next];
        if (path)
            path[n] = next;
        ++n;
        node = next;
    }
    out[n] = emit;
    for (int k = n + 1; k < N; ++k)
        out[k] = -1;
    if (path)
        for (int k = n; k < N; ++k)
            path[k] = -1;
    a->out_num[b] = n;
    free(rej);
    free(w);
}

typedef struct {
    const tree_args *a;
    int b0, b1;
} tree_slice;

static void *run_tree_slice(void *p)
{
    const tree_slice *s = (const tree_slice *)p;
    for (int b = s->b0; b < s->b1; ++b)
        tree_one(s->a, b);
    return NULL;
}

/* Entry point (host memory).  target [B, N, V]; parent, tokens, uniforms
 * [B, N]; num_nodes, temperature [B]; out_tokens, out_path [B, N]; out_num,
 * samp_margin, seq_status [B]; acc_margin [B, N].  Returns 0, or -1 on a bad
 * argument. */
int oracle_tree_verify(const void *target, int dtype, const int32_t *parent, const int32_t *tokens,
                       const int32_t *num_nodes, const float *uniforms, const float *temperature, int B, int N,
                       int V, int32_t *out_tokens, int32_t *out_num, int32_t *out_path, double *acc_margin,
                       double *samp_margin, int32_t *seq_status, int nthreads)
{
    if (B < 0 || N < 1 || V < 1 || (dtype != ORACLE_F32 && dtype != ORACLE_BF16))
        return -1;
    if (B == 0)
        return 0;
    if (!target || !parent || !tokens || !num_nodes || !uniforms || !temperature || !out_tokens || !out_num)
        return -1;
    tree_args a = {target, dtype, parent, tokens, num_nodes, uniforms, temperature, B, N, V,
                   out_tokens, out_num, out_path, acc_margin, samp_margin, seq_status};
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > B)
        nthreads = B;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    tree_slice *sl = (tree_slice *)malloc(sizeof(tree_slice) * (size_t)nthreads);
    if (!th || !sl) {
        free(th);
        free(sl);
        return -1;
    }
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        sl[t].a = &a;
        sl[t].b0 = (int)((long long)B * t / nthreads);
        sl[t].b1 = (int)((long long)B * (t + 1) / nthreads);
        if (nthreads > 1 && pthread_create(&th[started], NULL, run_tree_slice, &sl[t]) == 0)
            ++started;
        else
            run_tree_slice(&sl[t]);
    }
    for (int t = 0; t < started; ++t)
        pthread_join(th[t], NULL);
    free(th);
    free(sl);
    return 0;
}

/* ------------------------------------------------------------------------
 * Many draws from one decided row (test support): the same weights and
 * inverse CDF as the final sample of oracle_verify, for n uniforms at once.
 *   target_row, draft_row: V logits each (draft_row may be NULL)
 *   mode 0: p of the target row (a bonus row; the sampler's draw)
 *   mode 1: residual max(0, p - q), q = softmax(draft_row / T)
 *   mode 2: residual for a point-mass proposal at xn (p without xn)
 *   us[n]: uniforms in [0, 1); picks[n], margins[n] (margins may be NULL)
 *   mass (may be NULL): the total S of the weights
 * Returns 0, or -1 on a bad argument or a row with no finite normaliser.
 * ---------------------------------------------------------------------- */
int oracle_pick_many(const void *target_row, const void *draft_row, int dtype, int V, float temperature, int mode,
                     int xn, const float *us, int n, int32_t *picks, double *margins, double *mass)
{
    if (!target_row || V < 1 || n < 0 || (n > 0 && (!us || !picks)) || mode < 0 || mode > 2 ||
        (mode == 1 && !draft_row) || (dtype != ORACLE_F32 && dtype != ORACLE_BF16) ||
        !(temperature > 0.0f) || !temperature_is_valid(temperature))
        return -1;
    const double T = (double)temperature;
    softmax_norm st = row_softmax_norm(target_row, dtype, 0, V, T);
    softmax_norm sd = {0.0, 1.0};
    if (mode == 1)
        sd = row_softmax_norm(draft_row, dtype, 0, V, T);
    if (!norm_is_valid(st) || !norm_is_valid(sd))
        return -1;
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    double *C = (double *)malloc(sizeof(double) * (size_t)V);
    if (!w || !C) {
        free(w);
        free(C);
        return -1;
    }
    double S = decided_row_weights(target_row, mode == 1 ? draft_row : NULL, dtype, 0, 0, V, T, st, sd, mode != 0,
                                   mode == 2 ? xn : -1, w);
    double acc = 0.0;
    for (int j = 0; j < V; ++j) {
        acc += w[j];
        C[j] = acc;
    }
    if (mass)
        *mass = S;
    for (int i = 0; i < n; ++i) {
        double mg = 0.0;
        picks[i] = pick_by_cdf(w, C, V, S, (double)us[i], &mg);
        if (margins)
            margins[i] = mg;
    }
    free(w);
    free(C);
    return 0;
}
