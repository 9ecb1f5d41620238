/*
 * sv_oracle.c -- float64 CPU oracle for batched speculative-decoding verification.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow, obviously-correct implementation
 * that the CUDA library is checked against.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load it; the library never does.  It shares no code, header,
 * table or helper with the CUDA path.
 *
 * Sources (page title, section):
 *  [R1] "Speculative Decoding in Custom LLM Servicing: Implementing Draft Models in Rust",
 *       section "The Memory Bandwidth Wall and Speculative Math": accept x_i with probability
 *       min(1, p(x_i)/q(x_i)); at the first rejection discard the rest and draw from
 *       max(0, p - q) / sum max(0, p - q).
 *  [R2] same page, section "The Verification Algorithm": target probabilities are
 *       softmax(logits / temperature) over all K+1 rows; the loop stops at the first
 *       rejection; if every draft is accepted the extra token is drawn from row K.
 *  [R3] same page, section "Orchestrating the Inference Loop": the target appended K+1
 *       rows and keeps 1 + accepted of them (target_len = current - (K+1) + 1 + accepted);
 *       section "KV Cache Rollback Mechanics": rolling back forward is an error.
 *  [A1] "Adding Speculative Decoding", table "The existing base": greedy verification
 *       accepts while draft == argmax and the extra token is the argmax at the first
 *       mismatch; section "Verification and sampling" item 2: greedy is the degenerate
 *       (one-hot draft) case of the uniform-vs-ratio test.
 *  [F1] FreeToken PR #836, section "Design": every verify row samples with its own
 *       request's temperature, top-k, top-p and greedy flag; presence and frequency
 *       penalties count the drafts before a row as already generated.  Its drafts are
 *       argmax proposals, so it samples every verify row as a decode step would and keeps
 *       the prefix of drafts that equals those samples (the one-hot-draft scheme).
 *  [S2] "Speculative Decoding: Draft Model Sampling, Rejection Sampling & On-Device
 *       Acceleration", Key Topic 2 and Section 2: the same accept/residual formulas.
 *
 * Readings where the pages leave a step open (each one is also listed in the design notes):
 *  - accept iff u < min(1, p/q) with no epsilon in the denominator; q == 0 < p accepts,
 *    p == 0 always rejects.
 *  - penalties are additive: z_v = logit_v - presence*[c_v > 0] - frequency*c_v, where c_v
 *    counts v among d_0..d_{i-1} plus the request's prior history count of v (an optional
 *    input: distinct ascending ids with counts >= 1); they apply before temperature and
 *    filtering, greedy rows too.
 *  - top-k keeps every token whose scaled logit is >= the k-th largest (ties kept); k <= 0 or
 *    k >= V disables it.  top-p then keeps v iff the renormalised mass of tokens strictly
 *    more likely than v is < top_p; top_p >= 1 disables it.  The kept set is renormalised.
 *  - inverse CDF in token-index order: the smallest v whose running sum exceeds u * W;
 *    if rounding leaves none, the largest v with positive weight.
 *  - a residual with W == 0 falls back to drawing from p.
 *  - uniforms: slot 0 of row i is the accept test of draft i; slot 1 of the final row is
 *    the residual or extra-token draw.
 *  - greedy argmax breaks ties toward the lowest token id; greedy rows read neither q nor u.
 *  - one-hot-draft scheme [F1]: row i's sample is drawn with slot 1 (the draw slot) of its
 *    own uniforms, on every row 0..k; slot 0 is unused there.
 *
 * Near-tie bookkeeping (decisions whose float64 value lies within 1e-5 of a boundary, where
 * an fp32 implementation may legitimately decide the other way) is reported per request.
 *
 * Parity pins: tests/test_oracle_*.py check this file against closed forms, the pages'
 * worked examples, brute force on tiny vocabularies and a Monte Carlo distribution test.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define NEAR_TOL 1e-5
#define NEAR_W 1e-6

typedef struct sv_oracle_batch {
    int32_t B, k_max, V, total_rows;
    int32_t logits_bf16;          /* 1: target_logits holds bf16 bit patterns (uint16) */
    const void *target_logits;    /* [total_rows, V] */
    const float *draft_probs;     /* [total_rows - B, V] */
    const int32_t *draft_tokens;  /* [total_rows - B] */
    const int32_t *num_drafts;    /* [B] */
    const int32_t *row_offsets;   /* [B+1], or NULL: request b owns rows b*(k_max+1) .. */
    const float *temperature;     /* [B] */
    const int32_t *top_k;         /* [B] */
    const float *top_p;           /* [B] */
    const float *presence;        /* [B] or NULL */
    const float *frequency;       /* [B] or NULL */
    const uint8_t *greedy;        /* [B] */
    const float *uniforms;        /* [total_rows, 2] */
    /* prior history, or NULL: request b generated tokens prior_tokens[o_b .. o_{b+1}) (distinct,
     * ascending) prior_counts[] times each, o = prior_offsets */
    const int32_t *prior_offsets; /* [B+1] */
    const int32_t *prior_tokens;
    const int32_t *prior_counts;
    int32_t prior_len;            /* entries in prior_tokens / prior_counts */
} sv_oracle_batch;

typedef struct sv_oracle_diag {
    int32_t decisions;  /* accept tests + draws + greedy argmaxes + filter thresholds on the path */
    int32_t near_ties;  /* decisions within the near-tie band */
    int32_t error;      /* 0, or the device-data error code of the request */
    int32_t near_accept, near_cdf, near_filter, near_argmax, near_w;  /* near_ties by kind */
    /* where on the request's path the near-ties are: bit i of the 64-bit mask (lo | hi << 32)
     * is set when the decision of row i whether to keep draft i (accept test, greedy compare,
     * or the one-hot scheme's sample compare) is a near-tie; near_final when the final token's
     * decision (the residual, extra-token or argmax draw of the stopping row) is one */
    uint32_t near_rows_lo, near_rows_hi;
    int32_t near_final;
} sv_oracle_diag;

/* Records a near-tie at row i's keep decision (final = 0) or at the final token (final = 1). */
static void mark_near(sv_oracle_diag *d, int32_t i, int final) {
    if (final) {
        d->near_final = 1;
    } else if (i < 32) {
        d->near_rows_lo |= 1u << i;
    } else if (i < 64) {
        d->near_rows_hi |= 1u << (i - 32);
    }
}

enum { E_OK = 0, E_LAYOUT = 1, E_TOKEN = 2, E_TEMP = 3, E_TOPP = 4, E_UNIFORM = 5, E_PENALTY = 6, E_HISTORY = 8 };

/* ---------------------------------------------------------------------------------- */

static double logit_at(const sv_oracle_batch *in, int64_t row, int32_t v) {
    int64_t off = row * (int64_t)in->V + v;
    if (in->logits_bf16) {
        uint32_t bits = (uint32_t)((const uint16_t *)in->target_logits)[off] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float *)in->target_logits)[off];
}

static int64_t row_start(const sv_oracle_batch *in, int32_t b) {
    return in->row_offsets ? (int64_t)in->row_offsets[b] : (int64_t)b * (in->k_max + 1);
}

/* Checks the request's layout and the inputs its path reads; returns an error code.
 * `slot_lo` is the first uniform slot the path reads (0 for the accept-test scheme, 1 for
 * the one-hot scheme, which reads only the draw slot). */
static int check_request_slots(const sv_oracle_batch *in, int32_t b, int slot_lo) {
    int32_t k = in->num_drafts[b];
    int64_t r0 = row_start(in, b);
    int64_t cap;
    if (in->row_offsets) {
        int64_t r1 = in->row_offsets[b + 1];
        if (r0 < 0 || r1 > in->total_rows || r1 <= r0) return E_LAYOUT;
        cap = r1 - r0 - 1;
    } else {
        cap = in->k_max;
        if ((int64_t)(b + 1) * (in->k_max + 1) > in->total_rows) return E_LAYOUT;
    }
    if (k < 0 || k > in->k_max || k > cap) return E_LAYOUT;
    int64_t d0 = r0 - b;
    for (int32_t i = 0; i < k; i++) {
        int32_t d = in->draft_tokens[d0 + i];
        if (d < 0 || d >= in->V) return E_TOKEN;
    }
    if (in->presence && !isfinite(in->presence[b])) return E_PENALTY;
    if (in->frequency && !isfinite(in->frequency[b])) return E_PENALTY;
    if (in->prior_offsets) {
        /* the history: ascending distinct ids in [0, V), each with a count >= 1 */
        int32_t lo = in->prior_offsets[b], hi = in->prior_offsets[b + 1];
        if (lo < 0 || hi < lo || hi > in->prior_len || (b == 0 && lo != 0)) return E_HISTORY;
        for (int32_t j = lo; j < hi; j++) {
            int32_t x = in->prior_tokens[j];
            if (x < 0 || x >= in->V || in->prior_counts[j] < 1) return E_HISTORY;
            if (j > lo && in->prior_tokens[j - 1] >= x) return E_HISTORY;
        }
    }
    if (!in->greedy[b]) {
        float T = in->temperature[b];
        if (!(T > 0.0f) || !isfinite(T)) return E_TEMP;
        float P = in->top_p[b];
        if (!(P > 0.0f && P <= 1.0f)) return E_TOPP;
        for (int32_t i = 0; i <= k; i++)
            for (int s = slot_lo; s < 2; s++) {
                float u = in->uniforms[(r0 + i) * 2 + s];
                if (!(u >= 0.0f && u < 1.0f)) return E_UNIFORM;
            }
    }
    return E_OK;
}

static int check_request(const sv_oracle_batch *in, int32_t b) { return check_request_slots(in, b, 0); }

/* Count of token v in request b's prior history (0 without one). */
static int32_t prior_count(const sv_oracle_batch *in, int32_t b, int32_t v) {
    if (!in->prior_offsets) return 0;
    for (int32_t j = in->prior_offsets[b]; j < in->prior_offsets[b + 1]; j++)
        if (in->prior_tokens[j] == v) return in->prior_counts[j];
    return 0;
}

/* z_v for row i of request b: the logit minus the presence/frequency penalty of what the
 * request generated before the row -- its prior history and the drafts d_0..d_{i-1}, which
 * count as already generated [F1]: c_v = prior_v + #{j < i : d_j = v}.  Returns 1 when some
 * token of the row carries a nonzero penalty. */
static int row_logits(const sv_oracle_batch *in, int32_t b, int32_t i, double *z) {
    int64_t row = row_start(in, b) + i;
    for (int32_t v = 0; v < in->V; v++) z[v] = logit_at(in, row, v);
    double pres = in->presence ? in->presence[b] : 0.0;
    double freq = in->frequency ? in->frequency[b] : 0.0;
    if (pres == 0.0 && freq == 0.0) return 0;
    const int32_t *d = in->draft_tokens + (row_start(in, b) - b);
    const int32_t h0 = in->prior_offsets ? in->prior_offsets[b] : 0;
    const int32_t nh = in->prior_offsets ? in->prior_offsets[b + 1] - h0 : 0;
    int penalised = 0;
    /* every distinct token generated before the row: the history's, then the drafts' */
    for (int32_t e = 0; e < nh + i; e++) {
        int32_t v;
        if (e < nh) {
            v = in->prior_tokens[h0 + e];
        } else {
            int32_t j = e - nh;
            v = d[j];
            int seen = prior_count(in, b, v) > 0;
            for (int32_t t = 0; t < j; t++) seen |= (d[t] == v);
            if (seen) continue;             /* apply once per distinct token */
        }
        int32_t c = prior_count(in, b, v);
        for (int32_t t = 0; t < i; t++) c += (d[t] == v);
        double pen = pres * (c > 0 ? 1.0 : 0.0) + freq * (double)c;
        z[v] -= pen;
        if (pen != 0.0) penalised = 1;
    }
    return penalised;
}

static int cmp_desc(const void *a, const void *b) {
    double x = *(const double *)a, y = *(const double *)b;
    return (x < y) - (x > y);
}

static int close_rel(double a, double b) {
    double s = fabs(a) > 1.0 ? fabs(a) : 1.0;
    return fabs(a - b) <= NEAR_TOL * s;
}

/* Greedy row [A1]: the argmax of z with ties to the lowest id.  *near is set when the row
 * carries penalties and the runner-up is within the near-tie band of the maximum. */
static int32_t row_argmax(const double *z, int32_t V, int penalised, int *near) {
    int32_t best = 0;
    for (int32_t v = 1; v < V; v++)
        if (z[v] > z[best]) best = v;
    *near = 0;
    if (penalised) {
        for (int32_t v = 0; v < V; v++)
            if (v != best && close_rel(z[best], z[v]) && z[v] != z[best]) *near = 1;
    }
    return best;
}

/* Where an fp32 implementation may legitimately draw a row's kept set differently: the
 * z/T interval [lo, hi] of the value levels whose membership sits on a near-tie (lo > hi:
 * none), and their total mass as a share of the final kept mass. */
typedef struct row_amb {
    double lo, hi, mass;
} row_amb;

static void amb_add(row_amb *a, double level) {
    if (a->lo > a->hi) { a->lo = level; a->hi = level; return; }
    if (level < a->lo) a->lo = level;
    if (level > a->hi) a->hi = level;
}

/* Sampled row [R2][F1]: p = softmax(z / T) restricted to top-k, then to top-p, renormalised.
 * Writes p[0..V).  *decisions counts the filter thresholds of the row; *amb receives the
 * near-tie band of the cut.  Returns the number of tokens kept. */
static int32_t row_probs(const sv_oracle_batch *in, int32_t b, const double *z, int penalised,
                         double *p, double *scratch, int *decisions, row_amb *amb) {
    const int32_t V = in->V;
    const double T = in->temperature[b];
    const int32_t K = in->top_k[b];
    const double P = in->top_p[b];
    double *zs = scratch; /* V doubles */
    amb->lo = 1.0;
    amb->hi = 0.0;
    amb->mass = 0.0;

    for (int32_t v = 0; v < V; v++) p[v] = z[v] / T;          /* p[] holds z' for now */
    double m = p[0];
    for (int32_t v = 1; v < V; v++) if (p[v] > m) m = p[v];

    /* top-k threshold: the K-th largest scaled logit, ties kept */
    double tau = -INFINITY;
    if (K > 0 && K < V) {
        memcpy(zs, p, sizeof(double) * V);
        qsort(zs, V, sizeof(double), cmp_desc);
        tau = zs[K - 1];
        (*decisions)++;
        if (penalised) {   /* values near the cut may order differently in fp32 */
            for (int32_t j = K; j < V; j++)
                if (zs[j] < tau) {
                    if (close_rel(tau, zs[j])) { amb_add(amb, tau); amb_add(amb, zs[j]); }
                    break;
                }
        }
    }
    /* unnormalised weights of the top-k set */
    double ZK = 0.0;
    for (int32_t v = 0; v < V; v++) ZK += (p[v] >= tau) ? exp(p[v] - m) : 0.0;

    /* top-p: walk distinct values from the largest; a value is kept while the mass strictly
     * above it is < top_p (in units of the top-k mass) */
    if (P < 1.0) {
        int32_t n = 0;
        for (int32_t v = 0; v < V; v++) if (p[v] >= tau) zs[n++] = p[v];
        qsort(zs, n, sizeof(double), cmp_desc);
        double above = 0.0, last_kept = zs[0];
        int32_t j = 0;
        int cut = 0;
        double first_excl = 0.0;
        while (j < n) {
            double level = zs[j];
            int32_t c = 0;
            while (j + c < n && zs[j + c] == level) c++;
            double lm = (double)c * exp(level - m);
            /* near-tie: either end of this level's cumulative mass within 1e-5 of top_p */
            if (fabs(above / ZK - P) < NEAR_TOL || fabs((above + lm) / ZK - P) < NEAR_TOL) amb_add(amb, level);
            if (!cut && above / ZK < P) {
                last_kept = level;
            } else if (!cut) {
                cut = 1;
                first_excl = level;
                if (penalised && close_rel(last_kept, first_excl)) { amb_add(amb, last_kept); amb_add(amb, first_excl); }
            }
            if (cut && above / ZK - P >= NEAR_TOL) break;   /* past the band */
            above += lm;
            j += c;
        }
        (*decisions)++;
        tau = last_kept;
    }
    double Z = 0.0;
    int32_t kept = 0;
    for (int32_t v = 0; v < V; v++) {
        if (p[v] >= tau) { Z += exp(p[v] - m); kept++; }
    }
    if (amb->lo <= amb->hi) {
        double am = 0.0;
        for (int32_t v = 0; v < V; v++)
            if (p[v] >= amb->lo && p[v] <= amb->hi) am += exp(p[v] - m);
        amb->mass = am / Z;
    }
    for (int32_t v = 0; v < V; v++) p[v] = (p[v] >= tau) ? exp(p[v] - m) / Z : 0.0;
    return kept;
}

static int in_amb(const row_amb *a, double zprime) { return a->lo <= a->hi && zprime >= a->lo && zprime <= a->hi; }

/* Inverse CDF over w[0..V) in token-index order [R1]: the smallest v whose running sum is
 * > u * W, where W is the running sum's total; the largest positive-weight v if rounding
 * leaves none.  *near is set when the running sum at the boundary is within 1e-5 (of W) of
 * u * W (1), or within 1e-5 + shift (2): `shift` is how far (in units of W) the running sums
 * can move when the row's ambiguous kept-set levels flip (0 when there are none). */
static int32_t inverse_cdf(const double *w, int32_t V, double u, double shift, int *near) {
    double W = 0.0;
    for (int32_t v = 0; v < V; v++) W += w[v];
    double target = u * W, c = 0.0;
    *near = 0;
    for (int32_t v = 0; v < V; v++) {
        double prev = c;
        c += w[v];
        if (c > target) {
            const double dist = fmin(fabs(prev / W - u), fabs(c / W - u));
            if (dist < NEAR_TOL) *near = 1;
            else if (dist < NEAR_TOL + shift) *near = 2;
            return v;
        }
    }
    for (int32_t v = V - 1; v >= 0; v--)
        if (w[v] > 0.0) { *near = 1; return v; }
    *near = 1;
    return 0;
}

/* ---------------------------------------------------------------------------------- */
/* one request                                                                          */

static void verify_one(const sv_oracle_batch *in, int32_t b, int32_t *out_tok, int32_t *acc,
                       double *out_pq, uint8_t *pq_near, sv_oracle_diag *dg,
                       double *z, double *p, double *r, double *scratch) {
    const int32_t V = in->V;
    const int32_t kmax1 = in->k_max + 1;
    for (int32_t j = 0; j < kmax1; j++) out_tok[(int64_t)b * kmax1 + j] = -1;
    sv_oracle_diag d = {0, 0, 0, 0, 0, 0, 0, 0, 0u, 0u, 0};
    int err = check_request(in, b);
    const int64_t r0 = row_start(in, b), d0 = r0 - b;
    const int32_t k = in->num_drafts[b];
    if (err) {
        acc[b] = -1;
        if (out_pq && k >= 0 && k <= in->k_max && d0 >= 0)
            for (int32_t i = 0; i < k && d0 + i < in->total_rows - in->B; i++) {
                out_pq[(d0 + i) * 2] = NAN;
                out_pq[(d0 + i) * 2 + 1] = NAN;
            }
        d.error = err;
        if (dg) dg[b] = d;
        return;
    }
    const int32_t *drafts = in->draft_tokens + d0;
    int32_t a = k, token = -1;
    int decided = 0;

    if (in->greedy[b]) {
        /* [A1] accept while d_i == argmax_i; the output at the first mismatch (or row k) is
         * that row's argmax */
        for (int32_t i = 0; i <= k; i++) {
            int pen = row_logits(in, b, i, z), nt = 0;
            int32_t g = row_argmax(z, V, pen, &nt);
            if (i < k) {
                if (out_pq) { out_pq[(d0 + i) * 2] = NAN; out_pq[(d0 + i) * 2 + 1] = NAN; }
                if (pq_near) pq_near[d0 + i] = 0;
            }
            if (!decided) {
                d.decisions++;
                d.near_ties += nt;
                d.near_argmax += nt;
                const int stop = (i == k || drafts[i] != g);
                /* a near-tied argmax could move both the compare with the draft and, at the
                 * stopping row, the final token */
                if (nt && i < k) mark_near(&d, i, 0);
                if (nt && stop) mark_near(&d, i, 1);
                if (stop) { a = i; token = g; decided = 1; }
            }
        }
    } else {
        for (int32_t i = 0; i <= k; i++) {
            int pen = row_logits(in, b, i, z);
            int dec = 0;
            row_amb amb;
            row_probs(in, b, z, pen, p, scratch, &dec, &amb);
            if (i < k) {
                int32_t x = drafts[i];
                double px = p[x];
                double qx = (double)in->draft_probs[(d0 + i) * (int64_t)V + x];
                /* the draft's own membership in the kept set is on a near-tie */
                const int nt = in_amb(&amb, z[x] / in->temperature[b]);
                if (out_pq) { out_pq[(d0 + i) * 2] = px; out_pq[(d0 + i) * 2 + 1] = qx; }
                /* p(x) is not comparable when x's membership is ambiguous, or when flipping the
                 * ambiguous levels would move the normaliser enough to shift p(x) by 1e-6 */
                if (pq_near) pq_near[d0 + i] = (uint8_t)(nt || px * amb.mass >= 1e-6);
                if (decided) continue;
                d.decisions += dec + 1;
                double u = in->uniforms[(r0 + i) * 2 + 0];
                int accept, kind = nt ? 2 : 0;   /* near-tie kind: 1 accept band, 2 kept set */
                if (px > 0.0 && qx == 0.0) {
                    accept = 1;
                } else if (px > 0.0) {
                    double ratio = px / qx;
                    double thr = ratio < 1.0 ? ratio : 1.0;
                    accept = u < thr;
                    if (!kind && fabs(u - thr) < NEAR_TOL) kind = 1;
                    /* flipping an ambiguous level of the kept set moves Z, and with it
                     * p(x)/q(x), by up to amb.mass relative */
                    else if (!kind && fabs(u - thr) < NEAR_TOL + amb.mass * thr) kind = 2;
                } else {
                    accept = 0;
                }
                if (kind == 1) d.near_accept++;
                if (kind == 2) d.near_filter++;
                if (kind) {
                    d.near_ties++;
                    mark_near(&d, i, 0);
                }
                if (!accept) {
                    /* [R1] residual max(0, p - q) at the rejected row, normalised by its sum */
                    const float *q = in->draft_probs + (d0 + i) * (int64_t)V;
                    double W = 0.0;
                    for (int32_t v = 0; v < V; v++) {
                        double t = p[v] - (double)q[v];
                        r[v] = t > 0.0 ? t : 0.0;
                        W += r[v];
                    }
                    double u1 = in->uniforms[(r0 + i) * 2 + 1];
                    int cn = 0;
                    /* flipping the ambiguous levels moves p, hence r's running sums, by up to
                     * amb.mass (in units of p's total), i.e. amb.mass / W of r's */
                    if (W > 0.0) {
                        token = inverse_cdf(r, V, u1, amb.mass / W, &cn);
                    } else {
                        token = inverse_cdf(p, V, u1, amb.mass, &cn);   /* empty residual: draw from p */
                    }
                    if (W < NEAR_W) { cn = 1; d.near_w++; }
                    else if (cn == 1) d.near_cdf++;
                    else if (cn == 2) d.near_filter++;
                    cn = cn != 0;
                    d.decisions++;
                    d.near_ties += cn;
                    if (cn) mark_near(&d, i, 1);
                    a = i;
                    decided = 1;
                }
            } else if (!decided) {
                /* [R2] every draft accepted: the extra token comes from row k */
                int cn = 0;
                d.decisions += dec + 1;
                token = inverse_cdf(p, V, in->uniforms[(r0 + k) * 2 + 1], amb.mass, &cn);
                if (cn == 1) d.near_cdf++;
                if (cn == 2) d.near_filter++;
                cn = cn != 0;
                d.near_ties += cn;
                if (cn) mark_near(&d, k, 1);
                a = k;
                decided = 1;
            }
        }
    }
    for (int32_t j = 0; j < a; j++) out_tok[(int64_t)b * kmax1 + j] = drafts[j];
    out_tok[(int64_t)b * kmax1 + a] = token;
    acc[b] = a;
    if (dg) dg[b] = d;
}

/* One request under the one-hot-draft scheme [F1]: the drafts are argmax proposals (q_i is
 * one-hot at d_i), so every row i = 0..k is sampled as a decode step would sample it -- the
 * argmax for a greedy request, else t_i = inverse CDF of the filtered p_i at the row's draw
 * uniform u_{i,1} -- and the drafts are accepted while d_i == t_i.  The output at the first
 * mismatch, or at row k, is that row's own sample.  No q is read; slot 0 of the uniforms is
 * not read.  out_pq receives (p_i(d_i), 1): the one-hot draft puts mass 1 on its token. */
static void verify_one_onehot(const sv_oracle_batch *in, int32_t b, int32_t *out_tok, int32_t *acc,
                              double *out_pq, uint8_t *pq_near, sv_oracle_diag *dg,
                              double *z, double *p, double *scratch) {
    const int32_t V = in->V;
    const int32_t kmax1 = in->k_max + 1;
    for (int32_t j = 0; j < kmax1; j++) out_tok[(int64_t)b * kmax1 + j] = -1;
    sv_oracle_diag d = {0, 0, 0, 0, 0, 0, 0, 0, 0u, 0u, 0};
    int err = check_request_slots(in, b, 1);
    const int64_t r0 = row_start(in, b), d0 = r0 - b;
    const int32_t k = in->num_drafts[b];
    if (err) {
        acc[b] = -1;
        if (out_pq && k >= 0 && k <= in->k_max && d0 >= 0)
            for (int32_t i = 0; i < k && d0 + i < in->total_rows - in->B; i++) {
                out_pq[(d0 + i) * 2] = NAN;
                out_pq[(d0 + i) * 2 + 1] = NAN;
            }
        d.error = err;
        if (dg) dg[b] = d;
        return;
    }
    const int32_t *drafts = in->draft_tokens + d0;
    int32_t a = k, token = -1;
    int decided = 0;
    for (int32_t i = 0; i <= k; i++) {
        int pen = row_logits(in, b, i, z);
        int32_t t;
        int nt = 0, cn = 0, dec = 0;
        row_amb amb;
        if (in->greedy[b]) {
            t = row_argmax(z, V, pen, &nt);
            if (i < k) {
                if (out_pq) { out_pq[(d0 + i) * 2] = NAN; out_pq[(d0 + i) * 2 + 1] = NAN; }
                if (pq_near) pq_near[d0 + i] = 0;
            }
            if (decided) continue;
            d.decisions++;
            d.near_ties += nt;
            d.near_argmax += nt;
        } else {
            row_probs(in, b, z, pen, p, scratch, &dec, &amb);
            if (i < k) {
                int32_t x = drafts[i];
                if (out_pq) { out_pq[(d0 + i) * 2] = p[x]; out_pq[(d0 + i) * 2 + 1] = 1.0; }
                if (pq_near)
                    pq_near[d0 + i] = (uint8_t)(in_amb(&amb, z[x] / in->temperature[b]) || p[x] * amb.mass >= 1e-6);
            }
            if (decided) continue;
            /* tokens whose membership of the kept set is on a near-tie could move the boundary */
            t = inverse_cdf(p, V, in->uniforms[(r0 + i) * 2 + 1], amb.mass, &cn);
            if (cn == 1) d.near_cdf++;
            if (cn == 2) d.near_filter++;
            cn = cn != 0;
            d.decisions += dec + 1;
            d.near_ties += cn;
            nt = cn;
        }
        const int stop = (i == k || drafts[i] != t);
        /* a near-tied sample (or argmax) could move the compare with the draft and, at the
         * stopping row, the final token */
        if (nt && i < k) mark_near(&d, i, 0);
        if (nt && stop) mark_near(&d, i, 1);
        if (stop) {
            a = i;
            token = t;
            decided = 1;
        }
    }
    for (int32_t j = 0; j < a; j++) out_tok[(int64_t)b * kmax1 + j] = drafts[j];
    out_tok[(int64_t)b * kmax1 + a] = token;
    acc[b] = a;
    if (dg) dg[b] = d;
}

/* Verifies requests [b_lo, b_hi).  Output arrays are full-batch sized; only the rows of
 * these requests are written.  Safe to call concurrently on disjoint request ranges. */
int sv_oracle_verify(const sv_oracle_batch *in, int32_t b_lo, int32_t b_hi, int32_t *out_tokens,
                     int32_t *accept_len, double *out_pq, uint8_t *pq_near, sv_oracle_diag *diag) {
    if (!in || !out_tokens || !accept_len || in->V < 1 || b_lo < 0 || b_hi > in->B) return -1;
    size_t V = (size_t)in->V;
    double *buf = (double *)malloc(sizeof(double) * V * 4);
    if (!buf) return -2;
    for (int32_t b = b_lo; b < b_hi; b++)
        verify_one(in, b, out_tokens, accept_len, out_pq, pq_near, diag, buf, buf + V, buf + 2 * V,
                   buf + 3 * V);
    free(buf);
    return 0;
}

/* Verifies requests [b_lo, b_hi) under the one-hot-draft scheme (verify_one_onehot);
 * draft_probs is not read and may be NULL.  Same outputs and concurrency as
 * sv_oracle_verify. */
int sv_oracle_verify_onehot(const sv_oracle_batch *in, int32_t b_lo, int32_t b_hi, int32_t *out_tokens,
                            int32_t *accept_len, double *out_pq, uint8_t *pq_near, sv_oracle_diag *diag) {
    if (!in || !out_tokens || !accept_len || in->V < 1 || b_lo < 0 || b_hi > in->B) return -1;
    size_t V = (size_t)in->V;
    double *buf = (double *)malloc(sizeof(double) * V * 3);
    if (!buf) return -2;
    for (int32_t b = b_lo; b < b_hi; b++)
        verify_one_onehot(in, b, out_tokens, accept_len, out_pq, pq_near, diag, buf, buf + V, buf + 2 * V);
    free(buf);
    return 0;
}

/* The full distribution a row is sampled from: the filtered, renormalised target p for a
 * sampled request, or one-hot at the argmax for a greedy one.  Returns the kept count, or
 * a negative value on bad arguments. */
int32_t sv_oracle_row_probs(const sv_oracle_batch *in, int32_t b, int32_t i, double *p) {
    if (!in || !p || b < 0 || b >= in->B || i < 0 || i > in->num_drafts[b]) return -1;
    if (check_request(in, b) == E_LAYOUT) return -1;
    size_t V = (size_t)in->V;
    double *buf = (double *)malloc(sizeof(double) * V * 2);
    if (!buf) return -2;
    int pen = row_logits(in, b, i, buf);
    int32_t kept;
    if (in->greedy[b]) {
        int nt;
        int32_t g = row_argmax(buf, in->V, pen, &nt);
        for (size_t v = 0; v < V; v++) p[v] = 0.0;
        p[g] = 1.0;
        kept = 1;
    } else {
        int dec = 0;
        row_amb amb;
        kept = row_probs(in, b, buf, pen, p, buf + V, &dec, &amb);
    }
    free(buf);
    return kept;
}

/* The normalised residual max(0, p_i - q_i) / W at draft row i of request b (sampled
 * requests), with W returned through *W_out. */
int32_t sv_oracle_residual(const sv_oracle_batch *in, int32_t b, int32_t i, double *r, double *W_out) {
    if (!in || !r || b < 0 || b >= in->B || i < 0 || i >= in->num_drafts[b] || in->greedy[b]) return -1;
    size_t V = (size_t)in->V;
    double *buf = (double *)malloc(sizeof(double) * V * 3);
    if (!buf) return -2;
    int pen = row_logits(in, b, i, buf);
    int dec = 0;
    row_amb amb;
    row_probs(in, b, buf, pen, buf + V, buf + 2 * V, &dec, &amb);
    const float *q = in->draft_probs + (row_start(in, b) - b + i) * (int64_t)in->V;
    double W = 0.0;
    for (size_t v = 0; v < V; v++) {
        double t = buf[V + v] - (double)q[v];
        r[v] = t > 0.0 ? t : 0.0;
        W += r[v];
    }
    if (W > 0.0)
        for (size_t v = 0; v < V; v++) r[v] /= W;
    if (W_out) *W_out = W;
    free(buf);
    return 0;
}

/* Target KV rollback [R3]: the verify step appended k_b + 1 rows and keeps 1 + accept_len
 * of them: L' = L - (k_b + 1) + 1 + a.  A length that would move forward (a > k_b), a
 * negative accept length or a negative result is an error: that request's output is -1 and
 * the return value counts the errors. */
int32_t sv_oracle_rollback(const int32_t *kv_seq_len, const int32_t *accept_len,
                           const int32_t *num_drafts, int32_t B, int32_t *out_len) {
    int32_t errors = 0;
    for (int32_t b = 0; b < B; b++) {
        int64_t L = kv_seq_len[b], k = num_drafts[b], a = accept_len[b];
        int64_t t = L - (k + 1) + 1 + a;
        if (k < 0 || a < 0 || a > k || t < 0 || t > L) {
            out_len[b] = -1;
            errors++;
        } else {
            out_len[b] = (int32_t)t;
        }
    }
    return errors;
}
