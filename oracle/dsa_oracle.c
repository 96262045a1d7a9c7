/*
 * dsa_oracle.c -- CPU oracle for diagonal-aware sparse decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the decode path computes.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg load it; the CUDA library never
 * links, includes or calls it, and it shares no code with the CUDA library.
 *
 * Source: "Understanding and Exploiting Diagonal Attention Sparsity in
 * Autoregressive Image Generation" (arXiv 2609.19702), section 4,
 * Algorithm 1 "Diagonal-Aware Sparse Attention" with its three phases, the
 * detailed explanation of Fig. 12 (N_r = 7, N_att = 4), the cost analysis,
 * and section 5.1 "Our methods" for the Diagonal+sink4 variant.
 *
 * Representation follows the algorithm literally:
 *   - the decode cache is indexed by absolute decode position; eviction
 *     frees the row and leaves a NULL ("K[t - N_r] <- empty");
 *   - skip_idx is a list of absolute decode positions, every entry is
 *     incremented by one at each shift;
 *   - window is [max(0, t - N_r) .. t]; idx = window minus skip_idx minus
 *     evicted rows, ascending;
 *   - Attn(Q_t, K_p + K[idx], V_p + V[idx]) is softmax(q K^T / sqrt(d)) V
 *     over the prompt rows followed by the idx rows.
 * All arithmetic is fp64.  Inputs are whatever the caller passes (the tests
 * pass bf16- or fp32-rounded values widened to double).
 *
 * Readings where the page leaves a step open (each is listed in the design
 * notes of the repository):
 *   - phase 2 starts at t = N_att - 1 (the algorithm and the Fig. 12 example
 *     select at t = 3 for N_att = 4), t counts from 0;
 *   - the evicted row t - N_r is inside the literal window but holds nothing,
 *     so it is not attended: the live window has N_r rows;
 *   - the argmin is taken over the logits q.k of the attended decode rows
 *     idx (prompt rows excluded, the current token included); softmax is
 *     strictly increasing so this is the same choice as argmin of w;
 *   - exact ties go to the first entry of idx, i.e. the oldest position;
 *   - Diagonal+sink4: decode positions 0..sink-1 join the always-attended
 *     prompt; the algorithm then runs on positions >= sink with step
 *     t' = t - sink, window N_r - sink and budget N_att - sink, so the KV
 *     held stays <= N_r + L_p and the attended decode rows stay <= N_att.
 *     With N_att = N_r this is StreamingLLM with `sink` sinks.
 *
 * FP8 KV storage (orc_set_kv_fp8).  Section 6 (Related Works, "KV
 * quantization for LLM") calls KV quantization orthogonal to the method and
 * applicable on top of it, and fixes no scheme.  The
 * reading taken: every K and V row the cache holds (prompt rows, sink rows,
 * decode rows) is stored as OCP FP8 E4M3 codes with one fp32 scale per
 * stream for K and one for V; the stored code of an element x is the E4M3
 * value nearest to fp32(x) * fp32(1 / scale) (ties to the even code, beyond
 * the largest finite value 448 the value 448: "satfinite"), and attention
 * uses code * scale.  Everything after the store is the fp64 algorithm
 * above, unchanged.
 *
 * Near ties: a caller (the parity test) may pass the position its own
 * implementation selected.  If it differs from the oracle's argmin but its
 * logit is within 1e-4 * max(|a|, |b|, 1) of the minimum logit, the oracle
 * adopts it and continues from it (reported in orc_info.adopted); otherwise
 * the oracle keeps its own choice and reports a mismatch.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_NEAR_TIE_REL 1e-4

typedef struct orc_info {
    int phase;         /* 0 sink fill, 1 full attention, 2 grow skip set, 3 evict and shift */
    int t;             /* decode step (0-based) */
    int t_inner;       /* step of the inner algorithm (t - sink), -1 during sink fill */
    int n_prefix;      /* always-attended rows this step (prompt, plus sinks) */
    int n_idx;         /* attended decode rows of the inner algorithm */
    int selected;      /* inner position appended to skip_idx, -1 if none */
    int oracle_pick;   /* the oracle's own argmin position, -1 if no selection */
    int adopted;       /* 1: the caller's pick was adopted at a near tie */
    int mismatch;      /* 1: the caller's pick differs and is not a near tie */
    int live_rows;     /* decode rows held (prompt excluded) after the step */
    int n_skip;        /* |skip_idx| after the step */
    double min_logit;  /* lowest q.k over idx (selection steps only) */
    double pick_logit; /* q.k of the caller's pick (selection steps, if given) */
} orc_info;

typedef struct orc_stream {
    int d, L_p, N_r, N_att, sink;
    int Nr, Na;           /* window and budget of the inner algorithm */
    int t;                /* decode steps taken */
    int prefilled;
    int np;               /* rows in the always-attended prefix */
    double *Kp, *Vp;      /* [(L_p + sink) * d] */
    int cap;              /* slots in the position-indexed decode cache */
    double **K, **V;      /* by inner decode position; NULL after eviction */
    int *skip, n_skip;    /* skip_idx, absolute inner positions, insertion order */
    int *idx, n_idx;      /* idx of the last step */
    int live;             /* decode rows held */
    int fp8;              /* 1: rows are stored as E4M3 codes (see the header) */
    float k_scale, v_scale, k_inv, v_inv;
    int mutation;         /* planted mistake for the pin tests; 0 = faithful */
} orc_stream;

/* Planted mistakes.  Only the pin tests set these, to show that the pins
 * catch each kind of error; the faithful oracle runs with 0. */
enum {
    MUT_NONE = 0,
    MUT_NO_SHIFT = 1,        /* skip_idx is never shifted */
    MUT_ARGMAX = 2,          /* selects the highest logit */
    MUT_NO_PROMPT = 3,       /* prompt rows are not attended */
    MUT_NO_EVICT = 4,        /* the oldest row is never evicted */
    MUT_LATE_PHASE2 = 5,     /* phase 2 starts at t = N_att */
    MUT_SCALE = 6,           /* logits scaled by 1/d instead of 1/sqrt(d) */
    MUT_SKIP_NOW = 7,        /* the newly selected row is skipped in the same step */
    MUT_BUDGET = 8,          /* one selection too many */
    MUT_NEWEST_TIE = 9,      /* exact ties go to the newest position */
    MUT_FP8_SWAP = 10,       /* K rows quantized with the V scale and V rows with the K scale */
    MUT_FP8_SCALE = 11,      /* codes of x * scale instead of x / scale */
    MUT_FP8_TRUNC = 12,      /* codes rounded toward zero instead of to nearest */
    MUT_FP8_PROMPT = 13      /* prompt rows stored unquantized */
};

/* ---- OCP FP8 E4M3 ("E4M3FN"): 1 sign bit, 4 exponent bits (bias 7), 3
 * mantissa bits; no infinities, code 0x7F / 0xFF is NaN, so the largest
 * finite magnitude is 1.75 * 2^8 = 448; exponent field 0 holds the
 * subnormals m * 2^-9. */
double orc_e4m3_decode(unsigned char c)
{
    const int sgn = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    const double mag = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return sgn ? -mag : mag;
}

/* Nearest finite E4M3 value to y by exhaustive search over the 127
 * non-negative finite codes; an exact midpoint goes to the even code (the
 * one whose mantissa ends in 0); magnitudes beyond 448 give 448. */
unsigned char orc_e4m3_encode(float y)
{
    if (y != y) return 0x7F;
    const double a = fabs((double)y);
    if (a > 448.0) return (unsigned char)(126 | (signbit(y) ? 0x80 : 0));
    int best = 0;
    double berr = a;
    for (int c = 1; c < 127; ++c) {
        const double err = fabs(orc_e4m3_decode((unsigned char)c) - a);
        if (err < berr || (err == berr && (c & 1) == 0)) {
            berr = err;
            best = c;
        }
    }
    return (unsigned char)(best | (signbit(y) ? 0x80 : 0));
}

/* Largest-magnitude finite code not above |y| (planted mistake only). */
static unsigned char e4m3_trunc(float y)
{
    const double a = fabs((double)y);
    int best = 0;
    for (int c = 1; c < 127; ++c)
        if (orc_e4m3_decode((unsigned char)c) <= a) best = c;
    return (unsigned char)(best | (signbit(y) ? 0x80 : 0));
}

/* A stored row: x unchanged, or code * scale with code = E4M3(fp32(x) * inv).
 * `prompt` marks rows loaded by the prefill. */
static void store_row(const orc_stream *st, double *dst, const double *x, int is_v, int prompt)
{
    const int m = st->mutation;
    if (!st->fp8 || (prompt && m == MUT_FP8_PROMPT)) {
        for (int i = 0; i < st->d; ++i) dst[i] = x[i];
        return;
    }
    const int use_v = (m == MUT_FP8_SWAP) ? !is_v : is_v;
    const float scale = use_v ? st->v_scale : st->k_scale;
    const float inv = (m == MUT_FP8_SCALE) ? scale : (use_v ? st->v_inv : st->k_inv);
    for (int i = 0; i < st->d; ++i) {
        const float y = (float)x[i] * inv;
        const unsigned char c = (m == MUT_FP8_TRUNC) ? e4m3_trunc(y) : orc_e4m3_encode(y);
        dst[i] = orc_e4m3_decode(c) * (double)scale;
    }
}

static double dot(const double *a, const double *b, int d)
{
    double s = 0.0;
    for (int i = 0; i < d; ++i) s += a[i] * b[i];
    return s;
}

orc_stream *orc_create(int d, int L_p, int N_r, int N_att, int sink)
{
    if (d <= 0 || L_p < 0 || sink < 0 || N_att < 1 || N_att > N_r) return NULL;
    if (sink > 0 && (N_att <= sink || N_r <= sink)) return NULL;
    orc_stream *st = (orc_stream *)calloc(1, sizeof(orc_stream));
    if (!st) return NULL;
    st->d = d; st->L_p = L_p; st->N_r = N_r; st->N_att = N_att; st->sink = sink;
    st->Nr = N_r - sink;
    st->Na = N_att - sink;
    st->Kp = (double *)calloc((size_t)(L_p + sink) * d + 1, sizeof(double));
    st->Vp = (double *)calloc((size_t)(L_p + sink) * d + 1, sizeof(double));
    st->skip = (int *)calloc((size_t)st->Nr + 2, sizeof(int));
    st->idx = (int *)calloc((size_t)st->Nr + 2, sizeof(int));
    if (!st->Kp || !st->Vp || !st->skip || !st->idx) {
        free(st->Kp); free(st->Vp); free(st->skip); free(st->idx); free(st);
        return NULL;
    }
    return st;
}

void orc_destroy(orc_stream *st)
{
    if (!st) return;
    for (int j = 0; j < st->cap; ++j) { free(st->K[j]); free(st->V[j]); }
    free(st->K); free(st->V);
    free(st->Kp); free(st->Vp); free(st->skip); free(st->idx);
    free(st);
}

void orc_set_mutation(orc_stream *st, int m) { st->mutation = m; }

/* Stores rows as E4M3 codes with the given per-stream scales from the next
 * prefill on.  Returns -1 unless both scales are positive and finite. */
int orc_set_kv_fp8(orc_stream *st, float k_scale, float v_scale)
{
    if (!(k_scale > 0.0f) || !(v_scale > 0.0f) || isinf(k_scale) || isinf(v_scale)) return -1;
    st->fp8 = 1;
    st->k_scale = k_scale;
    st->v_scale = v_scale;
    st->k_inv = 1.0f / k_scale;
    st->v_inv = 1.0f / v_scale;
    return 0;
}

/* Loads the prompt KV (always attended in full) and resets the decode state. */
int orc_prefill(orc_stream *st, const double *Kp, const double *Vp)
{
    for (int j = 0; j < st->cap; ++j) {
        free(st->K[j]); free(st->V[j]);
        st->K[j] = st->V[j] = NULL;
    }
    for (int i = 0; i < st->L_p; ++i) {
        store_row(st, st->Kp + (size_t)i * st->d, Kp + (size_t)i * st->d, 0, 1);
        store_row(st, st->Vp + (size_t)i * st->d, Vp + (size_t)i * st->d, 1, 1);
    }
    st->np = st->L_p;
    st->t = 0;
    st->n_skip = 0;
    st->n_idx = 0;
    st->live = 0;
    st->prefilled = 1;
    return 0;
}

/* out = softmax(q [Kp ; K[idx]]^T / sqrt(d)) [Vp ; V[idx]] in fp64. */
static void attn(const orc_stream *st, const double *q, double *out)
{
    const int d = st->d;
    const int np = (st->mutation == MUT_NO_PROMPT) ? 0 : st->np;
    const int n = np + st->n_idx;
    const double scale = (st->mutation == MUT_SCALE) ? 1.0 / d : 1.0 / sqrt((double)d);
    double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    for (int i = 0; i < np; ++i) s[i] = dot(q, st->Kp + (size_t)i * d, d) * scale;
    for (int j = 0; j < st->n_idx; ++j) s[np + j] = dot(q, st->K[st->idx[j]], d) * scale;
    double m = -INFINITY;
    for (int i = 0; i < n; ++i) if (s[i] > m) m = s[i];
    double z = 0.0;
    for (int i = 0; i < n; ++i) { s[i] = exp(s[i] - m); z += s[i]; }
    for (int c = 0; c < d; ++c) out[c] = 0.0;
    for (int i = 0; i < n; ++i) {
        const double *v = (i < np) ? st->Vp + (size_t)i * d : st->V[st->idx[i - np]];
        const double w = s[i] / z;
        for (int c = 0; c < d; ++c) out[c] += w * v[c];
    }
    free(s);
}

static int in_skip(const orc_stream *st, int j)
{
    for (int i = 0; i < st->n_skip; ++i) if (st->skip[i] == j) return 1;
    return 0;
}

/* idx <- window - skip_idx, ascending, without evicted rows. */
static void build_idx(orc_stream *st, int tt)
{
    int lo = tt - st->Nr;
    if (lo < 0) lo = 0;
    st->n_idx = 0;
    for (int j = lo; j <= tt; ++j) {
        if (st->K[j] == NULL) continue;
        if (in_skip(st, j)) continue;
        st->idx[st->n_idx++] = j;
    }
}

static void shift_skip(orc_stream *st)
{
    if (st->mutation == MUT_NO_SHIFT) return;
    for (int i = 0; i < st->n_skip; ++i) st->skip[i] += 1;
}

static int ensure_cap(orc_stream *st, int need)
{
    if (need <= st->cap) return 0;
    int nc = st->cap ? st->cap : 64;
    while (nc < need) nc *= 2;
    double **K = (double **)realloc(st->K, sizeof(double *) * (size_t)nc);
    if (!K) return -1;
    st->K = K;
    double **V = (double **)realloc(st->V, sizeof(double *) * (size_t)nc);
    if (!V) return -1;
    st->V = V;
    for (int j = st->cap; j < nc; ++j) st->K[j] = st->V[j] = NULL;
    st->cap = nc;
    return 0;
}

/* One decode step.  `caller_pick` is the inner position the implementation
 * under test selected at this step (-1: none given).  Returns 0, or -1 on a
 * usage error (step before prefill, allocation failure). */
int orc_step(orc_stream *st, const double *q, const double *k, const double *v,
             double *out, int caller_pick, orc_info *info)
{
    const int d = st->d;
    orc_info inf;
    memset(&inf, 0, sizeof(inf));
    inf.selected = inf.oracle_pick = -1;
    inf.t = st->t;
    if (!st->prefilled) return -1;

    if (st->t < st->sink) {
        /* Diagonal+sink4: the first `sink` decode tokens join the prefix. */
        store_row(st, st->Kp + (size_t)st->np * d, k, 0, 0);
        store_row(st, st->Vp + (size_t)st->np * d, v, 1, 0);
        st->np += 1;
        st->n_idx = 0;
        attn(st, q, out);
        inf.phase = 0;
        inf.t_inner = -1;
    } else {
        const int tt = st->t - st->sink;
        const int Nr = st->Nr, Na = st->Na;
        if (ensure_cap(st, tt + 1)) return -1;
        st->K[tt] = (double *)malloc(sizeof(double) * d);
        st->V[tt] = (double *)malloc(sizeof(double) * d);
        if (!st->K[tt] || !st->V[tt]) return -1;
        store_row(st, st->K[tt], k, 0, 0);
        store_row(st, st->V[tt], v, 1, 0);
        st->live += 1;
        inf.t_inner = tt;

        const int phase1_end = (st->mutation == MUT_LATE_PHASE2) ? Na : Na - 1;
        if (tt < phase1_end) {
            /* Phase 1: full attention over the window. */
            inf.phase = 1;
            build_idx(st, tt);
            attn(st, q, out);
        } else if (tt < Nr || st->mutation == MUT_NO_EVICT) {
            /* Phase 2: shift, attend, and grow the diagonal skip set. */
            inf.phase = 2;
            shift_skip(st);
            build_idx(st, tt);
            int budget = Nr - Na + ((st->mutation == MUT_BUDGET) ? 1 : 0);
            int selecting = st->n_skip < budget && st->n_idx > 0;
            if (st->mutation == MUT_NO_EVICT && tt >= Nr) selecting = 0;
            int pick = -1;
            if (selecting) {
                /* j* = argmin of the logits q.k over idx; first (oldest) on ties */
                int jbest = 0;
                double best = dot(q, st->K[st->idx[0]], d);
                for (int j = 1; j < st->n_idx; ++j) {
                    double s = dot(q, st->K[st->idx[j]], d);
                    int better;
                    if (st->mutation == MUT_ARGMAX) better = s > best;
                    else if (st->mutation == MUT_NEWEST_TIE) better = s <= best;
                    else better = s < best;
                    if (better) { best = s; jbest = j; }
                }
                pick = st->idx[jbest];
                inf.oracle_pick = pick;
                inf.min_logit = best;
                if (caller_pick >= 0 && caller_pick != pick) {
                    int found = 0;
                    for (int j = 0; j < st->n_idx; ++j) found |= (st->idx[j] == caller_pick);
                    double s = found ? dot(q, st->K[caller_pick], d) : INFINITY;
                    inf.pick_logit = s;
                    double a = fabs(best), b = fabs(s);
                    double ref = a > b ? a : b;
                    if (ref < 1.0) ref = 1.0;
                    if (found && fabs(s - best) <= ORC_NEAR_TIE_REL * ref) {
                        pick = caller_pick;
                        inf.adopted = 1;
                    } else {
                        inf.mismatch = 1;
                    }
                } else if (caller_pick >= 0) {
                    inf.pick_logit = best;
                }
            }
            if (st->mutation == MUT_SKIP_NOW && pick >= 0) {
                st->skip[st->n_skip++] = pick;
                build_idx(st, tt);
                attn(st, q, out);
            } else {
                attn(st, q, out);
                if (pick >= 0) st->skip[st->n_skip++] = pick;
            }
            inf.selected = pick;
        } else {
            /* Phase 3: evict the oldest row, shift, attend. */
            inf.phase = 3;
            const int old = tt - Nr;
            free(st->K[old]); free(st->V[old]);
            st->K[old] = st->V[old] = NULL;
            st->live -= 1;
            shift_skip(st);
            build_idx(st, tt);
            attn(st, q, out);
        }
    }
    inf.n_prefix = (st->mutation == MUT_NO_PROMPT) ? 0 : st->np;
    inf.n_idx = st->n_idx;
    inf.live_rows = st->live + (st->np - st->L_p);
    inf.n_skip = st->n_skip;
    st->t += 1;
    if (info) *info = inf;
    return 0;
}

/* Inner positions in skip_idx, in insertion order.  Returns the count. */
int orc_get_skip(const orc_stream *st, int *dst, int cap)
{
    int n = st->n_skip < cap ? st->n_skip : cap;
    for (int i = 0; i < n; ++i) dst[i] = st->skip[i];
    return st->n_skip;
}

/* Inner positions attended at the last step, ascending.  Returns the count. */
int orc_get_idx(const orc_stream *st, int *dst, int cap)
{
    int n = st->n_idx < cap ? st->n_idx : cap;
    for (int i = 0; i < n; ++i) dst[i] = st->idx[i];
    return st->n_idx;
}

int orc_get_step(const orc_stream *st) { return st->t; }

/* One decode step for n independent streams (the page keeps a separate skip
 * set per head), optionally spread over `threads` host threads.  q, k, v and
 * out are [n, d]; picks is [n] or NULL; infos is [n] or NULL.  Returns the
 * number of streams whose step failed. */
int orc_step_batch(orc_stream **sts, int n, const double *q, const double *k,
                   const double *v, double *out, const int *picks,
                   orc_info *infos, int threads)
{
    int bad = 0;
#ifdef _OPENMP
    if (threads < 1) threads = 1;
#pragma omp parallel for num_threads(threads) schedule(dynamic, 1) reduction(+ : bad)
#endif
    for (int i = 0; i < n; ++i) {
        const int d = sts[i]->d;
        int r = orc_step(sts[i], q + (size_t)i * d, k + (size_t)i * d, v + (size_t)i * d,
                         out + (size_t)i * d, picks ? picks[i] : -1,
                         infos ? &infos[i] : NULL);
        bad += (r != 0);
    }
    (void)threads;
    return bad;
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- Diagnostics of dense decode attention over one stream's trace
 * (section 3.4 "Attention Sparsity Analysis": "Skewed attention toward
 * prompt and local tokens" with
 * Fig. 8, and "Diagonal attention sparsity pattern" with Fig. 10).
 *
 * Query i (decode step i, 0-based) attends the L_p prompt keys and decode
 * keys 0..i with weights w_i = softmax(q_i k^T / sqrt(d)).
 *   mass[3 i + 0..2]: the weight on the prompt keys, on the local keys (the
 *     most recent ceil(0.1 (i + 1)) decoded keys, the current one included)
 *     and on the middle keys (the other decoded keys);
 *   for each distance dist[k], summed over the queries i = 0 .. L_dec - 1 -
 *     dist[k]: vsum[k] += cos(w_i[0..i], w_{i+d}[0..i]) (vertical: the same
 *     keys) and dsum[k] += cos(w_i[0..i], w_{i+d}[d..i+d]) (diagonal: keys
 *     shifted by d), over decode keys only.
 * Returns 0, or -1 on bad arguments / allocation failure.
 * orc_diag_set_mutation plants a mistake for the pin tests (0: faithful):
 * 1 the local window is floor(0.1 (i + 1)) keys, 2 the diagonal shift is
 * applied to query i instead of i + d, 3 the score vectors include the
 * prompt keys. */
static int g_diag_mutation;
void orc_diag_set_mutation(int m) { g_diag_mutation = m; }

int orc_diag_stream(int d, int L_p, int L_dec, const double *Q, const double *Kp, const double *Kd,
                    int n_dist, const int *dist, double *mass, double *vsum, double *dsum)
{
    if (d < 1 || L_p < 0 || L_dec < 1 || n_dist < 0) return -1;
    const int pw = g_diag_mutation == 3 ? L_p : 0;  /* prompt columns kept in w (planted mistake only) */
    const int W = pw + L_dec;
    double *w = (double *)calloc((size_t)L_dec * W, sizeof(double)); /* weights of query i, row i */
    double *z = (double *)malloc(sizeof(double) * (size_t)(L_p + L_dec));
    if (!w || !z) { free(w); free(z); return -1; }
    const double scale = 1.0 / sqrt((double)d);
    for (int i = 0; i < L_dec; ++i) {
        const double *q = Q + (size_t)i * d;
        const int n = L_p + i + 1;
        double m = -INFINITY;
        for (int j = 0; j < n; ++j) {
            const double *k = j < L_p ? Kp + (size_t)j * d : Kd + (size_t)(j - L_p) * d;
            z[j] = dot(q, k, d) * scale;
            if (z[j] > m) m = z[j];
        }
        double total = 0.0;
        for (int j = 0; j < n; ++j) { z[j] = exp(z[j] - m); total += z[j]; }
        const int n_local = g_diag_mutation == 1 ? (i + 1) / 10 : (i + 1 + 9) / 10;
        double mp = 0.0, ml = 0.0, mm = 0.0;
        for (int j = 0; j < n; ++j) {
            const double p = z[j] / total;
            if (j < L_p) mp += p;
            else if (j - L_p > i - n_local) ml += p;
            else mm += p;
            if (j >= L_p - pw) w[(size_t)i * W + (j - (L_p - pw))] = p;
        }
        mass[3 * i] = mp; mass[3 * i + 1] = ml; mass[3 * i + 2] = mm;
    }
    for (int k = 0; k < n_dist; ++k) {
        const int dd = dist[k];
        vsum[k] = dsum[k] = 0.0;
        for (int i = 0; i + dd < L_dec; ++i) {
            const double *a = w + (size_t)i * W, *b = w + (size_t)(i + dd) * W;
            double aa = 0.0, bv = 0.0, bd = 0.0, ab_v = 0.0, ab_d = 0.0;
            for (int j = 0; j <= i + pw; ++j) {
                /* planted mistake 2: query i's keys shifted instead of query i + d's */
                const double ad = (g_diag_mutation == 2) ? (j + dd <= i + pw ? a[j + dd] : 0.0) : a[j];
                const double bdj = (g_diag_mutation == 2) ? b[j] : b[j + dd];
                aa += a[j] * a[j];
                bv += b[j] * b[j];
                bd += bdj * bdj;
                ab_v += a[j] * b[j];
                ab_d += ad * bdj;
            }
            vsum[k] += ab_v / sqrt(aa * bv);
            dsum[k] += ab_d / sqrt(aa * bd);
        }
    }
    free(w); free(z);
    return 0;
}
