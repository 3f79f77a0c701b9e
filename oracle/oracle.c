/*
 * oracle.c -- float64 CPU oracle for batched speculative-decoding verification.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct
 * statement of what the verification step computes.  Only tests/, the smoke
 * check in __graft_entry__.py and the CPU-baseline leg of bench.py may load it.
 * It shares no code, header, table or constant with the CUDA library, and the
 * library never calls it.
 *
 * Sources, cited by page title and section:
 *   [SD-FA] nextadmin.net lesson "Speculative Decoding (دیکودینگ گمانه‌زن):
 *           2-4x faster text generation" (Persian).
 *   [SD-EN] aiengineeringfromscratch.com, Phase 10 lesson 25
 *           "Speculative Decoding" (Persian translation, English code).
 *   [RL]    runelab.ai blog "Küçük bir model büyük olanı nasıl
 *           hızlandırır?" (Turkish).
 *   [DYNA]  lowest.today summary of "DynaSpec: Context-aware Dynamic
 *           Speculative Sampling for Large-Vocabulary Language Models".
 *
 * Notation follows [SD-FA] § Core algorithm: q is the TARGET distribution,
 * p is the DRAFT distribution, d_i the drafted tokens, K the draft length,
 * V the vocabulary size, T the temperature.  ([SD-EN] and [RL] swap the two
 * letters; their rules are the same after the swap.)
 *
 * Readings where the pages are silent or inconsistent (all listed in the
 * design notes as well):
 *   - the residual at a rejection uses the full draft distribution p_j at the
 *     rejected position ([SD-FA] § Core algorithm step 5; [SD-EN] § The
 *     exact rule), not the first-position draft or a scalar;
 *   - temperature divides both target and draft logits ([SD-EN] § Build it:
 *     both calls receive the temperature); draft probabilities given directly
 *     are used as given;
 *   - "sample" is inverse-CDF sampling in ascending token order: the smallest
 *     x with sum_{y<=x} r(y) > v*R; if rounding leaves no such x, the largest
 *     x with r(x) > 0;
 *   - a zero residual mass (q == p) falls back to sampling q_j
 *     ([SD-FA] § Step 2 divides by the sum and leaves this case open);
 *   - p_i(d_i) == 0 accepts ([SD-FA] § Step 1: the ratio is taken as
 *     infinite);
 *   - the uniforms are Philox4x32-10 words (Salmon, Moraes, Dror, Shaw,
 *     "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11) with counter
 *     (position, sequence, tag, 0) and key (seed low word, seed high word);
 *     word 0 is the accept uniform u_i, word 1 the sampling uniform v_i;
 *     a word w maps to ((w >> 8) + 0.5) * 2^-24;
 *   - greedy (T == 0) takes the first index of the maximum raw logit
 *     ([SD-EN] § Greedy case); when all K match, the bonus is argmax q_{K+1}
 *     ([SD-FA] § Core algorithm step 6);
 *   - data errors (NaN / +inf logits, an all -inf row, a token outside
 *     [0, V), a shortlist that is not ascending and unique inside [0, V)
 *     (or whose length is outside [1, S]),
 *     negative or non-finite draft probabilities) are checked at the positions
 *     the left-to-right rule examines, in the order: the position's shortlist,
 *     token, target row, draft row.  Logit rows are checked whole (their
 *     softmax needs every entry); given draft probabilities are checked where
 *     the rule reads them: p_i(d_i) at each examined position, and the whole
 *     row p_j at a rejection, whose residual uses it.  A sequence with an
 *     error gets accept_len = -code and every token -1.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F32 = 0, OR_BF16 = 1 };
enum { OR_OK = 0, OR_ERR_NONFINITE = 2, OR_ERR_TOKEN_RANGE = 3, OR_ERR_SHORTLIST = 4 };
enum { OR_TAG_VERIFY = 0 };

/* ------------------------------------------------------------------------ */
/* Philox4x32-10, from its published definition (SC'11, section 3 and
 * table 2): each round multiplies counter words 0 and 2 by the two round
 * constants, swaps and XORs the high halves with the other words and the key;
 * the key is bumped by the two Weyl constants between rounds.                 */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Uniform in (0, 1) from the top 24 bits n = w >> 8 of a word: (n + 0.5) 2^-24,
 * i.e. (2n + 1) 2^-25, exact in float64.  It needs 25 significant bits, so a
 * float32 holds it exactly only for n < 2^23.                                 */
double oracle_uniform24(uint32_t w)
{
    return ((double)(w >> 8) + 0.5) * (1.0 / 16777216.0);
}

/* Word `word` (0: accept uniform u, 1: sampling uniform v) for (seed, seq, pos). */
static double verify_uniform(uint64_t seed, int seq, int pos, int word)
{
    uint32_t ctr[4] = { (uint32_t)pos, (uint32_t)seq, (uint32_t)OR_TAG_VERIFY, 0u };
    uint32_t key[2] = { (uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32) };
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    return oracle_uniform24(out[word]);
}

/* ------------------------------------------------------------------------ */
/* Element access: float32 as is; bfloat16 bits shifted into a float32. Both
 * convert to float64 exactly.                                                 */
static double elem(const void *base, int dtype, size_t i)
{
    if (dtype == OR_F32)
        return (double)((const float *)base)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Temperature softmax of one row: out = softmax(z / T), with the maximum
 * subtracted before exponentiating ([SD-EN] § Build it: softmax of the logits
 * divided by the temperature).  Returns OR_ERR_NONFINITE for a NaN or +inf
 * logit or a row that is -inf everywhere; -inf entries get probability 0.
 * *lse receives log sum exp(z / T).                                           */
int oracle_softmax(const double *z, int n, double T, double *out, double *lse)
{
    double zmax = -INFINITY;
    for (int x = 0; x < n; ++x) {
        if (isnan(z[x]) || z[x] == INFINITY)
            return OR_ERR_NONFINITE;
        if (z[x] > zmax)
            zmax = z[x];
    }
    if (zmax == -INFINITY)
        return OR_ERR_NONFINITE;
    double sum = 0.0;
    for (int x = 0; x < n; ++x) {
        double e = exp((z[x] - zmax) / T);
        out[x] = e;
        sum += e;
    }
    for (int x = 0; x < n; ++x)
        out[x] /= sum;
    if (lse)
        *lse = zmax / T + log(sum);
    return OR_OK;
}

/* Acceptance probability of a drafted token: min(1, q(d) / p(d)), taken as 1
 * when p(d) == 0 ([SD-FA] § Step 1: accept/reject; [SD-EN] § The exact rule). */
double oracle_accept_prob(double q_d, double p_d)
{
    if (p_d > 0.0) {
        double ratio = q_d / p_d;
        return ratio < 1.0 ? ratio : 1.0;
    }
    return 1.0;
}

/* Residual at a rejection: r(x) = max(0, q(x) - p(x)) element by element;
 * returns R = sum_x r(x) ([SD-FA] § Step 2: residual distribution; [RL]
 * § single-position example: the replacements go to the words the target
 * likes more than the draft).                                                 */
double oracle_residual(const double *q, const double *p, int n, double *r)
{
    double R = 0.0;
    for (int x = 0; x < n; ++x) {
        double diff = q[x] - p[x];
        r[x] = diff > 0.0 ? diff : 0.0;
        R += r[x];
    }
    return R;
}

/* Inverse-CDF sample from the unnormalised weights r (total R) with uniform v:
 * the smallest x whose running sum exceeds v*R, accumulated in ascending x.
 * *margin receives the distance from v to the nearer edge of the chosen
 * token's interval in the normalised CDF (0 for the fallback).                */
int oracle_inverse_cdf(const double *r, int n, double R, double v, double *margin)
{
    double threshold = v * R;
    double cum = 0.0;
    for (int x = 0; x < n; ++x) {
        double before = cum;
        cum += r[x];
        if (cum > threshold) {
            if (margin) {
                double lo = v - before / R, hi = cum / R - v;
                *margin = lo < hi ? lo : hi;
            }
            return x;
        }
    }
    for (int x = n - 1; x >= 0; --x) {
        if (r[x] > 0.0) {
            if (margin)
                *margin = 0.0;
            return x;
        }
    }
    if (margin)
        *margin = 0.0;
    return n - 1;
}

/* First index of the maximum ([SD-EN] § Greedy case; ties to the lowest
 * index).  Returns -1 for NaN / +inf / an all -inf row.                       */
int oracle_argmax_first(const double *z, int n)
{
    int best = -1;
    double zbest = -INFINITY;
    for (int x = 0; x < n; ++x) {
        if (isnan(z[x]) || z[x] == INFINITY)
            return -1;
        if (z[x] > zbest) {
            zbest = z[x];
            best = x;
        }
    }
    return best;
}

/* ------------------------------------------------------------------------ */
struct job {
    const void *target; int tdt;        /* [B][K+1][V]                          */
    const void *draft; int ddt;         /* [B][K][V], or [B][K][S] on a shortlist */
    int draft_is_probs;                 /* draft holds probabilities (float32)  */
    const int32_t *shortlist; int S;    /* index lists (ascending), or NULL; S = draft row stride */
    long long sl_seq, sl_pos;           /* list of (b, i) at shortlist + b sl_seq + i sl_pos */
    const int32_t *sl_len;              /* [K] entries of the list at position i, or NULL (S) */
    const int32_t *tokens;              /* [B][K]                               */
    int B, K, V;
    double T;
    uint64_t seed;
    int32_t *out_tokens;                /* [B][K+1]                             */
    int32_t *out_accept_len;            /* [B]                                  */
    double *q_draft, *p_draft;          /* [B][K]   optional                    */
    double *residual_mass;              /* [B]      optional                    */
    double *row_lse;                    /* [B][2K+1] optional                   */
    double *accept_margin;              /* [B][K]   optional                    */
    double *sample_margin;              /* [B]      optional                    */
    int32_t *terminal;                  /* [B]      optional                    */
    const int32_t *seq_ids;             /* [B] sequence index for the uniforms, or NULL (= b) */
    int nthreads;
};

struct scratch { double *z, *q, *p, *r; };

/* The sequence index that keys the uniforms of batch row b. */
static int seq_of(const struct job *J, int b)
{
    return J->seq_ids ? J->seq_ids[b] : b;
}

/* The shortlist of position i of sequence b and its length ([DYNA] § Method 3:
 * the budget, hence the list, may depend on the position; a list shared by
 * every position or every sequence is the same layout with stride 0).        */
static const int32_t *sl_row(const struct job *J, int b, int i)
{
    return J->shortlist + (long long)b * J->sl_seq + (long long)i * J->sl_pos;
}
static int sl_n(const struct job *J, int i)
{
    return J->sl_len ? J->sl_len[i] : J->S;
}

/* q_i: softmax of target row (b, i). */
static int target_dist(const struct job *J, int b, int i, struct scratch *w, double *lse)
{
    size_t off = ((size_t)b * (J->K + 1) + i) * (size_t)J->V;
    for (int x = 0; x < J->V; ++x)
        w->z[x] = elem(J->target, J->tdt, off + x);
    return oracle_softmax(w->z, J->V, J->T, w->q, lse);
}

/* p_i: the draft distribution at position i over the full vocabulary.
 * Logits: softmax(z / T).  Probabilities: as given (finite, >= 0).
 * Shortlist ([DYNA] § Abstract and § Method 3: the drafter runs on the union
 * of the selected clusters while verification keeps the full vocabulary):
 * softmax over the S shortlisted logits, 0 for every other token.             */
static int draft_dist(const struct job *J, int b, int i, struct scratch *w, double *lse)
{
    int n = J->shortlist ? sl_n(J, i) : J->V;
    size_t off = ((size_t)b * J->K + i) * (size_t)(J->shortlist ? J->S : J->V);
    if (lse)
        *lse = NAN;
    if (J->draft_is_probs) {
        for (int x = 0; x < n; ++x)
            w->r[x] = elem(J->draft, OR_F32, off + x);
    } else {
        for (int x = 0; x < n; ++x)
            w->z[x] = elem(J->draft, J->ddt, off + x);
        int st = oracle_softmax(w->z, n, J->T, w->r, lse);
        if (st)
            return st;
    }
    if (!J->shortlist) {
        memcpy(w->p, w->r, sizeof(double) * (size_t)n);
    } else {
        const int32_t *idx = sl_row(J, b, i);
        for (int x = 0; x < J->V; ++x)
            w->p[x] = 0.0;
        for (int s = 0; s < n; ++s)
            w->p[idx[s]] = w->r[s];
    }
    return OR_OK;
}

/* A given draft probability is usable when it is finite and >= 0. */
static int prob_ok(double v)
{
    return v >= 0.0 && v != INFINITY;
}

/* Every entry of draft probability row (b, i) usable. */
static int prob_row_ok(const struct job *J, int b, int i)
{
    int n = J->shortlist ? sl_n(J, i) : J->V;
    size_t off = ((size_t)b * J->K + i) * (size_t)(J->shortlist ? J->S : J->V);
    for (int x = 0; x < n; ++x)
        if (!prob_ok(elem(J->draft, OR_F32, off + x)))
            return 0;
    return 1;
}

static int shortlist_ok(const struct job *J, int b, int i)
{
    const int32_t *idx = sl_row(J, b, i);
    const int n = sl_n(J, i);
    if (n < 1 || n > J->S)
        return 0;
    for (int s = 0; s < n; ++s) {
        if (idx[s] < 0 || idx[s] >= J->V)
            return 0;
        if (s > 0 && idx[s] <= idx[s - 1])
            return 0;
    }
    return 1;
}

static void emit_error(const struct job *J, int b, int code)
{
    for (int i = 0; i <= J->K; ++i)
        J->out_tokens[(size_t)b * (J->K + 1) + i] = -1;
    J->out_accept_len[b] = -code;
    if (J->terminal)
        J->terminal[b] = -1;
}

/* One verification round for sequence b ([SD-FA] § Core algorithm steps 4-6
 * and § Step 3; [SD-EN] § The exact rule and § Build it; [RL] § the exact
 * rule, points 1-3):
 *   for i = 1..K, left to right: accept d_i with probability
 *   min(1, q_i(d_i)/p_i(d_i)); at the first rejection j sample the replacement
 *   from the normalised residual (q_j - p_j)_+ and discard the rest; if every
 *   draft token is accepted, sample a bonus token from q_{K+1}.               */
static void verify_stochastic(const struct job *J, int b, struct scratch *w)
{
    const int K = J->K, V = J->V;
    int32_t *tok = J->out_tokens + (size_t)b * (K + 1);
    for (int i = 0; i <= K; ++i)
        tok[i] = -1;
    if (J->accept_margin)
        for (int i = 0; i < K; ++i)
            J->accept_margin[(size_t)b * K + i] = INFINITY;
    if (J->sample_margin)
        J->sample_margin[b] = INFINITY;
    if (J->residual_mass)
        J->residual_mass[b] = NAN;

    for (int i = 0; i < K; ++i) {
        /* the shortlist this position's draft uses, before its token */
        if (J->shortlist && !shortlist_ok(J, b, i)) {
            emit_error(J, b, OR_ERR_SHORTLIST);
            return;
        }
        int d = J->tokens[(size_t)b * K + i];
        if (d < 0 || d >= V) {
            emit_error(J, b, OR_ERR_TOKEN_RANGE);
            return;
        }
        if (target_dist(J, b, i, w, NULL) || draft_dist(J, b, i, w, NULL)
            || (J->draft_is_probs && !prob_ok(w->p[d]))) {
            emit_error(J, b, OR_ERR_NONFINITE);
            return;
        }
        double u = verify_uniform(J->seed, seq_of(J, b), i, 0);
        double a = oracle_accept_prob(w->q[d], w->p[d]);
        if (J->accept_margin && w->p[d] > 0.0)
            J->accept_margin[(size_t)b * K + i] = fabs(u - a);
        if (u < a) {
            tok[i] = d;
            continue;
        }
        /* First rejection at position i: residual sample, then stop. */
        if (J->draft_is_probs && !prob_row_ok(J, b, i)) {
            emit_error(J, b, OR_ERR_NONFINITE);
            return;
        }
        double R = oracle_residual(w->q, w->p, V, w->r);
        double v = verify_uniform(J->seed, seq_of(J, b), i, 1);
        double margin;
        int x;
        if (R > 0.0) {
            x = oracle_inverse_cdf(w->r, V, R, v, &margin);
        } else {
            double Rq = 0.0;
            for (int y = 0; y < V; ++y)
                Rq += w->q[y];
            x = oracle_inverse_cdf(w->q, V, Rq, v, &margin);
        }
        tok[i] = x;
        J->out_accept_len[b] = i;
        if (J->terminal)
            J->terminal[b] = i;
        if (J->residual_mass)
            J->residual_mass[b] = R;
        if (J->sample_margin)
            J->sample_margin[b] = margin;
        return;
    }
    /* Every draft token accepted: bonus token from q_{K+1}. */
    if (target_dist(J, b, K, w, NULL)) {
        emit_error(J, b, OR_ERR_NONFINITE);
        return;
    }
    double Rq = 0.0;
    for (int y = 0; y < V; ++y)
        Rq += w->q[y];
    double v = verify_uniform(J->seed, seq_of(J, b), K, 1), margin;
    tok[K] = oracle_inverse_cdf(w->q, V, Rq, v, &margin);
    J->out_accept_len[b] = K;
    if (J->terminal)
        J->terminal[b] = K;
    if (J->residual_mass)
        J->residual_mass[b] = Rq;
    if (J->sample_margin)
        J->sample_margin[b] = margin;
}

/* Per-position probabilities for every position (requested outputs only):
 * q_i(d_i), p_i(d_i) and the log-sum-exp of every row, NaN where a row or a
 * token is invalid.                                                            */
static void all_positions(const struct job *J, int b, struct scratch *w)
{
    const int K = J->K;
    for (int i = 0; i <= K; ++i) {
        int sl_bad = i < K && J->shortlist && !shortlist_ok(J, b, i);
        double lse_t = NAN, lse_d = NAN;
        int bad_t = target_dist(J, b, i, w, &lse_t);
        if (J->row_lse)
            J->row_lse[(size_t)b * (2 * K + 1) + i] = bad_t ? NAN : lse_t;
        if (i == K)
            break;
        int bad_d = sl_bad ? 1 : draft_dist(J, b, i, w, &lse_d);
        if (sl_bad)
            lse_d = NAN;
        if (J->row_lse)
            J->row_lse[(size_t)b * (2 * K + 1) + K + 1 + i] = bad_d ? NAN : lse_d;
        int d = J->tokens[(size_t)b * K + i];
        int ok = !bad_t && !bad_d && d >= 0 && d < J->V && (!J->draft_is_probs || prob_ok(w->p[d]));
        if (J->q_draft)
            J->q_draft[(size_t)b * K + i] = ok ? w->q[d] : NAN;
        if (J->p_draft)
            J->p_draft[(size_t)b * K + i] = ok ? w->p[d] : NAN;
    }
}

/* Greedy verification, T == 0 ([SD-EN] § Greedy case): accept d_i while
 * argmax q_i == d_i; at the first mismatch emit argmax q_i and stop; if all K
 * match, emit argmax q_{K+1}.  Draft rows are not used.                       */
static void verify_greedy(const struct job *J, int b, struct scratch *w)
{
    const int K = J->K, V = J->V;
    int32_t *tok = J->out_tokens + (size_t)b * (K + 1);
    if (J->residual_mass)
        J->residual_mass[b] = NAN;
    for (int i = 0; i <= K; ++i)
        tok[i] = -1;
    for (int i = 0; i <= K; ++i) {
        int d = -1;
        if (i < K) {
            d = J->tokens[(size_t)b * K + i];
            if (d < 0 || d >= V) {
                emit_error(J, b, OR_ERR_TOKEN_RANGE);
                return;
            }
        }
        size_t off = ((size_t)b * (K + 1) + i) * (size_t)V;
        for (int x = 0; x < V; ++x)
            w->z[x] = elem(J->target, J->tdt, off + x);
        int g = oracle_argmax_first(w->z, V);
        if (g < 0) {
            emit_error(J, b, OR_ERR_NONFINITE);
            return;
        }
        if (i < K && g == d) {
            tok[i] = d;
            continue;
        }
        tok[i] = g;
        J->out_accept_len[b] = i;
        if (J->terminal)
            J->terminal[b] = i;
        return;
    }
}

struct worker { const struct job *J; int t; };

static void *run_worker(void *arg)
{
    const struct worker *wk = (const struct worker *)arg;
    const struct job *J = wk->J;
    size_t n = (size_t)J->V;
    if (J->shortlist && (size_t)J->S > n)
        n = (size_t)J->S;
    struct scratch w;
    w.z = malloc(sizeof(double) * n);
    w.q = malloc(sizeof(double) * n);
    w.p = malloc(sizeof(double) * n);
    w.r = malloc(sizeof(double) * n);
    for (int b = wk->t; b < J->B; b += J->nthreads) {
        if (J->T == 0.0) {
            verify_greedy(J, b, &w);
        } else {
            verify_stochastic(J, b, &w);
            if (J->q_draft || J->p_draft || J->row_lse)
                all_positions(J, b, &w);
        }
    }
    free(w.z); free(w.q); free(w.p); free(w.r);
    return NULL;
}

/* Batched entry point: one verification round for each of B independent
 * sequences, split over `nthreads` host threads (one sequence at a time per
 * thread).  Host pointers.  The shortlist of position i of sequence b is the
 * sl_len[i] (all S when sl_len is NULL) entries at shortlist + b sl_seq +
 * i sl_pos; draft rows are [B][K][S].  Returns 0, or 1 for arguments that are
 * out of range.                                                               */
int oracle_verify_sl(const void *target, int tdt, const void *draft, int ddt, int draft_is_probs,
                     const int32_t *shortlist, int S, long long sl_seq, long long sl_pos, const int32_t *sl_len,
                     const int32_t *tokens, int B, int K, int V, double T, uint64_t seed,
                     int32_t *out_tokens, int32_t *out_accept_len,
                     double *q_draft, double *p_draft, double *residual_mass, double *row_lse,
                     double *accept_margin, double *sample_margin, int32_t *terminal,
                     const int32_t *seq_ids, int nthreads)
{
    if (B < 1 || K < 1 || V < 1 || !(T >= 0.0) || !target || !tokens || !out_tokens || !out_accept_len)
        return 1;
    if (T > 0.0 && !draft)
        return 1;
    if (shortlist && (S < 1 || S > V))
        return 1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > B)
        nthreads = B;
    struct job J = { target, tdt, draft, ddt, draft_is_probs, shortlist, S, sl_seq, sl_pos, sl_len, tokens, B, K, V,
                     T, seed, out_tokens, out_accept_len, q_draft, p_draft, residual_mass, row_lse,
                     accept_margin, sample_margin, terminal, seq_ids, nthreads };
    pthread_t *th = malloc(sizeof(pthread_t) * (size_t)nthreads);
    struct worker *wk = malloc(sizeof(struct worker) * (size_t)nthreads);
    for (int t = 0; t < nthreads; ++t) {
        wk[t].J = &J;
        wk[t].t = t;
        pthread_create(&th[t], NULL, run_worker, &wk[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        pthread_join(th[t], NULL);
    free(th);
    free(wk);
    return 0;
}

/* The per-sequence shortlist form: list b at shortlist + b S, all S entries. */
int oracle_verify(const void *target, int tdt, const void *draft, int ddt, int draft_is_probs,
                  const int32_t *shortlist, int S, const int32_t *tokens,
                  int B, int K, int V, double T, uint64_t seed,
                  int32_t *out_tokens, int32_t *out_accept_len,
                  double *q_draft, double *p_draft, double *residual_mass, double *row_lse,
                  double *accept_margin, double *sample_margin, int32_t *terminal,
                  const int32_t *seq_ids, int nthreads)
{
    return oracle_verify_sl(target, tdt, draft, ddt, draft_is_probs, shortlist, S, (long long)S, 0, NULL, tokens, B,
                            K, V, T, seed, out_tokens, out_accept_len, q_draft, p_draft, residual_mass, row_lse,
                            accept_margin, sample_margin, terminal, seq_ids, nthreads);
}
