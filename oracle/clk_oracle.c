/*
 * CPU oracle of the context-lookup speculative decoding step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness reference that the
 * CUDA path is compared against.  Only the test suite, the smoke entry point
 * and the benchmark's CPU-baseline / reference leg may load or run it; the
 * product library never links, loads or calls it, and it shares no code,
 * header, table or constant with that library.
 *
 * It computes every step from the plain definitions in the pages
 * (HyperQwen context-lookup article, section "lookup 草稿的原理：三步走"),
 * slowly and without any index:
 *
 *   Step 1 (lookup): the most recent earlier occurrence of the longest
 *     4..12-token suffix of the request's own history, overlap allowed, by a
 *     full scan of the history; the tokens that follow it are the draft
 *     (continued cyclically with period n - j past the end of history).
 *   Step 2 (fusion): head slots 1..7 take the lookup draft if the match is at
 *     least 8, or at least 6 with the draft model's first 2 proposals
 *     agreeing; otherwise they keep the draft model's proposals.  Tail slots
 *     8..15 take the lookup draft if the block is long and the match is at
 *     least 4.
 *   Step 3 (scheduler): the 16-token block is entered after 2 consecutive
 *     steps that have a match able to fill the tail and follow a nearly full
 *     step, and is left only after the match flag has stayed down for more
 *     than 3 steps (sticky 3).
 *   Greedy verification: row-wise argmax over the target logits (lowest
 *     index on ties), the accepted prefix up to the first mismatch, plus the
 *     target's own token at the first mismatch (the bonus token).
 *   Sampling verification (same section, closing paragraph): each draft is
 *     a point mass, accepted with the target's probability of it; the first
 *     rejection emits a sample of the target without that token, and a fully
 *     accepted block emits a sample of the last row (see or_sample_verify).
 *
 * Readings adopted where the pages are silent (each one a parameter):
 *   - ties on length go to the most recent occurrence; length first;
 *   - "nearly full" = accepted >= block - 1 - slack with slack 1;
 *   - the scheduler flag is "k >= tail threshold" on this step's lookup, and
 *     the near-full signal is the previous step's; at the first step there
 *     is no previous step;
 *   - unfilled slots hold the sentinel -1, which no argmax can equal.
 *
 * Argmax compares values as float32 (bf16 widens exactly): the first index
 * of the maximum wins, +0 equals -0, and if a row holds a NaN the first NaN
 * wins (torch.argmax convention).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <time.h>

#define OR_SENT (-1)
#define OR_BLOCK 16
#define OR_SHORT 0
#define OR_LONG 1

typedef struct or_params {
    int32_t min_k;           /* shortest suffix match that counts: 4 */
    int32_t max_k;           /* longest suffix length searched: 12 */
    int32_t head;            /* draft-model head slots: 7 */
    int32_t tail;            /* lookup-only tail slots: 8 */
    int32_t head_replace_k;  /* match that replaces the head outright: 8 */
    int32_t head_agree_k;    /* match that replaces it if the drafter agrees: 6 */
    int32_t head_agree_n;    /* leading proposals that must agree: 2 */
    int32_t tail_k;          /* match that fills the tail: 4 */
    int32_t enter_streak;    /* consecutive qualifying steps to enter: 2 */
    int32_t sticky;          /* flag-down steps tolerated in the long block: 3 */
    int32_t near_full_slack; /* rejected drafts still "nearly full": 1 */
} or_params;

typedef struct or_sched_state {
    int32_t mode;
    int32_t streak;
    int32_t miss;
    int32_t has_prev;
} or_sched_state;

/* Per-request counters, same order as the product's report. */
typedef struct or_counters {
    int64_t steps, hits, long_steps, drafted, accepted, emitted;
    int64_t accept_hist[2][16];
} or_counters;

void or_params_default(or_params* p)
{
    p->min_k = 4;
    p->max_k = 12;
    p->head = 7;
    p->tail = 8;
    p->head_replace_k = 8;
    p->head_agree_k = 6;
    p->head_agree_n = 2;
    p->tail_k = 4;
    p->enter_streak = 2;
    p->sticky = 3;
    p->near_full_slack = 1;
}

/* Step 1: longest k in [min_k, max_k] and then largest j with
 * h[j-k .. j-1] == h[n-k .. n-1] and k <= j <= n-1.  Full scan.
 * Returns k (0 when nothing matches) and writes j (-1 when nothing matches). */
int32_t or_lookup(const int32_t* h, int64_t n, int32_t min_k, int32_t max_k, int64_t* j_out)
{
    for (int32_t k = max_k; k >= min_k; --k) {
        for (int64_t j = n - 1; j >= k; --j) {
            int same = 1;
            for (int32_t i = 0; i < k; ++i) {
                if (h[j - k + i] != h[n - k + i]) {
                    same = 0;
                    break;
                }
            }
            if (same) {
                *j_out = j;
                return k;
            }
        }
    }
    *j_out = -1;
    return 0;
}

/* Step 1, copy: the 16 tokens that follow the match; past the end of the
 * history the copy continues from its own start (period n - j). */
void or_copy(const int32_t* h, int64_t n, int32_t k, int64_t j, int32_t* c)
{
    for (int64_t i = 0; i < OR_BLOCK; ++i) {
        if (k == 0)
            c[i] = OR_SENT;
        else if (j + i < n)
            c[i] = h[j + i];
        else
            c[i] = c[i - (n - j)];
    }
}

/* Step 3: one scheduler step.  Returns the block length for this step. */
int32_t or_sched(or_sched_state* s, int32_t k, int32_t prev_a, int32_t prev_L, const or_params* p)
{
    const int flag = k >= p->tail_k;
    const int near_full = s->has_prev && prev_a >= prev_L - 1 - p->near_full_slack;
    if (s->mode == OR_SHORT) {
        if (flag && near_full)
            s->streak += 1;
        else
            s->streak = 0;
        if (s->streak >= p->enter_streak) {
            s->mode = OR_LONG;
            s->miss = 0;
        }
    } else {
        if (flag)
            s->miss = 0;
        else
            s->miss += 1;
        if (s->miss > p->sticky) {
            s->mode = OR_SHORT;
            s->streak = 0;
        }
    }
    s->has_prev = 1;
    return s->mode == OR_LONG ? 1 + p->head + p->tail : 1 + p->head;
}

/* Step 2: the verify block.  blk[0] is the last committed token. */
void or_fuse(int32_t last, const int32_t* c, int32_t k, const int32_t* m, int32_t L, const or_params* p,
             int32_t* blk)
{
    int take_head = k >= p->head_replace_k;
    if (!take_head && k >= p->head_agree_k) {
        take_head = 1;
        for (int32_t i = 0; i < p->head_agree_n; ++i)
            if (c[i] != m[i]) take_head = 0;
    }
    const int fill_tail = (L == 1 + p->head + p->tail) && k >= p->tail_k;
    for (int32_t i = 0; i < OR_BLOCK; ++i) blk[i] = OR_SENT;
    blk[0] = last;
    for (int32_t i = 0; i < p->head; ++i) blk[1 + i] = take_head ? c[i] : m[i];
    for (int32_t i = 0; i < p->tail; ++i) blk[1 + p->head + i] = fill_tail ? c[p->head + i] : OR_SENT;
}

static float or_bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Greedy verification, one row: first index of the maximum. */
int32_t or_argmax_f32(const float* x, int64_t V)
{
    for (int64_t v = 0; v < V; ++v)
        if (isnan(x[v])) return (int32_t)v;
    int64_t best = 0;
    for (int64_t v = 1; v < V; ++v)
        if (x[v] > x[best]) best = v;
    return (int32_t)best;
}

int32_t or_argmax_bf16(const uint16_t* x, int64_t V)
{
    for (int64_t v = 0; v < V; ++v)
        if (isnan(or_bf16_value(x[v]))) return (int32_t)v;
    int64_t best = 0;
    float bv = or_bf16_value(x[0]);
    for (int64_t v = 1; v < V; ++v) {
        float f = or_bf16_value(x[v]);
        if (f > bv) {
            bv = f;
            best = v;
        }
    }
    return (int32_t)best;
}

/* Greedy verification: number of drafts accepted before the first mismatch. */
int32_t or_accept(const int32_t* blk, const int32_t* g, int32_t L)
{
    int32_t a = 0;
    while (a < L - 1 && blk[a + 1] == g[a]) a += 1;
    return a;
}

/* ------------------------------------------------------------------------ */
/* Sampling verification with point-mass drafts.                             */
/* ------------------------------------------------------------------------ */
/*
 * HyperQwen context-lookup article, closing paragraph of "lookup 草稿的原理：
 * 三步走": for a sampled request every position the lookup filled is treated
 * as a point mass on its proposed token, which the standard speculative
 * rejection sampler accepts as a proposal distribution, so the output has
 * exactly the distribution of sampling without speculation.
 *
 * Per row r (r < L) the target distribution is p_r = softmax(x_r * inv_temp).
 * With the proposal q = point mass on the draft c = blk[r + 1]:
 *   the draft is accepted with probability min(1, p_r(c) / q(c)) = p_r(c),
 *   i.e. iff u_acc[r] < p_r(c);
 *   at the first rejection the emitted token is a sample of the residual
 *   max(p_r - q, 0), normalised: p_r with c removed, drawn with u_smp[r];
 *   if all L - 1 drafts are accepted, the bonus token is a sample of p_{L-1}
 *   drawn with u_smp[L - 1].
 * A draft outside [0, V) (the sentinel: no proposal) has p_r(c) = 0: it is
 * rejected, and the residual is p_r itself.
 * A sample of weights w_0..w_{V-1} with the uniform u is the smallest v whose
 * running sum w_0 + .. + w_v exceeds u * (w_0 + .. + w_{V-1}); if rounding
 * leaves none, the last v of nonzero weight.
 * Everything is computed in double from the logits as given (float32, or
 * bf16 widened exactly); the logits are finite.
 */

/* Row r of the logits as doubles. */
static void or_row_values(const void* row, int32_t dtype, int64_t V, double* y)
{
    for (int64_t v = 0; v < V; ++v)
        y[v] = dtype == 0 ? (double)or_bf16_value(((const uint16_t*)row)[v]) : (double)((const float*)row)[v];
}

/* Unnormalised softmax weights e_v = exp(x_v * inv_temp - max) and their sum. */
static double or_softmax_weights(const void* row, int32_t dtype, int64_t V, double inv_temp, double* e)
{
    or_row_values(row, dtype, V, e);
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
        e[v] *= inv_temp;
        if (e[v] > m) m = e[v];
    }
    double z = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        e[v] = exp(e[v] - m);
        z += e[v];
    }
    return z;
}

/* Inverse-CDF sample of the weights e with token `excl` removed (excl outside
 * [0, V): nothing removed). */
int32_t or_sample_weights(const double* e, int64_t V, int32_t excl, double u)
{
    double total = 0.0;
    for (int64_t v = 0; v < V; ++v)
        if (v != excl) total += e[v];
    const double target = u * total;
    double run = 0.0;
    int64_t last = -1;
    for (int64_t v = 0; v < V; ++v) {
        if (v == excl) continue;
        run += e[v];
        if (e[v] > 0.0) last = v;
        if (run > target) return (int32_t)v;
    }
    return (int32_t)last;
}

/* One request: rows[r * row_stride ..] for r < L, block blk[16], uniforms
 * u[2 * r] (acceptance) and u[2 * r + 1] (sample).  Writes out_tok[16]
 * (emitted tokens, then OR_SENT) and returns the number of accepted drafts;
 * L outside 1..16 gives -1 and no tokens. */
int32_t or_sample_verify(const void* rows, int32_t dtype, int64_t row_stride, int64_t V, const int32_t* blk,
                         int32_t L, float inv_temp, const float* u, int32_t* out_tok)
{
    for (int i = 0; i < OR_BLOCK; ++i) out_tok[i] = OR_SENT;
    if (L < 1 || L > OR_BLOCK) return -1;
    const size_t esz = dtype == 0 ? sizeof(uint16_t) : sizeof(float);
    double* e = (double*)malloc((size_t)V * sizeof(double));
    if (e == NULL) return -1;
    int32_t a = 0;
    int32_t tok = OR_SENT;
    for (int32_t r = 0; r < L; ++r) {
        const void* row = (const char*)rows + (size_t)r * (size_t)row_stride * esz;
        const double z = or_softmax_weights(row, dtype, V, (double)inv_temp, e);
        if (r == L - 1) {
            tok = or_sample_weights(e, V, -1, (double)u[2 * r + 1]);
            break;
        }
        const int32_t c = blk[r + 1];
        const double pc = (c >= 0 && c < V) ? e[c] / z : 0.0;
        if ((double)u[2 * r] < pc) {
            out_tok[r] = c;
            a += 1;
            continue;
        }
        tok = or_sample_weights(e, V, c, (double)u[2 * r + 1]);
        break;
    }
    out_tok[a] = tok;
    free(e);
    return a;
}

/* ------------------------------------------------------------------------ */
/* Exact sampling verification: the same rule on fixed-point weights.        */
/* ------------------------------------------------------------------------ */
/*
 * The rule of or_sample_verify (accept iff u_acc < p_r(c); the first
 * rejection draws from p_r without c; a full acceptance draws from the last
 * row) with the target's weights defined as integers, so that every
 * acceptance and every draw is an integer comparison that two
 * implementations reach bit for bit.  Where floating point decides an
 * integer, both sides must take that decision in the same precision; here
 * that precision is float32 with fused multiply-adds, then integers.
 *
 * Row x (V entries, bf16 widened exactly or float32), inverse temperature t:
 *   s = fl32(t * fl32(log2 e)); the row is cut into chunks of 1024 entries
 *   (the last one ragged).  Chunk k's reference is R_k = ceil(fl32(M_k * s))
 *   with M_k its largest entry; a chunk of -inf only has no reference and
 *   weight 0.  Entry i of chunk k weighs q_i = Q(fma(x_i, s, -R_k)), where
 *   for d < -32: Q(d) = 0, else with n = rint(d) (ties to even) and
 *   r = d - n (exact, |r| <= 1/2):
 *     f = P(r), the degree-6 Taylor polynomial of 2^(r + 1/2) = sqrt(2) 2^r
 *         (coefficients sqrt(2) (ln 2)^k / k! rounded to float, evaluated by
 *         Horner's rule with fmaf), a float in [1, 2];
 *     m = bits(f) - bits(0.5f), i.e. f * 2^23 as an integer;
 *     Q(d) = floor(64 m / 2^-n + 1/2), the nearest integer (halves up).
 *   So q_i is 2^(z_i - R_k + 29.5) (z = x s) to within 2^-22 relative plus
 *   half a unit.  S_k = sum of the chunk's q_i (exact) and R = max_k R_k.
 *   Row units are 2^-12 of a unit of the reference R: a chunk's total in
 *   them is U(S_k, R - R_k), with U(v, e) = v 2^(12 - e) for e <= 12 and
 *   floor(v / 2^(e - 12)) above (0 from e - 12 >= 64); the row's total is
 *   T = sum_k U(S_k, R - R_k).  (The 12 guard bits keep the floors of the
 *   chunk totals far below one token's weight.)
 *   A row of more than 4,194,304 entries, or whose chunk maxima have
 *   |fl32(M_k s)| > 2^22 (or is NaN), or whose entries are all -inf, cannot
 *   be weighed: the request gets the empty result (as for an invalid
 *   length).
 * A uniform u becomes the integer k(u) = floor(u 2^24) clamped to
 * [0, 2^24 - 1] (NaN: 0); the generator's uniforms are multiples of 2^-24,
 * so k(u) = u 2^24 exactly.
 * Acceptance of a draft c in [0, V) at row r: with q_c its weight in its
 *   chunk kc and w = U(q_c, R - R_kc), accept iff
 *   floor(k(u_acc) T / 2^24) < w (i.e. u_acc < w / T).  A sentinel draft is
 *   rejected and removes nothing.
 * The draw with u_smp (residual after removing c, or the last row): the
 *   chunk weights become T'_k = U(S_k - [k = kc] q_c, R - R_k),
 *   T' = sum T'_k, t = floor(k(u_smp) T' / 2^24); the chunk is the first
 *   whose running sum of T'_k exceeds t, and inside it, with t_c the
 *   remainder t - (earlier chunks' T'_k) taken back to chunk units
 *   (times 2^(e - 12), or floor(/ 2^(12 - e)), e = R - R_k), the token is
 *   the first entry (c skipped) whose running sum of q_i exceeds t_c.  One
 *   always exists.
 */
#define OR_FX_CHUNK 1024
#define OR_FX_NOREF (-16777216) /* a chunk of -inf only */

/* Horner coefficients c[k] = sqrt(2) (ln 2)^k / k!, from the recurrence
 * t_0 = sqrt(2), t_{k+1} = t_k * ln2 / (k + 1) in double, each rounded to
 * float. */
static void or_fx_coefs(float c[7])
{
    double t = 1.4142135623730951;           /* sqrt(2), correctly rounded */
    const double ln2 = 0.6931471805599453;   /* ln 2, correctly rounded */
    for (int k = 0; k < 7; ++k) {
        c[k] = (float)t;
        t = t * ln2 / (double)(k + 1);
    }
}

static float or_row_value(const void* row, int32_t dtype, int64_t v)
{
    return dtype == 0 ? or_bf16_value(((const uint16_t*)row)[v]) : ((const float*)row)[v];
}

/* Q(d) of one entry with d = fma(x, s, -R). */
static uint64_t or_fx_q(float x, float s, float R, const float c[7])
{
    const float d = fmaf(x, s, -R);
    if (!(d >= -32.0f)) return 0;  /* also -inf */
    const float n = rintf(d);
    const float r = d - n;
    float f = c[6];
    for (int k = 5; k >= 0; --k) f = fmaf(f, r, c[k]);
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    const uint64_t m = (uint64_t)(bits - 0x3F000000u);
    const int sh = (int)(-n); /* 0..32: d <= 1/4 for every entry */
    return (((m << 7) >> sh) + 1) >> 1;
}

/* floor(k v / 2^24) for k < 2^24 and v < 2^62, without 128-bit products. */
static uint64_t or_fx_mulshift(uint32_t k, uint64_t v)
{
    return (uint64_t)k * (v >> 24) + (((uint64_t)k * (v & 0xFFFFFFu)) >> 24);
}

static uint32_t or_fx_unit(float u)
{
    const float v = u * 16777216.0f;
    if (!(v > 0.0f)) return 0;
    if (v >= 16777215.0f) return 16777215u;
    return (uint32_t)v;
}

#define OR_FX_GUARD 12
#define OR_FX_VMAX 4194304

/* U(v, e): a chunk quantity v in row units, e = R - R_k >= 0. */
static uint64_t or_fx_rowunits(uint64_t v, int32_t e)
{
    if (e <= OR_FX_GUARD) return v << (OR_FX_GUARD - e);
    return e - OR_FX_GUARD >= 64 ? 0 : v >> (e - OR_FX_GUARD);
}

/* A row-unit remainder back in chunk units. */
static uint64_t or_fx_chunkunits(uint64_t v, int32_t e)
{
    return e >= OR_FX_GUARD ? v << (e - OR_FX_GUARD) : v >> (OR_FX_GUARD - e);
}

/* Chunk references R[k] and totals S[k] of one row; returns -1 when the row
 * cannot be weighed. */
static int or_fx_row(const void* row, int32_t dtype, int64_t V, float s, const float c[7], uint64_t* S, int32_t* R)
{
    const int64_t nc = (V + OR_FX_CHUNK - 1) / OR_FX_CHUNK;
    int any = 0;
    for (int64_t k = 0; k < nc; ++k) {
        const int64_t v0 = k * OR_FX_CHUNK, v1 = v0 + OR_FX_CHUNK < V ? v0 + OR_FX_CHUNK : V;
        float M = -INFINITY;
        for (int64_t v = v0; v < v1; ++v) {
            const float x = or_row_value(row, dtype, v);
            if (x > M) M = x;
        }
        S[k] = 0;
        if (M == -INFINITY) {
            R[k] = OR_FX_NOREF;
            continue;
        }
        const float y = M * s;
        if (!(fabsf(y) <= 4194304.0f)) return -1;
        R[k] = (int32_t)ceilf(y);
        any = 1;
        for (int64_t v = v0; v < v1; ++v) S[k] += or_fx_q(or_row_value(row, dtype, v), s, (float)R[k], c);
    }
    return any ? 0 : -1;
}

static int32_t or_fx_ref(const int32_t* R, int64_t nc)
{
    int32_t m = OR_FX_NOREF;
    for (int64_t k = 0; k < nc; ++k)
        if (R[k] > m) m = R[k];
    return m;
}

/* The draw from a weighed row with token excl (weight qx) removed; excl
 * outside [0, V) removes nothing. */
static int32_t or_fx_draw(const void* row, int32_t dtype, int64_t V, float s, const float c[7], const uint64_t* S,
                          const int32_t* R, int32_t excl, uint64_t qx, float u)
{
    const int64_t nc = (V + OR_FX_CHUNK - 1) / OR_FX_CHUNK;
    const int32_t Rr = or_fx_ref(R, nc);
    const int64_t kx = (excl >= 0 && excl < V) ? excl / OR_FX_CHUNK : -1;
    uint64_t total = 0;
    for (int64_t k = 0; k < nc; ++k) total += or_fx_rowunits(S[k] - (k == kx ? qx : 0), Rr - R[k]);
    const uint64_t t = or_fx_mulshift(or_fx_unit(u), total);
    uint64_t before = 0;
    for (int64_t k = 0; k < nc; ++k) {
        const uint64_t tk = or_fx_rowunits(S[k] - (k == kx ? qx : 0), Rr - R[k]);
        if (before + tk > t) {
            const uint64_t tc = or_fx_chunkunits(t - before, Rr - R[k]);
            const int64_t v0 = k * OR_FX_CHUNK, v1 = v0 + OR_FX_CHUNK < V ? v0 + OR_FX_CHUNK : V;
            uint64_t run = 0;
            for (int64_t v = v0; v < v1; ++v) {
                if (v == excl) continue;
                run += or_fx_q(or_row_value(row, dtype, v), s, (float)R[k], c);
                if (run > tc) return (int32_t)v;
            }
            return OR_SENT; /* not reached: tc < the chunk's sum */
        }
        before += tk;
    }
    return OR_SENT; /* not reached: t < total */
}

/* One request, as or_sample_verify, on the fixed-point weights.  Returns the
 * number of accepted drafts, or -1 (and no tokens) for an invalid L or
 * temperature or a row that cannot be weighed. */
int32_t or_sample_verify_exact(const void* rows, int32_t dtype, int64_t row_stride, int64_t V, const int32_t* blk,
                               int32_t L, float inv_temp, const float* u, int32_t* out_tok)
{
    for (int i = 0; i < OR_BLOCK; ++i) out_tok[i] = OR_SENT;
    if (L < 1 || L > OR_BLOCK || V < 1 || V > OR_FX_VMAX) return -1;
    if (!(inv_temp > 0.0f && inv_temp < INFINITY)) return -1;
    const size_t rb = (size_t)row_stride * (dtype == 0 ? sizeof(uint16_t) : sizeof(float)); /* bytes per row */
    const int64_t nc = (V + OR_FX_CHUNK - 1) / OR_FX_CHUNK;
    const float s = inv_temp * 1.44269504088896341f;
    float c[7];
    or_fx_coefs(c);
    uint64_t* S = (uint64_t*)malloc((size_t)(nc * L) * sizeof(uint64_t));
    int32_t* R = (int32_t*)malloc((size_t)(nc * L) * sizeof(int32_t));
    if (S == NULL || R == NULL) {
        free(S);
        free(R);
        return -1;
    }
    /* every row of the block must be weighable, whichever rows are used */
    for (int32_t r = 0; r < L; ++r) {
        const void* row = (const char*)rows + (size_t)r * rb;
        if (or_fx_row(row, dtype, V, s, c, S + r * nc, R + r * nc) != 0) {
            free(S);
            free(R);
            return -1;
        }
    }
    int32_t a = 0, tok = OR_SENT;
    for (int32_t r = 0; r < L; ++r) {
        const void* row = (const char*)rows + (size_t)r * rb;
        const uint64_t* Sr = S + r * nc;
        const int32_t* Rrow = R + r * nc;
        if (r == L - 1) {
            tok = or_fx_draw(row, dtype, V, s, c, Sr, Rrow, -1, 0, u[2 * r + 1]);
            break;
        }
        const int32_t cd = blk[r + 1];
        if (cd >= 0 && cd < V) {
            const int32_t Rr = or_fx_ref(Rrow, nc);
            uint64_t T = 0;
            for (int64_t k = 0; k < nc; ++k) T += or_fx_rowunits(Sr[k], Rr - Rrow[k]);
            const int64_t kc = cd / OR_FX_CHUNK;
            const uint64_t qc = or_fx_q(or_row_value(row, dtype, cd), s, (float)Rrow[kc], c);
            const uint64_t w = or_fx_rowunits(qc, Rr - Rrow[kc]);
            if (or_fx_mulshift(or_fx_unit(u[2 * r]), T) < w) {
                out_tok[r] = cd;
                a += 1;
                continue;
            }
            tok = or_fx_draw(row, dtype, V, s, c, Sr, Rrow, cd, qc, u[2 * r + 1]);
        } else {
            tok = or_fx_draw(row, dtype, V, s, c, Sr, Rrow, -1, 0, u[2 * r + 1]);
        }
        break;
    }
    out_tok[a] = tok;
    free(S);
    free(R);
    return a;
}

/* Test access to the pieces of the exact rule (one entry's weight, a row's
 * chunk references and totals, the uniform's integer). */
uint64_t or_fx_weight(float x, float s, int32_t R)
{
    float c[7];
    or_fx_coefs(c);
    return or_fx_q(x, s, (float)R, c);
}

int or_fx_chunks(const void* row, int32_t dtype, int64_t V, float inv_temp, uint64_t* S, int32_t* R)
{
    float c[7];
    or_fx_coefs(c);
    return or_fx_row(row, dtype, V, inv_temp * 1.44269504088896341f, c, S, R);
}

void or_fx_poly_coefs(float* out) { or_fx_coefs(out); }

/* ------------------------------------------------------------------------ */
/* Whole decode loop over a set of requests.                                 */
/* ------------------------------------------------------------------------ */

/* Input providers (the synthetic target and draft model). */
typedef void (*or_logits_fn)(const void* ctx, int32_t b, int64_t P, void* out_row);
typedef void (*or_head_fn)(const void* ctx, int32_t b, int32_t t, int64_t n, int32_t* out);
/* The 16 x 2 sampling uniforms of step t of request b ([16][2]). */
typedef void (*or_uniform_fn)(const void* ctx, int32_t b, int32_t t, float* out);

typedef struct or_run_args {
    const or_params* params;
    int32_t n_req;          /* requests simulated */
    const int32_t* req_ids; /* their ids, passed to the providers */
    const int32_t* prompt;  /* CSR over the n_req requests */
    const int64_t* prompt_off;
    int32_t steps;
    int32_t V;
    int32_t dtype; /* 0 = bf16, 1 = fp32 */
    int32_t threads;
    const void* gen_ctx;
    or_logits_fn logits_fn;
    or_head_fn head_fn;
    or_uniform_fn uniform_fn; /* sampling verification only */
    float inv_temp;           /* > 0: sampling verification at this 1/temperature; 0: greedy */
    int32_t exact;            /* sampling on the fixed-point weights (or_sample_verify_exact) */
    /* outputs, indexed [t][i] or [t][i][16] with i the request's position */
    int32_t* rec_k;
    int32_t* rec_j;
    int32_t* rec_L;
    int32_t* rec_a;
    int32_t* rec_c;
    int32_t* rec_blk;
    int32_t* rec_g;
    int32_t* hist_out;          /* CSR by hist_off: capacity per request */
    const int64_t* hist_off;    /* n_req + 1 */
    int64_t* hist_len;          /* n_req */
    or_counters* counters;      /* n_req */
    /* timing: steps before timed_from are not timed; then nanoseconds in the
     * method's own work and in the providers (filled) */
    int32_t timed_from;
    int32_t pad;
    int64_t method_ns;
    int64_t provider_ns;
    /* the method's time split (timed steps, summed over threads):
     * lookup + copy (full scan), scheduler + fusion, verification */
    int64_t lookup_ns;
    int64_t sched_fuse_ns;
    int64_t verify_ns;
} or_run_args;

typedef struct or_shared {
    or_run_args* a;
    int32_t next;
    pthread_mutex_t mu;
    int32_t error;
} or_shared;

static int64_t or_now_ns(void)
{
    struct timespec ts;
    clock_gettime(CLOCK_MONOTONIC, &ts);
    return (int64_t)ts.tv_sec * 1000000000LL + ts.tv_nsec;
}

static int or_run_request(or_run_args* a, int32_t i, int64_t* method_ns, int64_t* provider_ns, int64_t* part_ns)
{
    const or_params* p = a->params;
    const int32_t b = a->req_ids[i];
    const int64_t n0 = a->prompt_off[i + 1] - a->prompt_off[i];
    const int64_t cap = a->hist_off[i + 1] - a->hist_off[i];
    const size_t esz = a->dtype == 0 ? 2 : 4;
    int32_t* h = a->hist_out + a->hist_off[i];
    const int sampling = a->inv_temp > 0.0f;
    /* greedy: one row at a time; sampling: the block's rows together */
    void* row = malloc((size_t)a->V * esz * (sampling ? OR_BLOCK : 1));
    if (!row) return -1;
    if (n0 > cap || n0 < 1) {
        free(row);
        return -2;
    }
    memcpy(h, a->prompt + a->prompt_off[i], (size_t)n0 * sizeof(int32_t));
    int64_t n = n0;
    or_sched_state st = {OR_SHORT, 0, 0, 0};
    or_counters* cnt = &a->counters[i];
    memset(cnt, 0, sizeof *cnt);
    int32_t prev_a = 0, prev_L = 0;
    const int32_t long_L = 1 + p->head + p->tail;
    int rc = 0;

    int64_t start_ns = or_now_ns();
    int64_t prov = 0;
    for (int32_t t = 0; t < a->steps; ++t) {
        if (t == a->timed_from) {
            start_ns = or_now_ns();
            prov = 0;
        }
        int32_t c[OR_BLOCK], m[OR_BLOCK], blk[OR_BLOCK], g[OR_BLOCK];
        int64_t j;
        const int64_t p0 = or_now_ns();
        int32_t k = or_lookup(h, n, p->min_k, p->max_k, &j);
        or_copy(h, n, k, j, c);
        const int64_t p1 = or_now_ns();
        int32_t L = or_sched(&st, k, prev_a, prev_L, p);
        int64_t u0 = or_now_ns();
        a->head_fn(a->gen_ctx, b, t, n, m);
        const int64_t head_ns = or_now_ns() - u0;
        prov += head_ns;
        or_fuse(h[n - 1], c, k, m, L, p, blk);
        const int64_t p2 = or_now_ns();
        const int64_t prov_before_verify = prov;
        for (int32_t r = 0; r < OR_BLOCK; ++r) g[r] = OR_SENT;
        int32_t acc;
        if (sampling) {
            /* g: the emitted tokens (accepted drafts, then the drawn token) */
            float u[2 * OR_BLOCK];
            u0 = or_now_ns();
            for (int32_t r = 0; r < L; ++r) a->logits_fn(a->gen_ctx, b, n + r, (char*)row + (size_t)r * a->V * esz);
            a->uniform_fn(a->gen_ctx, b, t, u);
            prov += or_now_ns() - u0;
            acc = a->exact ? or_sample_verify_exact(row, a->dtype, a->V, a->V, blk, L, a->inv_temp, u, g)
                           : or_sample_verify(row, a->dtype, a->V, a->V, blk, L, a->inv_temp, u, g);
            if (acc < 0) {
                rc = -3;
                break;
            }
        } else {
            for (int32_t r = 0; r < L; ++r) {
                u0 = or_now_ns();
                a->logits_fn(a->gen_ctx, b, n + r, row);
                prov += or_now_ns() - u0;
                g[r] = a->dtype == 0 ? or_argmax_bf16((const uint16_t*)row, a->V)
                                     : or_argmax_f32((const float*)row, a->V);
            }
            acc = or_accept(blk, g, L);
        }
        if (t >= a->timed_from) {
            const int64_t p3 = or_now_ns();
            part_ns[0] += p1 - p0;
            part_ns[1] += (p2 - p1) - head_ns;
            part_ns[2] += (p3 - p2) - (prov - prov_before_verify);
        }
        if (n + acc + 1 > cap) {
            rc = -2;
            break;
        }
        for (int32_t r = 0; r <= acc; ++r) h[n + r] = g[r];
        n += acc + 1;
        cnt->steps += 1;
        cnt->hits += (k >= p->min_k);
        cnt->long_steps += (p->tail > 0 && L == long_L); /* with no tail there is no long block */
        cnt->drafted += p->head + ((L == long_L && k >= p->tail_k) ? p->tail : 0);
        cnt->accepted += acc;
        cnt->emitted += acc + 1;
        cnt->accept_hist[p->tail > 0 && L == long_L][acc] += 1;
        prev_a = acc;
        prev_L = L;

        const int64_t o = (int64_t)t * a->n_req + i;
        a->rec_k[o] = k;
        a->rec_j[o] = (int32_t)j;
        a->rec_L[o] = L;
        a->rec_a[o] = acc;
        memcpy(a->rec_c + o * OR_BLOCK, c, sizeof c);
        memcpy(a->rec_blk + o * OR_BLOCK, blk, sizeof blk);
        memcpy(a->rec_g + o * OR_BLOCK, g, sizeof g);
    }
    *provider_ns += prov;
    *method_ns += (or_now_ns() - start_ns) - prov;
    a->hist_len[i] = n;
    free(row);
    return rc;
}

static void* or_worker(void* arg)
{
    or_shared* sh = (or_shared*)arg;
    int64_t meth = 0, prov = 0;
    int64_t part[3] = {0, 0, 0};
    for (;;) {
        pthread_mutex_lock(&sh->mu);
        int32_t i = sh->next++;
        pthread_mutex_unlock(&sh->mu);
        if (i >= sh->a->n_req) break;
        int rc = or_run_request(sh->a, i, &meth, &prov, part);
        if (rc != 0) {
            pthread_mutex_lock(&sh->mu);
            if (sh->error == 0) sh->error = rc;
            pthread_mutex_unlock(&sh->mu);
        }
    }
    pthread_mutex_lock(&sh->mu);
    sh->a->method_ns += meth;
    sh->a->provider_ns += prov;
    sh->a->lookup_ns += part[0];
    sh->a->sched_fuse_ns += part[1];
    sh->a->verify_ns += part[2];
    pthread_mutex_unlock(&sh->mu);
    return NULL;
}

/* Runs the decode loop for every request, `threads` requests at a time.
 * Returns 0, -1 (out of memory), -2 (history capacity) or -3 (a sampled block
 * that cannot be weighed: see or_sample_verify_exact). */
int or_run(or_run_args* a)
{
    or_shared sh;
    sh.a = a;
    sh.next = 0;
    sh.error = 0;
    a->method_ns = 0;
    a->provider_ns = 0;
    a->lookup_ns = 0;
    a->sched_fuse_ns = 0;
    a->verify_ns = 0;
    pthread_mutex_init(&sh.mu, NULL);
    int nt = a->threads < 1 ? 1 : a->threads;
    if (nt > a->n_req) nt = a->n_req < 1 ? 1 : a->n_req;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
    if (!th) return -1;
    for (int i = 0; i < nt; ++i) pthread_create(&th[i], NULL, or_worker, &sh);
    for (int i = 0; i < nt; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&sh.mu);
    return sh.error;
}

size_t or_counters_size(void) { return sizeof(or_counters); }
size_t or_run_args_size(void) { return sizeof(or_run_args); }
