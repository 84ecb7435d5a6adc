/*
 * gdn_oracle.c -- plain fp64 CPU oracle for the Gated DeltaNet decode step.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load this library.  The CUDA
 * path shares no code, header, table or helper with it, and it never reads
 * anything the CUDA path produced.
 *
 * Every quantity is carried in double precision, every loop is written out,
 * and nothing is blocked, fused or reordered beyond what the definitions say.
 *
 * Sources (the web pages describing the method):
 *  - "mstar PR #1139" (twin slots for the GDN state pool; the decode-only
 *    causal_conv1d_decode), sections "Why" and "What changed": the GDN rule is
 *    the recurrent state update of a decode step (one token a row); a request
 *    holds two slots, a decode step reads the state from one and writes the
 *    next state to the other, commit swaps them; prefill and split walks keep
 *    the state in place; the decode conv is the conv-state update for one
 *    token a row, with a write slot, optional bias and activation.
 *  - "mstar PR #1127" (resident decode planning), section "What changed":
 *    padding rows sit on row/slot 0, which stays zero (SINK_SLOT).
 *  - "mstar PR #965" (mixed steps), section "What changed": dropped padding
 *    rows only ever address the null slot, so every real row's output and
 *    state is unchanged by them.
 *  The pages name the rule but print no formula for it.  The formulas below
 *  are the standard gated delta rule of Gated DeltaNet:
 *      alpha = exp(-exp(A_log) * softplus(a + dt_bias)),   beta = sigmoid(b)
 *      q^ = q / sqrt(sum q^2 + eps) / sqrt(dk),            k^ = k / sqrt(sum k^2 + eps)
 *      S' = alpha * S * (I - beta * k^ k^T) + beta * v k^T,   o = S' q^
 *  with S in R^{dv x dk}.  Readings where the sources are silent:
 *      eps = 1e-6 inside the square root; softplus(x) = log1p(exp(x)), and x
 *      itself above 20; v head h reads qk head h / (Hv/Hk); the conv window
 *      holds the previous W-1 inputs oldest first, tap W-1 multiplies the
 *      current token; channels are packed [q | k | v], head-major; a row whose
 *      read slot is 0 is padding: no state or conv traffic, output zero.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_L2_EPS 1e-6

/* ------------------------------------------------------------------------ */
/* Scalar pieces                                                             */
/* ------------------------------------------------------------------------ */

/* softplus(x) = log(1 + e^x); above 20 the value is x to within 2e-9. */
double gdn_oracle_softplus(double x)
{
    if (x > 20.0)
        return x;
    return log1p(exp(x));
}

/* Decay gate: alpha = exp(-exp(A_log) * softplus(a + dt_bias)).  The pages
 * name the gates of the rule ("mstar PR #1139", "Why") but print no formula;
 * this is the standard Gated DeltaNet decay. */
double gdn_oracle_alpha(double A_log, double a, double dt_bias)
{
    double decay_rate = exp(A_log);
    double dt = gdn_oracle_softplus(a + dt_bias);
    double g = decay_rate * dt;
    if (decay_rate == 0.0)
        g = 0.0; /* 0 * inf: a zero decay rate means no decay at all */
    return exp(-g);
}

/* Write strength: beta = sigmoid(b) = 1 / (1 + e^-b) (standard Gated
 * DeltaNet, as for alpha). */
double gdn_oracle_beta(double b)
{
    return 1.0 / (1.0 + exp(-b));
}

/*
 * Round a double to the nearest bfloat16 value (ties to even), returned as a
 * double.  bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 stored
 * fraction bits, so 8 significant bits for normal values and a fixed spacing
 * of 2^-133 below 2^-126.  Overflow past the largest finite value rounds to
 * infinity.
 */
double gdn_oracle_round_bf16(double x)
{
    if (x == 0.0 || isnan(x) || isinf(x))
        return x;
    int e2;
    frexp(x, &e2);              /* |x| in [2^(e2-1), 2^e2) */
    int e = e2 - 1;             /* |x| in [2^e, 2^(e+1)) */
    if (e < -126)
        e = -126;               /* subnormal range: fixed spacing */
    double spacing = ldexp(1.0, e - 7);
    double r = nearbyint(x / spacing) * spacing; /* exact steps; default mode is ties-to-even */
    double largest = ldexp(255.0 / 128.0, 127);  /* (2 - 2^-7) * 2^127 */
    if (fabs(r) > largest)
        return x > 0 ? INFINITY : -INFINITY;
    return r;
}

/* Elementwise gdn_oracle_round_bf16 over n values. */
void gdn_oracle_round_bf16_array(const double *x, double *y, long n)
{
    for (long i = 0; i < n; ++i)
        y[i] = gdn_oracle_round_bf16(x[i]);
}

/* Round a double to the nearest binary32 value. */
double gdn_oracle_round_f32(double x)
{
    return (double)(float)x;
}

/* ------------------------------------------------------------------------ */
/* L2 normalisation                                                          */
/* ------------------------------------------------------------------------ */

/* y = x / sqrt(sum_i x_i^2 + eps) * scale */
void gdn_oracle_l2norm(const double *x, int n, double eps, double scale, double *y)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i)
        ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss + eps);
    for (int i = 0; i < n; ++i)
        y[i] = x[i] * inv * scale;
}

/* ------------------------------------------------------------------------ */
/* The gated delta rule for one (row, value head), literal matrix form       */
/* ------------------------------------------------------------------------ */

/*
 * S, S_new: [dv][dk] row-major (S maps a key vector to a value vector).
 *   M      = I - beta * khat khat^T             (dk x dk)
 *   S_new  = alpha * (S M) + beta * v khat^T     (dv x dk)
 *   o      = S_new qhat                          (dv)
 * S_new may not alias S.  The rule the pages name ("mstar PR #1139", "Why":
 * the recurrent state update of one token), in the standard gated delta
 * form stated at the top of this file.
 */
void gdn_oracle_rule(int dk, int dv, const double *S, const double *qhat, const double *khat,
                     const double *v, double alpha, double beta, double *S_new, double *o)
{
    double *M = (double *)malloc(sizeof(double) * (size_t)dk * (size_t)dk);
    for (int l = 0; l < dk; ++l)
        for (int j = 0; j < dk; ++j)
            M[(size_t)l * dk + j] = (l == j ? 1.0 : 0.0) - beta * khat[l] * khat[j];

    for (int i = 0; i < dv; ++i) {
        for (int j = 0; j < dk; ++j) {
            double sm = 0.0;
            for (int l = 0; l < dk; ++l)
                sm += S[(size_t)i * dk + l] * M[(size_t)l * dk + j];
            S_new[(size_t)i * dk + j] = alpha * sm + beta * v[i] * khat[j];
        }
    }
    for (int i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int j = 0; j < dk; ++j)
            acc += S_new[(size_t)i * dk + j] * qhat[j];
        o[i] = acc;
    }
    free(M);
}

/*
 * One (row, value head) of the decode step from raw inputs: normalise q and k,
 * form the gates, apply the rule.
 */
void gdn_oracle_head(int dk, int dv, const double *S, const double *q, const double *k,
                     const double *v, double a, double b, double A_log, double dt_bias,
                     double *S_new, double *o)
{
    double *qhat = (double *)malloc(sizeof(double) * (size_t)dk);
    double *khat = (double *)malloc(sizeof(double) * (size_t)dk);
    gdn_oracle_l2norm(q, dk, ORACLE_L2_EPS, 1.0 / sqrt((double)dk), qhat);
    gdn_oracle_l2norm(k, dk, ORACLE_L2_EPS, 1.0, khat);
    double alpha = gdn_oracle_alpha(A_log, a, dt_bias);
    double beta = gdn_oracle_beta(b);
    gdn_oracle_rule(dk, dv, S, qhat, khat, v, alpha, beta, S_new, o);
    free(qhat);
    free(khat);
}

/* ------------------------------------------------------------------------ */
/* Decode step over a slot-indexed state pool                                */
/* ------------------------------------------------------------------------ */

/*
 * pool:  [num_slots][hv][dv][dk]; slot 0 is the null slot.
 * q, k:  [rows][hk][dk]   v: [rows][hv][dv]   a, b: [rows][hv]
 * A_log, dt_bias: [hv]    out: [rows][hv][dv]
 * Row r is padding when read_slot[r] == 0: out[r] = 0, nothing else.
 * Otherwise the state is read from read_slot[r] and written to write_slot[r]
 * (twin) or back to read_slot[r] (keep_in_place).  A slot outside
 * [0, num_slots), a twin write to slot 0, or a twin write slot equal to the
 * read slot (a twin step writes the other slot) makes the row count as bad:
 * its output is zero and nothing is written.  Returns the number of bad rows.
 * Rows must name distinct slots (a precondition of the method).  Twin slots
 * follow "mstar PR #1139", "What changed" (read one slot, write the other);
 * padding on slot 0 follows "mstar PR #1127" and "mstar PR #965", "What
 * changed" (padding rows address only the null slot, which stays zero).
 */
int gdn_oracle_step(int rows, int hk, int hv, int dk, int dv, int num_slots,
                    const double *q, const double *k, const double *v,
                    const double *a, const double *b, const double *A_log, const double *dt_bias,
                    double *pool, const int32_t *read_slot, const int32_t *write_slot,
                    int keep_in_place, double *out, int nthreads)
{
    const int group = hv / hk;
    const size_t head_elems = (size_t)dv * dk;
    const size_t slot_elems = (size_t)hv * head_elems;
    int bad = 0;
    int *row_ok = (int *)malloc(sizeof(int) * (size_t)(rows > 0 ? rows : 1));
    for (int r = 0; r < rows; ++r) {
        int rs = read_slot[r];
        int ws = keep_in_place ? rs : write_slot[r];
        if (rs == 0) {
            row_ok[r] = 0;
        } else if (rs < 0 || rs >= num_slots || ws <= 0 || ws >= num_slots ||
                   (!keep_in_place && ws == rs)) {
            row_ok[r] = 0;
            ++bad;
        } else {
            row_ok[r] = 1;
        }
    }
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (long u = 0; u < (long)rows * hv; ++u) {
        int r = (int)(u / hv);
        int h = (int)(u % hv);
        double *o = out + ((size_t)r * hv + h) * dv;
        if (!row_ok[r]) {
            for (int i = 0; i < dv; ++i)
                o[i] = 0.0;
            continue;
        }
        int g = h / group;
        int rs = read_slot[r];
        int ws = keep_in_place ? rs : write_slot[r];
        double *S_new = (double *)malloc(sizeof(double) * head_elems);
        gdn_oracle_head(dk, dv, pool + (size_t)rs * slot_elems + (size_t)h * head_elems,
                        q + ((size_t)r * hk + g) * dk, k + ((size_t)r * hk + g) * dk,
                        v + ((size_t)r * hv + h) * dv, a[(size_t)r * hv + h], b[(size_t)r * hv + h],
                        A_log[h], dt_bias[h], S_new, o);
        memcpy(pool + (size_t)ws * slot_elems + (size_t)h * head_elems, S_new,
               sizeof(double) * head_elems);
        free(S_new);
    }
    free(row_ok);
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Depthwise causal conv, one token a row                                    */
/* ------------------------------------------------------------------------ */

/*
 * win: [W-1][C], the previous W-1 inputs, oldest first.  x: [C], this token.
 * w: [C][W]; tap W-1 multiplies x.  bias may be NULL.
 *   pre[c]  = bias[c] + sum_{j<W-1} w[c][j] * win[j][c] + w[c][W-1] * x[c]
 *   y[c]    = silu(pre[c]) = pre / (1 + e^-pre)   (or pre itself when silu == 0)
 *   new_win = [win[1], ..., win[W-2], x]
 * The conv-state update for one token ("mstar PR #1139", "What changed":
 * causal_conv1d_decode, with optional bias and activation).
 */
void gdn_oracle_conv_row(int C, int W, const double *win, const double *x, const double *w,
                         const double *bias, int silu, double *y, double *new_win)
{
    for (int c = 0; c < C; ++c) {
        double pre = bias ? bias[c] : 0.0;
        for (int j = 0; j < W - 1; ++j)
            pre += w[(size_t)c * W + j] * win[(size_t)j * C + c];
        pre += w[(size_t)c * W + (W - 1)] * x[c];
        y[c] = silu ? pre / (1.0 + exp(-pre)) : pre;
    }
    for (int j = 0; j + 1 < W - 1; ++j)
        for (int c = 0; c < C; ++c)
            new_win[(size_t)j * C + c] = win[(size_t)(j + 1) * C + c];
    for (int c = 0; c < C; ++c)
        new_win[(size_t)(W - 2) * C + c] = x[c];
}

/*
 * Conv decode over a slot-indexed conv pool [num_slots][W-1][C].
 * x: [rows][C], y: [rows][C].  write_slot == NULL means in place.
 * Padding rows (read slot 0) give y = 0 and touch no slot.  Bad slots as in
 * gdn_oracle_step (with a write slot given, it must differ from the read
 * slot).  Returns the number of bad rows.  The write slot follows "mstar PR
 * #1139", "What changed" (the decode conv with a write slot).
 */
int gdn_oracle_conv_step(int rows, int C, int W, int num_slots, const double *x,
                         double *conv_pool, const int32_t *read_slot, const int32_t *write_slot,
                         const double *w, const double *bias, int silu, double *y)
{
    const size_t slot_elems = (size_t)(W - 1) * C;
    double *new_win = (double *)malloc(sizeof(double) * (slot_elems > 0 ? slot_elems : 1));
    int bad = 0;
    for (int r = 0; r < rows; ++r) {
        int rs = read_slot[r];
        int ws = write_slot ? write_slot[r] : rs;
        double *yr = y + (size_t)r * C;
        if (rs == 0 || rs < 0 || rs >= num_slots || ws <= 0 || ws >= num_slots ||
            (write_slot && ws == rs)) {
            if (rs != 0)
                ++bad;
            for (int c = 0; c < C; ++c)
                yr[c] = 0.0;
            continue;
        }
        gdn_oracle_conv_row(C, W, conv_pool + (size_t)rs * slot_elems, x + (size_t)r * C, w, bias,
                            silu, yr, new_win);
        memcpy(conv_pool + (size_t)ws * slot_elems, new_win, sizeof(double) * slot_elems);
    }
    free(new_win);
    return bad;
}

/* ------------------------------------------------------------------------ */
/* The whole layer: conv, round to the activation type, split, rule          */
/* ------------------------------------------------------------------------ */

/*
 * x: [rows][C] with C = 2*hk*dk + hv*dv, packed [q | k | v], head-major.
 * The conv output is rounded to the activation type (act_bf16 = 1: bfloat16,
 * 0: binary32), as it would be when stored between two separate kernels,
 * then split into q, k, v and fed to the decode step.  Both pools use the
 * same read and write slots.  Returns the number of bad rows.  The pages run
 * the conv and the rule as separate kernels ("mstar PR #1139", "What
 * changed"); this is that composition, step by step.
 */
int gdn_oracle_layer(int rows, int hk, int hv, int dk, int dv, int W, int num_slots,
                     const double *x, double *conv_pool, const double *w, const double *bias,
                     int silu, const double *a, const double *b, const double *A_log,
                     const double *dt_bias, double *pool, const int32_t *read_slot,
                     const int32_t *write_slot, int keep_in_place, int act_bf16, double *out,
                     int nthreads)
{
    const int C = 2 * hk * dk + hv * dv;
    double *y = (double *)malloc(sizeof(double) * (size_t)(rows > 0 ? rows : 1) * C);
    double *q = (double *)malloc(sizeof(double) * (size_t)(rows > 0 ? rows : 1) * hk * dk);
    double *k = (double *)malloc(sizeof(double) * (size_t)(rows > 0 ? rows : 1) * hk * dk);
    double *v = (double *)malloc(sizeof(double) * (size_t)(rows > 0 ? rows : 1) * hv * dv);
    int bad = gdn_oracle_conv_step(rows, C, W, num_slots, x, conv_pool, read_slot,
                                   keep_in_place ? NULL : write_slot, w, bias, silu, y);
    for (int r = 0; r < rows; ++r) {
        for (int c = 0; c < C; ++c) {
            double t = y[(size_t)r * C + c];
            y[(size_t)r * C + c] = act_bf16 ? gdn_oracle_round_bf16(t) : gdn_oracle_round_f32(t);
        }
        const double *yr = y + (size_t)r * C;
        for (int i = 0; i < hk * dk; ++i) {
            q[(size_t)r * hk * dk + i] = yr[i];
            k[(size_t)r * hk * dk + i] = yr[hk * dk + i];
        }
        for (int i = 0; i < hv * dv; ++i)
            v[(size_t)r * hv * dv + i] = yr[2 * hk * dk + i];
    }
    int bad2 = gdn_oracle_step(rows, hk, hv, dk, dv, num_slots, q, k, v, a, b, A_log, dt_bias,
                               pool, read_slot, write_slot, keep_in_place, out, nthreads);
    free(y);
    free(q);
    free(k);
    free(v);
    return bad > bad2 ? bad : bad2;
}

/* ------------------------------------------------------------------------ */
/* Many tokens a row: prefill and speculative verification                   */
/* ------------------------------------------------------------------------ */

/*
 * Sequence r holds tokens [cu_seqlens[r], cu_seqlens[r+1]) of the packed
 * inputs q, k: [T][hk][dk]   v: [T][hv][dv]   a, b: [T][hv]   out: [T][hv][dv].
 * For each real sequence and value head the decode rule is applied token
 * after token, in order, starting from the state in read_slot[r]; o_t comes
 * from the state after token t ("mstar PR #1139", "Why": prefill keeps the
 * state in place; the rule is the recurrent update of one token).  The final
 * state goes to write_slot[r] (twin), or back to read_slot[r] when write_slot
 * is NULL (in place).  When token_slot ([T]) is given, the state after token t
 * goes to token_slot[t] instead: a state a token, as speculative verification
 * keeps them ("mstar PR #1139", "What changed": speculative decoding holds a
 * state per token); write_slot is then ignored and the read slot left alone.
 * Padding (read slot 0): outputs zero, nothing written.  Bad: a slot outside
 * [0, num_slots), a write or token slot 0, a twin write slot equal to the read
 * slot, a token slot equal to the read slot; outputs zero, nothing written.
 * Returns the number of bad sequences.  Sequences must name distinct slots.
 */
static int prefill_seq_ok(int r, int num_slots, const int32_t *cu_seqlens, const int32_t *read_slot,
                          const int32_t *write_slot, const int32_t *token_slot, int *bad)
{
    int rs = read_slot[r];
    if (rs == 0)
        return 0;
    int ok = rs > 0 && rs < num_slots;
    if (token_slot) {
        for (int t = cu_seqlens[r]; t < cu_seqlens[r + 1]; ++t)
            if (token_slot[t] <= 0 || token_slot[t] >= num_slots || token_slot[t] == rs)
                ok = 0;
    } else if (write_slot) {
        int ws = write_slot[r];
        if (ws <= 0 || ws >= num_slots || ws == rs)
            ok = 0;
    }
    if (!ok)
        ++*bad;
    return ok;
}

int gdn_oracle_prefill(int nseq, int hk, int hv, int dk, int dv, int num_slots,
                       const int32_t *cu_seqlens, const double *q, const double *k, const double *v,
                       const double *a, const double *b, const double *A_log, const double *dt_bias,
                       double *pool, const int32_t *read_slot, const int32_t *write_slot,
                       const int32_t *token_slot, double *out, int nthreads)
{
    const int group = hv / hk;
    const size_t head_elems = (size_t)dv * dk;
    const size_t slot_elems = (size_t)hv * head_elems;
    int bad = 0;
    int *seq_ok = (int *)malloc(sizeof(int) * (size_t)(nseq > 0 ? nseq : 1));
    for (int r = 0; r < nseq; ++r)
        seq_ok[r] = prefill_seq_ok(r, num_slots, cu_seqlens, read_slot, write_slot, token_slot, &bad);
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (long u = 0; u < (long)nseq * hv; ++u) {
        int r = (int)(u / hv);
        int h = (int)(u % hv);
        int g = h / group;
        if (!seq_ok[r]) {
            for (int t = cu_seqlens[r]; t < cu_seqlens[r + 1]; ++t)
                for (int i = 0; i < dv; ++i)
                    out[((size_t)t * hv + h) * dv + i] = 0.0;
            continue;
        }
        int rs = read_slot[r];
        double *S = (double *)malloc(sizeof(double) * head_elems);
        double *S_new = (double *)malloc(sizeof(double) * head_elems);
        memcpy(S, pool + (size_t)rs * slot_elems + (size_t)h * head_elems, sizeof(double) * head_elems);
        for (int t = cu_seqlens[r]; t < cu_seqlens[r + 1]; ++t) {
            gdn_oracle_head(dk, dv, S, q + ((size_t)t * hk + g) * dk, k + ((size_t)t * hk + g) * dk,
                            v + ((size_t)t * hv + h) * dv, a[(size_t)t * hv + h], b[(size_t)t * hv + h],
                            A_log[h], dt_bias[h], S_new, out + ((size_t)t * hv + h) * dv);
            memcpy(S, S_new, sizeof(double) * head_elems);
            if (token_slot)
                memcpy(pool + (size_t)token_slot[t] * slot_elems + (size_t)h * head_elems, S,
                       sizeof(double) * head_elems);
        }
        if (!token_slot) {
            int ws = write_slot ? write_slot[r] : rs;
            memcpy(pool + (size_t)ws * slot_elems + (size_t)h * head_elems, S, sizeof(double) * head_elems);
        }
        free(S);
        free(S_new);
    }
    free(seq_ok);
    return bad;
}

/*
 * The depthwise causal conv over many tokens a row.  Sequence r's tokens
 * x[cu_seqlens[r] .. cu_seqlens[r+1]) ([T][C]) continue the window held in
 * read_slot[r]: each token sees the W-1 inputs before it, from the window and
 * then from the sequence itself; y: [T][C].  The window after the last token
 * goes to write_slot[r] (NULL: in place), or, with token_slot ([T]), the
 * window after token t goes to token_slot[t].  Padding and bad sequences as
 * in gdn_oracle_prefill.  Returns the number of bad sequences.
 */
int gdn_oracle_conv_prefill(int nseq, int C, int W, int num_slots, const int32_t *cu_seqlens,
                            const double *x, double *conv_pool, const int32_t *read_slot,
                            const int32_t *write_slot, const int32_t *token_slot, const double *w,
                            const double *bias, int silu, double *y)
{
    const size_t slot_elems = (size_t)(W - 1) * C;
    double *win = (double *)malloc(sizeof(double) * (slot_elems > 0 ? slot_elems : 1));
    double *new_win = (double *)malloc(sizeof(double) * (slot_elems > 0 ? slot_elems : 1));
    int bad = 0;
    for (int r = 0; r < nseq; ++r) {
        if (!prefill_seq_ok(r, num_slots, cu_seqlens, read_slot, write_slot, token_slot, &bad)) {
            for (int t = cu_seqlens[r]; t < cu_seqlens[r + 1]; ++t)
                for (int c = 0; c < C; ++c)
                    y[(size_t)t * C + c] = 0.0;
            continue;
        }
        int rs = read_slot[r];
        memcpy(win, conv_pool + (size_t)rs * slot_elems, sizeof(double) * slot_elems);
        for (int t = cu_seqlens[r]; t < cu_seqlens[r + 1]; ++t) {
            gdn_oracle_conv_row(C, W, win, x + (size_t)t * C, w, bias, silu, y + (size_t)t * C, new_win);
            memcpy(win, new_win, sizeof(double) * slot_elems);
            if (token_slot)
                memcpy(conv_pool + (size_t)token_slot[t] * slot_elems, win, sizeof(double) * slot_elems);
        }
        if (!token_slot) {
            int ws = write_slot ? write_slot[r] : rs;
            memcpy(conv_pool + (size_t)ws * slot_elems, win, sizeof(double) * slot_elems);
        }
    }
    free(win);
    free(new_win);
    return bad;
}

/*
 * Snapshots and forks: slot dst[i] of a pool receives a copy of slot src[i]
 * ("mstar PR #1139", "What changed": prefix-cache snapshots of the conv window
 * and the state; "mstar PR #965", "What changed": prefix-cache checkpoints).
 * pool: [num_slots][slot_elems].  A source outside [0, num_slots) or a
 * destination outside [1, num_slots) (the null slot is never written) makes
 * the pair bad: it is skipped.  Destinations must be distinct and no
 * destination may be a source (then the order of the copies does not
 * matter).  Returns the number of bad pairs.
 */
int gdn_oracle_copy_slots(int num_slots, long slot_elems, double *pool, const int32_t *src,
                          const int32_t *dst, int n)
{
    int bad = 0;
    for (int i = 0; i < n; ++i) {
        if (src[i] < 0 || src[i] >= num_slots || dst[i] <= 0 || dst[i] >= num_slots) {
            ++bad;
            continue;
        }
        for (long e = 0; e < slot_elems; ++e)
            pool[(size_t)dst[i] * slot_elems + e] = pool[(size_t)src[i] * slot_elems + e];
    }
    return bad;
}

/* Commit of a twin step: the read and write slot of every row trade places
 * ("mstar PR #1139", "What changed": commit swaps the two slots). */
void gdn_oracle_commit(int rows, int32_t *read_slot, int32_t *write_slot)
{
    for (int r = 0; r < rows; ++r) {
        int32_t t = read_slot[r];
        read_slot[r] = write_slot[r];
        write_slot[r] = t;
    }
}

/* Threads an OpenMP region would use (1 without OpenMP). */
int gdn_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
