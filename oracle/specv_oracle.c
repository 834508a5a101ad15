/*
 * specv_oracle.c -- plain, slow, float64 CPU oracle for the batched
 * speculative-decoding verify step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker that the CUDA path is
 * compared against.  Only the tests, the smoke check and the benchmark's CPU
 * baseline leg may load it; the product library never links, imports or
 * calls it, and it shares no code, header, table or helper with the CUDA
 * sources.  It is written for a reader who wants to check it against the
 * pages by eye: one row at a time, one position at a time, every sum a plain
 * left-to-right loop in double precision, in the order the pages give.
 *
 * Sources (page title, section):
 *  [A] "LLM Inference & Speculative Decoding: From Roofline Physics to
 *      Lossless Acceleration" -- s.2 "Speculative Decoding: Exact Modified
 *      Rejection Sampling Proof" (acceptance rule, residual distribution,
 *      bonus token, PyTorch verification step with its q clamp) and s.4
 *      "Failure Modes" (greedy T = 0 rule, FP32-or-better arithmetic).
 *  [B] "Speculative Decoding: Mathematical Foundations, Distribution
 *      Preservation Proofs, ..." -- "The Modified Rejection Sampling
 *      Algorithm" (stop at the first rejection, discard later drafts, bonus
 *      token) and "Greedy Decoding Equivalence".
 *  [C] "Speculative decoding." (learn-cs lesson) -- "First: what an output
 *      distribution is" (softmax of logits / T, sampling by laying the
 *      probabilities end to end), "Draft, then verify", "The acceptance rule".
 *  [D] "Speculative Decoding: Draft, Verify, Accept" -- demo script part B
 *      (residual with a zero-mass fallback to p, inverse-CDF sampling).
 *
 * Readings where the pages leave a step open (the plainest reading that the
 * rest of the pages support, with the reason beside each):
 *  - accept iff u < min(1, p(x)/max(q(x), 1e-12))  (strict '<' and the clamp
 *    follow the code of [A] s.2 and [D]);
 *  - inverse CDF: the token is the smallest v, in vocabulary order, with
 *    u * W < sum_{w<=v} weight(w), W = sum of all weights; if no v qualifies
 *    the last v with positive weight is taken;
 *  - residual mass W = 0: sample from p_j instead ([D] residual()) and set
 *    the informational status bit 16;
 *  - uniforms U[b,i,0] drive the accept test at position i < k, U[j,1] the
 *    residual or bonus draw at the stop position j;
 *  - temperature divides the target logits only; q is used as given;
 *  - T == 0 selects the greedy rule of [A] s.4 / [C] (argmax, lowest index
 *    on ties); any other T must be a finite normal positive float;
 *  - data errors end the row's walk at the position where they are met
 *    (bits: 1 non-finite logits, 2 draft token out of range, 4 uniform not
 *    in [0,1), 8 bad temperature, 32 q value NaN, negative or infinite);
 *    an error row reports num_accepted = 0 and out_tokens = -1.
 */
#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ST_NONFINITE 1
#define ST_TOKEN_RANGE 2
#define ST_UNIFORM_RANGE 4
#define ST_TEMPERATURE 8
#define ST_ZERO_RESIDUAL 16
#define ST_Q_INVALID 32
#define ST_FILTER 1024 /* warped verification: top_k outside [1, 4096] or top_p outside (0, 1] */
#define ST_ERROR_MASK (ST_NONFINITE | ST_TOKEN_RANGE | ST_UNIFORM_RANGE | ST_TEMPERATURE | ST_Q_INVALID | ST_FILTER)

/* Exact decoding of one stored logit to double. dtype 0 = float32,
 * dtype 1 = bfloat16 (the upper 16 bits of a float32). */
static double logit_at(int dtype, const void *base, int64_t idx) {
    if (dtype == 1) {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float *)base)[idx];
}

/* ---------------------------------------------------------------- step 1
 * Target distribution at one position: p(v) = exp((l(v) - M) / T) / s with
 * M = max_v l(v) and s = sum_v exp((l(v) - M) / T)  ([C] "First: what an
 * output distribution is": softmax of the logits, temperature divides them
 * first).  Subtracting M leaves p unchanged and keeps exp() finite.
 * Returns 0 if the row is usable, ST_NONFINITE if a logit is NaN or +inf,
 * or every logit is -inf (then p does not exist).
 * e_out (nullable) receives exp((l - M)/T) for every v.                   */
int specv_oracle_softmax_stats(int dtype, const void *row, int64_t V, double T,
                               double *M_out, double *s_out, double *e_out) {
    double M = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
        double l = logit_at(dtype, row, v);
        if (isnan(l) || l == INFINITY) {
            *M_out = NAN;
            *s_out = NAN;
            return ST_NONFINITE;
        }
        if (l > M) M = l;
    }
    if (M == -INFINITY) {
        *M_out = M;
        *s_out = NAN;
        return ST_NONFINITE;
    }
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        double e = exp((logit_at(dtype, row, v) - M) / T);
        if (e_out) e_out[v] = e;
        s += e;
    }
    *M_out = M;
    *s_out = s;
    return 0;
}

/* Greedy target token: argmax_v l(v), the lowest index among equal maxima
 * ([A] s.4 fix for T = 0; [C] "The acceptance rule", greedy case).
 * Returns ST_NONFINITE if any logit is NaN (the argmax is then undefined).  */
int specv_oracle_argmax(int dtype, const void *row, int64_t V, int64_t *arg_out, double *max_out) {
    int64_t best = 0;
    double bestv = logit_at(dtype, row, 0);
    if (isnan(bestv)) return ST_NONFINITE;
    for (int64_t v = 1; v < V; ++v) {
        double l = logit_at(dtype, row, v);
        if (isnan(l)) return ST_NONFINITE;
        if (l > bestv) {
            bestv = l;
            best = v;
        }
    }
    *arg_out = best;
    *max_out = bestv;
    return 0;
}

/* ---------------------------------------------------------------- step 4
 * Residual weights r(v) = max(0, p(v) - q(v)) and their total
 * S = sum_v r(v)  ([A] s.2 residual distribution; [B] P'(x); [D] residual()).
 * The normaliser is applied by the sampler, which compares u * S with the
 * running sum of r.  Returns ST_Q_INVALID if some q(v) is NaN, negative or
 * infinite.                                                                */
int specv_oracle_residual(const double *p, const float *q, int64_t V, double *r_out, double *S_out) {
    double S = 0.0;
    int st = 0;
    for (int64_t v = 0; v < V; ++v) {
        double qv = (double)q[v];
        if (!(qv >= 0.0 && qv <= (double)FLT_MAX)) st = ST_Q_INVALID;
        double r = p[v] - qv;
        if (r < 0.0) r = 0.0;
        r_out[v] = r;
        S += r;
    }
    *S_out = S;
    return st;
}

/* The residual for a one-hot draft, q = the point mass at the draft token x
 * ([C] "One guess (lookup)": keep x with probability p(x), otherwise sample
 * from p with x removed; "N-gram and prompt lookup": q is one-hot).  It is
 * the same definition r(v) = max(0, p(v) - q(v)) with q(x) = 1 and q(v) = 0
 * elsewhere: r(v) = p(v) for v != x and r(x) = max(0, p(x) - 1) = 0.        */
int specv_oracle_residual_onehot(const double *p, int64_t V, int64_t x, double *r_out, double *S_out) {
    double S = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        double r = p[v] - (v == x ? 1.0 : 0.0);
        if (r < 0.0) r = 0.0;
        r_out[v] = r;
        S += r;
    }
    *S_out = S;
    return 0;
}

/* Inverse-CDF sampling over non-negative weights w[0..V): lay the weights
 * end to end in vocabulary order and take the slot that u * W lands in
 * ([C] "First: what an output distribution is", sampling; [D] sample()).
 * W is the sum of w in the same order.  The token is the smallest v with
 * u * W < C(v), C(v) = w[0] + ... + w[v]; if none qualifies the last v with
 * positive weight is returned.  lo/hi (nullable) receive C(v-1)/W and C(v)/W
 * of the returned token, the edges of its slot on [0,1).                  */
int64_t specv_oracle_inverse_cdf(const double *w, int64_t V, double u, double *lo, double *hi) {
    double W = 0.0;
    for (int64_t v = 0; v < V; ++v) W += w[v];
    double target = u * W;
    double C = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        double before = C;
        C += w[v];
        if (target < C) {
            if (lo) *lo = before / W;
            if (hi) *hi = C / W;
            return v;
        }
    }
    int64_t last = V - 1;
    while (last > 0 && !(w[last] > 0.0)) --last;
    if (lo) *lo = 1.0;
    if (hi) *hi = 1.0;
    return last;
}

/* ---------------------------------------------------------------- the row */

typedef struct {
    int dtype;
    const void *logits;        /* [B, k+1, V] */
    const float *q;            /* [B, k, V] or NULL when every row is greedy */
    const int32_t *x;          /* [B, k] */
    const float *u;            /* [B, k+1, 2] or NULL when every row is greedy */
    const float *T;            /* [B] or NULL: every row greedy */
    int64_t B;
    int k;
    int64_t V;
    int32_t *num_accepted;     /* [B] */
    int32_t *out_tokens;       /* [B, k+1] */
    int32_t *row_status;       /* [B] */
    double *p_at_draft;        /* [B, k] nullable */
    double *q_at_draft;        /* [B, k] nullable */
    double *row_max;           /* [B, k+1] nullable */
    double *row_sumexp;        /* [B, k+1] nullable */
    double *residual_mass;     /* [B] nullable */
    int32_t *boundary;         /* [B] nullable: 0, or 1 + 2*i + slot of U[b,i,slot] */
    double eps;
} job_t;

static int temperature_ok(float T) { return T == 0.0f || (T >= FLT_MIN && T <= FLT_MAX); }

static int uniform_ok(float u) { return u >= 0.0f && u < 1.0f; }

static void note_boundary(const job_t *J, int64_t b, int i, int slot, double u, double edge) {
    if (!J->boundary || J->boundary[b] != 0) return;
    if (fabs(u - edge) <= J->eps) J->boundary[b] = 1 + 2 * i + slot;
}

static void finish_error(const job_t *J, int64_t b, int status) {
    J->row_status[b] = status;
    J->num_accepted[b] = 0;
    for (int i = 0; i <= J->k; ++i) J->out_tokens[b * (J->k + 1) + i] = -1;
}

static void finish_ok(const job_t *J, int64_t b, int j, int64_t token, int status) {
    const int k = J->k;
    J->row_status[b] = status;
    J->num_accepted[b] = j;
    for (int i = 0; i < j; ++i) J->out_tokens[b * (k + 1) + i] = J->x[b * k + i];
    J->out_tokens[b * (k + 1) + j] = (int32_t)token;
    for (int i = j + 1; i <= k; ++i) J->out_tokens[b * (k + 1) + i] = -1;
}

static const void *row_ptr(const job_t *J, int64_t b, int i) {
    int64_t off = (b * (J->k + 1) + i) * J->V;
    return J->dtype == 1 ? (const void *)((const uint16_t *)J->logits + off)
                         : (const void *)((const float *)J->logits + off);
}

/* Debug intermediates for every position, independent of the walk:
 * row_max = M_i, row_sumexp = s_i (0 for greedy rows), p_at_draft =
 * p_i(x_i), q_at_draft = q_i(x_i) (0 for greedy rows or out-of-range x).  */
static void fill_debug(const job_t *J, int64_t b, int greedy, double T) {
    const int k = J->k;
    for (int i = 0; i <= k; ++i) {
        const void *row = row_ptr(J, b, i);
        double M = NAN, s = 0.0;
        if (greedy) {
            int64_t a;
            if (specv_oracle_argmax(J->dtype, row, J->V, &a, &M) != 0) M = NAN;
        } else {
            specv_oracle_softmax_stats(J->dtype, row, J->V, T, &M, &s, NULL);
        }
        if (J->row_max) J->row_max[b * (k + 1) + i] = M;
        if (J->row_sumexp) J->row_sumexp[b * (k + 1) + i] = greedy ? 0.0 : s;
        if (i == k) continue;
        int32_t x = J->x[b * k + i];
        double p = 0.0, q = 0.0;
        if (!greedy && x >= 0 && x < J->V) {
            p = exp((logit_at(J->dtype, row, x) - M) / T) / s;
            q = J->q ? (double)J->q[(b * k + i) * J->V + x] : 1.0; /* one-hot draft: q(x) = 1 */
        }
        if (J->p_at_draft) J->p_at_draft[b * k + i] = p;
        if (J->q_at_draft) J->q_at_draft[b * k + i] = q;
    }
}

/* Greedy verification ([A] s.4; [B] "Greedy Decoding Equivalence"; [C]
 * "The acceptance rule", greedy case): keep x_i while it equals the target
 * argmax a_i; at the first mismatch emit a_i; if all k match, emit a_k.   */
static void verify_greedy_row(const job_t *J, int64_t b) {
    const int k = J->k;
    for (int i = 0; i <= k; ++i) {
        int st = 0;
        int32_t x = -1;
        if (i < k) {
            x = J->x[b * k + i];
            if (x < 0 || x >= J->V) st |= ST_TOKEN_RANGE;
        }
        int64_t a;
        double M;
        st |= specv_oracle_argmax(J->dtype, row_ptr(J, b, i), J->V, &a, &M);
        if (st) {
            finish_error(J, b, st);
            return;
        }
        if (i == k || x != a) {
            finish_ok(J, b, i, a, 0);
            return;
        }
    }
}

/* Sampled verification, the modified rejection sampling of [A] s.2 and
 * [B], in the order of [C] "Draft, then verify": accept left to right,
 * stop at the first rejection, then fix (residual) or bonus.              */
static void verify_sampled_row(const job_t *J, int64_t b, double T, double *buf_p, double *buf_w) {
    const int k = J->k;
    const int64_t V = J->V;
    int j = k; /* stop position: first rejection, or k when all are kept */
    for (int i = 0; i < k; ++i) {
        int st = 0;
        int32_t x = J->x[b * k + i];
        float u = J->u[(b * (k + 1) + i) * 2 + 0];
        if (x < 0 || x >= V) st |= ST_TOKEN_RANGE;
        if (!uniform_ok(u)) st |= ST_UNIFORM_RANGE;
        double M, s;
        st |= specv_oracle_softmax_stats(J->dtype, row_ptr(J, b, i), V, T, &M, &s, NULL);
        double q = 0.0;
        if (x >= 0 && x < V) {
            q = J->q ? (double)J->q[(b * k + i) * V + x] : 1.0; /* one-hot draft: q(x) = 1 */
            if (!(q >= 0.0 && q <= (double)FLT_MAX)) st |= ST_Q_INVALID;
        }
        if (st) {
            finish_error(J, b, st);
            return;
        }
        /* p_i(x) and the acceptance probability min(1, p/q), q clamped
         * below at 1e-12 as in the verification step of [A] s.2. */
        double p = exp((logit_at(J->dtype, row_ptr(J, b, i), x) - M) / T) / s;
        double rho = p / (q > 1e-12 ? q : 1e-12);
        if (rho > 1.0) rho = 1.0;
        note_boundary(J, b, i, 0, (double)u, rho);
        if (!((double)u < rho)) {
            j = i;
            break;
        }
    }

    float u1 = J->u[(b * (k + 1) + j) * 2 + 1];
    double M, s;
    int st = specv_oracle_softmax_stats(J->dtype, row_ptr(J, b, j), V, T, &M, &s, buf_w);
    if (!uniform_ok(u1)) st |= ST_UNIFORM_RANGE;
    if (st) {
        finish_error(J, b, st);
        return;
    }
    int status = 0;
    int64_t token;
    double lo, hi;
    if (j == k) {
        /* Bonus token: sample from p_{k+1} = e / s.  The unnormalised
         * weights e give the same slots as p. */
        token = specv_oracle_inverse_cdf(buf_w, V, (double)u1, &lo, &hi);
        if (J->residual_mass) J->residual_mass[b] = 0.0;
    } else {
        for (int64_t v = 0; v < V; ++v) buf_p[v] = buf_w[v] / s;
        double S;
        int qst = J->q ? specv_oracle_residual(buf_p, J->q + (b * k + j) * V, V, buf_w, &S)
                       : specv_oracle_residual_onehot(buf_p, V, (int64_t)J->x[b * k + j], buf_w, &S);
        if (qst) {
            finish_error(J, b, qst);
            return;
        }
        if (J->residual_mass) J->residual_mass[b] = S;
        if (S > 0.0) {
            token = specv_oracle_inverse_cdf(buf_w, V, (double)u1, &lo, &hi);
        } else {
            /* zero residual mass: fall back to p ([D] residual()) */
            status |= ST_ZERO_RESIDUAL;
            token = specv_oracle_inverse_cdf(buf_p, V, (double)u1, &lo, &hi);
        }
    }
    note_boundary(J, b, j, 1, (double)u1, lo);
    note_boundary(J, b, j, 1, (double)u1, hi);
    finish_ok(J, b, j, token, status);
}

typedef struct {
    const job_t *J;
    int64_t b0, b1;
    int err;
} range_t;

static void *run_range(void *arg) {
    range_t *R = (range_t *)arg;
    const job_t *J = R->J;
    double *buf_p = (double *)malloc(sizeof(double) * (size_t)J->V);
    double *buf_w = (double *)malloc(sizeof(double) * (size_t)J->V);
    if (!buf_p || !buf_w) {
        free(buf_p);
        free(buf_w);
        R->err = 1;
        return NULL;
    }
    for (int64_t b = R->b0; b < R->b1; ++b) {
        if (J->boundary) J->boundary[b] = 0;
        if (J->residual_mass) J->residual_mass[b] = 0.0;
        float Tf = J->T ? J->T[b] : 0.0f;
        int greedy = (Tf == 0.0f);
        if (J->p_at_draft || J->q_at_draft || J->row_max || J->row_sumexp)
            fill_debug(J, b, greedy || !temperature_ok(Tf), (double)Tf);
        if (!temperature_ok(Tf)) {
            finish_error(J, b, ST_TEMPERATURE);
            continue;
        }
        if (greedy)
            verify_greedy_row(J, b);
        else
            verify_sampled_row(J, b, (double)Tf, buf_p, buf_w);
    }
    free(buf_p);
    free(buf_w);
    return NULL;
}

/* The whole batch.  Rows are independent; nthreads > 1 splits them into
 * contiguous ranges, one per POSIX thread (nthreads <= 0: one per online
 * core).  Returns 0, or -1 on a bad argument, -2 if memory ran out.       */
int specv_oracle_verify(int dtype, const void *logits, const float *q, const int32_t *x,
                        const float *u, const float *T, int64_t B, int k, int64_t V,
                        int32_t *num_accepted, int32_t *out_tokens, int32_t *row_status,
                        double *p_at_draft, double *q_at_draft, double *row_max,
                        double *row_sumexp, double *residual_mass, int32_t *boundary,
                        double boundary_eps, int nthreads) {
    if (B < 0 || k < 1 || V < 1 || (dtype != 0 && dtype != 1)) return -1;
    if (!logits || !x || !num_accepted || !out_tokens || !row_status) return -1;
    if (T && !u) return -1; /* q may be NULL: one-hot drafts */
    job_t J = {dtype, logits, q, x, u, T, B, k, V, num_accepted, out_tokens, row_status,
               p_at_draft, q_at_draft, row_max, row_sumexp, residual_mass, boundary, boundary_eps};
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if ((int64_t)nthreads > B) nthreads = B > 0 ? (int)B : 1;
    range_t *R = (range_t *)calloc((size_t)nthreads, sizeof(range_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!R || !th) {
        free(R);
        free(th);
        return -2;
    }
    for (int t = 0; t < nthreads; ++t) {
        R[t].J = &J;
        R[t].b0 = B * t / nthreads;
        R[t].b1 = B * (t + 1) / nthreads;
    }
    int err = 0;
    if (nthreads == 1) {
        run_range(&R[0]);
        err = R[0].err;
    } else {
        for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, run_range, &R[t]);
        for (int t = 0; t < nthreads; ++t) {
            pthread_join(th[t], NULL);
            err |= R[t].err;
        }
    }
    free(R);
    free(th);
    return err ? -2 : 0;
}

/* ---------------------------------------------------------------- rollback
 * Paged KV-cache bookkeeping after verification, row by row in batch order
 * ([A] s.1 "PagedKVCacheManager", rollback_to): a row whose cache holds
 * seq_len positions, the last k of them the drafts, keeps
 *   target_len = seq_len - (k - num_accepted)
 * positions; its block table keeps ceil(target_len / block_size) blocks
 * (0 for an empty sequence) and the rest are popped from the end, each one
 * appended to the free list as it is popped.  A row whose num_accepted is
 * outside [0, k], whose target length would be negative, or whose block
 * count is out of [0, max_blocks] is left as it is and gets status 128.
 * If the free list cannot take every freed block, nothing changes and every
 * row gets status 256.  Popped table entries are set to -1.             */
int specv_oracle_rollback(const int32_t *num_accepted, int64_t B, int k, int32_t *seq_lens,
                          int32_t *block_tables, int max_blocks, int32_t *num_blocks, int block_size,
                          int32_t *free_list, int64_t free_capacity, int32_t *free_count,
                          int32_t *row_status) {
    if (B < 0 || k < 0 || max_blocks < 0 || block_size < 1 || !num_accepted || !seq_lens ||
        !block_tables || !num_blocks || !free_count || (!free_list && free_capacity > 0))
        return -1;
    /* the free list's room is checked against the whole batch first */
    int64_t total = 0;
    for (int64_t b = 0; b < B; ++b) {
        int32_t n = num_accepted[b], len = seq_lens[b], nb = num_blocks[b];
        if (n < 0 || n > k || len - (k - n) < 0 || nb < 0 || nb > max_blocks) continue;
        int64_t target = (int64_t)len - (k - n);
        int64_t needed = target > 0 ? (target + block_size - 1) / block_size : 0;
        if (nb > needed) total += nb - needed;
    }
    if ((int64_t)*free_count + total > free_capacity) {
        if (row_status)
            for (int64_t b = 0; b < B; ++b) row_status[b] = 256;
        return 0;
    }
    for (int64_t b = 0; b < B; ++b) {
        int32_t n = num_accepted[b], len = seq_lens[b];
        int32_t *table = block_tables + b * max_blocks;
        if (n < 0 || n > k || len - (k - n) < 0 || num_blocks[b] < 0 || num_blocks[b] > max_blocks) {
            if (row_status) row_status[b] = 128;
            continue;
        }
        int64_t target = (int64_t)len - (k - n);
        int64_t needed = target > 0 ? (target + block_size - 1) / block_size : 0;
        while (num_blocks[b] > needed) {
            int32_t freed = table[num_blocks[b] - 1]; /* pop */
            table[num_blocks[b] - 1] = -1;
            num_blocks[b] -= 1;
            free_list[(*free_count)++] = freed; /* append */
        }
        seq_lens[b] = (int32_t)target;
        if (row_status) row_status[b] = 0;
    }
    return 0;
}

/* ---------------------------------------------------------------- tree
 * Greedy verification of a draft tree ([A] s.3 "Multi-Draft Tree
 * Speculation"; [B] "SpecInfer and Tree-Based Verification": the target
 * scores every node in one pass and the longest accepted path is kept).
 * Row b holds M draft nodes: token[i] and parent[i] in [-1, i) (-1: a child
 * of the prefix).  Logit row 0 is the target's prediction after the prefix,
 * row 1 + i its prediction after node i.  Node i is accepted iff its parent
 * is (the prefix always is) and token[i] equals the argmax (lowest index on
 * ties) of its parent's row.  The deepest accepted node wins, the lowest
 * index among equally deep ones; the row emits the tokens of its path from
 * the prefix down, then the argmax of its own row (the bonus; row 0 when no
 * node is accepted).  num_accepted = the path length.  Errors (no tokens
 * emitted, num_accepted 0): a NaN logit in any of the M + 1 rows (bit 1), a
 * token outside [0, V) (bit 2), a parent outside [-1, i) (bit 512).        */
int specv_oracle_tree_greedy(int dtype, const void *logits, const int32_t *tokens, const int32_t *parents,
                             int64_t B, int M, int64_t V, int32_t *num_accepted, int32_t *out_tokens,
                             int32_t *path, int32_t *row_status) {
    if (B < 0 || M < 1 || M > 4096 || V < 1 || (dtype != 0 && dtype != 1)) return -1;
    if (!logits || !tokens || !parents || !num_accepted || !out_tokens || !row_status) return -1;
    int64_t *amax = (int64_t *)malloc(sizeof(int64_t) * (size_t)(M + 1));
    int *acc = (int *)malloc(sizeof(int) * (size_t)M);
    int *depth = (int *)malloc(sizeof(int) * (size_t)M);
    if (!amax || !acc || !depth) {
        free(amax);
        free(acc);
        free(depth);
        return -2;
    }
    const size_t esz = dtype == 1 ? 2 : 4;
    for (int64_t b = 0; b < B; ++b) {
        const int32_t *tok = tokens + b * M, *par = parents + b * M;
        int st = 0;
        for (int r = 0; r <= M; ++r) {
            const void *row = (const unsigned char *)logits + ((size_t)b * (M + 1) + r) * (size_t)V * esz;
            double mx;
            st |= specv_oracle_argmax(dtype, row, V, &amax[r], &mx);
        }
        for (int i = 0; i < M; ++i) {
            if (tok[i] < 0 || tok[i] >= V) st |= ST_TOKEN_RANGE;
            if (par[i] < -1 || par[i] >= i) st |= 512;
        }
        for (int i = 0; i <= M; ++i) out_tokens[b * (M + 1) + i] = -1;
        if (path)
            for (int i = 0; i < M; ++i) path[b * M + i] = -1;
        row_status[b] = st;
        if (st) {
            num_accepted[b] = 0;
            continue;
        }
        int best = -1;
        for (int i = 0; i < M; ++i) {
            const int p = par[i];
            const int parent_ok = p < 0 ? 1 : acc[p];
            acc[i] = parent_ok && (int64_t)tok[i] == amax[p + 1];
            depth[i] = p < 0 ? 0 : depth[p] + 1;
            if (acc[i] && (best < 0 || depth[i] > depth[best])) best = i;
        }
        const int n = best < 0 ? 0 : depth[best] + 1;
        num_accepted[b] = n;
        for (int node = best, d = n - 1; node >= 0; node = par[node], --d) {
            out_tokens[b * (M + 1) + d] = tok[node];
            if (path) path[b * M + d] = node;
        }
        out_tokens[b * (M + 1) + n] = (int32_t)amax[best + 1];
    }
    free(amax);
    free(acc);
    free(depth);
    return 0;
}

/* ---------------------------------------------------------------- warping
 * Sampled verification with top-k / top-p applied to the target p before
 * the rule ([C] "Why the output is exactly p": temperature, top-k and top-p
 * have to be applied to p before the rule; [D] "The rejection-sampling
 * correctness argument": the rule composes with anything that changes p).
 * The pages name the filters but do not define them; the readings here:
 *   top-k: the K entries with the largest logits, the lower index first
 *          among equal logits (exactly min(K, V) entries);
 *   top-p: within those, in the same order, the shortest prefix whose mass
 *          (renormalised over the K entries) reaches top_p (at least one
 *          entry; top_p >= 1 keeps all K);
 *   p'   = exp((l - M) / T) on the kept set P, renormalised; 0 elsewhere.
 * The rule then runs on p' exactly as in verify_sampled_row; the residual
 * max(0, p' - q) lives on P only (q is read there and at the draft tokens,
 * and only there is it checked), and the inverse CDF walks P in vocabulary
 * order.  q == NULL: one-hot drafts.  Greedy rows (T = 0) are unaffected:
 * the argmax is always kept.                                              */
typedef struct {
    double *val;
    int64_t *idx;
    double *e;
    int n;
} kept_t;

/* P of one row: returns ST_NONFINITE for a NaN / +inf logit or an all -inf
 * row, else 0; fills kept->(val, idx, e) in rank order and the kept count. */
static int warp_row(int dtype, const void *row, int64_t V, double T, int K, double top_p, kept_t *kp,
                    double *S_out) {
    int cnt = 0;
    if (K > V) K = (int)V;
    for (int64_t v = 0; v < V; ++v) {
        double l = logit_at(dtype, row, v);
        if (isnan(l) || l == INFINITY) return ST_NONFINITE;
        if (cnt == K && !(l > kp->val[cnt - 1])) continue;
        int pos = cnt < K ? cnt : K - 1;
        if (cnt < K) ++cnt;
        while (pos > 0 && l > kp->val[pos - 1]) { /* equal values keep the lower index first */
            kp->val[pos] = kp->val[pos - 1];
            kp->idx[pos] = kp->idx[pos - 1];
            --pos;
        }
        kp->val[pos] = l;
        kp->idx[pos] = v;
    }
    double M = kp->val[0];
    if (M == -INFINITY) return ST_NONFINITE;
    double SK = 0.0;
    for (int r = 0; r < cnt; ++r) {
        kp->e[r] = exp((kp->val[r] - M) / T);
        SK += kp->e[r];
    }
    int n = cnt;
    if (top_p < 1.0) {
        double c = 0.0;
        for (n = 0; n < cnt;) {
            c += kp->e[n];
            ++n;
            if (c >= top_p * SK) break;
        }
    }
    double S = 0.0;
    for (int r = 0; r < n; ++r) S += kp->e[r];
    kp->n = n;
    *S_out = S;
    return 0;
}

/* Inverse CDF over the kept entries in vocabulary order: the smallest index
 * v with u * W < (sum of w over kept entries with index <= v); else the last
 * kept index with positive weight.  w[r] belongs to kp->idx[r].            */
static int64_t kept_inverse_cdf(const kept_t *kp, const double *w, double u, double *lo, double *hi) {
    int order[4096] = {0};
    int n = kp->n;
    for (int r = 0; r < n; ++r) order[r] = r;
    for (int a = 1; a < n; ++a) { /* insertion sort by index */
        int t = order[a], b = a;
        while (b > 0 && kp->idx[order[b - 1]] > kp->idx[t]) {
            order[b] = order[b - 1];
            --b;
        }
        order[b] = t;
    }
    double W = 0.0;
    for (int r = 0; r < n; ++r) W += w[order[r]];
    double target = u * W, C = 0.0;
    for (int r = 0; r < n; ++r) {
        double before = C;
        C += w[order[r]];
        if (target < C) {
            *lo = before / W;
            *hi = C / W;
            return kp->idx[order[r]];
        }
    }
    int last = n - 1;
    while (last > 0 && !(w[order[last]] > 0.0)) --last;
    *lo = *hi = 1.0;
    return kp->idx[order[last]];
}

int specv_oracle_verify_warped(int dtype, const void *logits, const float *q, const int32_t *x, const float *u,
                               const float *T, const int32_t *top_k, const float *top_p, int64_t B, int k,
                               int64_t V, int32_t *num_accepted, int32_t *out_tokens, int32_t *row_status,
                               int32_t *boundary, double boundary_eps) {
    if (B < 0 || k < 1 || V < 1 || (dtype != 0 && dtype != 1)) return -1;
    if (!logits || !x || !u || !T || !top_k || !top_p || !num_accepted || !out_tokens || !row_status) return -1;
    kept_t kp;
    kp.n = 0;
    kp.val = (double *)malloc(sizeof(double) * 4096);
    kp.idx = (int64_t *)malloc(sizeof(int64_t) * 4096);
    kp.e = (double *)malloc(sizeof(double) * 4096);
    double *w = (double *)malloc(sizeof(double) * 4096);
    if (!kp.val || !kp.idx || !kp.e || !w) {
        free(kp.val), free(kp.idx), free(kp.e), free(w);
        return -2;
    }
    const size_t esz = dtype == 1 ? 2 : 4;
    job_t J = {dtype, logits, q, x, u, T, B, k, V, num_accepted, out_tokens, row_status,
               NULL, NULL, NULL, NULL, NULL, boundary, boundary_eps};
    for (int64_t b = 0; b < B; ++b) {
        if (boundary) boundary[b] = 0;
        float Tf = T[b];
        if (!temperature_ok(Tf)) {
            finish_error(&J, b, ST_TEMPERATURE);
            continue;
        }
        if (Tf == 0.0f) {
            verify_greedy_row(&J, b);
            continue;
        }
        int K = top_k[b];
        float tp = top_p[b];
        if (K < 1 || K > 4096 || !(tp > 0.0f && tp <= 1.0f)) {
            finish_error(&J, b, ST_FILTER);
            continue;
        }
        int j = k, st = 0;
        double S = 0.0;
        for (int i = 0; i <= k; ++i) {
            const void *row = (const unsigned char *)logits + ((size_t)b * (k + 1) + i) * (size_t)V * esz;
            st = warp_row(dtype, row, V, (double)Tf, K, (double)tp, &kp, &S);
            if (i == k) break;
            int32_t xi = x[b * k + i];
            float ui = u[(b * (k + 1) + i) * 2];
            if (xi < 0 || xi >= V) st |= ST_TOKEN_RANGE;
            if (!uniform_ok(ui)) st |= ST_UNIFORM_RANGE;
            double qx = 0.0;
            if (xi >= 0 && xi < V) {
                qx = q ? (double)q[(b * k + i) * V + xi] : 1.0;
                if (!(qx >= 0.0 && qx <= (double)FLT_MAX)) st |= ST_Q_INVALID;
            }
            if (st) break;
            double px = 0.0;
            for (int r = 0; r < kp.n; ++r)
                if (kp.idx[r] == xi) px = kp.e[r] / S;
            double rho = px / (qx > 1e-12 ? qx : 1e-12);
            if (rho > 1.0) rho = 1.0;
            note_boundary(&J, b, i, 0, (double)ui, rho);
            if (!((double)ui < rho)) {
                j = i;
                break;
            }
        }
        float u1 = u[(b * (k + 1) + j) * 2 + 1];
        if (!st && !uniform_ok(u1)) st |= ST_UNIFORM_RANGE;
        if (st) {
            finish_error(&J, b, st);
            continue;
        }
        int status = 0;
        double lo = 0.0, hi = 1.0;
        int64_t token;
        for (int r = 0; r < kp.n; ++r) w[r] = kp.e[r] / S; /* p' on P */
        if (j < k) {
            double Wr = 0.0;
            const int32_t xj = x[b * k + j];
            for (int r = 0; r < kp.n; ++r) {
                double qv = q ? (double)q[(b * k + j) * V + kp.idx[r]] : (kp.idx[r] == xj ? 1.0 : 0.0);
                if (!(qv >= 0.0 && qv <= (double)FLT_MAX)) st |= ST_Q_INVALID;
                double r_ = kp.e[r] / S - qv;
                w[r] = r_ > 0.0 ? r_ : 0.0;
                Wr += w[r];
            }
            if (st) {
                finish_error(&J, b, st);
                continue;
            }
            if (!(Wr > 0.0)) {
                status |= ST_ZERO_RESIDUAL;
                for (int r = 0; r < kp.n; ++r) w[r] = kp.e[r] / S;
            }
        }
        token = kept_inverse_cdf(&kp, w, (double)u1, &lo, &hi);
        note_boundary(&J, b, j, 1, (double)u1, lo);
        note_boundary(&J, b, j, 1, (double)u1, hi);
        finish_ok(&J, b, j, token, status);
    }
    free(kp.val), free(kp.idx), free(kp.e), free(w);
    return 0;
}
