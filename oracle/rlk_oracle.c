/*
 * rlk_oracle.c -- plain fp64 CPU oracle for the fused linear selected-token
 * log-prob, its backward, the masked dlogp audit and the GRPO clipped-ratio
 * upstream gradient.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * Every routine is the plain definition written out with explicit loops in
 * IEEE double, single-threaded, in ascending index order, with no blocking,
 * fusion or reordering.  Inputs that are bf16 on the GPU are handed in as
 * doubles holding the exact bf16 values (the conversion is exact), so every
 * product h*W below is exact and only the sums round (in fp64).
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared (no fast-math), so that the
 * compiler neither fuses multiply-adds nor reassociates sums.
 *
 * Sources (page title, section):
 *  - "RL-Kernel Roadmap (2026)", P0.2 "Typical Fused Operators": the fused
 *    linear log-prob that never lands [B,S,V] logits, with a tile-recompute
 *    backward.
 *  - "RL-Kernel integration roadmap for vime", Operator Integration Plan,
 *    "linear_logp / lm_head + logp": inputs (hidden states, target ids,
 *    active masks, LM-head weight, vocab size, rollout temperature), the
 *    max / sum-exp / selected-target-logit statistics, full-gradient
 *    backward from dlogits.
 *  - "RL-Kernel Roadmap (2026)", backlog: fused entropy, and chunked
 *    full-vocab / distillation KL fused with lm_head (forward and reverse KL
 *    over the whole distribution).
 *  - "RL-Kernel integration roadmap for vime", Consistency Contract: dlogp =
 *    recomputed - old; every metric over active tokens only; max_abs_dlogp
 *    is the primary metric; approx_kl0 = mean(exp(dlogp) - 1 - dlogp);
 *    active-token count; worst-token location.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - temperature divides the logits before the softmax: z = s / T;
 *  - inactive rows get logp = 0, lse = 0, dh = 0 and add nothing to dW;
 *  - an active row whose target lies outside [0, V) gets logp = NaN and is
 *    counted in the return value;
 *  - audit ties in max|d| go to the lowest token index; a NaN |d| ranks
 *    above every number; with no active token: count 0, max 0, index -1,
 *    mean = kl = NaN (0/0);
 *  - GRPO loss: L = -(1/Na) * sum_active min(r*A, clip(r, 1-eps, 1+eps)*A),
 *    r = exp(logp - old), a token-mean over the active tokens.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

/* s = sum_k a[k] * b[k], ascending k, one fp64 accumulator. */
static double dot(const double* a, const double* b, int64_t n) {
    double s = 0.0;
    for (int64_t k = 0; k < n; ++k) s += a[k] * b[k];
    return s;
}

static int row_active(const uint8_t* mask, int64_t t) {
    return mask == NULL || mask[t] != 0;
}

/*
 * Forward.  For every active row t:
 *   z[v]    = (h_t . W_v) / T                       for v in [0, V)
 *   M       = max_v z[v]
 *   LSE_t   = M + log( sum_v exp(z[v] - M) )
 *   logp_t  = z[y_t] - LSE_t
 * Inactive rows: logp = 0, lse = 0.  lse may be NULL.
 * Returns the number of active rows whose target is outside [0, V)
 * (their logp is NaN), or -1 if the scratch row cannot be allocated.
 */
int64_t rlk_oracle_linear_logp_fwd(const double* h, const double* w,
                                   const int64_t* y, const uint8_t* mask,
                                   int64_t n, int64_t hdim, int64_t vocab,
                                   double temperature,
                                   double* logp, double* lse) {
    double* z = (double*)malloc((size_t)(vocab > 0 ? vocab : 1) * sizeof(double));
    if (z == NULL) return -1;
    int64_t bad = 0;
    for (int64_t t = 0; t < n; ++t) {
        if (!row_active(mask, t)) {
            logp[t] = 0.0;
            if (lse) lse[t] = 0.0;
            continue;
        }
        const double* ht = h + t * hdim;
        for (int64_t v = 0; v < vocab; ++v) z[v] = dot(ht, w + v * hdim, hdim) / temperature;
        double m = -INFINITY;
        for (int64_t v = 0; v < vocab; ++v) if (z[v] > m) m = z[v];
        double sum = 0.0;
        for (int64_t v = 0; v < vocab; ++v) sum += exp(z[v] - m);
        double l = m + log(sum);
        if (lse) lse[t] = l;
        if (y[t] < 0 || y[t] >= vocab) {
            logp[t] = NAN;
            ++bad;
        } else {
            logp[t] = z[y[t]] - l;
        }
    }
    free(z);
    return bad;
}

/*
 * Backward, rows [row_begin, row_end) of dL/dh for L = sum_t g_t * logp_t.
 * With p[v] = exp(z[v] - LSE_t) (LSE_t from the forward above) and
 *   G[t][v] = g_t * (delta(v, y_t) - p[v]) / T,
 *   dh_t    = sum_v G[t][v] * W_v               (ascending v)
 * Inactive rows and rows with an invalid target get dh_t = 0.
 * dh points at the first output row (row_begin), row-major [.., H].
 */
void rlk_oracle_linear_logp_bwd_dh(const double* h, const double* w,
                                   const int64_t* y, const uint8_t* mask,
                                   const double* g, const double* lse,
                                   int64_t n, int64_t hdim, int64_t vocab,
                                   double temperature,
                                   int64_t row_begin, int64_t row_end,
                                   double* dh) {
    (void)n;
    for (int64_t t = row_begin; t < row_end; ++t) {
        double* out = dh + (t - row_begin) * hdim;
        for (int64_t k = 0; k < hdim; ++k) out[k] = 0.0;
        if (!row_active(mask, t) || y[t] < 0 || y[t] >= vocab) continue;
        const double* ht = h + t * hdim;
        for (int64_t v = 0; v < vocab; ++v) {
            double z = dot(ht, w + v * hdim, hdim) / temperature;
            double p = exp(z - lse[t]);
            double delta = (v == y[t]) ? 1.0 : 0.0;
            double G = g[t] * (delta - p) / temperature;
            const double* wv = w + v * hdim;
            for (int64_t k = 0; k < hdim; ++k) out[k] += G * wv[k];
        }
    }
}

/*
 * Backward, rows [v_begin, v_end) of dL/dW:
 *   dW_v = sum_t G[t][v] * h_t                  (ascending t, active rows)
 * with G as above.  dw points at the first output row (v_begin).
 */
void rlk_oracle_linear_logp_bwd_dw(const double* h, const double* w,
                                   const int64_t* y, const uint8_t* mask,
                                   const double* g, const double* lse,
                                   int64_t n, int64_t hdim, int64_t vocab,
                                   double temperature,
                                   int64_t v_begin, int64_t v_end,
                                   double* dw) {
    for (int64_t v = v_begin; v < v_end; ++v) {
        double* out = dw + (v - v_begin) * hdim;
        for (int64_t k = 0; k < hdim; ++k) out[k] = 0.0;
        const double* wv = w + v * hdim;
        for (int64_t t = 0; t < n; ++t) {
            if (!row_active(mask, t) || y[t] < 0 || y[t] >= vocab) continue;
            const double* ht = h + t * hdim;
            double z = dot(ht, wv, hdim) / temperature;
            double p = exp(z - lse[t]);
            double delta = (v == y[t]) ? 1.0 : 0.0;
            double G = g[t] * (delta - p) / temperature;
            for (int64_t k = 0; k < hdim; ++k) out[k] += G * ht[k];
        }
    }
}

typedef struct {
    int64_t active_count;
    int64_t argmax_index;
    double max_abs_dlogp;
    double mean_dlogp;
    double approx_kl;
} rlk_oracle_audit_t;

/*
 * Masked dlogp audit over active tokens, ascending t:
 *   d_t       = logp_new[t] - logp_old[t]         (exact in double)
 *   count     = #active
 *   max|d|    and the first index attaining it (NaN ranks highest), ranked on
 *             the fp32 difference of the two fp32 logps (one IEEE subtraction,
 *             i.e. d_t rounded once to float): the worst token is an index
 *             decided by floating point, so it is decided in the precision of
 *             the logps themselves; two tokens whose exact |d| differ below
 *             fp32 resolution tie, and the first wins
 *   mean      = sum d / count
 *   approx_kl = sum (exp(d) - 1 - d) / count, evaluated as expm1(d) - d
 */
void rlk_oracle_dlogp_audit(const float* logp_new, const float* logp_old,
                            const uint8_t* mask, int64_t n,
                            rlk_oracle_audit_t* out) {
    int64_t count = 0, arg = -1;
    double best = 0.0, sum_d = 0.0, sum_kl = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        if (!row_active(mask, t)) continue;
        double d = (double)logp_new[t] - (double)logp_old[t];
        const float d32 = logp_new[t] - logp_old[t];   /* float operands: an fp32 subtraction */
        double a = fabs((double)d32);
        if (arg < 0) {
            best = a;
            arg = t;
        } else if (isnan(a) ? !isnan(best) : (!isnan(best) && a > best)) {
            best = a;
            arg = t;
        }
        ++count;
        sum_d += d;
        sum_kl += expm1(d) - d;
    }
    out->active_count = count;
    out->argmax_index = arg;
    out->max_abs_dlogp = count ? best : 0.0;
    out->mean_dlogp = sum_d / (double)count;
    out->approx_kl = sum_kl / (double)count;
}

/*
 * GRPO / PPO clipped-ratio objective and its per-token gradient.
 *   r_t   = exp(logp_t - old_t)
 *   L     = -(1/Na) * sum_active min(r_t * A_t, clip(r_t, 1-eps, 1+eps) * A_t)
 *   g_t   = dL/dlogp_t = -(A_t * r_t) / Na  where the unclipped term is the
 *           one selected by the min (always when r_t lies inside the clip
 *           interval), 0 where the clipped constant is selected, 0 on
 *           inactive tokens.
 * Returns L (NaN when no token is active).
 */
double rlk_oracle_grpo_clip_grad(const double* logp, const double* old,
                                 const double* adv, const uint8_t* mask,
                                 int64_t n, double eps, double* g) {
    int64_t na = 0;
    for (int64_t t = 0; t < n; ++t) na += row_active(mask, t) ? 1 : 0;
    double total = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        g[t] = 0.0;
        if (!row_active(mask, t)) continue;
        double r = exp(logp[t] - old[t]);
        double rc = r < 1.0 - eps ? 1.0 - eps : (r > 1.0 + eps ? 1.0 + eps : r);
        double unclipped = r * adv[t];
        double clipped = rc * adv[t];
        int take_unclipped = (unclipped <= clipped);
        total += take_unclipped ? unclipped : clipped;
        if (take_unclipped) g[t] = -(adv[t] * r) / (double)na;
    }
    return -total / (double)na;
}

typedef struct {
    int64_t active_count;
    int64_t clipped_count;
    int64_t outside_count;
    double loss;
    double mean_ratio;
} rlk_oracle_grpo_t;

/*
 * Clipped-ratio policy-gradient fragment with explicit clip range and
 * aggregation scale ("RL-Kernel integration roadmap for vime", RL Loss
 * Operators: the caller owns aggregation and clipping range; "RL-Kernel
 * Roadmap (2026)", backlog: fused PPO clip loss, ratio-clip-aggregate
 * primitive).  For active t, with r_t = exp(logp_t - old_t):
 *   term_t  = min(r_t A_t, clip(r_t, 1 - eps_low, 1 + eps_high) A_t)
 *   L       = -scale * sum_active term_t
 *   g_t     = -scale * A_t * r_t   where the unclipped product is the one the
 *             min selects (always inside the clip range), else 0; 0 inactive
 *   clipped = #active with the clipped constant selected and r_t outside the
 *             range (zero gradient); outside = #active with r_t outside the range
 *   mean_ratio = sum_active r_t / #active
 * With eps_low = eps_high = eps and scale = 1/#active this is
 * rlk_oracle_grpo_clip_grad.
 */
void rlk_oracle_grpo_clip(const double* logp, const double* old, const double* adv,
                          const uint8_t* mask, int64_t n, double eps_low, double eps_high,
                          double scale, double* g, rlk_oracle_grpo_t* out) {
    int64_t na = 0, clipped = 0, outside = 0;
    double total = 0.0, rsum = 0.0;
    const double lo = 1.0 - eps_low, hi = 1.0 + eps_high;
    for (int64_t t = 0; t < n; ++t) {
        g[t] = 0.0;
        if (!row_active(mask, t)) continue;
        double r = exp(logp[t] - old[t]);
        double rc = r < lo ? lo : (r > hi ? hi : r);
        double unclipped = r * adv[t];
        double clippedv = rc * adv[t];
        int take_unclipped = (unclipped <= clippedv);
        int out_of_range = (r < lo || r > hi);
        ++na;
        rsum += r;
        total += take_unclipped ? unclipped : clippedv;
        if (take_unclipped) g[t] = -scale * adv[t] * r;
        if (out_of_range) ++outside;
        if (!take_unclipped && out_of_range) ++clipped;
    }
    out->active_count = na;
    out->clipped_count = clipped;
    out->outside_count = outside;
    out->loss = -scale * total;
    out->mean_ratio = rsum / (double)na;
}

/*
 * Selected-token logp from given logits ("RL-Kernel integration roadmap for
 * vime", logp Reference Scoring: log-softmax over existing logits, the same
 * active mask and temperature as linear_logp, dense or indexed rows).
 * Output row i scores logits row r_i = rows[i] (or i when rows is NULL):
 *   z[v]   = logits[r_i][v] / T
 *   lse_i  = M + log( sum_v exp(z[v] - M) ),  M = max_v z[v]
 *   logp_i = z[y[r_i]] - lse_i   when row r_i is active, else logp_i = lse_i = 0
 * logits is [N][stride] (row stride in elements); targets and mask are indexed
 * by logits row.  Returns the number of active rows with a target outside
 * [0, V) (their logp is NaN).
 */
int64_t rlk_oracle_logp_from_logits(const double* logits, int64_t stride, int64_t vocab,
                                    const int64_t* rows, int64_t m, const int64_t* y,
                                    const uint8_t* mask, double temperature,
                                    double* logp, double* lse) {
    int64_t bad = 0;
    for (int64_t i = 0; i < m; ++i) {
        const int64_t r = rows ? rows[i] : i;
        if (!row_active(mask, r)) {
            logp[i] = 0.0;
            if (lse) lse[i] = 0.0;
            continue;
        }
        const double* z = logits + r * stride;
        double mx = -INFINITY;
        for (int64_t v = 0; v < vocab; ++v) if (z[v] / temperature > mx) mx = z[v] / temperature;
        double sum = 0.0;
        for (int64_t v = 0; v < vocab; ++v) sum += exp(z[v] / temperature - mx);
        const double l = mx + log(sum);
        if (lse) lse[i] = l;
        if (y[r] < 0 || y[r] >= vocab) {
            logp[i] = NAN;
            ++bad;
        } else {
            logp[i] = z[y[r]] / temperature - l;
        }
    }
    return bad;
}

/*
 * Entropy of the temperature-scaled softmax, next to logp ("RL-Kernel
 * Roadmap (2026)", backlog: fused entropy / entropy-bonus kernel; "RL-Kernel
 * integration roadmap for vime", linear_logp: entropy requests).  For every
 * active row, with z[v] = (h_t . W_v) / T and log p[v] = z[v] - LSE_t:
 *   entropy_t = - sum_v p[v] * log p[v]
 * logp and lse as in rlk_oracle_linear_logp_fwd; inactive rows give 0.
 */
int64_t rlk_oracle_linear_logp_entropy_fwd(const double* h, const double* w,
                                           const int64_t* y, const uint8_t* mask,
                                           int64_t n, int64_t hdim, int64_t vocab,
                                           double temperature, double* logp, double* lse,
                                           double* entropy) {
    double* z = (double*)malloc((size_t)(vocab > 0 ? vocab : 1) * sizeof(double));
    if (z == NULL) return -1;
    int64_t bad = 0;
    for (int64_t t = 0; t < n; ++t) {
        if (!row_active(mask, t)) {
            logp[t] = 0.0;
            lse[t] = 0.0;
            entropy[t] = 0.0;
            continue;
        }
        const double* ht = h + t * hdim;
        for (int64_t v = 0; v < vocab; ++v) z[v] = dot(ht, w + v * hdim, hdim) / temperature;
        double m = -INFINITY;
        for (int64_t v = 0; v < vocab; ++v) if (z[v] > m) m = z[v];
        double sum = 0.0;
        for (int64_t v = 0; v < vocab; ++v) sum += exp(z[v] - m);
        double l = m + log(sum);
        lse[t] = l;
        double ent = 0.0;
        for (int64_t v = 0; v < vocab; ++v) {
            double lp = z[v] - l;
            ent -= exp(lp) * lp;
        }
        entropy[t] = ent;
        if (y[t] < 0 || y[t] >= vocab) {
            logp[t] = NAN;
            ++bad;
        } else {
            logp[t] = z[y[t]] - l;
        }
    }
    free(z);
    return bad;
}

/*
 * Backward of L = sum_t g_t logp_t + sum_t gH_t entropy_t.  With
 * log p[v] = z[v] - LSE_t and the forward's entropy_t:
 *   dlogp_t/dz_v    = delta(v, y_t) - p[v]
 *   dentropy_t/dz_v = -p[v] * (log p[v] + entropy_t)
 *   G[t][v] = ( g_t (delta - p[v]) - gH_t p[v] (log p[v] + entropy_t) ) / T
 * dh rows [row_begin, row_end) and dW rows [v_begin, v_end) as in the logp-only
 * backward (ascending v for dh, ascending t for dW).
 */
static double entropy_coef(double g, double gh, double delta, double lp, double ent,
                           double temperature) {
    double p = exp(lp);
    return (g * (delta - p) - gh * p * (lp + ent)) / temperature;
}

void rlk_oracle_linear_logp_entropy_bwd_dh(const double* h, const double* w,
                                           const int64_t* y, const uint8_t* mask,
                                           const double* g, const double* gh,
                                           const double* lse, const double* ent,
                                           int64_t n, int64_t hdim, int64_t vocab,
                                           double temperature, int64_t row_begin,
                                           int64_t row_end, double* dh) {
    (void)n;
    for (int64_t t = row_begin; t < row_end; ++t) {
        double* out = dh + (t - row_begin) * hdim;
        for (int64_t k = 0; k < hdim; ++k) out[k] = 0.0;
        if (!row_active(mask, t) || y[t] < 0 || y[t] >= vocab) continue;
        const double* ht = h + t * hdim;
        for (int64_t v = 0; v < vocab; ++v) {
            double lp = dot(ht, w + v * hdim, hdim) / temperature - lse[t];
            double G = entropy_coef(g[t], gh[t], v == y[t] ? 1.0 : 0.0, lp, ent[t], temperature);
            const double* wv = w + v * hdim;
            for (int64_t k = 0; k < hdim; ++k) out[k] += G * wv[k];
        }
    }
}

void rlk_oracle_linear_logp_entropy_bwd_dw(const double* h, const double* w,
                                           const int64_t* y, const uint8_t* mask,
                                           const double* g, const double* gh,
                                           const double* lse, const double* ent,
                                           int64_t n, int64_t hdim, int64_t vocab,
                                           double temperature, int64_t v_begin,
                                           int64_t v_end, double* dw) {
    for (int64_t v = v_begin; v < v_end; ++v) {
        double* out = dw + (v - v_begin) * hdim;
        for (int64_t k = 0; k < hdim; ++k) out[k] = 0.0;
        const double* wv = w + v * hdim;
        for (int64_t t = 0; t < n; ++t) {
            if (!row_active(mask, t) || y[t] < 0 || y[t] >= vocab) continue;
            const double* ht = h + t * hdim;
            double lp = dot(ht, wv, hdim) / temperature - lse[t];
            double G = entropy_coef(g[t], gh[t], v == y[t] ? 1.0 : 0.0, lp, ent[t], temperature);
            for (int64_t k = 0; k < hdim; ++k) out[k] += G * ht[k];
        }
    }
}

typedef struct {
    int64_t active_count;
    int64_t argmax_index;
    int64_t argmax_seq;
    int64_t argmax_pos;
    int64_t clip_count;
    double mean_dlogp;
    double mean_abs_dlogp;
    double mean_ratio;
    double approx_kl;
    double max_abs_dlogp;
    double p50_abs_dlogp;
    double p90_abs_dlogp;
    double p99_abs_dlogp;
    double clipfrac;
} rlk_oracle_audit_ext_t;

static int cmp_abs(const void* a, const void* b) {
    double x = *(const double*)a, y = *(const double*)b;
    int nx = isnan(x), ny = isnan(y);
    if (nx || ny) return nx - ny;          /* NaN sorts above every number */
    return (x > y) - (x < y);
}

/* nearest rank: the value at 1-based rank ceil(p * count) of the ascending order */
static double nearest_rank(const double* sorted, int64_t count, int64_t num, int64_t den) {
    if (count == 0) return NAN;
    int64_t rank = (num * count + den - 1) / den;
    if (rank < 1) rank = 1;
    return sorted[rank - 1];
}

/*
 * The Consistency Contract's minimum diagnostics ("RL-Kernel integration
 * roadmap for vime"): over active tokens, with d = new - old,
 *   mean d, mean |d|, max |d| (first index), p50 / p90 / p99 of |d| (nearest
 *   rank), mean ratio0 = mean exp(d), approx_kl0 = mean(exp(d) - 1 - d),
 *   clip count = #{|exp(d) - 1| > eps} and clipfrac0 = clip count / count,
 *   and the worst token's sequence and position, from seq_offsets[0..num_seqs]
 *   (sequence s holds tokens [seq_offsets[s], seq_offsets[s+1])) when given.
 * Ties and NaN as in rlk_oracle_dlogp_audit.  Returns -1 if the scratch array
 * cannot be allocated.
 */
int rlk_oracle_dlogp_audit_ext(const float* logp_new, const float* logp_old, const uint8_t* mask,
                               int64_t n, const int64_t* seq_offsets, int64_t num_seqs,
                               double eps, rlk_oracle_audit_ext_t* out) {
    double* absd = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    if (absd == NULL) return -1;
    rlk_oracle_audit_t base;
    rlk_oracle_dlogp_audit(logp_new, logp_old, mask, n, &base);
    int64_t count = 0, clip = 0;
    double sum_abs = 0.0, sum_ratio = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        if (!row_active(mask, t)) continue;
        double d = (double)logp_new[t] - (double)logp_old[t];
        double r = exp(d);
        absd[count++] = fabs(d);
        sum_abs += fabs(d);
        sum_ratio += r;
        if (fabs(r - 1.0) > eps) ++clip;
    }
    qsort(absd, (size_t)count, sizeof(double), cmp_abs);
    out->active_count = count;
    out->argmax_index = base.argmax_index;
    out->argmax_seq = -1;
    out->argmax_pos = -1;
    if (seq_offsets != NULL && base.argmax_index >= 0) {
        for (int64_t s = 0; s < num_seqs; ++s) {
            if (base.argmax_index >= seq_offsets[s] && base.argmax_index < seq_offsets[s + 1]) {
                out->argmax_seq = s;
                out->argmax_pos = base.argmax_index - seq_offsets[s];
                break;
            }
        }
    }
    out->clip_count = clip;
    out->mean_dlogp = base.mean_dlogp;
    out->mean_abs_dlogp = sum_abs / (double)count;
    out->mean_ratio = sum_ratio / (double)count;
    out->approx_kl = base.approx_kl;
    out->max_abs_dlogp = base.max_abs_dlogp;
    out->p50_abs_dlogp = nearest_rank(absd, count, 50, 100);
    out->p90_abs_dlogp = nearest_rank(absd, count, 90, 100);
    out->p99_abs_dlogp = nearest_rank(absd, count, 99, 100);
    out->clipfrac = (double)clip / (double)count;
    free(absd);
    return 0;
}

/*
 * Full-vocabulary KL between the policy head and a reference head ("RL-Kernel
 * Roadmap (2026)", backlog: chunked full-vocab KL / distillation KL fused with
 * lm_head, forward and reverse KL beyond the sampled token).  For every
 * active row t, with the policy logits z[v] = (h_t . W_v) / T and the
 * reference logits r[v] = (hr_t . Wr_v) / Tr over the same vocabulary:
 *   log p[v] = z[v] - LSE(z),  log q[v] = r[v] - LSE(r)
 *   kl_t     = sum_v p[v] (log p[v] - log q[v])         KL(p || q)
 *   kl_rev_t = sum_v q[v] (log q[v] - log p[v])         KL(q || p)
 * Inactive rows: every output 0.  The reference hidden size may differ.
 */
static double logsumexp(const double* z, int64_t vocab) {
    double m = -INFINITY;
    for (int64_t v = 0; v < vocab; ++v) if (z[v] > m) m = z[v];
    double sum = 0.0;
    for (int64_t v = 0; v < vocab; ++v) sum += exp(z[v] - m);
    return m + log(sum);
}

int64_t rlk_oracle_linear_kl_fwd(const double* h, const double* w, const double* hr,
                                 const double* wr, const uint8_t* mask, int64_t n, int64_t hdim,
                                 int64_t hrdim, int64_t vocab, double temperature,
                                 double temperature_ref, double* kl, double* kl_rev, double* lse,
                                 double* lse_ref) {
    double* z = (double*)malloc((size_t)(vocab > 0 ? vocab : 1) * sizeof(double));
    double* r = (double*)malloc((size_t)(vocab > 0 ? vocab : 1) * sizeof(double));
    if (z == NULL || r == NULL) {
        free(z);
        free(r);
        return -1;
    }
    for (int64_t t = 0; t < n; ++t) {
        if (!row_active(mask, t)) {
            kl[t] = kl_rev[t] = lse[t] = lse_ref[t] = 0.0;
            continue;
        }
        for (int64_t v = 0; v < vocab; ++v) {
            z[v] = dot(h + t * hdim, w + v * hdim, hdim) / temperature;
            r[v] = dot(hr + t * hrdim, wr + v * hrdim, hrdim) / temperature_ref;
        }
        const double lz = logsumexp(z, vocab), lr = logsumexp(r, vocab);
        double f = 0.0, b = 0.0;
        for (int64_t v = 0; v < vocab; ++v) {
            const double lp = z[v] - lz, lq = r[v] - lr;
            f += exp(lp) * (lp - lq);
            b += exp(lq) * (lq - lp);
        }
        kl[t] = f;
        kl_rev[t] = b;
        lse[t] = lz;
        lse_ref[t] = lr;
    }
    free(z);
    free(r);
    return 0;
}

/*
 * Backward of L = sum_t (g_t kl_t + gr_t kl_rev_t) with respect to the policy
 * head only (the reference is fixed).  With l[v] = log p[v] - log q[v]:
 *   dkl_t/dz_v     = p[v] (l[v] - kl_t)
 *   dkl_rev_t/dz_v = p[v] - q[v]
 *   G[t][v] = ( g_t p[v] (l[v] - kl_t) + gr_t (p[v] - q[v]) ) / T
 *   dh_t = sum_v G[t][v] W_v (ascending v),  dW_v = sum_t G[t][v] h_t
 * (ascending t).  lse, lse_ref and kl are the forward's outputs.
 */
static double kl_coef(const double* h, const double* w, const double* hr, const double* wr,
                      int64_t t, int64_t v, int64_t hdim, int64_t hrdim, double temperature,
                      double temperature_ref, double g, double gr, double lse, double lse_ref,
                      double kl) {
    const double lp = dot(h + t * hdim, w + v * hdim, hdim) / temperature - lse;
    const double lq = dot(hr + t * hrdim, wr + v * hrdim, hrdim) / temperature_ref - lse_ref;
    const double p = exp(lp), q = exp(lq);
    return (g * p * ((lp - lq) - kl) + gr * (p - q)) / temperature;
}

void rlk_oracle_linear_kl_bwd_dh(const double* h, const double* w, const double* hr,
                                 const double* wr, const uint8_t* mask, const double* g,
                                 const double* gr, const double* lse, const double* lse_ref,
                                 const double* kl, int64_t n, int64_t hdim, int64_t hrdim,
                                 int64_t vocab, double temperature, double temperature_ref,
                                 int64_t row_begin, int64_t row_end, double* dh) {
    (void)n;
    for (int64_t t = row_begin; t < row_end; ++t) {
        double* out = dh + (t - row_begin) * hdim;
        for (int64_t k = 0; k < hdim; ++k) out[k] = 0.0;
        if (!row_active(mask, t)) continue;
        for (int64_t v = 0; v < vocab; ++v) {
            const double G = kl_coef(h, w, hr, wr, t, v, hdim, hrdim, temperature,
                                     temperature_ref, g[t], gr[t], lse[t], lse_ref[t], kl[t]);
            const double* wv = w + v * hdim;
            for (int64_t k = 0; k < hdim; ++k) out[k] += G * wv[k];
        }
    }
}

void rlk_oracle_linear_kl_bwd_dw(const double* h, const double* w, const double* hr,
                                 const double* wr, const uint8_t* mask, const double* g,
                                 const double* gr, const double* lse, const double* lse_ref,
                                 const double* kl, int64_t n, int64_t hdim, int64_t hrdim,
                                 int64_t vocab, double temperature, double temperature_ref,
                                 int64_t v_begin, int64_t v_end, double* dw) {
    (void)vocab;
    for (int64_t v = v_begin; v < v_end; ++v) {
        double* out = dw + (v - v_begin) * hdim;
        for (int64_t k = 0; k < hdim; ++k) out[k] = 0.0;
        for (int64_t t = 0; t < n; ++t) {
            if (!row_active(mask, t)) continue;
            const double G = kl_coef(h, w, hr, wr, t, v, hdim, hrdim, temperature,
                                     temperature_ref, g[t], gr[t], lse[t], lse_ref[t], kl[t]);
            const double* ht = h + t * hdim;
            for (int64_t k = 0; k < hdim; ++k) out[k] += G * ht[k];
        }
    }
}
