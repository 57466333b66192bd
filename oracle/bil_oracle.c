/*
 * Selected-token log-probability: the CPU oracle.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test-suite, the smoke check
 * and the benchmark's CPU-baseline leg load this library.  It shares no code,
 * header, table or constant with the CUDA library; the two meet only in the
 * seeded input bytes they are both given.
 *
 * Plain, slow and in float64 throughout.  Each function states the passage of
 * the pages it follows:
 *
 *  - "Batch-Invariant LogP" operator page, section "Reference Semantics":
 *      out[row] = log_softmax(float(logits[row, :]))[target[row]]
 *      ignored rows (target == ignore_index): out = 0, grad row = 0
 *      a non-ignored target outside [0, V) is invalid.
 *  - same page, section "Tensor Parallel", steps 1-6: per fixed vocab tile t a
 *    (max m_t, sum-exp s_t) partial; all tiles merged in one fixed order as
 *    LSE = M + log(sum_t s_t * exp(m_t - M)), M = max_t m_t; the target logit
 *    is copied from the tile that owns it; logp = target_logit - LSE.
 *  - same page, section "Batch-Invariance": the backward is computed per row
 *    tile from the saved per-row LSE:  d[c] = g * (onehot(target)[c] - p[c]),
 *    p[c] = exp(x[c] - LSE).
 *
 * The tile method is an exact rewrite of log-softmax in real arithmetic
 * ("RL-Kernel x vime x AMD: Achieving Bitwise Consistency Between Training
 * and Rollout", section "The Shared Normalization Structure of Attention and
 * Logprob": the merged result depends only on the set of all blocks), so the
 * forward and backward here compute the plain definition over the whole row;
 * the tile-partial and merge entry points exist so that the GPU's split mode
 * can be checked piece by piece.
 *
 *  - "[RFC][ROCm] End-to-end optimization of bitwise VIME R/R beyond native
 *    P/P", section "Workstream 3: fused ROCm LM-head and linear logp": an
 *    optional full-vocabulary entropy output, and a temperature applied to the
 *    logits at one fixed point.  Here z = x / temperature (float64 division),
 *    p = softmax(z), logp = z_t - LSE(z), entropy H = -sum_c p_c log p_c, and
 *    the backward of g * logp + g_H * H with respect to x is
 *      (1 / temperature) * (g * ([c == t] - p_c) - g_H * p_c * (z_c - LSE + H)).
 *    (dH/dz_c = -p_c (log p_c + H) follows from H = -sum_j p_j log p_j and
 *    dp_j/dz_c = p_j ([j == c] - p_c).)
 *
 * Readings taken where the pages are silent (each is listed with its reason in
 * the design notes):
 *  - ignored rows: lse = 0 and their logits are never read;
 *  - out-of-range target on an active row: logp = NaN and the row is counted
 *    as an error (the return value), nothing outside the row is read;
 *  - a row whose entries are all -inf: LSE = -inf, logp = NaN;
 *  - NaN anywhere in a row makes that row's LSE and logp NaN;
 *  - ignored rows have entropy 0 and a zero gradient whatever g_H is.
 *
 * Element types: 0 = float32, 1 = bfloat16, 2 = float16, 3 = float64 (the
 * exact products of the LM-head projection below).  Every input value is
 * widened to double exactly.
 *
 *  - same RFC, same section: the fused LM-head and linear logp.  The logits are
 *    the projection z[r, c] = sum_k hidden[r, k] * weight[c, k] of the row's
 *    hidden state onto the LM-head rows (weight stored [vocab, hidden], one row
 *    per token), and everything after that is the operator above applied to z.
 *    bil_oracle_linear_logits forms z in float64, summing k = 0, 1, ... in
 *    order; the products of two bf16/fp16 values are exact in double.
 *
 * Build: gcc -O2 -std=c11 -fopenmp -shared -fPIC (no -ffast-math: the order of
 * every sum below is the order written).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F16 2
#define ORACLE_F64 3

/* ---- exact widening of one stored element to double ---------------------- */

static double from_bf16_bits(uint16_t h) {
    /* bfloat16 is the upper half of an IEEE binary32 word. */
    uint32_t w = (uint32_t)h << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

static double from_f16_bits(uint16_t h) {
    /* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24); /* subnormal: frac * 2^-14 * 2^-10 */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(frac + 1024), expo - 25); /* 1.frac * 2^(expo-15) */
    }
    return sign ? -v : v;
}

/* One row of stored logits, as the softmax sees it: z_c = x_c / temperature. */
typedef struct {
    const void *base;
    int dtype;
    int64_t row, ld;
    double temperature;
} RowView;

static double load_raw(const void *base, int dtype, int64_t row, int64_t ld, int64_t col) {
    int64_t i = row * ld + col;
    if (dtype == ORACLE_BF16) {
        return from_bf16_bits(((const uint16_t *)base)[i]);
    }
    if (dtype == ORACLE_F16) {
        return from_f16_bits(((const uint16_t *)base)[i]);
    }
    if (dtype == ORACLE_F64) {
        return ((const double *)base)[i];
    }
    return (double)((const float *)base)[i];
}

static double z_at(const RowView *v, int64_t col) {
    double x = load_raw(v->base, v->dtype, v->row, v->ld, col);
#ifdef BIL_ORACLE_MUTANT_TEMPERATURE_MULTIPLIES
    return v->temperature == 1.0 ? x : x * v->temperature;
#else
    return v->temperature == 1.0 ? x : x / v->temperature;
#endif
}

/* ---- log-sum-exp over columns [c0, c1) of one row --------------------------
 * The definition log(sum_c exp(z_c)), evaluated with the usual shift by the
 * maximum so that nothing overflows.  Returns the maximum in *m_out, the
 * shifted sum sum_c exp(z_c - max) in *s_out and, when u_out is not NULL,
 * sum_c exp(z_c - max) * (z_c - max) in *u_out (what the entropy needs).  A
 * range whose entries are all -inf has max -inf and sums 0.  A NaN entry never
 * wins the max (comparisons with NaN are false) and makes the sums NaN. */
static void max_and_sumexp(const RowView *v, int64_t c0, int64_t c1, double *m_out, double *s_out,
                           double *u_out) {
    double m = -INFINITY;
    for (int64_t c = c0; c < c1; ++c) {
        double z = z_at(v, c);
        if (z > m) {
            m = z;
        }
    }
    double s = 0.0, u = 0.0;
    if (m != -INFINITY) {
        for (int64_t c = c0; c < c1; ++c) {
#ifdef BIL_ORACLE_MUTANT_SUM_SKIPS_FIRST
            if (c == c0) continue;
#endif
            double d = z_at(v, c) - m;
#ifdef BIL_ORACLE_MUTANT_NO_SHIFT_SIGN
            double e = exp(-d);
#else
            double e = exp(d);
#endif
            s += e;
            if (e != 0.0) { /* p log p -> 0 as p -> 0: an -inf logit adds nothing */
#ifdef BIL_ORACLE_MUTANT_PART_ENT_UNWEIGHTED
                u += d;
#else
                u += e * d;
#endif
            }
        }
    } else {
        /* every entry is -inf (or the range is empty of finite values);
         * a NaN entry still poisons the sums */
#ifndef BIL_ORACLE_MUTANT_NAN_NOT_PROPAGATED
        for (int64_t c = c0; c < c1; ++c) {
            if (isnan(z_at(v, c))) {
                s = NAN;
                u = NAN;
            }
        }
#endif
    }
    *m_out = m;
    *s_out = s;
    if (u_out != NULL) {
        *u_out = u;
    }
}

static double row_lse(const RowView *v, int64_t vocab) {
    double m, s;
    max_and_sumexp(v, 0, vocab, &m, &s, NULL);
    if (m == -INFINITY && s == 0.0) {
        return -INFINITY;
    }
#ifdef BIL_ORACLE_MUTANT_LSE_DROPS_MAX
    return log(s);
#else
    return m + log(s);
#endif
}

/* Entropy of the row's distribution by its definition, -sum_c p_c log p_c
 * with p_c = exp(z_c - L) and log p_c = z_c - L (L: the row's LSE). */
static double row_entropy(const RowView *v, int64_t vocab, double L) {
    double h = 0.0;
    for (int64_t c = 0; c < vocab; ++c) {
        double lp = z_at(v, c) - L;
        double p = exp(lp);
        if (p != 0.0) {
#ifdef BIL_ORACLE_MUTANT_ENTROPY_SIGN
            h += p * lp;
#else
            h -= p * lp;
#endif
        } else if (isnan(lp)) {
            h = NAN;
        }
    }
    return h;
}

/* ---- LM-head projection --------------------------------------------------------
 * "Workstream 3: fused ROCm LM-head and linear logp": the logits of row r are
 * z[r, c] = sum_{k=0}^{H-1} hidden[r, k] * weight[c, k], for the hidden state
 * hidden [n_rows, H] (row stride ld_h) and the LM-head weight [vocab, H] (row
 * stride ld_w), both of element type dtype.  z is written as float64 to
 * [n_rows, ld_z]; the sum runs over k in increasing order. */
void bil_oracle_linear_logits(const void *hidden, const void *weight, int dtype, int64_t n_rows,
                              int64_t hidden_size, int64_t ld_h, int64_t vocab, int64_t ld_w,
                              double *z, int64_t ld_z) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        for (int64_t c = 0; c < vocab; ++c) {
            double acc = 0.0;
#ifdef BIL_ORACLE_MUTANT_LINEAR_DROPS_LAST_K
            for (int64_t k = 0; k + 1 < hidden_size; ++k) {
#else
            for (int64_t k = 0; k < hidden_size; ++k) {
#endif
#ifdef BIL_ORACLE_MUTANT_LINEAR_TRANSPOSED
                /* weight read as [H, vocab] */
                double w = load_raw(weight, dtype, k % vocab, ld_w, c % hidden_size);
#else
                double w = load_raw(weight, dtype, c, ld_w, k);
#endif
                acc += load_raw(hidden, dtype, r, ld_h, k) * w;
            }
            z[r * ld_z + c] = acc;
        }
    }
}

int bil_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- forward -----------------------------------------------------------------
 * "Reference Semantics": logp[r] = z[r, t_r] - LSE(z[r, :]) for active rows,
 * 0 for ignored rows.  lse[r] receives the row's LSE (0 for ignored rows);
 * entropy[r] (when entropy is not NULL) the row's entropy (0 for ignored rows).
 * Returns the number of active rows whose target lies outside [0, vocab);
 * those rows get logp = NaN. */
int64_t bil_oracle_logp_fwd(const void *logits, int dtype, int64_t n_rows, int64_t vocab,
                            int64_t ld, const int64_t *target_ids, int64_t ignore_index,
                            double temperature, double *logp, double *lse, double *entropy) {
    int64_t bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (int64_t r = 0; r < n_rows; ++r) {
        RowView v = {logits, dtype, r, ld, temperature};
        int64_t t = target_ids[r];
#ifndef BIL_ORACLE_MUTANT_IGNORE_NOT_ZEROED
        if (t == ignore_index) {
            logp[r] = 0.0;
            lse[r] = 0.0;
            if (entropy != NULL) {
                entropy[r] = 0.0;
            }
            continue;
        }
#endif
        double L = row_lse(&v, vocab);
        lse[r] = L;
        if (entropy != NULL) {
            entropy[r] = row_entropy(&v, vocab, L);
        }
#ifdef BIL_ORACLE_MUTANT_RANGE_ALLOWS_VOCAB
        if (t < 0 || t > vocab) {
#else
        if (t < 0 || t >= vocab) {
#endif
            logp[r] = NAN;
            bad += 1;
            continue;
        }
#if defined(BIL_ORACLE_MUTANT_TARGET_OFF_BY_ONE)
        double zt = z_at(&v, t + 1 < vocab ? t + 1 : t);
#else
        double zt = z_at(&v, t);
#endif
#ifdef BIL_ORACLE_MUTANT_SIGN
        logp[r] = L - zt;
#else
        logp[r] = zt - L;
#endif
    }
    return bad;
}

/* ---- tile partials -------------------------------------------------------------
 * "Tensor Parallel", steps 1-2 and 5: the vocabulary is split into fixed tiles
 * of tile_v columns; tile t covers columns [t*tile_v, min((t+1)*tile_v, V)).
 * For every row and every tile t in [tile_begin, tile_end):
 *   part_max[r*ld_part + t] = max of the tile, part_sum[...] = sum exp(z - max),
 *   part_ent[...] (when not NULL) = sum exp(z - max) * (z - max).
 * The target logit z_t is copied (never summed) into target_logit[r] when the
 * row's target lies in one of these tiles.  Ignored rows get (-inf, 0, 0) and
 * their logits are not read.  Columns are global column indices of the full
 * row held in `logits`. */
void bil_oracle_tile_partials(const void *logits, int dtype, int64_t n_rows, int64_t vocab,
                              int64_t ld, int64_t tile_v, int64_t tile_begin,
                              int64_t tile_end, const int64_t *target_ids,
                              int64_t ignore_index, double temperature, double *part_max,
                              double *part_sum, double *part_ent, int64_t ld_part,
                              double *target_logit) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        RowView v = {logits, dtype, r, ld, temperature};
        int64_t t_id = target_ids[r];
        for (int64_t t = tile_begin; t < tile_end; ++t) {
            double m = -INFINITY, s = 0.0, u = 0.0;
            if (t_id != ignore_index) {
                int64_t c0 = t * tile_v;
#ifdef BIL_ORACLE_MUTANT_TILE_IGNORES_VOCAB
                int64_t c1 = c0 + tile_v;
#else
                int64_t c1 = c0 + tile_v < vocab ? c0 + tile_v : vocab;
#endif
                max_and_sumexp(&v, c0, c1, &m, &s, &u);
                if (t_id >= c0 && t_id < c1) {
#ifdef BIL_ORACLE_MUTANT_TARGET_LOGIT_UNSCALED
                    target_logit[r] = load_raw(v.base, v.dtype, v.row, v.ld, t_id);
#else
                    target_logit[r] = z_at(&v, t_id);
#endif
                }
            }
            part_max[r * ld_part + t] = m;
            part_sum[r * ld_part + t] = s;
            if (part_ent != NULL) {
                part_ent[r * ld_part + t] = u;
            }
        }
    }
}

/* ---- fixed-order merge -----------------------------------------------------------
 * "Tensor Parallel", steps 4 and 6:
 *   M = max_t m_t,  w_t = exp(m_t - M),  S = sum_{t=0..T-1} s_t w_t,
 *   LSE = M + log S,  logp = target_logit - LSE;  ignored rows give 0.
 * Entropy from the same partials (an exact rewrite of -sum_c p_c log p_c: with
 * d_c = z_c - m_t inside tile t, log p_c = d_c + (m_t - M) - log S):
 *   H = log S - (1/S) sum_t w_t (u_t + (m_t - M) s_t).
 * Returns the number of active rows whose target lies outside [0, vocab)
 * (their logp is NaN). */
int64_t bil_oracle_merge(const double *part_max, const double *part_sum, const double *part_ent,
                         int64_t n_rows, int64_t num_tiles, int64_t ld_part,
                         const double *target_logit, const int64_t *target_ids,
                         int64_t ignore_index, int64_t vocab, double *logp, double *lse,
                         double *entropy) {
    int64_t bad = 0;
#pragma omp parallel for schedule(static) reduction(+ : bad)
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t t_id = target_ids[r];
        if (t_id == ignore_index) {
            logp[r] = 0.0;
            lse[r] = 0.0;
            if (entropy != NULL) {
                entropy[r] = 0.0;
            }
            continue;
        }
        const double *m = part_max + r * ld_part;
        const double *s = part_sum + r * ld_part;
        double M = -INFINITY;
        for (int64_t t = 0; t < num_tiles; ++t) {
            if (m[t] > M) {
                M = m[t];
            }
        }
        double L, H = NAN;
        if (M == -INFINITY) {
            L = -INFINITY;
            for (int64_t t = 0; t < num_tiles; ++t) {
                if (isnan(s[t])) {
                    L = NAN;
                }
            }
        } else {
            double S = 0.0, U = 0.0;
            for (int64_t t = 0; t < num_tiles; ++t) {
#ifdef BIL_ORACLE_MUTANT_MERGE_TRANSPOSED
                double w = exp(M - m[t]);
#else
                double w = exp(m[t] - M);
#endif
                S += s[t] * w;
                if (part_ent != NULL && s[t] != 0.0) { /* an empty tile adds nothing */
#ifdef BIL_ORACLE_MUTANT_MERGE_ENTROPY_DROPS_SHIFT
                    U += w * part_ent[r * ld_part + t];
#else
                    U += w * (part_ent[r * ld_part + t] + (m[t] - M) * s[t]);
#endif
                }
            }
            L = M + log(S);
            H = log(S) - U / S;
        }
        lse[r] = L;
        if (entropy != NULL) {
            entropy[r] = H;
        }
        if (t_id < 0 || t_id >= vocab) {
            logp[r] = NAN;
            bad += 1;
        } else {
            logp[r] = target_logit[r] - L;
        }
    }
    return bad;
}

/* ---- backward --------------------------------------------------------------------
 * "Batch-Invariance" (the backward reuses the per-row LSE) and "Reference
 * Semantics" (ignored rows receive zero gradient):
 *   dlogits[r, c] = (1/T) * (g[r] * ([c == t_r] - p_c) - gH[r] * p_c * (z_c - LSE + H))
 * with p_c = exp(z_c - LSE), T the temperature; the second term only when
 * grad_entropy is not NULL.  LSE and H are the oracle's own float64 values,
 * recomputed here from the row.  Output is float64, row stride ld_out;
 * columns [vocab, out_cols) of every row are written as 0.  Returns the
 * number of active rows with an out-of-range target (their gradient row is
 * NaN). */
int64_t bil_oracle_logp_bwd(const void *logits, int dtype, int64_t n_rows, int64_t vocab,
                            int64_t ld, const int64_t *target_ids, int64_t ignore_index,
                            double temperature, const double *grad_logp,
                            const double *grad_entropy, double *dlogits, int64_t ld_out,
                            int64_t out_cols) {
    int64_t bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (int64_t r = 0; r < n_rows; ++r) {
        RowView v = {logits, dtype, r, ld, temperature};
        double *d = dlogits + r * ld_out;
        int64_t t_id = target_ids[r];
        for (int64_t c = vocab; c < out_cols; ++c) {
            d[c] = 0.0;
        }
        if (t_id == ignore_index) {
            for (int64_t c = 0; c < vocab; ++c) {
                d[c] = 0.0;
            }
            continue;
        }
        if (t_id < 0 || t_id >= vocab) {
            for (int64_t c = 0; c < vocab; ++c) {
                d[c] = NAN;
            }
            bad += 1;
            continue;
        }
        double L = row_lse(&v, vocab);
        double H = grad_entropy != NULL ? row_entropy(&v, vocab, L) : 0.0;
        double g = grad_logp[r];
        double gh = grad_entropy != NULL ? grad_entropy[r] : 0.0;
        for (int64_t c = 0; c < vocab; ++c) {
            double z = z_at(&v, c);
            double p = exp(z - L);
            double onehot = (c == t_id) ? 1.0 : 0.0;
#if defined(BIL_ORACLE_MUTANT_BWD_SIGN)
            double dz = g * (p - onehot);
#elif defined(BIL_ORACLE_MUTANT_BWD_NO_G)
            double dz = onehot - p;
#else
            double dz = g * (onehot - p);
#endif
            if (grad_entropy != NULL && p != 0.0) { /* p (log p + H) -> 0 as p -> 0 */
#ifdef BIL_ORACLE_MUTANT_BWD_ENTROPY_SIGN
                dz += gh * p * (z - L + H);
#else
                dz -= gh * p * (z - L + H);
#endif
            }
#ifdef BIL_ORACLE_MUTANT_BWD_TEMPERATURE_DROPPED
            d[c] = dz;
#else
            d[c] = temperature == 1.0 ? dz : dz / temperature;
#endif
        }
    }
    return bad;
}

/* ---- LM-head backward ----------------------------------------------------------
 * "Workstream 3: fused ROCm LM-head and linear logp", the autograd actor path:
 * the gradient of g * logp + g_H * H with respect to the hidden states and the
 * LM-head weight.  dZ = d(g logp + g_H H)/dz is bil_oracle_logp_bwd applied to
 * the float64 projection z = hidden . weight^T (bil_oracle_linear_logits), and
 * the chain rule through z gives
 *   dhidden[r, k] = sum_c dZ[r, c] * weight[c, k]    (c = 0, 1, ... in order)
 *   dweight[c, k] = sum_r dZ[r, c] * hidden[r, k]    (r = 0, 1, ... in order)
 * for dhidden [n_rows, hidden_size] and dweight [vocab, hidden_size] (both
 * row-major, float64).  dZ is also written to dz [n_rows, vocab] when dz is not
 * NULL.  Returns the number of active rows with an invalid target (their
 * dZ rows, and so every gradient, are NaN), or -1 if memory ran out. */
int64_t bil_oracle_linear_bwd(const void *hidden, const void *weight, int dtype, int64_t n_rows,
                              int64_t hidden_size, int64_t ld_h, int64_t vocab, int64_t ld_w,
                              const int64_t *target_ids, int64_t ignore_index, double temperature,
                              const double *grad_logp, const double *grad_entropy,
                              double *dhidden, double *dweight, double *dz) {
    double *z = malloc(sizeof(double) * (size_t)(n_rows * vocab > 0 ? n_rows * vocab : 1));
    double *d = dz != NULL ? dz : malloc(sizeof(double) * (size_t)(n_rows * vocab > 0 ? n_rows * vocab : 1));
    if (z == NULL || d == NULL) {
        free(z);
        if (dz == NULL) free(d);
        return -1;
    }
    bil_oracle_linear_logits(hidden, weight, dtype, n_rows, hidden_size, ld_h, vocab, ld_w, z, vocab);
    int64_t bad = bil_oracle_logp_bwd(z, ORACLE_F64, n_rows, vocab, vocab, target_ids, ignore_index,
                                      temperature, grad_logp, grad_entropy, d, vocab, vocab);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        for (int64_t k = 0; k < hidden_size; ++k) {
            double acc = 0.0;
            for (int64_t c = 0; c < vocab; ++c) {
#ifdef BIL_ORACLE_MUTANT_LINEAR_BWD_DX_TRANSPOSED
                acc += d[r * vocab + c] * load_raw(weight, dtype, k % vocab, ld_w, c % hidden_size);
#else
                acc += d[r * vocab + c] * load_raw(weight, dtype, c, ld_w, k);
#endif
            }
            dhidden[r * hidden_size + k] = acc;
        }
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t c = 0; c < vocab; ++c) {
        for (int64_t k = 0; k < hidden_size; ++k) {
            double acc = 0.0;
            for (int64_t r = 0; r < n_rows; ++r) {
#ifdef BIL_ORACLE_MUTANT_LINEAR_BWD_DW_ROW_SHIFT
                acc += d[r * vocab + c] * load_raw(hidden, dtype, (r + 1) % n_rows, ld_h, k);
#else
                acc += d[r * vocab + c] * load_raw(hidden, dtype, r, ld_h, k);
#endif
            }
            dweight[c * hidden_size + k] = acc;
        }
    }
    free(z);
    if (dz == NULL) free(d);
    return bad;
}

/* ---- element widening, exposed so that tests can pin it to library routines --- */
void bil_oracle_widen(const void *src, int dtype, int64_t count, double *dst) {
    for (int64_t i = 0; i < count; ++i) {
#ifdef BIL_ORACLE_MUTANT_BF16_WIDEN
        if (dtype == ORACLE_BF16) {
            uint32_t w = (uint32_t)((const uint16_t *)src)[i] << 15;
            float f;
            memcpy(&f, &w, sizeof f);
            dst[i] = f;
            continue;
        }
#endif
        dst[i] = load_raw(src, dtype, 0, 0, i);
    }
}
