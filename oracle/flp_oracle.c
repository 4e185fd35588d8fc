/*
 * flp_oracle.c - plain, slow, fp64 CPU reference for the fused linear
 * log-prob / cross-entropy LM head.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this library.  It shares no code, header, table or
 * helper with the CUDA path, and the CUDA path never calls it.
 *
 * What it computes is the plain definition of the method, with every logit
 * materialised in fp64:
 *
 *   z_ij       = s * sum_k X_ik W_jk                      (scaled classifier GEMM)
 *   LSE_i      = log sum_j exp(z_ij)
 *   p_ij       = exp(z_ij - LSE_i)
 *   logprob_i  = z_{i,y_i} - LSE_i
 *   entropy_i  = LSE_i - sum_j p_ij z_ij
 *   dZ_ij      = s * [ g_lp_i (1[j = y_i] - p_ij) + g_ent_i p_ij (sum_k p_ik z_ik - z_ij) ]
 *   dX         = dZ W,     dW = dZ^T X
 *
 * Sources (the pages are web text; each function below names the passage it
 * follows):
 *  - "Triton MoE improvements and chunked GRPO improvements" (Liger-Kernel
 *    pull request 1294), section "Chunked Triton GRPO loss": the lm_head
 *    projection fused into the loss with an online logsumexp, so the logits
 *    are never stored; "Kernel design notes": the backward recomputes the
 *    logits tiles into grad_logits, then grad_hidden = grad_logits . W and
 *    grad_weight += grad_logits^T . hidden.
 *  - Liger-Kernel v0.8.3 test/transformers page (the native SM100 fused scaled
 *    linear cross-entropy commit), section "Summary": classifier GEMM fused
 *    with NLL/LSE and optional entropy; "Correctness": ignored targets.
 *  - "perf(megatron): autotune fused LM-head Triton kernels" (SkyRL pull
 *    request 2141), sections "Summary" and "Overview": optional entropy,
 *    log-sum-exp started from the true row maximum (-inf initialisation).
 *
 * Readings taken where the pages are silent (each is also listed in the
 * design notes of the repository):
 *  - the scale s multiplies the fp32/fp64 accumulator, so every output is over
 *    the scaled logits and the gradients carry the factor s;
 *  - a row whose target equals ignore_index has logprob = 0, entropy = 0 and a
 *    zero dZ row; its LSE is still reported;
 *  - a target outside [0, V) that is not ignore_index is a contract violation:
 *    logprob is NaN for that row and the call returns FLPO_BAD_TARGET;
 *  - grad_logprob is the upstream gradient of logprob (not of the NLL), so
 *    dZ carries g_lp * (onehot - p);
 *  - with compute_entropy = 0 no entropy is produced and g_ent is ignored.
 *
 * No blocking, fusion or reordering beyond the definitions: each row's logits
 * are formed in full, the max shift is the textbook one, and the GEMMs are
 * plain triple loops.  OpenMP only splits independent rows (or, for dW,
 * independent vocabulary rows).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define FLPO_OK 0
#define FLPO_BAD_TARGET 5
#define FLPO_INVALID_ARG 1
#define FLPO_NO_MEMORY 7

/* Element type of an input matrix. */
#define FLPO_BF16 1
#define FLPO_F64 2

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t h) {
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round a binary32 to bf16, round-to-nearest-even (NaN kept quiet). */
static uint16_t float_to_bf16_rne(float f) {
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    if ((bits & 0x7f800000u) == 0x7f800000u && (bits & 0x007fffffu) != 0)
        return (uint16_t)((bits >> 16) | 0x0040u);
    uint32_t lsb = (bits >> 16) & 1u;
    bits += 0x7fffu + lsb;
    return (uint16_t)(bits >> 16);
}

static double get_elem(const void* base, int type, int64_t idx) {
    if (type == FLPO_BF16) return bf16_to_double(((const uint16_t*)base)[idx]);
    return ((const double*)base)[idx];
}

/* z_j = s * <X_i, W_j> for every j in [0, V): the full, materialised logit row. */
static void logits_row(const void* X, const void* W, int type, int64_t i, int64_t H,
                       int64_t V, double s, double* xrow, double* z) {
    for (int64_t k = 0; k < H; ++k) xrow[k] = get_elem(X, type, i * H + k);
    for (int64_t j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int64_t k = 0; k < H; ++k) acc += xrow[k] * get_elem(W, type, j * H + k);
        z[j] = s * acc;
    }
}

/* Per-row statistics from the materialised row, by definition.
 * The max shift starts from the true row maximum, as the SkyRL page's
 * "Correctness" section prescribes for strongly negative rows. */
typedef struct {
    double lse;
    double sum_pz; /* sum_j p_j z_j */
} row_stats;

static row_stats stats_from_logits(const double* z, int64_t V) {
    double m = -INFINITY;
    for (int64_t j = 0; j < V; ++j)
        if (z[j] > m) m = z[j];
    double se = 0.0;
    for (int64_t j = 0; j < V; ++j) se += exp(z[j] - m);
    row_stats r;
    r.lse = m + log(se);
    double spz = 0.0;
    for (int64_t j = 0; j < V; ++j) spz += exp(z[j] - r.lse) * z[j];
    r.sum_pz = spz;
    return r;
}

static int target_ok(int64_t y, int64_t V) { return y >= 0 && y < V; }

/* logprob and entropy of one row from its logits and statistics; ignored rows
 * give 0 and 0, an out-of-range target NaN (returns 0 then, else 1). */
static int row_outputs(const double* z, row_stats st, int64_t y, int64_t ignore_index, int64_t V,
                       double* lp, double* ent) {
    *ent = st.lse - st.sum_pz;
    if (y == ignore_index) {
        *lp = 0.0;
        *ent = 0.0;
        return 1;
    }
    if (!target_ok(y, V)) {
        *lp = NAN;
        return 0;
    }
    *lp = z[y] - st.lse;
    return 1;
}

/*
 * Forward outputs for the rows listed in `rows` (all rows when rows == NULL).
 * Output k belongs to row rows[k].  entropy may be NULL when compute_entropy
 * is 0.  Follows the Liger-Kernel native commit's "Summary" (NLL/LSE and
 * optional entropy) and the SkyRL page's "Overview" (entropy optional).
 */
static int forward_impl(const void* X, const void* W, int type, const int64_t* y, int64_t M,
                        int64_t H, int64_t V, int64_t ignore_index, double s,
                        int compute_entropy, const int64_t* rows, int64_t nrows,
                        double* logprob, double* lse, double* entropy) {
    if (M < 0 || H < 1 || V < 1 || nrows < 0) return FLPO_INVALID_ARG;
    if (rows == NULL && nrows != M) return FLPO_INVALID_ARG;
    int status = FLPO_OK;
#pragma omp parallel
    {
        double* xrow = (double*)malloc(sizeof(double) * (size_t)H);
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
#pragma omp for schedule(dynamic, 1)
        for (int64_t k = 0; k < nrows; ++k) {
            int64_t i = rows ? rows[k] : k;
            if (i < 0 || i >= M) {
#pragma omp atomic write
                status = FLPO_INVALID_ARG;
                continue;
            }
            logits_row(X, W, type, i, H, V, s, xrow, z);
            row_stats st = stats_from_logits(z, V);
            if (lse) lse[k] = st.lse;
            double lp, ent;
            if (!row_outputs(z, st, y[i], ignore_index, V, &lp, &ent)) {
#pragma omp atomic write
                status = FLPO_BAD_TARGET;
            }
            if (logprob) logprob[k] = lp;
            if (compute_entropy && entropy) entropy[k] = ent;
        }
        free(xrow);
        free(z);
    }
    return status;
}

/*
 * Backward for the rows listed in `rows` (all rows when rows == NULL): every
 * listed row's logits are recomputed (the "Kernel design notes" of the chunked
 * GRPO page), its dZ row is formed from the definition above, and
 *   dX_rows[k, :] = sum_j dZ[rows[k], j] W[j, :]        (when dX_rows != NULL)
 *   dW[j, :]      = sum_k dZ[rows[k], j] X[rows[k], :]  (when dW != NULL)
 * Rows that are not listed contribute nothing to dW, which equals a backward
 * whose upstream gradients are zero on those rows.
 *
 * round_dz_bf16 = 1 rounds each dZ value to fp32 and then to bf16 (RNE) before
 * the two contractions, mirroring the rounding point of the bf16 GEMM operands
 * that the chunked PPO backward of the same page adopts; 0 keeps fp64.
 */
static int backward_impl(const void* X, const void* W, int type, const int64_t* y, int64_t M,
                         int64_t H, int64_t V, int64_t ignore_index, double s,
                         int compute_entropy, const double* g_lp, const double* g_ent,
                         const int64_t* rows, int64_t nrows, int round_dz_bf16,
                         double* dX_rows, double* dW) {
    if (M < 0 || H < 1 || V < 1 || nrows < 0) return FLPO_INVALID_ARG;
    if (rows == NULL && nrows != M) return FLPO_INVALID_ARG;
    for (int64_t k = 0; k < nrows; ++k) {
        int64_t i = rows ? rows[k] : k;
        if (i < 0 || i >= M) return FLPO_INVALID_ARG;
    }
    double* dZ = (double*)malloc(sizeof(double) * (size_t)(nrows > 0 ? nrows : 1) * (size_t)V);
    if (!dZ) return FLPO_NO_MEMORY;
    int status = FLPO_OK;
#pragma omp parallel
    {
        double* xrow = (double*)malloc(sizeof(double) * (size_t)H);
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
#pragma omp for schedule(dynamic, 1)
        for (int64_t k = 0; k < nrows; ++k) {
            int64_t i = rows ? rows[k] : k;
            double* dz = dZ + k * V;
            double glp = g_lp ? g_lp[i] : 0.0;
            double gent = (compute_entropy && g_ent) ? g_ent[i] : 0.0;
            if (y[i] == ignore_index) {
                for (int64_t j = 0; j < V; ++j) dz[j] = 0.0;
                continue;
            }
            if (!target_ok(y[i], V)) {
#pragma omp atomic write
                status = FLPO_BAD_TARGET;
            }
            logits_row(X, W, type, i, H, V, s, xrow, z);
            row_stats st = stats_from_logits(z, V);
            for (int64_t j = 0; j < V; ++j) {
                double p = exp(z[j] - st.lse);
                double onehot = (j == y[i]) ? 1.0 : 0.0;
                dz[j] = s * (glp * (onehot - p) + gent * p * (st.sum_pz - z[j]));
            }
            if (round_dz_bf16)
                for (int64_t j = 0; j < V; ++j)
                    dz[j] = bf16_to_double(float_to_bf16_rne((float)dz[j]));
        }
        free(xrow);
        free(z);
    }
    if (dX_rows) {
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t k = 0; k < nrows; ++k) {
            const double* dz = dZ + k * V;
            double* out = dX_rows + k * H;
            for (int64_t h = 0; h < H; ++h) out[h] = 0.0;
            for (int64_t j = 0; j < V; ++j) {
                if (dz[j] == 0.0) continue;
                for (int64_t h = 0; h < H; ++h) out[h] += dz[j] * get_elem(W, type, j * H + h);
            }
        }
    }
    if (dW) {
#pragma omp parallel for schedule(dynamic, 16)
        for (int64_t j = 0; j < V; ++j) {
            double* out = dW + j * H;
            for (int64_t h = 0; h < H; ++h) out[h] = 0.0;
            for (int64_t k = 0; k < nrows; ++k) {
                int64_t i = rows ? rows[k] : k;
                double d = dZ[k * V + j];
                if (d == 0.0) continue;
                for (int64_t h = 0; h < H; ++h) out[h] += d * get_elem(X, type, i * H + h);
            }
        }
    }
    free(dZ);
    return status;
}

/*
 * dW restricted to the vocabulary rows listed in `cols`, with every row's
 * upstream gradient live:
 *   dW_cols[c, :] = sum_i dZ[i, cols[c]] X[i, :]      over all rows i in [0, M)
 * Each dZ entry needs its row's LSE and sum_j p_ij z_ij, hence every row's full
 * logit row (the same forward definitions as above); only the listed columns
 * of dZ are kept.  This is the sampled form of the backward for problems whose
 * full fp64 dW does not fit a test's time budget.  round_dz_bf16 as in
 * backward_impl.  Since every row's logits are formed anyway, the forward
 * outputs of every row can be returned too (logprob, lse, entropy: each may
 * be NULL), by the same definitions as forward_impl.
 */
static int backward_dw_cols_impl(const void* X, const void* W, int type, const int64_t* y,
                                 int64_t M, int64_t H, int64_t V, int64_t ignore_index,
                                 double s, int compute_entropy, const double* g_lp,
                                 const double* g_ent, const int64_t* cols, int64_t ncols,
                                 int round_dz_bf16, double* dW_cols, double* logprob,
                                 double* lse, double* entropy) {
    if (M < 0 || H < 1 || V < 1 || ncols < 0 || (ncols > 0 && !cols)) return FLPO_INVALID_ARG;
    for (int64_t c = 0; c < ncols; ++c)
        if (cols[c] < 0 || cols[c] >= V) return FLPO_INVALID_ARG;
    /* dZ[i, cols[c]] for every row i: M x ncols */
    double* dZ = (double*)malloc(sizeof(double) * (size_t)(M > 0 ? M : 1) * (size_t)(ncols > 0 ? ncols : 1));
    if (!dZ) return FLPO_NO_MEMORY;
    int status = FLPO_OK;
#pragma omp parallel
    {
        double* xrow = (double*)malloc(sizeof(double) * (size_t)H);
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < M; ++i) {
            double* dz = dZ + i * ncols;
            double glp = g_lp ? g_lp[i] : 0.0;
            double gent = (compute_entropy && g_ent) ? g_ent[i] : 0.0;
            logits_row(X, W, type, i, H, V, s, xrow, z);
            row_stats st = stats_from_logits(z, V);
            double lp, ent;
            if (!row_outputs(z, st, y[i], ignore_index, V, &lp, &ent)) {
#pragma omp atomic write
                status = FLPO_BAD_TARGET;
            }
            if (logprob) logprob[i] = lp;
            if (lse) lse[i] = st.lse;
            if (compute_entropy && entropy) entropy[i] = ent;
            if (y[i] == ignore_index) {  /* an ignored row's dZ row is zero */
                for (int64_t c = 0; c < ncols; ++c) dz[c] = 0.0;
                continue;
            }
            for (int64_t c = 0; c < ncols; ++c) {
                int64_t j = cols[c];
                double p = exp(z[j] - st.lse);
                double onehot = (j == y[i]) ? 1.0 : 0.0;
                double v = s * (glp * (onehot - p) + gent * p * (st.sum_pz - z[j]));
                dz[c] = round_dz_bf16 ? bf16_to_double(float_to_bf16_rne((float)v)) : v;
            }
        }
        free(xrow);
        free(z);
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t c = 0; c < ncols; ++c) {
        double* out = dW_cols + c * H;
        for (int64_t h = 0; h < H; ++h) out[h] = 0.0;
        for (int64_t i = 0; i < M; ++i) {
            double d = dZ[i * ncols + c];
            if (d == 0.0) continue;
            for (int64_t h = 0; h < H; ++h) out[h] += d * get_elem(X, type, i * H + h);
        }
    }
    free(dZ);
    return status;
}

/* ---- exported entry points (ctypes) ---- */

int flpo_forward_bf16(const uint16_t* X, const uint16_t* W, const int64_t* y, int64_t M,
                      int64_t H, int64_t V, int64_t ignore_index, double s,
                      int compute_entropy, const int64_t* rows, int64_t nrows,
                      double* logprob, double* lse, double* entropy) {
    return forward_impl(X, W, FLPO_BF16, y, M, H, V, ignore_index, s, compute_entropy, rows,
                        nrows, logprob, lse, entropy);
}

int flpo_forward_f64(const double* X, const double* W, const int64_t* y, int64_t M, int64_t H,
                     int64_t V, int64_t ignore_index, double s, int compute_entropy,
                     const int64_t* rows, int64_t nrows, double* logprob, double* lse,
                     double* entropy) {
    return forward_impl(X, W, FLPO_F64, y, M, H, V, ignore_index, s, compute_entropy, rows,
                        nrows, logprob, lse, entropy);
}

int flpo_backward_bf16(const uint16_t* X, const uint16_t* W, const int64_t* y, int64_t M,
                       int64_t H, int64_t V, int64_t ignore_index, double s,
                       int compute_entropy, const double* g_lp, const double* g_ent,
                       const int64_t* rows, int64_t nrows, int round_dz_bf16, double* dX_rows,
                       double* dW) {
    return backward_impl(X, W, FLPO_BF16, y, M, H, V, ignore_index, s, compute_entropy, g_lp,
                         g_ent, rows, nrows, round_dz_bf16, dX_rows, dW);
}

int flpo_backward_f64(const double* X, const double* W, const int64_t* y, int64_t M,
                      int64_t H, int64_t V, int64_t ignore_index, double s,
                      int compute_entropy, const double* g_lp, const double* g_ent,
                      const int64_t* rows, int64_t nrows, int round_dz_bf16, double* dX_rows,
                      double* dW) {
    return backward_impl(X, W, FLPO_F64, y, M, H, V, ignore_index, s, compute_entropy, g_lp,
                         g_ent, rows, nrows, round_dz_bf16, dX_rows, dW);
}

int flpo_backward_dw_cols_bf16(const uint16_t* X, const uint16_t* W, const int64_t* y,
                               int64_t M, int64_t H, int64_t V, int64_t ignore_index, double s,
                               int compute_entropy, const double* g_lp, const double* g_ent,
                               const int64_t* cols, int64_t ncols, int round_dz_bf16,
                               double* dW_cols, double* logprob, double* lse, double* entropy) {
    return backward_dw_cols_impl(X, W, FLPO_BF16, y, M, H, V, ignore_index, s, compute_entropy,
                                 g_lp, g_ent, cols, ncols, round_dz_bf16, dW_cols, logprob, lse,
                                 entropy);
}

int flpo_backward_dw_cols_f64(const double* X, const double* W, const int64_t* y, int64_t M,
                              int64_t H, int64_t V, int64_t ignore_index, double s,
                              int compute_entropy, const double* g_lp, const double* g_ent,
                              const int64_t* cols, int64_t ncols, int round_dz_bf16,
                              double* dW_cols, double* logprob, double* lse, double* entropy) {
    return backward_dw_cols_impl(X, W, FLPO_F64, y, M, H, V, ignore_index, s, compute_entropy,
                                 g_lp, g_ent, cols, ncols, round_dz_bf16, dW_cols, logprob, lse,
                                 entropy);
}

/* The oracle's binary32 -> bf16 rounding (round to nearest, ties to even),
 * exported so that tests can pin it bit for bit. */
void flpo_round_bf16(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = float_to_bf16_rne(in[i]);
}

/* Threads OpenMP will use for the parallel regions above. */
int flpo_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Loss heads on the per-row log-probs (the chunked GRPO loss of "Triton MoE
 * improvements and chunked GRPO improvements", section "Chunked Triton GRPO
 * loss": a loss on top of the lm_head's per-token log-probs, aggregated over
 * the valid tokens).  Rows whose target is ignore_index are not tokens of the
 * loss.  With N valid rows:
 *
 *   kind 1 (token-mean NLL):  loss = -(1/N) sum_i lp_i
 *   kind 2 (clipped surrogate, token-level ratio, token-mean):
 *       r_i    = exp(lp_i - old_i)
 *       surr_i = min(r_i A_i, clip(r_i, 1 - eps_low, 1 + eps_high) A_i)
 *       kl_i   = exp(ref_i - lp_i) - (ref_i - lp_i) - 1      (when ref given)
 *       loss   = (1/N) sum_i [ -surr_i + beta kl_i ]
 *
 * Outputs: per-row loss terms (0 on ignored rows), the scalar loss, and the
 * gradient of the scalar loss with respect to each row's log-prob (the
 * upstream gradient the backward takes).  The gradient is the derivative of
 * the definition: the min picks r A unless the clipped term is strictly
 * smaller, and a clipped ratio has zero derivative.
 */
int flpo_loss(const double* lp, const int64_t* y, int64_t M, int64_t ignore_index, int kind,
              const double* old_lp, const double* adv, const double* ref_lp, double eps_low,
              double eps_high, double beta, double* per_row, double* grad, double* loss) {
    if (M < 0 || (kind != 1 && kind != 2 && kind != 3)) return FLPO_INVALID_ARG;
    if (kind == 3) {
        /* kind 3 (token-sum NLL): loss = -sum_i lp_i over the valid rows, no
         * normalisation; d loss / d lp_i = -1 on a valid row. */
        double total = 0.0;
        for (int64_t i = 0; i < M; ++i) {
            int valid = y[i] != ignore_index;
            if (per_row) per_row[i] = valid ? -lp[i] : 0.0;
            if (grad) grad[i] = valid ? -1.0 : 0.0;
            if (valid) total += -lp[i];
        }
        if (loss) *loss = total;
        return FLPO_OK;
    }
    if (kind == 2 && (!old_lp || !adv)) return FLPO_INVALID_ARG;
    int64_t n = 0;
    for (int64_t i = 0; i < M; ++i)
        if (y[i] != ignore_index) ++n;
    double total = 0.0;
    for (int64_t i = 0; i < M; ++i) {
        double term = 0.0, g = 0.0;
        if (y[i] != ignore_index) {
            if (kind == 1) {
                term = -lp[i];
                g = -1.0;
            } else {
                double r = exp(lp[i] - old_lp[i]);
                double lo = 1.0 - eps_low, hi = 1.0 + eps_high;
                double rc = r < lo ? lo : (r > hi ? hi : r);
                double s1 = r * adv[i], s2 = rc * adv[i];
                double surr = s1 <= s2 ? s1 : s2;
                double dsurr = s1 <= s2 ? r * adv[i] : 0.0;
                term = -surr;
                g = -dsurr;
                if (ref_lp && beta != 0.0) {
                    double d = ref_lp[i] - lp[i];
                    term += beta * (exp(d) - d - 1.0);
                    g += beta * (1.0 - exp(d));
                }
            }
        }
        if (per_row) per_row[i] = term;
        total += term;
        if (grad) grad[i] = n > 0 ? g / (double)n : 0.0;
    }
    if (loss) *loss = n > 0 ? total / (double)n : 0.0;
    return FLPO_OK;
}

/*
 * Policy-gradient loss over sequences (the chunked GRPO page: "Setup" runs
 * loss_type="dapo" with importance_sampling_level="sequence" and
 * num_items_in_batch; "Correctness" lists the grpo / bnpo / dr_grpo / dapo
 * aggregations with token- and sequence-level importance sampling).  The page
 * names these options without defining them; the readings taken here:
 *
 *   rows [off[b], off[b+1]) form sequence b (b < B); a row is a token of the
 *   loss when its target is not ignore_index; n_b = tokens of sequence b,
 *   N = sum_b n_b.  off == NULL means one sequence of all M rows.
 *   ratio, token level:    log r_t = lp_t - old_t
 *   ratio, sequence level: log r_t = (1/n_b) sum_{u in b} (lp_u - old_u)  (every t in b)
 *   term_t = -min(r_t A_t, clip(r_t, 1 - eps_low, 1 + eps_high) A_t)
 *            + beta (exp(ref_t - lp_t) - (ref_t - lp_t) - 1)   (KL only when ref given)
 *   aggregation 0, token mean (bnpo):     loss = (1/N) sum_t term_t
 *   aggregation 1, sequence mean (grpo):  loss = (1/B) sum_b (1/max(n_b, 1)) sum_{t in b} term_t
 *   aggregation 2, sum over a normaliser (dapo: num_items_in_batch; dr_grpo:
 *                 B x the longest completion):  loss = (1/D) sum_t term_t,
 *                 D = normalizer when > 0, else N
 *
 * Outputs: per-token terms (0 on rows that are not tokens), the scalar loss,
 * and d loss / d lp_t.  Each token's weight in the loss is c_t (1/N,
 * 1/(B max(n_b, 1)) or 1/D); the min picks r A unless the clipped term is
 * strictly smaller, and a clipped ratio has zero derivative.  With a
 * sequence-level ratio every term of sequence b depends on every lp_u of b
 * through log r_b, whose derivative with respect to lp_u is 1/n_b.
 */
int flpo_policy_loss(const double* lp, const int64_t* y, int64_t M, int64_t ignore_index,
                     const int64_t* off, int64_t B, const double* old_lp, const double* adv,
                     const double* ref_lp, double eps_low, double eps_high, double beta,
                     int is_level, int aggregation, double normalizer, double* per_row,
                     double* grad, double* loss) {
    if (M < 0 || !old_lp || !adv || (is_level != 0 && is_level != 1) || aggregation < 0 ||
        aggregation > 2)
        return FLPO_INVALID_ARG;
    int64_t one_seq[2] = {0, M};
    if (!off) {
        off = one_seq;
        B = 1;
    }
    if (B < 1) return FLPO_INVALID_ARG;
    for (int64_t b = 0; b < B; ++b)
        if (off[b] < 0 || off[b + 1] < off[b] || off[b + 1] > M) return FLPO_INVALID_ARG;
    for (int64_t i = 0; i < M; ++i) {
        if (per_row) per_row[i] = 0.0;
        if (grad) grad[i] = 0.0;
    }
    int64_t N = 0;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t t = off[b]; t < off[b + 1]; ++t)
            if (y[t] != ignore_index) ++N;
    double D = (aggregation == 2 && normalizer > 0.0) ? normalizer : (double)N;
    double total = 0.0;
    double lo = 1.0 - eps_low, hi = 1.0 + eps_high;
    for (int64_t b = 0; b < B; ++b) {
        int64_t nb = 0;
        double sum_log = 0.0;
        for (int64_t t = off[b]; t < off[b + 1]; ++t)
            if (y[t] != ignore_index) {
                ++nb;
                sum_log += lp[t] - old_lp[t];
            }
        double seq_log_r = nb > 0 ? sum_log / (double)nb : 0.0;
        double c;
        if (aggregation == 0) c = N > 0 ? 1.0 / (double)N : 0.0;
        else if (aggregation == 1) c = 1.0 / ((double)B * (double)(nb > 0 ? nb : 1));
        else c = D > 0.0 ? 1.0 / D : 0.0;
        double G = 0.0; /* sum over the tokens of b of c * d term_t / d log r_b */
        for (int64_t t = off[b]; t < off[b + 1]; ++t) {
            if (y[t] == ignore_index) continue;
            double log_r = is_level == 1 ? seq_log_r : lp[t] - old_lp[t];
            double r = exp(log_r);
            double rc = r < lo ? lo : (r > hi ? hi : r);
            double s1 = r * adv[t], s2 = rc * adv[t];
            double term = -(s1 <= s2 ? s1 : s2);
            double dterm_dlogr = s1 <= s2 ? -r * adv[t] : 0.0;
            double g_kl = 0.0;
            if (ref_lp && beta != 0.0) {
                double d = ref_lp[t] - lp[t];
                term += beta * (exp(d) - d - 1.0);
                g_kl = beta * (1.0 - exp(d));
            }
            if (per_row) per_row[t] = term;
            total += c * term;
            if (is_level == 1) {
                G += c * dterm_dlogr;
                if (grad) grad[t] = c * g_kl;
            } else if (grad) {
                grad[t] = c * (dterm_dlogr + g_kl);
            }
        }
        if (is_level == 1 && grad && nb > 0)
            for (int64_t t = off[b]; t < off[b + 1]; ++t)
                if (y[t] != ignore_index) grad[t] += G / (double)nb;
    }
    if (loss) *loss = total;
    return FLPO_OK;
}
