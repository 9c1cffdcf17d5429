/*
 * Reference oracle for the fused attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into a small CPU library
 * that the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load.  The product path (the CUDA library) never links, calls or reads it,
 * and this file shares no code, header or constant with the CUDA path.
 *
 * What it computes (fp64 throughout, one query row at a time):
 *
 *   s_j   = scale * sum_c q[i][c] * k[j][c]        for every key j < N
 *   s_j   = -inf                                   if causal and j > i
 *   m     = max_j s_j
 *   p_j   = exp(s_j - m)
 *   l     = sum_j p_j
 *   O[i]  = sum_j p_j * v[j] / l
 *   LSE_i = m + ln(l)
 *
 * Source: "Warp specialization" concept card (wikillm), section
 * "Implementation sketch": the consumer returns output / row_sum and
 * row_max + log(row_sum); its loop over key blocks only reschedules this
 * computation ("they change the schedule of the loop, not its result"), so
 * with the whole score row in one block the recurrence collapses to the
 * plain definition above.  The pages do not define the scale factor, the
 * causal mask or the layout; the readings taken here are:
 *   - scale multiplies Q.K^T before the max, the mask and the exponential,
 *     so LSE is the natural-log logsumexp of the scaled scores;
 *   - causal means key j is visible to query i iff j <= i (square,
 *     top-left aligned lower-triangular mask);
 *   - tensors are contiguous [B, H, N, d] row-major, LSE is [B, H, N].
 *
 * A second entry point runs the card's blockwise recurrence itself (running
 * max, rescale of the old sum and output by exp(row_max - new_max), then
 * output / row_sum at the end), so the tests can check the two forms
 * against each other.  That form is only used for self-checks.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Number of threads the parallel loops will use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One query row, direct (materialised) form.  q_row: [d]; k, v: [N, d] of
 * one (b, h); o_row: [d].  Returns the LSE.  `srow` is caller scratch [N]. */
static double attn_row_direct(const double* q_row, const double* k, const double* v,
                              double* o_row, double* srow, int64_t N, int64_t d,
                              double scale, int causal, int64_t i) {
    /* scores, with the causal mask applied before the max */
    for (int64_t j = 0; j < N; ++j) {
        if (causal && j > i) {
            srow[j] = -INFINITY;
            continue;
        }
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c) acc += q_row[c] * k[j * d + c];
        srow[j] = scale * acc;
    }
    /* row max */
    double m = -INFINITY;
    for (int64_t j = 0; j < N; ++j)
        if (srow[j] > m) m = srow[j];
    /* exponentials and their sum; a row with every key masked has no
       finite score, then the subtraction reference is 0 so that
       (-inf) - (-inf) never appears */
    double ref = isinf(m) && m < 0 ? 0.0 : m;
    double l = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        srow[j] = exp(srow[j] - ref);
        l += srow[j];
    }
    /* O = P V / l */
    for (int64_t c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int64_t j = 0; j < N; ++j) acc += srow[j] * v[j * d + c];
        o_row[c] = acc / l;
    }
    return ref + log(l);
}

/*
 * Direct oracle.
 *   q, k, v : [B, H, N, d] fp64 (the values the GPU reads, upcast exactly)
 *   rows    : NULL for every row, else n_rows query indices in [0, N) that
 *             are computed for every (b, h)
 *   o       : [B, H, R, d] with R = N (rows == NULL) or n_rows
 *   lse     : [B, H, R]
 *   n_threads <= 0 uses the OpenMP default.
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_attn_fwd(const double* q, const double* k, const double* v,
                    double* o, double* lse,
                    int64_t B, int64_t H, int64_t N, int64_t d,
                    double scale, int causal,
                    const int64_t* rows, int64_t n_rows, int n_threads) {
    if (!q || !k || !v || !o || !lse || B < 1 || H < 1 || N < 1 || d < 1) return -1;
    int64_t R = rows ? n_rows : N;
    if (R < 1) return -1;
    if (rows)
        for (int64_t r = 0; r < R; ++r)
            if (rows[r] < 0 || rows[r] >= N) return -1;
    int64_t total = B * H * R;
    int failed = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
#endif
    {
        double* srow = (double*)malloc((size_t)N * sizeof(double));
        if (!srow) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 16)
#endif
            for (int64_t t = 0; t < total; ++t) {
                int64_t bh = t / R, r = t % R;
                int64_t i = rows ? rows[r] : r;
                const double* qh = q + bh * N * d;
                const double* kh = k + bh * N * d;
                const double* vh = v + bh * N * d;
                lse[t] = attn_row_direct(qh + i * d, kh, vh, o + t * d, srow,
                                         N, d, scale, causal, i);
            }
            free(srow);
        }
    }
    (void)n_threads;
    return failed ? -1 : 0;
}

/*
 * Blockwise form: the card's consumer loop ("Warp specialization",
 * section "Implementation sketch") for one query row, over key blocks of
 * Bc keys.  Per block j: scores of the block; new_max = max(row_max,
 * rowmax(scores)); probs = exp(scores - new_max); row_sum =
 * exp(row_max - new_max) * row_sum + rowsum(probs); output =
 * exp(row_max - new_max) * output + probs @ values_j; row_max = new_max.
 * The rescale multiplies the OLD output by exp(row_max - new_max), the
 * form the card states agrees with the normalising sum (it rejects the
 * inverse factor).  Initial state: output 0, row_max -inf, row_sum 0.
 * While row_max is still -inf (every key so far masked), 0 is used as the
 * subtraction reference so that no (-inf) - (-inf) is formed.
 * Same arguments and layout as oracle_attn_fwd, plus Bc >= 1.
 */
int oracle_attn_fwd_blockwise(const double* q, const double* k, const double* v,
                              double* o, double* lse,
                              int64_t B, int64_t H, int64_t N, int64_t d,
                              double scale, int causal, int64_t Bc) {
    if (!q || !k || !v || !o || !lse || B < 1 || H < 1 || N < 1 || d < 1 || Bc < 1)
        return -1;
    double* scores = (double*)malloc((size_t)Bc * sizeof(double));
    double* out = (double*)malloc((size_t)d * sizeof(double));
    if (!scores || !out) {
        free(scores);
        free(out);
        return -1;
    }
    for (int64_t bh = 0; bh < B * H; ++bh) {
        const double* qh = q + bh * N * d;
        const double* kh = k + bh * N * d;
        const double* vh = v + bh * N * d;
        for (int64_t i = 0; i < N; ++i) {
            double row_max = -INFINITY, row_sum = 0.0;
            for (int64_t c = 0; c < d; ++c) out[c] = 0.0;
            for (int64_t j0 = 0; j0 < N; j0 += Bc) {
                int64_t nb = N - j0 < Bc ? N - j0 : Bc;
                double blk_max = -INFINITY;
                for (int64_t jj = 0; jj < nb; ++jj) {
                    int64_t j = j0 + jj;
                    double s;
                    if (causal && j > i) {
                        s = -INFINITY;
                    } else {
                        double acc = 0.0;
                        for (int64_t c = 0; c < d; ++c) acc += qh[i * d + c] * kh[j * d + c];
                        s = scale * acc;
                    }
                    scores[jj] = s;
                    if (s > blk_max) blk_max = s;
                }
                double new_max = row_max > blk_max ? row_max : blk_max;
                double ref = isinf(new_max) && new_max < 0 ? 0.0 : new_max;
                /* exp(row_max - new_max); 0 when row_max is still -inf */
                double alpha = exp(row_max - ref);
                double blk_sum = 0.0;
                for (int64_t jj = 0; jj < nb; ++jj) {
                    scores[jj] = exp(scores[jj] - ref);
                    blk_sum += scores[jj];
                }
                row_sum = alpha * row_sum + blk_sum;
                for (int64_t c = 0; c < d; ++c) {
                    double acc = 0.0;
                    for (int64_t jj = 0; jj < nb; ++jj) acc += scores[jj] * vh[(j0 + jj) * d + c];
                    out[c] = alpha * out[c] + acc;
                }
                row_max = new_max;
            }
            double ref = isinf(row_max) && row_max < 0 ? 0.0 : row_max;
            for (int64_t c = 0; c < d; ++c) o[(bh * N + i) * d + c] = out[c] / row_sum;
            lse[bh * N + i] = ref + log(row_sum);
        }
    }
    free(scores);
    free(out);
    return 0;
}

/*
 * Backward pass of the same function, fp64, per (b, h) (test infrastructure
 * only, like the rest of this file).  For the loss gradient dO = dL/dO the
 * gradients follow from differentiating the definition above:
 *
 *   P_ij  = exp(s_ij - LSE_i)                  (0 where masked)
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . v_j
 *   D_i   = sum_j P_ij dP_ij                   (= dO_i . O_i)
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale * sum_j dS_ij k_j
 *   dK_j  = scale * sum_i dS_ij q_i
 *
 * The logsumexp output of the forward is what makes this computable block
 * by block without the running max ("Warp specialization" concept card,
 * section "Implementation sketch": the consumer returns row_max +
 * log(row_sum) next to the output).  Here every score row is materialised
 * and LSE is recomputed exactly.  Arrays are [B, H, N, d]; all of dq, dk,
 * dv are written.  Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_attn_bwd(const double* q, const double* k, const double* v, const double* dout,
                    double* dq, double* dk, double* dv,
                    int64_t B, int64_t H, int64_t N, int64_t d, double scale, int causal,
                    int n_threads) {
    if (!q || !k || !v || !dout || !dq || !dk || !dv || B < 1 || H < 1 || N < 1 || d < 1)
        return -1;
    int failed = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t bh = 0; bh < B * H; ++bh) {
        const double* qh = q + bh * N * d;
        const double* kh = k + bh * N * d;
        const double* vh = v + bh * N * d;
        const double* doh = dout + bh * N * d;
        double* dqh = dq + bh * N * d;
        double* dkh = dk + bh * N * d;
        double* dvh = dv + bh * N * d;
        double* prow = (double*)malloc((size_t)N * sizeof(double));
        double* dprow = (double*)malloc((size_t)N * sizeof(double));
        if (!prow || !dprow) {
            free(prow);
            free(dprow);
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
            continue;
        }
        for (int64_t x = 0; x < N * d; ++x) {
            dqh[x] = 0.0;
            dkh[x] = 0.0;
            dvh[x] = 0.0;
        }
        for (int64_t i = 0; i < N; ++i) {
            /* scores, max, LSE of row i */
            double m = -INFINITY;
            for (int64_t j = 0; j < N; ++j) {
                if (causal && j > i) {
                    prow[j] = -INFINITY;
                    continue;
                }
                double acc = 0.0;
                for (int64_t c = 0; c < d; ++c) acc += qh[i * d + c] * kh[j * d + c];
                prow[j] = scale * acc;
                if (prow[j] > m) m = prow[j];
            }
            double l = 0.0;
            for (int64_t j = 0; j < N; ++j) l += exp(prow[j] - m);
            double lse = m + log(l);
            /* P, dP, D */
            double D = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                prow[j] = exp(prow[j] - lse);
                double acc = 0.0;
                for (int64_t c = 0; c < d; ++c) acc += doh[i * d + c] * vh[j * d + c];
                dprow[j] = acc;
                D += prow[j] * acc;
            }
            /* accumulate the three gradients */
            for (int64_t j = 0; j < N; ++j) {
                double pij = prow[j];
                if (pij == 0.0) continue;
                double ds = pij * (dprow[j] - D);
                for (int64_t c = 0; c < d; ++c) {
                    dvh[j * d + c] += pij * doh[i * d + c];
                    dqh[i * d + c] += scale * ds * kh[j * d + c];
                    dkh[j * d + c] += scale * ds * qh[i * d + c];
                }
            }
        }
        free(prow);
        free(dprow);
    }
    (void)n_threads;
    return failed ? -1 : 0;
}
