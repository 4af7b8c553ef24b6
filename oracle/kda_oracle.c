/*
 * Plain CPU oracle for the chunkwise Kimi Delta Attention (KDA) forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no source, header, table or helper with
 * the CUDA library.
 *
 * What it computes (fp64 throughout, one token at a time, no chunking):
 *
 *   For every sequence n (tokens cu[n] .. cu[n+1]-1) and every head h, with a
 *   V-first state S in R^{V x K}:
 *
 *     q^ = q / sqrt(sum q^2 + eps) / sqrt(K)       L2-normalised query, scaled
 *     k^ = k / sqrt(sum k^2 + eps)                 L2-normalised key
 *     g  = lower_bound * sigmoid(g_raw)            per-channel log-decay (K)
 *     b  = sigmoid(beta_raw)                       scalar write strength
 *     S  <- S * Diag(exp g) * (I - b k^ k^T) + b v k^T
 *     o  = S q^                                    (state after the update)
 *
 *   S starts from the sequence's initial state when has_init[n] is set and
 *   from zeros otherwise (the initial state is then never read, so NaN in it
 *   cannot leak).  The state after the last token is the sequence's final
 *   state; an empty sequence returns its initial state (zeros without one).
 *
 * Sources.  ROCm/aiter PR #4741 "[FlyDSL] Add gfx950 Kimi Delta Attention
 * prefill kernel", Summary and "Optimizations Applied": q/k L2 norm, the
 * lower-bounded-sigmoid gate, the beta sigmoid, V-first state, padded tokens
 * (beta = 0, g = 0) leave the state unchanged.  ROCm/aiter PR #5754 "Technical
 * Details": has_initial_state = false starts from zero and never reads the slot;
 * the final state goes back to the same pool row.  ROCm/aiter PR #5249 "What":
 * accumulation is fp32 or better whatever the storage dtype.  The recurrence
 * itself (the update and output lines above) is not printed on those pages;
 * it is the gated delta rule with per-channel decay exactly as written above.
 *
 * The update is evaluated in the algebraically identical rank-1 form
 *     S' = S Diag(exp g);  S = S' + b (v - S' k^) k^T
 * which is the same expression with the product expanded (no reordering beyond
 * distributing the matrix product).  Each V row of S evolves independently
 * given (k^, g, b, v[row]), so the work is split over (sequence, head, block of
 * V rows) with OpenMP; the arithmetic of every row is the same whatever the
 * thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef KDA_ORACLE_ROW_BLOCK
#define KDA_ORACLE_ROW_BLOCK 16
#endif

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Number of OpenMP threads a parallel region of the oracle will use. */
int kda_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Per-token quantities of one (token, head): normalised q and k, the decay
 * factors exp(g) per channel and the scalar beta.
 */
static void token_prep(const double* q, const double* k, const double* g_raw,
                       double beta_raw, int K, double lower_bound, double eps,
                       double* qn, double* kn, double* decay, double* beta) {
    double sq = 0.0, sk = 0.0;
    for (int c = 0; c < K; ++c) {
        sq += q[c] * q[c];
        sk += k[c] * k[c];
    }
    double rq = 1.0 / sqrt(sq + eps) / sqrt((double)K);
    double rk = 1.0 / sqrt(sk + eps);
    for (int c = 0; c < K; ++c) {
        qn[c] = q[c] * rq;
        kn[c] = k[c] * rk;
        decay[c] = exp(lower_bound * sigmoid(g_raw[c]));
    }
    *beta = sigmoid(beta_raw);
}

/*
 * kda_oracle_forward
 *
 *   q, k      [T][H][K]   fp64
 *   v         [T][H][V]   fp64
 *   g_raw     [T][H][K]   fp64, raw (pre-activation) gate
 *   beta_raw  [T][H]      fp64, raw (pre-activation) beta
 *   cu        [N+1]       sequence bounds, cu[0] = 0, non-decreasing, cu[N] = T
 *   init      [N][H][V][K] initial states (read only where has_init[n] != 0;
 *                         may be NULL when no flag is set)
 *   has_init  [N]
 *   out       [T][H][V]   written for every token
 *   final     [N][H][V][K] written for every sequence (empty ones included)
 *
 * Returns 0, or -1 on an argument error.
 */
int kda_oracle_forward(int64_t T, int32_t H, int32_t K, int32_t V,
                       const double* q, const double* k, const double* v,
                       const double* g_raw, const double* beta_raw,
                       int32_t N, const int64_t* cu,
                       const double* init, const uint8_t* has_init,
                       double lower_bound, double eps,
                       double* out, double* final_state) {
    if (T < 0 || H <= 0 || K <= 0 || V <= 0 || N < 0) return -1;
    if (cu == NULL || out == NULL || final_state == NULL) return -1;
    if (cu[0] != 0 || cu[N] != T) return -1;
    for (int32_t n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return -1;
    for (int32_t n = 0; n < N; ++n)
        if (has_init && has_init[n] && init == NULL) return -1;

    const int RB = KDA_ORACLE_ROW_BLOCK;
    const int nblk = (V + RB - 1) / RB;
    const int64_t items = (int64_t)N * H * nblk;
    int bad = 0;

#pragma omp parallel
    {
        double* qn = (double*)malloc(sizeof(double) * K);
        double* kn = (double*)malloc(sizeof(double) * K);
        double* dec = (double*)malloc(sizeof(double) * K);
        double* S = (double*)malloc(sizeof(double) * (size_t)RB * K);
        if (!qn || !kn || !dec || !S) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t it = 0; it < items; ++it) {
            if (bad) continue;
            const int32_t n = (int32_t)(it / ((int64_t)H * nblk));
            const int32_t h = (int32_t)((it / nblk) % H);
            const int v0 = (int)(it % nblk) * RB;
            const int nv = (V - v0 < RB) ? (V - v0) : RB;

            /* initial state rows v0 .. v0+nv-1 */
            const size_t plane = (size_t)V * K;
            const size_t sbase = ((size_t)n * H + h) * plane + (size_t)v0 * K;
            if (has_init && has_init[n]) {
                memcpy(S, init + sbase, sizeof(double) * (size_t)nv * K);
            } else {
                memset(S, 0, sizeof(double) * (size_t)nv * K);
            }

            for (int64_t t = cu[n]; t < cu[n + 1]; ++t) {
                const size_t tk = ((size_t)t * H + h) * K;
                const size_t tv = ((size_t)t * H + h) * V;
                double beta;
                token_prep(q + tk, k + tk, g_raw + tk, beta_raw[(size_t)t * H + h],
                           K, lower_bound, eps, qn, kn, dec, &beta);
                for (int r = 0; r < nv; ++r) {
                    double* s = S + (size_t)r * K;
                    /* S' = S Diag(exp g): decay scales the K columns */
                    for (int c = 0; c < K; ++c) s[c] *= dec[c];
                    /* delta write: S = S' + b (v - S' k^) k^T */
                    double sk = 0.0;
                    for (int c = 0; c < K; ++c) sk += s[c] * kn[c];
                    const double d = beta * (v[tv + v0 + r] - sk);
                    for (int c = 0; c < K; ++c) s[c] += d * kn[c];
                    /* o = S q^ with the updated state */
                    double o = 0.0;
                    for (int c = 0; c < K; ++c) o += s[c] * qn[c];
                    out[tv + v0 + r] = o;
                }
            }
            memcpy(final_state + sbase, S, sizeof(double) * (size_t)nv * K);
        }
        free(qn);
        free(kn);
        free(dec);
        free(S);
    }
    return bad ? -2 : 0;
}
