/*
 * kda_oracle.c -- plain, slow f64 CPU oracle for the Kimi Delta Attention
 * (KDA) forward.  TEST INFRASTRUCTURE ONLY: tests, the smoke check and the
 * bench's CPU-baseline leg may call it; the product path never does.
 *
 * It shares no code, header or constant with the CUDA library.  Every step
 * is written from the method's statement, token by token, with no blocking,
 * fusion or reordering:
 *
 *   gate   (kdafix-2026-10-02, "Fix 1 -- decay form"):
 *          g = -exp(A_log_h) * softplus(z + dt_bias_h)   per key channel,
 *          softplus evaluated first, then the -exp(A_log) multiplier;
 *          alpha = exp(g) in (0, 1], g <= 0.
 *   step   (per (b, h), state S is K x V):
 *          S <- diag(alpha_t) S
 *          u  = v_t - S^T k_t
 *          S <- S + beta_t k_t u^T
 *          o_t = S^T (scale * q_t)
 *          (kdafix-2026-10-02, "Fix 2 -- read scale": the scale is folded
 *          into q and enters only the read, never the state.)
 *
 * Layouts are head-major and contiguous:
 *   q, k, z, g : (B, H, T, K)     v, o : (B, H, T, V)     beta : (B, H, T)
 *   h0, hT     : (B, H, K, V)     A_log : (H)             dt_bias : (H, K)
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - softplus(x) = max(x, 0) + log1p(exp(-|x|)), exact (no threshold cut);
 *   - no clamp on A_log;
 *   - u uses the decayed state, o uses the post-update state.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

/* softplus(x) = log(1 + e^x), written so that neither branch overflows. */
double kda_oracle_softplus(double x) {
    return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

/* g[b,h,t,c] = -exp(A_log[h]) * softplus(z[b,h,t,c] + dt_bias[h,c]). */
void kda_oracle_gate(int B, int H, int T, int K, const double* z,
                     const double* A_log, const double* dt_bias, double* g) {
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            const double mult = exp(A_log[h]);
            for (int t = 0; t < T; ++t) {
                size_t row = (((size_t)b * H + h) * T + t) * K;
                for (int c = 0; c < K; ++c) {
                    double sp = kda_oracle_softplus(z[row + c] + dt_bias[(size_t)h * K + c]);
                    g[row + c] = -(mult * sp);
                }
            }
        }
}

/*
 * Token-by-token recurrence for the (b, h) pairs with flat index
 * bh in [bh_begin, bh_end), given the log decay g (B,H,T,K).
 * h0 may be NULL (zero initial state); hT may be NULL.
 */
void kda_oracle_recurrent_range(int B, int H, int T, int K, int V,
                                const double* q, const double* k, const double* v,
                                const double* g, const double* beta, double scale,
                                const double* h0, double* o, double* hT,
                                int bh_begin, int bh_end) {
    (void)B;
    double* S = (double*)malloc(sizeof(double) * (size_t)K * V);
    double* u = (double*)malloc(sizeof(double) * (size_t)V);
    double* qs = (double*)malloc(sizeof(double) * (size_t)K);
    for (int bh = bh_begin; bh < bh_end; ++bh) {
        (void)H;
        const size_t sidx = (size_t)bh * K * V;
        if (h0) memcpy(S, h0 + sidx, sizeof(double) * (size_t)K * V);
        else memset(S, 0, sizeof(double) * (size_t)K * V);
        for (int t = 0; t < T; ++t) {
            const size_t kr = ((size_t)bh * T + t) * K;
            const size_t vr = ((size_t)bh * T + t) * V;
            const double bt = beta[(size_t)bh * T + t];
            /* S <- diag(alpha_t) S */
            for (int c = 0; c < K; ++c) {
                double a = exp(g[kr + c]);
                for (int j = 0; j < V; ++j) S[(size_t)c * V + j] *= a;
            }
            /* u = v_t - S^T k_t */
            for (int j = 0; j < V; ++j) {
                double acc = 0.0;
                for (int c = 0; c < K; ++c) acc += S[(size_t)c * V + j] * k[kr + c];
                u[j] = v[vr + j] - acc;
            }
            /* S <- S + beta_t k_t u^T */
            for (int c = 0; c < K; ++c)
                for (int j = 0; j < V; ++j) S[(size_t)c * V + j] += bt * k[kr + c] * u[j];
            /* o_t = S^T (scale q_t) */
            for (int c = 0; c < K; ++c) qs[c] = scale * q[kr + c];
            for (int j = 0; j < V; ++j) {
                double acc = 0.0;
                for (int c = 0; c < K; ++c) acc += S[(size_t)c * V + j] * qs[c];
                o[vr + j] = acc;
            }
        }
        if (hT) memcpy(hT + sidx, S, sizeof(double) * (size_t)K * V);
    }
    free(S);
    free(u);
    free(qs);
}

/*
 * Full forward for (b, h) in [bh_begin, bh_end): the gate evaluated per token
 * from z, A_log and dt_bias, then the same recurrence.  This is the routine the
 * CPU baseline times; it allocates only O(K + V) scratch per token.
 */
void kda_oracle_forward_range(int B, int H, int T, int K, int V,
                              const double* q, const double* k, const double* v,
                              const double* z, const double* beta,
                              const double* A_log, const double* dt_bias, double scale,
                              const double* h0, double* o, double* hT,
                              int bh_begin, int bh_end) {
    double* gt = (double*)malloc(sizeof(double) * (size_t)T * K);
    for (int bh = bh_begin; bh < bh_end; ++bh) {
        const int h = bh % H;
        const double mult = exp(A_log[h]);
        for (int t = 0; t < T; ++t) {
            const size_t kr = ((size_t)bh * T + t) * K;
            for (int c = 0; c < K; ++c)
                gt[(size_t)t * K + c] =
                    -(mult * kda_oracle_softplus(z[kr + c] + dt_bias[(size_t)h * K + c]));
        }
        /* Run the recurrence on this single (b, h) with its gate: offset the
         * pointers so the pair sits at flat index 0 of a one-pair problem. */
        kda_oracle_recurrent_range(1, 1, T, K, V, q + (size_t)bh * T * K, k + (size_t)bh * T * K,
                                   v + (size_t)bh * T * V, gt, beta + (size_t)bh * T, scale,
                                   h0 ? h0 + (size_t)bh * K * V : NULL, o + (size_t)bh * T * V,
                                   hT ? hT + (size_t)bh * K * V : NULL, 0, 1);
    }
    free(gt);
}
