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

/*
 * Gradients of the same forward (the backward pass), f64, token by token in reverse.
 *
 * The loss is any scalar L whose adjoints with respect to the outputs are given:
 * d_o = dL/do (B,H,T,V) and dhT = dL/dhT (B,H,K,V, NULL = 0).  Every input gets its
 * adjoint by reverse-mode differentiation of the steps above, taken in the opposite order
 * (the kda-adjoint-2026-10-01 page names the backward of this forward and its gradients dq,
 * dk, dv, dg, dbeta and the state gradient; the steps below are the chain rule applied to
 * the forward as stated, nothing else).  For token t, with S the state entering it,
 * alpha = exp(g_t), Sd = diag(alpha) S, u = v_t - Sd^T k_t, Sn = Sd + beta_t k_t u^T and the
 * adjoint dSn of Sn:
 *
 *   dSn   += (scale q_t) d_o_t^T              dq_t  = scale Sn d_o_t
 *   du     = beta_t dSn^T k_t                 dbeta_t = k_t^T dSn u
 *   dk_t   = beta_t dSn u - Sd du             dv_t  = du
 *   dSd    = dSn - k_t du^T                   dalpha = rowsum(S .* dSd)
 *   dS     = diag(alpha) dSd                  dg_t  = alpha .* dalpha
 *
 * and through the gate x = z + dt_bias_h, g = -exp(A_log_h) softplus(x):
 *   dz = dg (-exp(A_log_h)) sigmoid(x),  ddt_bias_h += dz,  dA_log_h += dg g.
 * dh0 is dS after token 0.  dA_log and ddt_bias are returned per (b, h) (dA_part (B*H),
 * ddt_part (B*H, K)); the caller sums them over b.  dg (B,H,T,K), the gradient with respect
 * to the log decay itself, is written when `dg_out` is not NULL.
 *
 * The states entering each token are recomputed forward from copies kept every 16 tokens
 * (storage only: the arithmetic of each step is the forward's).  `mutant` plants a known
 * mistake for the tests that check the pins catch it: 0 none, 1 drops the -Sd du term of
 * dk, 2 takes dalpha against the decayed state Sd instead of S, 3 omits diag(alpha) in dS.
 */
static double kda_oracle_sigmoid(double x) {
    if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
    const double e = exp(x);
    return e / (1.0 + e);
}

/* one forward token step in place: S <- Sn; u (V) is left in `u` */
static void kda_oracle_step(int K, int V, double* S, double* u, const double* alpha,
                            const double* kt, const double* vt, double bt) {
    for (int c = 0; c < K; ++c)
        for (int j = 0; j < V; ++j) S[(size_t)c * V + j] *= alpha[c];
    for (int j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int c = 0; c < K; ++c) acc += S[(size_t)c * V + j] * kt[c];
        u[j] = vt[j] - acc;
    }
    for (int c = 0; c < K; ++c)
        for (int j = 0; j < V; ++j) S[(size_t)c * V + j] += bt * kt[c] * u[j];
}

void kda_oracle_backward_range(int B, int H, int T, int K, int V,
                               const double* q, const double* k, const double* v,
                               const double* z, const double* beta,
                               const double* A_log, const double* dt_bias, double scale,
                               const double* h0, const double* d_o, const double* dhT,
                               double* dq, double* dk, double* dv, double* dz, double* dg_out,
                               double* dbeta, double* dA_part, double* ddt_part, double* dh0,
                               int mutant, int bh_begin, int bh_end) {
    (void)B;
    const int L = 16;
    const int nck = (T + L - 1) / L;
    const size_t KV = (size_t)K * V;
    double* ck = (double*)malloc(sizeof(double) * KV * (size_t)(nck > 0 ? nck : 1));
    double* blk = (double*)malloc(sizeof(double) * KV * (size_t)(L + 1));
    double* S = (double*)malloc(sizeof(double) * KV);
    double* Sd = (double*)malloc(sizeof(double) * KV);
    double* dS = (double*)malloc(sizeof(double) * KV);
    double* u = (double*)malloc(sizeof(double) * (size_t)V);
    double* du = (double*)malloc(sizeof(double) * (size_t)V);
    double* g = (double*)malloc(sizeof(double) * (size_t)T * K);
    double* sg = (double*)malloc(sizeof(double) * (size_t)T * K);
    double* alpha = (double*)malloc(sizeof(double) * (size_t)T * K);
    for (int bh = bh_begin; bh < bh_end; ++bh) {
        const int h = bh % H;
        const double mult = exp(A_log[h]);
        const double* qb = q + (size_t)bh * T * K;
        const double* kb = k + (size_t)bh * T * K;
        const double* vb = v + (size_t)bh * T * V;
        const double* zb = z + (size_t)bh * T * K;
        const double* bb = beta + (size_t)bh * T;
        const double* ob = d_o + (size_t)bh * T * V;
        /* gate, alpha and the sigmoid of the gate's argument */
        for (int t = 0; t < T; ++t)
            for (int c = 0; c < K; ++c) {
                const double x = zb[(size_t)t * K + c] + dt_bias[(size_t)h * K + c];
                g[(size_t)t * K + c] = -(mult * kda_oracle_softplus(x));
                sg[(size_t)t * K + c] = kda_oracle_sigmoid(x);
                alpha[(size_t)t * K + c] = exp(g[(size_t)t * K + c]);
            }
        /* forward: the state entering tokens 0, L, 2L, ... */
        if (h0) memcpy(S, h0 + (size_t)bh * KV, sizeof(double) * KV);
        else memset(S, 0, sizeof(double) * KV);
        for (int t = 0; t < T; ++t) {
            if (t % L == 0) memcpy(ck + (size_t)(t / L) * KV, S, sizeof(double) * KV);
            kda_oracle_step(K, V, S, u, alpha + (size_t)t * K, kb + (size_t)t * K,
                            vb + (size_t)t * V, bb[t]);
        }
        /* reverse */
        if (dhT) memcpy(dS, dhT + (size_t)bh * KV, sizeof(double) * KV);
        else memset(dS, 0, sizeof(double) * KV);
        double dA = 0.0;
        double* ddt = ddt_part + (size_t)bh * K;
        for (int c = 0; c < K; ++c) ddt[c] = 0.0;
        for (int n = nck - 1; n >= 0; --n) {
            const int t0 = n * L, t1 = (t0 + L < T) ? t0 + L : T;
            /* blk[i] = state entering token t0 + i, i = 0 .. t1 - t0 */
            memcpy(blk, ck + (size_t)n * KV, sizeof(double) * KV);
            for (int t = t0; t < t1; ++t) {
                memcpy(blk + (size_t)(t - t0 + 1) * KV, blk + (size_t)(t - t0) * KV,
                       sizeof(double) * KV);
                kda_oracle_step(K, V, blk + (size_t)(t - t0 + 1) * KV, u, alpha + (size_t)t * K,
                                kb + (size_t)t * K, vb + (size_t)t * V, bb[t]);
            }
            for (int t = t1 - 1; t >= t0; --t) {
                const double* Sp = blk + (size_t)(t - t0) * KV;     /* entering token t */
                const double* Sn = blk + (size_t)(t - t0 + 1) * KV; /* after token t */
                const double* kt = kb + (size_t)t * K;
                const double* qt = qb + (size_t)t * K;
                const double* dot = ob + (size_t)t * V;
                const double* at = alpha + (size_t)t * K;
                const double bt = bb[t];
                /* Sd and u again (the forward's own steps) */
                for (int c = 0; c < K; ++c)
                    for (int j = 0; j < V; ++j) Sd[(size_t)c * V + j] = Sp[(size_t)c * V + j] * at[c];
                for (int j = 0; j < V; ++j) {
                    double acc = 0.0;
                    for (int c = 0; c < K; ++c) acc += Sd[(size_t)c * V + j] * kt[c];
                    u[j] = vb[(size_t)t * V + j] - acc;
                }
                /* o_t = Sn^T (scale q_t) */
                for (int c = 0; c < K; ++c) {
                    double acc = 0.0;
                    for (int j = 0; j < V; ++j) {
                        dS[(size_t)c * V + j] += scale * qt[c] * dot[j];
                        acc += Sn[(size_t)c * V + j] * dot[j];
                    }
                    dq[((size_t)bh * T + t) * K + c] = scale * acc;
                }
                /* Sn = Sd + beta_t k_t u^T */
                double db = 0.0;
                for (int j = 0; j < V; ++j) {
                    double acc = 0.0;
                    for (int c = 0; c < K; ++c) acc += kt[c] * dS[(size_t)c * V + j];
                    du[j] = bt * acc;
                    db += acc * u[j];
                }
                dbeta[(size_t)bh * T + t] = db;
                for (int c = 0; c < K; ++c) {
                    double a1 = 0.0, a2 = 0.0;
                    for (int j = 0; j < V; ++j) {
                        a1 += dS[(size_t)c * V + j] * u[j];
                        a2 += Sd[(size_t)c * V + j] * du[j];
                    }
                    dk[((size_t)bh * T + t) * K + c] = bt * a1 - (mutant == 1 ? 0.0 : a2);
                }
                /* u = v_t - Sd^T k_t */
                for (int j = 0; j < V; ++j) dv[((size_t)bh * T + t) * V + j] = du[j];
                for (int c = 0; c < K; ++c)
                    for (int j = 0; j < V; ++j) dS[(size_t)c * V + j] -= kt[c] * du[j];
                /* Sd = diag(alpha) S, alpha = exp(g), gate */
                for (int c = 0; c < K; ++c) {
                    const double* Sa = (mutant == 2) ? Sd : Sp;
                    double dal = 0.0;
                    for (int j = 0; j < V; ++j) dal += Sa[(size_t)c * V + j] * dS[(size_t)c * V + j];
                    if (mutant != 3)
                        for (int j = 0; j < V; ++j) dS[(size_t)c * V + j] *= at[c];
                    const size_t gi = (size_t)t * K + c;
                    const double dg = at[c] * dal;
                    const double dzc = dg * (-mult) * sg[gi];
                    dz[((size_t)bh * T + t) * K + c] = dzc;
                    if (dg_out) dg_out[((size_t)bh * T + t) * K + c] = dg;
                    ddt[c] += dzc;
                    dA += dg * g[gi];
                }
            }
        }
        dA_part[bh] = dA;
        if (dh0) memcpy(dh0 + (size_t)bh * KV, dS, sizeof(double) * KV);
    }
    free(ck); free(blk); free(S); free(Sd); free(dS); free(u); free(du);
    free(g); free(sg); free(alpha);
}
