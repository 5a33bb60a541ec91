/*
 * Plain fp64 CPU oracle for the per-token recurrent-state update of
 * linear-attention decoding: Gated DeltaNet (GDN), Kimi Delta Attention (KDA)
 * and RWKV6.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header or constant with the CUDA
 * library.  Every function is the eager definition, written out step by step,
 * with no blocking, fusion or reordering: one (batch, head) pair at a time,
 * one token at a time.
 *
 * Sources.  The DeltaLog page ("DeltaLog: Deferred Materialization of Recurrent
 * States for Linear Attention Decoding", section "Problem: the state-update
 * tax") describes eager decoding: every token rewrites the whole d_k x d_v
 * state.  Its "Kernel implementation" section names the three operators and
 * what distinguishes them (GDN: one scalar decay per head plus the delta-rule
 * correction; KDA: one decay per key channel plus the delta rule; RWKV6: one
 * decay per key channel and raw-value updates, no delta rule).  The pages print
 * no formulas; the update rules below are the ones the decode workloads state:
 *
 *   GDN   u_t = beta_t (v_t - alpha_t S_{t-1} k_t),  S_t = alpha_t S_{t-1} + u_t k_t^T,
 *         o_t = scale * S_t q_t,  alpha_t = exp(g_t)
 *   KDA   S_t = S_{t-1} Diag(alpha_t) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *         o_t = scale * S_t q_t,  alpha_t = exp(g_t) per key channel
 *   RWKV6 (key-major form of the workload)  S_t = Diag(w_t) S_{t-1} + k_t v_t^T,
 *         o_t = r_t^T (S_{t-1} + Diag(bonus) k_t v_t^T),  w_t = exp(g_t)
 *
 * Layout.  The state is stored value-major, S[dv][dk] (row = value index),
 * which is what the products S k, u k^T and S q in the GDN rule require.  The
 * RWKV6 rule is written key-major on the pages; oracle_rwkv6 applies it to the
 * transposed (value-major) state and oracle_rwkv6_keymajor applies it exactly
 * as written; a test checks that the two agree.
 *
 * Array layouts (all fp64, C order):
 *   S0, S_final          [BH][dv][dk]
 *   q, k (r for RWKV6)   [T][BH][dk]
 *   v                    [T][BH][dv]
 *   g                    [T][BH]      (GDN)   or [T][BH][dk] (KDA, RWKV6)
 *   beta                 [T][BH]      (GDN, KDA)
 *   bonus                [BH][dk]     (RWKV6)
 *   o                    [T][BH][dv]
 *   S_snap               [n_snap][BH][dv][dk]: state after step snap_t[i]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static void snap_state(const double *S, int64_t bh, int64_t BH, int dk, int dv,
                       int64_t t, int n_snap, const int64_t *snap_t, double *S_snap) {
    for (int i = 0; i < n_snap; ++i) {
        if (snap_t[i] == t) {
            memcpy(S_snap + ((int64_t)i * BH + bh) * dv * dk, S,
                   sizeof(double) * (size_t)dv * dk);
        }
    }
}

/* Gated DeltaNet, eager: one rank-1 delta-rule update of the whole state per
 * token, followed by the read-out with the updated state. */
void oracle_gdn(int64_t BH, int64_t T, int dk, int dv, double scale,
                const double *S0, const double *q, const double *k,
                const double *v, const double *g, const double *beta,
                double *o, double *S_final,
                int n_snap, const int64_t *snap_t, double *S_snap) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *S = (double *)malloc(sizeof(double) * (size_t)dv * dk);
        double *Sk = (double *)malloc(sizeof(double) * (size_t)dv);
        double *u = (double *)malloc(sizeof(double) * (size_t)dv);
        memcpy(S, S0 + bh * dv * dk, sizeof(double) * (size_t)dv * dk);
        for (int64_t t = 0; t < T; ++t) {
            const double *qt = q + (t * BH + bh) * dk;
            const double *kt = k + (t * BH + bh) * dk;
            const double *vt = v + (t * BH + bh) * dv;
            const double alpha = exp(g[t * BH + bh]);
            const double b = beta[t * BH + bh];
            /* S_{t-1} k_t */
            for (int r = 0; r < dv; ++r) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += S[r * dk + i] * kt[i];
                Sk[r] = acc;
            }
            /* u_t = beta_t (v_t - alpha_t S_{t-1} k_t) */
            for (int r = 0; r < dv; ++r) u[r] = b * (vt[r] - alpha * Sk[r]);
            /* S_t = alpha_t S_{t-1} + u_t k_t^T */
            for (int r = 0; r < dv; ++r)
                for (int i = 0; i < dk; ++i)
                    S[r * dk + i] = alpha * S[r * dk + i] + u[r] * kt[i];
            /* o_t = scale * S_t q_t */
            double *ot = o + (t * BH + bh) * dv;
            for (int r = 0; r < dv; ++r) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += S[r * dk + i] * qt[i];
                ot[r] = scale * acc;
            }
            if (n_snap > 0) snap_state(S, bh, BH, dk, dv, t, n_snap, snap_t, S_snap);
        }
        if (S_final) memcpy(S_final + bh * dv * dk, S, sizeof(double) * (size_t)dv * dk);
        free(S);
        free(Sk);
        free(u);
    }
}

/* Kimi Delta Attention, eager, literally as the rule is written: the d_k x d_k
 * transition P_t = Diag(alpha_t) (I - beta_t k_t k_t^T) is formed explicitly and
 * the state is multiplied by it, then beta_t v_t k_t^T is added.  (No use is
 * made of the rank-1 structure; that is what makes it an independent check of
 * any factorised implementation.) */
void oracle_kda(int64_t BH, int64_t T, int dk, int dv, double scale,
                const double *S0, const double *q, const double *k,
                const double *v, const double *g, const double *beta,
                double *o, double *S_final,
                int n_snap, const int64_t *snap_t, double *S_snap) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *S = (double *)malloc(sizeof(double) * (size_t)dv * dk);
        double *Sn = (double *)malloc(sizeof(double) * (size_t)dv * dk);
        double *P = (double *)malloc(sizeof(double) * (size_t)dk * dk);
        memcpy(S, S0 + bh * dv * dk, sizeof(double) * (size_t)dv * dk);
        for (int64_t t = 0; t < T; ++t) {
            const double *qt = q + (t * BH + bh) * dk;
            const double *kt = k + (t * BH + bh) * dk;
            const double *vt = v + (t * BH + bh) * dv;
            const double *gt = g + (t * BH + bh) * dk;
            const double b = beta[t * BH + bh];
            /* P = Diag(alpha) (I - beta k k^T):  P[i][j] = alpha_i (delta_ij - beta k_i k_j) */
            for (int i = 0; i < dk; ++i) {
                const double ai = exp(gt[i]);
                for (int j = 0; j < dk; ++j)
                    P[i * dk + j] = ai * ((i == j ? 1.0 : 0.0) - b * kt[i] * kt[j]);
            }
            /* S_t = S_{t-1} P + beta v k^T */
            for (int r = 0; r < dv; ++r) {
                for (int j = 0; j < dk; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; ++i) acc += S[r * dk + i] * P[i * dk + j];
                    Sn[r * dk + j] = acc + b * vt[r] * kt[j];
                }
            }
            double *tmp = S; S = Sn; Sn = tmp;
            double *ot = o + (t * BH + bh) * dv;
            for (int r = 0; r < dv; ++r) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += S[r * dk + i] * qt[i];
                ot[r] = scale * acc;
            }
            if (n_snap > 0) snap_state(S, bh, BH, dk, dv, t, n_snap, snap_t, S_snap);
        }
        if (S_final) memcpy(S_final + bh * dv * dk, S, sizeof(double) * (size_t)dv * dk);
        free(S);
        free(Sn);
        free(P);
    }
}

/* RWKV6, eager, on the value-major state (the key-major rule transposed):
 *   o_t = scale * (S_{t-1} r_t + (sum_i r_i bonus_i k_i) v_t)
 *   S_t = S_{t-1} Diag(w_t) + v_t k_t^T                                   */
void oracle_rwkv6(int64_t BH, int64_t T, int dk, int dv, double scale,
                  const double *S0, const double *r, const double *k,
                  const double *v, const double *g, const double *bonus,
                  double *o, double *S_final,
                  int n_snap, const int64_t *snap_t, double *S_snap) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *S = (double *)malloc(sizeof(double) * (size_t)dv * dk);
        memcpy(S, S0 + bh * dv * dk, sizeof(double) * (size_t)dv * dk);
        const double *ub = bonus + bh * dk;
        for (int64_t t = 0; t < T; ++t) {
            const double *rt = r + (t * BH + bh) * dk;
            const double *kt = k + (t * BH + bh) * dk;
            const double *vt = v + (t * BH + bh) * dv;
            const double *gt = g + (t * BH + bh) * dk;
            double cb = 0.0;
            for (int i = 0; i < dk; ++i) cb += rt[i] * ub[i] * kt[i];
            double *ot = o + (t * BH + bh) * dv;
            for (int c = 0; c < dv; ++c) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += S[c * dk + i] * rt[i];
                ot[c] = scale * (acc + cb * vt[c]);
            }
            for (int c = 0; c < dv; ++c)
                for (int i = 0; i < dk; ++i)
                    S[c * dk + i] = S[c * dk + i] * exp(gt[i]) + vt[c] * kt[i];
            if (n_snap > 0) snap_state(S, bh, BH, dk, dv, t, n_snap, snap_t, S_snap);
        }
        if (S_final) memcpy(S_final + bh * dv * dk, S, sizeof(double) * (size_t)dv * dk);
        free(S);
    }
}

/* RWKV6 exactly as the workload writes it, on a key-major state Z[dk][dv]:
 *   o_t = scale * r_t^T (Z_{t-1} + Diag(bonus) k_t v_t^T)
 *   Z_t = Diag(w_t) Z_{t-1} + k_t v_t^T
 * S0 and S_final are given value-major ([dv][dk]) so that results compare
 * directly with oracle_rwkv6; the transposition happens here, on entry and exit. */
void oracle_rwkv6_keymajor(int64_t BH, int64_t T, int dk, int dv, double scale,
                           const double *S0, const double *r, const double *k,
                           const double *v, const double *g, const double *bonus,
                           double *o, double *S_final) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *Z = (double *)malloc(sizeof(double) * (size_t)dk * dv);
        for (int c = 0; c < dv; ++c)
            for (int i = 0; i < dk; ++i) Z[i * dv + c] = S0[bh * dv * dk + c * dk + i];
        const double *ub = bonus + bh * dk;
        for (int64_t t = 0; t < T; ++t) {
            const double *rt = r + (t * BH + bh) * dk;
            const double *kt = k + (t * BH + bh) * dk;
            const double *vt = v + (t * BH + bh) * dv;
            const double *gt = g + (t * BH + bh) * dk;
            double *ot = o + (t * BH + bh) * dv;
            for (int c = 0; c < dv; ++c) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i)
                    acc += rt[i] * (Z[i * dv + c] + ub[i] * kt[i] * vt[c]);
                ot[c] = scale * acc;
            }
            for (int i = 0; i < dk; ++i) {
                const double wi = exp(gt[i]);
                for (int c = 0; c < dv; ++c) Z[i * dv + c] = wi * Z[i * dv + c] + kt[i] * vt[c];
            }
        }
        if (S_final)
            for (int c = 0; c < dv; ++c)
                for (int i = 0; i < dk; ++i) S_final[bh * dv * dk + c * dk + i] = Z[i * dv + c];
        free(Z);
    }
}
