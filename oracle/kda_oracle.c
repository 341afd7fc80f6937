/*
 * kda_oracle.c -- fp64 CPU oracle for the Kimi Delta Attention recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * definition that the CUDA library is checked against.  Only the tests, the
 * smoke check and the CPU-baseline leg of the benchmark may load it; the
 * library itself never calls it and has no CPU fallback.
 *
 * It shares no code, header or constant with the CUDA path.  It is a plain
 * token-by-token loop in double precision, one (sequence, head) at a time,
 * with OpenMP over the independent (sequence, head) pairs.
 *
 * What it computes (all citations are to the source pages):
 *
 *   S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     -- "Understanding Kimi Delta Attention" (pyshine), section
 *        "The KDA Recurrence: Scalar Gate vs Channel-wise Gate", KDA equation.
 *   S is dk x dv; Diag(alpha_t) scales the ROWS of S, one row per key channel
 *     -- "kimi delta attn from first principles" (aryagxr), section "KDA",
 *        step 1 ("each row of the memory matrix S gets its own decay factor").
 *   o_t = S_t^T q_t, read from the UPDATED state with the query
 *     -- same page, section "KDA" (output gate paragraph, o_t = S_t^T q_t).
 *   alpha_t = exp(log_alpha_t), natural log, one value per key channel.
 *   Each packed sequence starts from its own S0 (zeros if none is given) and
 *   returns its final state -- "Kimi Delta Attention (KDA)" (codewithdark),
 *   section "KV Caching Challenges & vLLM Contribution" (states stored at
 *   prefix boundaries).
 *
 * The update is evaluated literally as written: decay the rows, then apply
 * the rank-1 erase (I - beta k k^T) to the decayed state, then add the
 * rank-1 write.  It is deliberately NOT the factorised "u = beta(v - S'^T k)"
 * form the GPU decode kernel uses, so that the two are independent.
 *
 * Inputs are the exact values the GPU consumed (bf16/fp32 widened to float32
 * by the caller, which is exact), read as float and widened to double here.
 *
 * Parity pins (tests/test_oracle_pins.py): brute-force matrix products on
 * T <= 8, the Gated DeltaNet reduction, identity and pure-decay closed forms,
 * erase-then-write, the orthonormal-key linear-attention closed form, the
 * DeltaNet error-correction form, a hand-worked d = 2 example, and the
 * split / varlen / decode composition invariants.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* One token of the recurrence on a dk x dv row-major double state S.
 * Sd, kS: caller-provided scratch of dk*dv and dv doubles. */
static void kda_token(double *S, double *Sd, double *kS, int dk, int dv,
                      const float *q, const float *k, const float *v,
                      const float *log_alpha, double beta, double *o) {
    /* Diag(alpha_t) S_{t-1}: row r (key channel r) scaled by exp(log_alpha[r]) */
    for (int r = 0; r < dk; ++r) {
        double a = exp((double)log_alpha[r]);
        for (int j = 0; j < dv; ++j) Sd[(size_t)r * dv + j] = a * S[(size_t)r * dv + j];
    }
    /* k^T (Diag(alpha) S): the row vector the erase term removes */
    for (int j = 0; j < dv; ++j) kS[j] = 0.0;
    for (int r = 0; r < dk; ++r) {
        double kr = (double)k[r];
        for (int j = 0; j < dv; ++j) kS[j] += kr * Sd[(size_t)r * dv + j];
    }
    /* (I - beta k k^T) Sd + beta k v^T */
    for (int r = 0; r < dk; ++r) {
        double bk = beta * (double)k[r];
        for (int j = 0; j < dv; ++j)
            S[(size_t)r * dv + j] = Sd[(size_t)r * dv + j] - bk * kS[j] + bk * (double)v[j];
    }
    /* o_t = S_t^T q_t */
    if (o) {
        for (int j = 0; j < dv; ++j) o[j] = 0.0;
        for (int r = 0; r < dk; ++r) {
            double qr = (double)q[r];
            for (int j = 0; j < dv; ++j) o[j] += qr * S[(size_t)r * dv + j];
        }
    }
}

/*
 * Prefill over packed variable-length sequences.
 *   q, k, log_alpha : [T_total, H, dk] float     v : [T_total, H, dv] float
 *   beta            : [T_total, H] float
 *   S0              : [N, H, dk, dv] float or NULL (zeros)
 *   cu_seqlens      : [N + 1] int32, cu_seqlens[0] = 0, non-decreasing
 *   o               : [T_total, H, dv] double (out)
 *   S_final         : [N, H, dk, dv] double (out) or NULL
 * Returns 0, or -1 on a malformed cu_seqlens / allocation failure.
 */
int oracle_kda_prefill(const float *q, const float *k, const float *v,
                       const float *log_alpha, const float *beta, const float *S0,
                       const int32_t *cu_seqlens, int32_t N, int32_t H,
                       int32_t dk, int32_t dv, double *o, double *S_final,
                       int32_t nthreads) {
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
    if (N > 0 && cu_seqlens[0] != 0) return -1;
    for (int n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    int err = 0;
    long units = (long)N * H;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
#endif
    for (long u = 0; u < units; ++u) {
        int n = (int)(u / H), h = (int)(u % H);
        double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
        double *Sd = (double *)malloc(sizeof(double) * (size_t)dk * dv);
        double *kS = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!S || !Sd || !kS) {
            err |= 1;
        } else {
            size_t sidx = ((size_t)n * H + h) * (size_t)dk * dv;
            for (size_t e = 0; e < (size_t)dk * dv; ++e) S[e] = S0 ? (double)S0[sidx + e] : 0.0;
            for (int64_t t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
                size_t th = (size_t)t * H + h;
                kda_token(S, Sd, kS, dk, dv, q + th * dk, k + th * dk, v + th * dv,
                          log_alpha + th * dk, (double)beta[th], o + th * dv);
            }
            if (S_final) memcpy(S_final + sidx, S, sizeof(double) * (size_t)dk * dv);
        }
        free(S);
        free(Sd);
        free(kS);
    }
    return err ? -1 : 0;
}

/*
 * One decode step: the same token update applied once to each of N
 * sequences, on the state slot state_indices[n] (identity when NULL).
 *   q, k, log_alpha : [N, H, dk] float     v : [N, H, dv] float
 *   beta            : [N, H] float
 *   S               : [num_slots, H, dk, dv] double, updated in place
 *   o               : [N, H, dv] double (out)
 * Returns 0, or -1 when a slot index is out of range.
 */
int oracle_kda_decode_step(const float *q, const float *k, const float *v,
                           const float *log_alpha, const float *beta, double *S,
                           int32_t num_slots, const int32_t *state_indices,
                           int32_t N, int32_t H, int32_t dk, int32_t dv, double *o,
                           int32_t nthreads) {
    for (int n = 0; n < N; ++n) {
        int32_t slot = state_indices ? state_indices[n] : n;
        if (slot < 0 || slot >= num_slots) return -1;
    }
    int err = 0;
    long units = (long)N * H;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static) reduction(| : err)
#endif
    for (long u = 0; u < units; ++u) {
        int n = (int)(u / H), h = (int)(u % H);
        int32_t slot = state_indices ? state_indices[n] : n;
        double *Sd = (double *)malloc(sizeof(double) * (size_t)dk * dv);
        double *kS = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!Sd || !kS) {
            err |= 1;
        } else {
            size_t th = (size_t)n * H + h;
            double *Sslot = S + ((size_t)slot * H + h) * (size_t)dk * dv;
            kda_token(Sslot, Sd, kS, dk, dv, q + th * dk, k + th * dk, v + th * dv,
                      log_alpha + th * dk, (double)beta[th], o + th * dv);
        }
        free(Sd);
        free(kS);
    }
    return err ? -1 : 0;
}

/* Threads OpenMP will use for a given request (for reporting). */
int32_t oracle_num_threads(int32_t requested) {
#ifdef _OPENMP
    if (requested > 0) return requested;
    return (int32_t)omp_get_max_threads();
#else
    (void)requested;
    return 1;
#endif
}


/*
 * Reverse-mode gradient of the prefill above, for a loss
 *   L = sum_t <o_t, dO_t> + sum_n <S_final_n, dS_final_n>,
 * taken through the same literal update, step by step in reverse:
 *   S_t = Sd - beta k (Sd^T k)^T + beta k v^T,  Sd = Diag(exp(log_alpha)) S_{t-1},
 *   o_t = S_t^T q.
 * The adjoint of S (Sbar, dk x dv) starts at dS_final and is carried back to
 * dS0.  Forward states are kept for every token of the sequence (test sizes).
 *   dO, dS_final : double, shapes as o and S_final (dS_final may be NULL = 0)
 *   dq, dk, dlog_alpha : [T_total, H, dk] double (out); dv : [T_total, H, dv]
 *   dbeta : [T_total, H] double (out);  dS0 : [N, H, dk, dv] double or NULL
 * Returns 0, or -1 on a malformed cu_seqlens / allocation failure.
 */
int oracle_kda_prefill_backward(const float *q, const float *k, const float *v,
                                const float *log_alpha, const float *beta, const float *S0,
                                const int32_t *cu_seqlens, int32_t N, int32_t H,
                                int32_t dk, int32_t dv, const double *dO, const double *dS_final,
                                double *dq, double *dkk, double *dvv, double *dla, double *dbeta,
                                double *dS0, int32_t nthreads) {
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
    if (N > 0 && cu_seqlens[0] != 0) return -1;
    for (int n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    int err = 0;
    long units = (long)N * H;
    const size_t M = (size_t)dk * dv;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
#endif
    for (long u = 0; u < units; ++u) {
        int n = (int)(u / H), h = (int)(u % H);
        int64_t t0 = cu_seqlens[n], L = cu_seqlens[n + 1] - t0;
        double *Sall = (double *)malloc(sizeof(double) * M * (size_t)(L + 1)); /* S_{-1} .. S_{L-1} */
        double *Sd = (double *)malloc(sizeof(double) * M);
        double *Sb = (double *)malloc(sizeof(double) * M);  /* adjoint of S_t */
        double *Sdb = (double *)malloc(sizeof(double) * M); /* adjoint of Sd */
        double *kS = (double *)malloc(sizeof(double) * dv);
        double *kSb = (double *)malloc(sizeof(double) * dv);
        if (!Sall || !Sd || !Sb || !Sdb || !kS || !kSb) {
            err |= 1;
        } else {
            size_t sidx = ((size_t)n * H + h) * M;
            for (size_t e = 0; e < M; ++e) Sall[e] = S0 ? (double)S0[sidx + e] : 0.0;
            /* forward, keeping every state */
            for (int64_t i = 0; i < L; ++i) {
                size_t th = (size_t)(t0 + i) * H + h;
                double *Sp = Sall + (size_t)i * M, *Sn = Sall + (size_t)(i + 1) * M;
                memcpy(Sn, Sp, sizeof(double) * M);
                kda_token(Sn, Sd, kS, dk, dv, q + th * dk, k + th * dk, v + th * dv, log_alpha + th * dk,
                          (double)beta[th], NULL);
            }
            for (size_t e = 0; e < M; ++e) Sb[e] = dS_final ? dS_final[sidx + e] : 0.0;
            /* reverse */
            for (int64_t i = L - 1; i >= 0; --i) {
                size_t th = (size_t)(t0 + i) * H + h;
                const float *qt = q + th * dk, *kt = k + th * dk, *vt = v + th * dv, *lat = log_alpha + th * dk;
                const double *ob = dO + th * dv;
                const double b = (double)beta[th];
                const double *Sp = Sall + (size_t)i * M, *St = Sall + (size_t)(i + 1) * M;
                /* recompute Sd and kS = Sd^T k of this token */
                for (int r = 0; r < dk; ++r) {
                    double a = exp((double)lat[r]);
                    for (int j = 0; j < dv; ++j) Sd[(size_t)r * dv + j] = a * Sp[(size_t)r * dv + j];
                }
                for (int j = 0; j < dv; ++j) kS[j] = 0.0;
                for (int r = 0; r < dk; ++r)
                    for (int j = 0; j < dv; ++j) kS[j] += (double)kt[r] * Sd[(size_t)r * dv + j];
                /* o = S_t^T q: Sbar += q obar^T, qbar = S_t obar */
                for (int r = 0; r < dk; ++r) {
                    double acc = 0.0;
                    for (int j = 0; j < dv; ++j) {
                        Sb[(size_t)r * dv + j] += (double)qt[r] * ob[j];
                        acc += St[(size_t)r * dv + j] * ob[j];
                    }
                    dq[th * dk + r] = acc;
                }
                /* S_t = Sd - b k kS^T + b k v^T */
                double betabar = 0.0;
                for (int r = 0; r < dk; ++r) {
                    double acc = 0.0;
                    for (int j = 0; j < dv; ++j) acc += Sb[(size_t)r * dv + j] * ((double)vt[j] - kS[j]);
                    dkk[th * dk + r] = b * acc;          /* from the k of the outer products */
                    betabar += (double)kt[r] * acc;
                }
                dbeta[th] = betabar;
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int r = 0; r < dk; ++r) acc += Sb[(size_t)r * dv + j] * (double)kt[r];
                    kSb[j] = -b * acc;                   /* adjoint of kS */
                    dvv[th * dv + j] = b * acc;
                }
                /* Sd: direct term plus kS = Sd^T k */
                for (int r = 0; r < dk; ++r) {
                    double acc = 0.0;
                    for (int j = 0; j < dv; ++j) {
                        Sdb[(size_t)r * dv + j] = Sb[(size_t)r * dv + j] + (double)kt[r] * kSb[j];
                        acc += Sd[(size_t)r * dv + j] * kSb[j];
                    }
                    dkk[th * dk + r] += acc;
                }
                /* Sd = Diag(exp(log_alpha)) S_{t-1} */
                for (int r = 0; r < dk; ++r) {
                    double a = exp((double)lat[r]), acc = 0.0;
                    for (int j = 0; j < dv; ++j) {
                        acc += Sdb[(size_t)r * dv + j] * Sd[(size_t)r * dv + j];
                        Sb[(size_t)r * dv + j] = a * Sdb[(size_t)r * dv + j];
                    }
                    dla[th * dk + r] = acc;
                }
            }
            if (dS0) memcpy(dS0 + sidx, Sb, sizeof(double) * M);
        }
        free(Sall);
        free(Sd);
        free(Sb);
        free(Sdb);
        free(kS);
        free(kSb);
    }
    return err ? -1 : 0;
}
