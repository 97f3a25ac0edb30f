/*
 * la_oracle.c -- plain, slow fp64 CPU oracle for causal linear attention with
 * the feature map phi(x) = elu(x) + 1.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (page title, section):
 *   [KAT]  "Transformers은 RNN이다 — 선형 어텐션으로 빠른 Autoregressive
 *          Transformer 만들기" (irregular6612 blog digest), sections "Methods"
 *          and "핵심 구성요소" items 1-4.
 *   [REV]  "[논문 리뷰] Transformers are RNNs: Fast Autoregressive Transformers
 *          with Linear Attention" (velog review), sections 3.2 Linearized
 *          Attention, 3.3 Feature Maps, 3.4 Causal Masking, 3.5 Gradient
 *          Computation, 3.6 Transformers and RNNs.
 *   [WIKI] "선형 어텐션" (itwiki), sections "결합 법칙으로 순서 바꾸기",
 *          "인과 마스킹과 순환형", "계산 형태 비교" (table of forms) and
 *          "구현" (the parallel / recurrent / chunked forms).
 *
 * Layout (all row-major, fp64): q,k [BH][N][Dk], v,o,dO [BH][N][Dv],
 * decode state S [BH][Dk][Dv], z [BH][Dk].  BH = B*H heads are independent.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - ELU uses alpha = 1 (the pages never state alpha; the default ELU).
 *   - No 1/sqrt(D) scale and no epsilon in the denominator (neither appears in
 *     the linear forms).
 *   - The causal sum includes the diagonal, j <= i.
 *   - The gradient formulas are lost from [REV] 3.5; the backward here is the
 *     chain rule applied to the definition (bwd_direct) and its cumulative-sum
 *     rewriting (bwd_recurrent).
 *
 * Parity pins (tests/test_oracle.py): direct == recurrence == chunked; N=1,
 * constant V, identical keys, Dk=1, non-causal == causal at i=N, convex hull,
 * affine covariance, decode vs numpy K^T V, finite differences for every
 * backward (the non-causal one in its direct and its associative form),
 * gradient invariants, and phi against the library ELU.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define IDX3(h, i, d, n, dd) (((size_t)(h) * (size_t)(n) + (size_t)(i)) * (size_t)(dd) + (size_t)(d))

/*
 * phi(x) = elu(x) + 1 with alpha = 1, strictly positive.  [KAT] 핵심 구성요소 1;
 * [REV] 3.3; [WIKI] 결합 법칙.  For x > 0, elu(x) = x so phi(x) = x + 1.  For
 * x <= 0, elu(x) = exp(x) - 1 so phi(x) = exp(x) exactly; it is evaluated as
 * exp(x) because (exp(x) - 1) + 1 cancels for large negative x.
 */
static double phi(double x) { return x > 0.0 ? x + 1.0 : exp(x); }

/* d phi / dx: 1 for x > 0, exp(x) otherwise (continuous at 0 with value 1). */
static double dphi(double x) { return x > 0.0 ? 1.0 : exp(x); }

void oracle_phi(const double* x, double* y, long n) {
    for (long i = 0; i < n; ++i) y[i] = phi(x[i]);
}

void oracle_dphi(const double* x, double* y, long n) {
    for (long i = 0; i < n; ++i) y[i] = dphi(x[i]);
}

/* phi applied to one head's [N][D] slice into a fresh buffer. */
static double* phi_slice(const double* x, int h, int N, int D) {
    double* y = (double*)malloc(sizeof(double) * (size_t)N * (size_t)D);
    const double* src = x + IDX3(h, 0, 0, N, D);
    for (size_t t = 0; t < (size_t)N * (size_t)D; ++t) y[t] = phi(src[t]);
    return y;
}

static double dot(const double* a, const double* b, int n) {
    double s = 0.0;
    for (int d = 0; d < n; ++d) s += a[d] * b[d];
    return s;
}

/*
 * Generalised attention written out directly, O(N^2) per head:
 *   o_i = sum_{j in J(i)} sim(q_i,k_j) v_j / sum_{j in J(i)} sim(q_i,k_j),
 *   sim(q,k) = phi(q)^T phi(k),
 * with J(i) = {j <= i} (causal) or all j (non-causal).
 * [KAT] Methods (generalised attention, kernel feature map); [WIKI] 결합 법칙
 * (first display); the parallel masked form of [WIKI] 구현.
 */
static void attention_direct(const double* q, const double* k, const double* v, double* o,
                             int BH, int N, int Dk, int Dv, int causal) {
#pragma omp parallel for schedule(dynamic)
    for (int h = 0; h < BH; ++h) {
        double* qt = phi_slice(q, h, N, Dk);
        double* kt = phi_slice(k, h, N, Dk);
        const double* vh = v + IDX3(h, 0, 0, N, Dv);
        double* num = (double*)malloc(sizeof(double) * (size_t)Dv);
        for (int i = 0; i < N; ++i) {
            int jend = causal ? i : N - 1;
            double den = 0.0;
            for (int m = 0; m < Dv; ++m) num[m] = 0.0;
            for (int j = 0; j <= jend; ++j) {
                double w = dot(qt + (size_t)i * Dk, kt + (size_t)j * Dk, Dk);
                den += w;
                for (int m = 0; m < Dv; ++m) num[m] += w * vh[(size_t)j * Dv + m];
            }
            double* oi = o + IDX3(h, i, 0, N, Dv);
            for (int m = 0; m < Dv; ++m) oi[m] = num[m] / den;
        }
        free(num);
        free(qt);
        free(kt);
    }
}

void oracle_causal_direct(const double* q, const double* k, const double* v, double* o,
                          int BH, int N, int Dk, int Dv) {
    attention_direct(q, k, v, o, BH, N, Dk, Dv, 1);
}

void oracle_noncausal_direct(const double* q, const double* k, const double* v, double* o,
                             int BH, int N, int Dk, int Dv) {
    attention_direct(q, k, v, o, BH, N, Dk, Dv, 0);
}

/*
 * Non-causal form by associativity: S = phi(K)^T V (Dk x Dv), z = phi(K)^T 1,
 * o_i = phi(q_i)^T S / phi(q_i)^T z.  [KAT] 핵심 구성요소 2; [REV] 3.2.
 */
void oracle_noncausal_assoc(const double* q, const double* k, const double* v, double* o,
                            int BH, int N, int Dk, int Dv) {
#pragma omp parallel for schedule(dynamic)
    for (int h = 0; h < BH; ++h) {
        double* S = (double*)calloc((size_t)Dk * (size_t)Dv, sizeof(double));
        double* z = (double*)calloc((size_t)Dk, sizeof(double));
        double* qt = (double*)malloc(sizeof(double) * (size_t)Dk);
        for (int j = 0; j < N; ++j) {
            const double* kj = k + IDX3(h, j, 0, N, Dk);
            const double* vj = v + IDX3(h, j, 0, N, Dv);
            for (int d = 0; d < Dk; ++d) {
                double kt = phi(kj[d]);
                z[d] += kt;
                for (int m = 0; m < Dv; ++m) S[(size_t)d * Dv + m] += kt * vj[m];
            }
        }
        for (int i = 0; i < N; ++i) {
            const double* qi = q + IDX3(h, i, 0, N, Dk);
            for (int d = 0; d < Dk; ++d) qt[d] = phi(qi[d]);
            double den = dot(qt, z, Dk);
            double* oi = o + IDX3(h, i, 0, N, Dv);
            for (int m = 0; m < Dv; ++m) {
                double num = 0.0;
                for (int d = 0; d < Dk; ++d) num += qt[d] * S[(size_t)d * Dv + m];
                oi[m] = num / den;
            }
        }
        free(S);
        free(z);
        free(qt);
    }
}

/*
 * One recurrent step per head, state updated first and then read (j <= i):
 *   S <- S + phi(k) v^T,  z <- z + phi(k),  out = phi(q)^T S / phi(q)^T z.
 * [KAT] 핵심 구성요소 4 (RNN view); [REV] 3.6; [WIKI] 인과 마스킹과 순환형.
 * q,k [BH][Dk], v,out [BH][Dv], S [BH][Dk][Dv], z [BH][Dk]; S and z in place.
 */
void oracle_recurrent_step(const double* q, const double* k, const double* v,
                           double* S, double* z, double* out, int BH, int Dk, int Dv) {
    for (int h = 0; h < BH; ++h) {
        const double* qh = q + (size_t)h * Dk;
        const double* kh = k + (size_t)h * Dk;
        const double* vh = v + (size_t)h * Dv;
        double* Sh = S + (size_t)h * Dk * Dv;
        double* zh = z + (size_t)h * Dk;
        for (int d = 0; d < Dk; ++d) {
            double kt = phi(kh[d]);
            zh[d] += kt;
            for (int m = 0; m < Dv; ++m) Sh[(size_t)d * Dv + m] += kt * vh[m];
        }
        double den = 0.0;
        for (int d = 0; d < Dk; ++d) den += phi(qh[d]) * zh[d];
        for (int m = 0; m < Dv; ++m) {
            double num = 0.0;
            for (int d = 0; d < Dk; ++d) num += phi(qh[d]) * Sh[(size_t)d * Dv + m];
            out[(size_t)h * Dv + m] = num / den;
        }
    }
}

/*
 * Causal attention by the recurrence, O(N Dk Dv) per head: the step above run
 * from S = 0, z = 0 over i = 1..N.  [KAT] 핵심 구성요소 3-4; [WIKI] 구현
 * (recurrent form).
 */
void oracle_causal_recurrent(const double* q, const double* k, const double* v, double* o,
                             int BH, int N, int Dk, int Dv) {
#pragma omp parallel for schedule(dynamic)
    for (int h = 0; h < BH; ++h) {
        double* S = (double*)calloc((size_t)Dk * (size_t)Dv, sizeof(double));
        double* z = (double*)calloc((size_t)Dk, sizeof(double));
        for (int i = 0; i < N; ++i)
            oracle_recurrent_step(q + IDX3(h, i, 0, N, Dk), k + IDX3(h, i, 0, N, Dk),
                                  v + IDX3(h, i, 0, N, Dv), S, z, o + IDX3(h, i, 0, N, Dv),
                                  1, Dk, Dv);
        free(S);
        free(z);
    }
}

/*
 * Chunked form: inside a chunk of C positions the masked product
 * (phi(Q_c) phi(K_c)^T * tril) is formed explicitly; between chunks the state
 * (S, z) is carried.  A short last chunk is handled by its own length.
 * [WIKI] 계산 형태 비교 (chunked row) and 구현 (chunked form).
 */
void oracle_causal_chunked(const double* q, const double* k, const double* v, double* o,
                           int BH, int N, int Dk, int Dv, int C) {
#pragma omp parallel for schedule(dynamic)
    for (int h = 0; h < BH; ++h) {
        double* qt = phi_slice(q, h, N, Dk);
        double* kt = phi_slice(k, h, N, Dk);
        const double* vh = v + IDX3(h, 0, 0, N, Dv);
        double* S = (double*)calloc((size_t)Dk * (size_t)Dv, sizeof(double));
        double* z = (double*)calloc((size_t)Dk, sizeof(double));
        double* A = (double*)malloc(sizeof(double) * (size_t)C * (size_t)C);
        for (int s = 0; s < N; s += C) {
            int n = (N - s) < C ? (N - s) : C;
            /* intra = (Qc Kc^T) masked to its lower triangle incl. the diagonal */
            for (int a = 0; a < n; ++a)
                for (int b = 0; b < n; ++b)
                    A[(size_t)a * C + b] =
                        (b <= a) ? dot(qt + (size_t)(s + a) * Dk, kt + (size_t)(s + b) * Dk, Dk) : 0.0;
            for (int a = 0; a < n; ++a) {
                const double* qa = qt + (size_t)(s + a) * Dk;
                double den = dot(qa, z, Dk);
                for (int b = 0; b < n; ++b) den += A[(size_t)a * C + b];
                double* oa = o + IDX3(h, s + a, 0, N, Dv);
                for (int m = 0; m < Dv; ++m) {
                    double num = 0.0;
                    for (int d = 0; d < Dk; ++d) num += qa[d] * S[(size_t)d * Dv + m];
                    for (int b = 0; b < n; ++b) num += A[(size_t)a * C + b] * vh[(size_t)(s + b) * Dv + m];
                    oa[m] = num / den;
                }
            }
            /* state passed to the next chunk: S += Kc^T Vc, z += Kc^T 1 */
            for (int b = 0; b < n; ++b) {
                const double* kb = kt + (size_t)(s + b) * Dk;
                const double* vb = vh + (size_t)(s + b) * Dv;
                for (int d = 0; d < Dk; ++d) {
                    z[d] += kb[d];
                    for (int m = 0; m < Dv; ++m) S[(size_t)d * Dv + m] += kb[d] * vb[m];
                }
            }
        }
        free(A);
        free(S);
        free(z);
        free(qt);
        free(kt);
    }
}

/*
 * Backward of the causal form, direct O(N^2) version.  With
 * w_ij = phi(q_i)^T phi(k_j) (j <= i), den_i = sum_j w_ij and
 * o_i = sum_j w_ij v_j / den_i, the loss L = sum_i dO_i . o_i gives
 *   dL/dw_ij = dO_i . (v_j - o_i) / den_i,
 *   dL/dv_j  = sum_{i >= j} w_ij dO_i / den_i,
 *   dphi(q_i) = sum_{j <= i} (dL/dw_ij) phi(k_j),
 *   dphi(k_j) = sum_{i >= j} (dL/dw_ij) phi(q_i),
 * and dq = dphi(q) * phi'(q), dk = dphi(k) * phi'(k) elementwise.  This is
 * the chain rule applied to the definition; [REV] 3.5 states only that the
 * gradient is itself a cumulative sum (its formulas did not survive).
 */
void oracle_causal_bwd_direct(const double* q, const double* k, const double* v, const double* dO,
                              double* dq, double* dk, double* dv, int BH, int N, int Dk, int Dv) {
#pragma omp parallel for schedule(dynamic)
    for (int h = 0; h < BH; ++h) {
        double* qt = phi_slice(q, h, N, Dk);
        double* kt = phi_slice(k, h, N, Dk);
        const double* vh = v + IDX3(h, 0, 0, N, Dv);
        const double* dOh = dO + IDX3(h, 0, 0, N, Dv);
        double* den = (double*)malloc(sizeof(double) * (size_t)N);
        double* oh = (double*)malloc(sizeof(double) * (size_t)N * Dv);
        double* dqt = (double*)calloc((size_t)N * Dk, sizeof(double));
        double* dkt = (double*)calloc((size_t)N * Dk, sizeof(double));
        double* dvh = dv + IDX3(h, 0, 0, N, Dv);
        for (size_t t = 0; t < (size_t)N * Dv; ++t) dvh[t] = 0.0;
        /* forward quantities */
        for (int i = 0; i < N; ++i) {
            double dsum = 0.0;
            for (int m = 0; m < Dv; ++m) oh[(size_t)i * Dv + m] = 0.0;
            for (int j = 0; j <= i; ++j) {
                double w = dot(qt + (size_t)i * Dk, kt + (size_t)j * Dk, Dk);
                dsum += w;
                for (int m = 0; m < Dv; ++m) oh[(size_t)i * Dv + m] += w * vh[(size_t)j * Dv + m];
            }
            den[i] = dsum;
            for (int m = 0; m < Dv; ++m) oh[(size_t)i * Dv + m] /= dsum;
        }
        /* pairwise gradient terms */
        for (int i = 0; i < N; ++i) {
            const double* dOi = dOh + (size_t)i * Dv;
            const double* oi = oh + (size_t)i * Dv;
            for (int j = 0; j <= i; ++j) {
                const double* vj = vh + (size_t)j * Dv;
                double w = dot(qt + (size_t)i * Dk, kt + (size_t)j * Dk, Dk);
                double gw = 0.0;
                for (int m = 0; m < Dv; ++m) gw += dOi[m] * (vj[m] - oi[m]);
                gw /= den[i];
                for (int d = 0; d < Dk; ++d) {
                    dqt[(size_t)i * Dk + d] += gw * kt[(size_t)j * Dk + d];
                    dkt[(size_t)j * Dk + d] += gw * qt[(size_t)i * Dk + d];
                }
                for (int m = 0; m < Dv; ++m) dvh[(size_t)j * Dv + m] += w * dOi[m] / den[i];
            }
        }
        const double* qh = q + IDX3(h, 0, 0, N, Dk);
        const double* kh = k + IDX3(h, 0, 0, N, Dk);
        for (size_t t = 0; t < (size_t)N * Dk; ++t) {
            dq[IDX3(h, 0, 0, N, Dk) + t] = dqt[t] * dphi(qh[t]);
            dk[IDX3(h, 0, 0, N, Dk) + t] = dkt[t] * dphi(kh[t]);
        }
        free(qt); free(kt); free(den); free(oh); free(dqt); free(dkt);
    }
}

/*
 * Backward of the causal form by cumulative sums, O(N Dk Dv) per head and no
 * per-position state stored.  Forward sweep (S_i, z_i running):
 *   den_i = phi(q_i)^T z_i,  o_i = phi(q_i)^T S_i / den_i,
 *   P_i = dO_i / den_i,      g_i = -(dO_i . o_i) / den_i,
 *   dphi(q_i) = S_i P_i + g_i z_i.
 * Reverse sweep (R_j = sum_{i>=j} phi(q_i) P_i^T, r_j = sum_{i>=j} g_i phi(q_i)):
 *   dphi(k_j) = R_j v_j + r_j,  dv_j = R_j^T phi(k_j).
 * Only P (N x Dv) and g (N) are kept between the sweeps.  [REV] 3.5 (gradient
 * as cumulative sums, linear memory); [KAT] Methods (학습 line).
 */
void oracle_causal_bwd_recurrent(const double* q, const double* k, const double* v, const double* dO,
                                 double* dq, double* dk, double* dv, int BH, int N, int Dk, int Dv) {
#pragma omp parallel for schedule(dynamic)
    for (int h = 0; h < BH; ++h) {
        double* S = (double*)calloc((size_t)Dk * Dv, sizeof(double));
        double* z = (double*)calloc((size_t)Dk, sizeof(double));
        double* P = (double*)malloc(sizeof(double) * (size_t)N * Dv);
        double* g = (double*)malloc(sizeof(double) * (size_t)N);
        double* qt = (double*)malloc(sizeof(double) * (size_t)Dk);
        double* kt = (double*)malloc(sizeof(double) * (size_t)Dk);
        double* num = (double*)malloc(sizeof(double) * (size_t)Dv);
        for (int i = 0; i < N; ++i) {
            const double* qi = q + IDX3(h, i, 0, N, Dk);
            const double* ki = k + IDX3(h, i, 0, N, Dk);
            const double* vi = v + IDX3(h, i, 0, N, Dv);
            const double* dOi = dO + IDX3(h, i, 0, N, Dv);
            for (int d = 0; d < Dk; ++d) { qt[d] = phi(qi[d]); kt[d] = phi(ki[d]); }
            for (int d = 0; d < Dk; ++d) {
                z[d] += kt[d];
                for (int m = 0; m < Dv; ++m) S[(size_t)d * Dv + m] += kt[d] * vi[m];
            }
            double den = dot(qt, z, Dk);
            double od = 0.0;
            for (int m = 0; m < Dv; ++m) {
                double s = 0.0;
                for (int d = 0; d < Dk; ++d) s += qt[d] * S[(size_t)d * Dv + m];
                num[m] = s;
                od += dOi[m] * (s / den);
            }
            g[i] = -od / den;
            for (int m = 0; m < Dv; ++m) P[(size_t)i * Dv + m] = dOi[m] / den;
            double* dqi = dq + IDX3(h, i, 0, N, Dk);
            for (int d = 0; d < Dk; ++d) {
                double s = g[i] * z[d];
                for (int m = 0; m < Dv; ++m) s += S[(size_t)d * Dv + m] * P[(size_t)i * Dv + m];
                dqi[d] = s * dphi(qi[d]);
            }
        }
        double* R = S; /* reuse the buffer for the reverse state */
        double* r = z;
        memset(R, 0, sizeof(double) * (size_t)Dk * Dv);
        memset(r, 0, sizeof(double) * (size_t)Dk);
        for (int j = N - 1; j >= 0; --j) {
            const double* qj = q + IDX3(h, j, 0, N, Dk);
            const double* kj = k + IDX3(h, j, 0, N, Dk);
            const double* vj = v + IDX3(h, j, 0, N, Dv);
            for (int d = 0; d < Dk; ++d) { qt[d] = phi(qj[d]); kt[d] = phi(kj[d]); }
            for (int d = 0; d < Dk; ++d) {
                r[d] += g[j] * qt[d];
                for (int m = 0; m < Dv; ++m) R[(size_t)d * Dv + m] += qt[d] * P[(size_t)j * Dv + m];
            }
            double* dkj = dk + IDX3(h, j, 0, N, Dk);
            for (int d = 0; d < Dk; ++d) {
                double s = r[d];
                for (int m = 0; m < Dv; ++m) s += R[(size_t)d * Dv + m] * vj[m];
                dkj[d] = s * dphi(kj[d]);
            }
            double* dvj = dv + IDX3(h, j, 0, N, Dv);
            for (int m = 0; m < Dv; ++m) {
                double s = 0.0;
                for (int d = 0; d < Dk; ++d) s += R[(size_t)d * Dv + m] * kt[d];
                dvj[m] = s;
            }
        }
        free(S); free(z); free(P); free(g); free(qt); free(kt); free(num);
    }
}

/*
 * Backward of the non-causal form, direct O(N^2): the same chain rule as
 * oracle_causal_bwd_direct with every j paired with every i.
 * [KAT] 핵심 구성요소 2 (the non-causal form being differentiated).
 */
void oracle_noncausal_bwd_direct(const double* q, const double* k, const double* v, const double* dO,
                                 double* dq, double* dk, double* dv, int BH, int N, int Dk, int Dv) {
#pragma omp parallel for schedule(dynamic)
    for (int h = 0; h < BH; ++h) {
        double* qt = phi_slice(q, h, N, Dk);
        double* kt = phi_slice(k, h, N, Dk);
        const double* vh = v + IDX3(h, 0, 0, N, Dv);
        const double* dOh = dO + IDX3(h, 0, 0, N, Dv);
        double* den = (double*)malloc(sizeof(double) * (size_t)N);
        double* oh = (double*)malloc(sizeof(double) * (size_t)N * Dv);
        double* dqt = (double*)calloc((size_t)N * Dk, sizeof(double));
        double* dkt = (double*)calloc((size_t)N * Dk, sizeof(double));
        double* dvh = dv + IDX3(h, 0, 0, N, Dv);
        for (size_t t = 0; t < (size_t)N * Dv; ++t) dvh[t] = 0.0;
        for (int i = 0; i < N; ++i) {
            double dsum = 0.0;
            for (int m = 0; m < Dv; ++m) oh[(size_t)i * Dv + m] = 0.0;
            for (int j = 0; j < N; ++j) {
                double w = dot(qt + (size_t)i * Dk, kt + (size_t)j * Dk, Dk);
                dsum += w;
                for (int m = 0; m < Dv; ++m) oh[(size_t)i * Dv + m] += w * vh[(size_t)j * Dv + m];
            }
            den[i] = dsum;
            for (int m = 0; m < Dv; ++m) oh[(size_t)i * Dv + m] /= dsum;
        }
        for (int i = 0; i < N; ++i) {
            const double* dOi = dOh + (size_t)i * Dv;
            const double* oi = oh + (size_t)i * Dv;
            for (int j = 0; j < N; ++j) {
                const double* vj = vh + (size_t)j * Dv;
                double w = dot(qt + (size_t)i * Dk, kt + (size_t)j * Dk, Dk);
                double gw = 0.0;
                for (int m = 0; m < Dv; ++m) gw += dOi[m] * (vj[m] - oi[m]);
                gw /= den[i];
                for (int d = 0; d < Dk; ++d) {
                    dqt[(size_t)i * Dk + d] += gw * kt[(size_t)j * Dk + d];
                    dkt[(size_t)j * Dk + d] += gw * qt[(size_t)i * Dk + d];
                }
                for (int m = 0; m < Dv; ++m) dvh[(size_t)j * Dv + m] += w * dOi[m] / den[i];
            }
        }
        const double* qh = q + IDX3(h, 0, 0, N, Dk);
        const double* kh = k + IDX3(h, 0, 0, N, Dk);
        for (size_t t = 0; t < (size_t)N * Dk; ++t) {
            dq[IDX3(h, 0, 0, N, Dk) + t] = dqt[t] * dphi(qh[t]);
            dk[IDX3(h, 0, 0, N, Dk) + t] = dkt[t] * dphi(kh[t]);
        }
        free(qt); free(kt); free(den); free(oh); free(dqt); free(dkt);
    }
}

/*
 * Backward of the non-causal form through its totals, O(N Dk Dv) per head: the chain
 * rule of oracle_noncausal_bwd_direct with the sums over keys (for q) and over queries
 * (for k and v) taken once.  With S = sum_j phi(k_j) v_j^T and z = sum_j phi(k_j)
 * ([KAT] 핵심 구성요소 2; [REV] 3.2), for every i: den_i = phi(q_i) . z,
 * o_i = phi(q_i)^T S / den_i, P_i = dO_i / den_i, g_i = -P_i . o_i, so that
 * dL/dw_ij = P_i . v_j + g_i and
 *   dphi(q_i) = sum_j phi(k_j) (P_i . v_j + g_i) = S P_i + g_i z;
 * then with R = sum_i phi(q_i) P_i^T and r = sum_i g_i phi(q_i):
 *   dphi(k_j) = sum_i phi(q_i) (P_i . v_j + g_i) = R v_j + r,   dv_j = R^T phi(k_j).
 */
void oracle_noncausal_bwd_assoc(const double* q, const double* k, const double* v, const double* dO,
                                double* dq, double* dk, double* dv, int BH, int N, int Dk, int Dv) {
#pragma omp parallel for schedule(dynamic)
    for (int h = 0; h < BH; ++h) {
        double* qt = phi_slice(q, h, N, Dk);
        double* kt = phi_slice(k, h, N, Dk);
        const double* vh = v + IDX3(h, 0, 0, N, Dv);
        const double* dOh = dO + IDX3(h, 0, 0, N, Dv);
        const double* qh = q + IDX3(h, 0, 0, N, Dk);
        const double* kh = k + IDX3(h, 0, 0, N, Dk);
        double* S = (double*)calloc((size_t)Dk * Dv, sizeof(double));
        double* z = (double*)calloc((size_t)Dk, sizeof(double));
        double* R = (double*)calloc((size_t)Dk * Dv, sizeof(double));
        double* r = (double*)calloc((size_t)Dk, sizeof(double));
        double* P = (double*)malloc(sizeof(double) * (size_t)Dv);
        double* num = (double*)malloc(sizeof(double) * (size_t)Dv);
        for (int j = 0; j < N; ++j)
            for (int d = 0; d < Dk; ++d) {
                const double kd = kt[(size_t)j * Dk + d];
                z[d] += kd;
                for (int m = 0; m < Dv; ++m) S[(size_t)d * Dv + m] += kd * vh[(size_t)j * Dv + m];
            }
        for (int i = 0; i < N; ++i) {
            const double* qi = qt + (size_t)i * Dk;
            const double den = dot(qi, z, Dk);
            for (int m = 0; m < Dv; ++m) num[m] = 0.0;
            for (int d = 0; d < Dk; ++d)
                for (int m = 0; m < Dv; ++m) num[m] += qi[d] * S[(size_t)d * Dv + m];
            double g = 0.0;
            for (int m = 0; m < Dv; ++m) {
                P[m] = dOh[(size_t)i * Dv + m] / den;
                g -= P[m] * num[m] / den;
            }
            for (int d = 0; d < Dk; ++d) {
                double sp = 0.0;
                for (int m = 0; m < Dv; ++m) sp += S[(size_t)d * Dv + m] * P[m];
                dq[IDX3(h, i, d, N, Dk)] = (sp + g * z[d]) * dphi(qh[(size_t)i * Dk + d]);
                r[d] += g * qi[d];
                for (int m = 0; m < Dv; ++m) R[(size_t)d * Dv + m] += qi[d] * P[m];
            }
        }
        for (int j = 0; j < N; ++j) {
            const double* kj = kt + (size_t)j * Dk;
            const double* vj = vh + (size_t)j * Dv;
            for (int d = 0; d < Dk; ++d) {
                double rv = r[d];
                for (int m = 0; m < Dv; ++m) rv += R[(size_t)d * Dv + m] * vj[m];
                dk[IDX3(h, j, d, N, Dk)] = rv * dphi(kh[(size_t)j * Dk + d]);
            }
            for (int m = 0; m < Dv; ++m) {
                double s = 0.0;
                for (int d = 0; d < Dk; ++d) s += R[(size_t)d * Dv + m] * kj[d];
                dv[IDX3(h, j, m, N, Dv)] = s;
            }
        }
        free(qt); free(kt); free(S); free(z); free(R); free(r); free(P); free(num);
    }
}

/* ------------------------------------------------------------------ retention
 * The decayed variant in [WIKI] "발전: 감쇠, 게이트, 델타 규칙" (RetNet row):
 * S_t = gamma S_{t-1} + v_t k_t^T with a fixed decay gamma per head, read as
 * o_t = S_t q_t (column convention).  Here S is kept as Dk x Dv, so
 * S_t = gamma S_{t-1} + k_t v_t^T and o_t = S_t^T q_t.  Per [WIKI] "항등 사상"
 * the queries and keys enter as they are (no feature map) and there is no
 * denominator (RetNet normalises the head output outside the attention).
 * gamma[h] is the decay of flat head h (h = b*H + head), 0 <= gamma <= 1.
 * 0^0 is taken as 1 (the j = i term always has weight 1).
 */
static double powi(double g, int m) {
    double r = 1.0;
    for (int i = 0; i < m; ++i) r *= g;
    return r;
}

/* Direct form, O(N^2) per head: o_i = sum_{j <= i} gamma^(i-j) (q_i . k_j) v_j. */
void oracle_retention_direct(const double* q, const double* k, const double* v, const double* gamma, double* o,
                             int BH, int N, int Dk, int Dv) {
#pragma omp parallel for schedule(dynamic)
    for (int h = 0; h < BH; ++h) {
        for (int i = 0; i < N; ++i) {
            double* oi = o + IDX3(h, i, 0, N, Dv);
            for (int m = 0; m < Dv; ++m) oi[m] = 0.0;
            for (int j = 0; j <= i; ++j) {
                const double w = powi(gamma[h], i - j) * dot(q + IDX3(h, i, 0, N, Dk), k + IDX3(h, j, 0, N, Dk), Dk);
                const double* vj = v + IDX3(h, j, 0, N, Dv);
                for (int m = 0; m < Dv; ++m) oi[m] += w * vj[m];
            }
        }
    }
}

/* One recurrent step for every head: S <- gamma S + k v^T, then out = S^T q. */
void oracle_retention_step(const double* q, const double* k, const double* v, const double* gamma, double* S,
                           double* out, int BH, int Dk, int Dv) {
    for (int h = 0; h < BH; ++h) {
        const double* qh = q + (size_t)h * Dk;
        const double* kh = k + (size_t)h * Dk;
        const double* vh = v + (size_t)h * Dv;
        double* Sh = S + (size_t)h * Dk * Dv;
        for (int d = 0; d < Dk; ++d)
            for (int m = 0; m < Dv; ++m) Sh[(size_t)d * Dv + m] = gamma[h] * Sh[(size_t)d * Dv + m] + kh[d] * vh[m];
        for (int m = 0; m < Dv; ++m) {
            double acc = 0.0;
            for (int d = 0; d < Dk; ++d) acc += qh[d] * Sh[(size_t)d * Dv + m];
            out[(size_t)h * Dv + m] = acc;
        }
    }
}

/* The recurrence from S = 0 over i = 1..N. */
void oracle_retention_recurrent(const double* q, const double* k, const double* v, const double* gamma, double* o,
                                int BH, int N, int Dk, int Dv) {
#pragma omp parallel for schedule(dynamic)
    for (int h = 0; h < BH; ++h) {
        double* S = (double*)calloc((size_t)Dk * (size_t)Dv, sizeof(double));
        for (int i = 0; i < N; ++i)
            oracle_retention_step(q + IDX3(h, i, 0, N, Dk), k + IDX3(h, i, 0, N, Dk), v + IDX3(h, i, 0, N, Dv),
                                  gamma + h, S, o + IDX3(h, i, 0, N, Dv), 1, Dk, Dv);
        free(S);
    }
}

/*
 * Chunked form: inside a chunk of C positions starting at s, the product
 * (Q_c K_c^T) weighted by gamma^(a-b) on its lower triangle, plus the carried
 * state read as gamma^(a+1) q_a^T S; then S <- gamma^n S + sum_b gamma^(n-1-b)
 * k_b v_b^T for a chunk of n positions (a, b counted from the chunk start).
 */
void oracle_retention_chunked(const double* q, const double* k, const double* v, const double* gamma, double* o,
                              int BH, int N, int Dk, int Dv, int C) {
#pragma omp parallel for schedule(dynamic)
    for (int h = 0; h < BH; ++h) {
        const double g = gamma[h];
        double* S = (double*)calloc((size_t)Dk * (size_t)Dv, sizeof(double));
        for (int s = 0; s < N; s += C) {
            int n = (N - s) < C ? (N - s) : C;
            for (int a = 0; a < n; ++a) {
                const double* qa = q + IDX3(h, s + a, 0, N, Dk);
                double* oa = o + IDX3(h, s + a, 0, N, Dv);
                const double carry = powi(g, a + 1);
                for (int m = 0; m < Dv; ++m) {
                    double acc = 0.0;
                    for (int d = 0; d < Dk; ++d) acc += qa[d] * S[(size_t)d * Dv + m];
                    oa[m] = carry * acc;
                }
                for (int b = 0; b <= a; ++b) {
                    const double w = powi(g, a - b) * dot(qa, k + IDX3(h, s + b, 0, N, Dk), Dk);
                    const double* vb = v + IDX3(h, s + b, 0, N, Dv);
                    for (int m = 0; m < Dv; ++m) oa[m] += w * vb[m];
                }
            }
            const double gn = powi(g, n);
            for (size_t e = 0; e < (size_t)Dk * Dv; ++e) S[e] *= gn;
            for (int b = 0; b < n; ++b) {
                const double w = powi(g, n - 1 - b);
                const double* kb = k + IDX3(h, s + b, 0, N, Dk);
                const double* vb = v + IDX3(h, s + b, 0, N, Dv);
                for (int d = 0; d < Dk; ++d)
                    for (int m = 0; m < Dv; ++m) S[(size_t)d * Dv + m] += w * kb[d] * vb[m];
            }
        }
        free(S);
    }
}
