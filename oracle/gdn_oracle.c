/*
 * FP64 CPU oracle for the Gated DeltaNet prefill recurrence and its gated
 * RMSNorm output.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * bench's CPU-baseline leg call it; the product path (the CUDA library and its
 * Python binding) never does.  It shares no code, header, table or constant with
 * the CUDA path.
 *
 * Sources (web pages, cited by title and section):
 *   [P413]  "#413 prefill: DeltaNet recurrence with the three value heads of a key
 *           head in one thread", sections "What changes" and "Exactness".
 *   [P1372] "#1372 DeltaNet recurrence: STRATA_GDN_CHUNKED=1 - the prompt's
 *           recurrence in 32-token chunks", section "What it does".
 *
 * The recurrence, per value head h with key head kh = h % n_kh ([P413] "What
 * changes": heads qh, qh+16, qh+32 share key head qh), state S in R^{d x d}
 * (row i = key dim, column j = value dim), per token t:
 *     S     <- exp(g_t) S                       (decay; g <= 0)
 *     delta  = beta_t (v_t - S^T k_t)           (the "kv sum" and the delta rule)
 *     S     <- S + k_t delta^T
 *     o_t    = S^T q_t                          (the "output sum")
 * Readings where the pages leave a step open: the kv sum is taken on the decayed
 * state (the chunked form's D = T beta (v - e^gamma S0^T k) of [P1372] fixes
 * this), and the output uses the updated state (the chunked form's P includes
 * the diagonal term).
 *
 * Everything here is plain loops in double precision, in the order the
 * definitions are written; no blocking, fusion or reordering.  Pins (tests
 * under tests/test_oracle*.py): the T=1 closed form, beta=0/g=0 identity,
 * decay-only, exact recall with orthonormal keys, linearity, the chunked form
 * against the sequential one on tiny T, exact rational brute force, and the
 * FP16 rounding against numpy's conversion.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_NO_MEM (-3)

static int check_shapes(int64_t T, int n_kh, int n_vh, int d) {
    if (T < 0 || n_kh <= 0 || n_vh <= 0 || d <= 0) return ORACLE_BAD_ARG;
    if (n_vh % n_kh != 0) return ORACLE_BAD_ARG;
    return ORACLE_OK;
}

/*
 * Sequential recurrence ([P413] "What changes"; the per-token definition above).
 *
 * q, k   : [T][n_kh][d]  float (the same FP32 values the GPU path receives)
 * v      : [T][n_vh][d]  float
 * g, beta: [T][n_vh]     float
 * S_in   : [n_vh][d][d]  double, S[h][i][j], i = key dim, j = value dim
 * S_out  : [n_vh][d][d]  double (may alias S_in)
 * o      : [T][n_vh][d]  double
 * nthreads: value heads are independent; > 1 spreads them over OpenMP threads.
 */
int oracle_gdn_recurrence(const float* q, const float* k, const float* v,
                          const float* g, const float* beta,
                          const double* S_in, double* S_out, double* o,
                          int64_t T, int n_kh, int n_vh, int d, int nthreads) {
    int rc = check_shapes(T, n_kh, n_vh, d);
    if (rc != ORACLE_OK) return rc;
    int failed = 0;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int h = 0; h < n_vh; ++h) {
        const int kh = h % n_kh;
        const size_t dd = (size_t)d * d;
        double* S = (double*)malloc(dd * sizeof(double));
        double* kv = (double*)malloc((size_t)d * sizeof(double));
        double* delta = (double*)malloc((size_t)d * sizeof(double));
        if (!S || !kv || !delta) {
            free(S); free(kv); free(delta);
#pragma omp atomic write
            failed = 1;
            continue;
        }
        memcpy(S, S_in + (size_t)h * dd, dd * sizeof(double));
        for (int64_t t = 0; t < T; ++t) {
            const float* kt = k + ((size_t)t * n_kh + kh) * d;
            const float* qt = q + ((size_t)t * n_kh + kh) * d;
            const float* vt = v + ((size_t)t * n_vh + h) * d;
            const double a = exp((double)g[(size_t)t * n_vh + h]);
            const double b = (double)beta[(size_t)t * n_vh + h];
            /* S <- e^g S */
            for (size_t e = 0; e < dd; ++e) S[e] *= a;
            /* kv = S^T k */
            for (int j = 0; j < d; ++j) {
                double s = 0.0;
                for (int i = 0; i < d; ++i) s += S[(size_t)i * d + j] * (double)kt[i];
                kv[j] = s;
            }
            /* delta = beta (v - kv) */
            for (int j = 0; j < d; ++j) delta[j] = b * ((double)vt[j] - kv[j]);
            /* S <- S + k delta^T */
            for (int i = 0; i < d; ++i)
                for (int j = 0; j < d; ++j) S[(size_t)i * d + j] += (double)kt[i] * delta[j];
            /* o = S^T q */
            double* ot = o + ((size_t)t * n_vh + h) * d;
            for (int j = 0; j < d; ++j) {
                double s = 0.0;
                for (int i = 0; i < d; ++i) s += S[(size_t)i * d + j] * (double)qt[i];
                ot[j] = s;
            }
        }
        memcpy(S_out + (size_t)h * dd, S, dd * sizeof(double));
        free(S); free(kv); free(delta);
    }
    return failed ? ORACLE_NO_MEM : ORACLE_OK;
}

/*
 * The chunked WY form, in FP64, written from [P1372] "What it does" (chunk C):
 *   gamma_t = sum of g_s for s <= t inside the chunk (the gate's running sum);
 *   A[t][i] = beta_t e^{gamma_t - gamma_i} (k_t . k_i)   for i < t;
 *   Tm      = (I + A)^{-1}                               (forward substitution);
 *   D       = Tm . U,  U_t = beta_t (v_t - e^{gamma_t} S0^T k_t);
 *   o_t     = e^{gamma_t} S0^T q_t + sum_{i<=t} e^{gamma_t - gamma_i} (q_t . k_i) D_i;
 *   S_end   = e^{gamma_last} S0 + sum_i e^{gamma_last - gamma_i} k_i D_i^T.
 * The last two lines are the "small matmuls" the page leaves unwritten; they
 * follow from unrolling the per-token definition inside the chunk.  A last
 * chunk shorter than C is a chunk of its own length.  Used only to cross-check
 * the algebra against oracle_gdn_recurrence; it is not the reference.
 */
int oracle_gdn_chunked(const float* q, const float* k, const float* v,
                       const float* g, const float* beta,
                       const double* S_in, double* S_out, double* o,
                       int64_t T, int n_kh, int n_vh, int d, int C, int nthreads) {
    int rc = check_shapes(T, n_kh, n_vh, d);
    if (rc != ORACLE_OK) return rc;
    if (C <= 0) return ORACLE_BAD_ARG;
    int failed = 0;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int h = 0; h < n_vh; ++h) {
        const int kh = h % n_kh;
        const size_t dd = (size_t)d * d;
        double* S = (double*)malloc(dd * sizeof(double));
        double* Snew = (double*)malloc(dd * sizeof(double));
        double* gam = (double*)malloc((size_t)C * sizeof(double));
        double* A = (double*)malloc((size_t)C * C * sizeof(double));
        double* Tm = (double*)malloc((size_t)C * C * sizeof(double));
        double* U = (double*)malloc((size_t)C * d * sizeof(double));
        double* D = (double*)malloc((size_t)C * d * sizeof(double));
        if (!S || !Snew || !gam || !A || !Tm || !U || !D) {
            free(S); free(Snew); free(gam); free(A); free(Tm); free(U); free(D);
#pragma omp atomic write
            failed = 1;
            continue;
        }
        memcpy(S, S_in + (size_t)h * dd, dd * sizeof(double));
        for (int64_t t0 = 0; t0 < T; t0 += C) {
            const int n = (int)((T - t0) < C ? (T - t0) : C);
            /* token t of the chunk is absolute token t0 + t */
#define KROW(t) (k + ((size_t)(t0 + (t)) * n_kh + kh) * d)
#define QROW(t) (q + ((size_t)(t0 + (t)) * n_kh + kh) * d)
#define VROW(t) (v + ((size_t)(t0 + (t)) * n_vh + h) * d)
#define GATE(t) ((double)g[(size_t)(t0 + (t)) * n_vh + h])
#define BETA(t) ((double)beta[(size_t)(t0 + (t)) * n_vh + h])
            /* gamma: running sum of the gate inside the chunk */
            double run = 0.0;
            for (int t = 0; t < n; ++t) { run += GATE(t); gam[t] = run; }
            /* A (strictly lower triangular) */
            for (int t = 0; t < n; ++t)
                for (int i = 0; i < n; ++i) {
                    double a = 0.0;
                    if (i < t) {
                        double kk = 0.0;
                        for (int c = 0; c < d; ++c) kk += (double)KROW(t)[c] * (double)KROW(i)[c];
                        a = BETA(t) * exp(gam[t] - gam[i]) * kk;
                    }
                    A[(size_t)t * C + i] = a;
                }
            /* Tm = (I + A)^{-1}: solve (I + A) Tm = I row by row (forward substitution) */
            for (int t = 0; t < n; ++t)
                for (int j = 0; j < n; ++j) {
                    double s = (t == j) ? 1.0 : 0.0;
                    for (int i = 0; i < t; ++i) s -= A[(size_t)t * C + i] * Tm[(size_t)i * C + j];
                    Tm[(size_t)t * C + j] = s;
                }
            /* U_t = beta_t (v_t - e^{gamma_t} S0^T k_t) */
            for (int t = 0; t < n; ++t) {
                const double eg = exp(gam[t]);
                for (int j = 0; j < d; ++j) {
                    double sk = 0.0;
                    for (int i = 0; i < d; ++i) sk += S[(size_t)i * d + j] * (double)KROW(t)[i];
                    U[(size_t)t * d + j] = BETA(t) * ((double)VROW(t)[j] - eg * sk);
                }
            }
            /* D = Tm U */
            for (int t = 0; t < n; ++t)
                for (int j = 0; j < d; ++j) {
                    double s = 0.0;
                    for (int i = 0; i < n; ++i) s += Tm[(size_t)t * C + i] * U[(size_t)i * d + j];
                    D[(size_t)t * d + j] = s;
                }
            /* o_t = e^{gamma_t} S0^T q_t + sum_{i<=t} e^{gamma_t-gamma_i} (q_t.k_i) D_i */
            for (int t = 0; t < n; ++t) {
                const double eg = exp(gam[t]);
                double* ot = o + ((size_t)(t0 + t) * n_vh + h) * d;
                for (int j = 0; j < d; ++j) {
                    double sq = 0.0;
                    for (int i = 0; i < d; ++i) sq += S[(size_t)i * d + j] * (double)QROW(t)[i];
                    ot[j] = eg * sq;
                }
                for (int i = 0; i <= t; ++i) {
                    double qk = 0.0;
                    for (int c = 0; c < d; ++c) qk += (double)QROW(t)[c] * (double)KROW(i)[c];
                    const double p = exp(gam[t] - gam[i]) * qk;
                    for (int j = 0; j < d; ++j) ot[j] += p * D[(size_t)i * d + j];
                }
            }
            /* S_end = e^{gamma_last} S0 + sum_i e^{gamma_last - gamma_i} k_i D_i^T */
            const double glast = gam[n - 1];
            for (size_t e = 0; e < dd; ++e) Snew[e] = exp(glast) * S[e];
            for (int i = 0; i < n; ++i) {
                const double r = exp(glast - gam[i]);
                for (int a = 0; a < d; ++a)
                    for (int j = 0; j < d; ++j)
                        Snew[(size_t)a * d + j] += r * (double)KROW(i)[a] * D[(size_t)i * d + j];
            }
            memcpy(S, Snew, dd * sizeof(double));
#undef KROW
#undef QROW
#undef VROW
#undef GATE
#undef BETA
        }
        memcpy(S_out + (size_t)h * dd, S, dd * sizeof(double));
        free(S); free(Snew); free(gam); free(A); free(Tm); free(U); free(D);
    }
    return failed ? ORACLE_NO_MEM : ORACLE_OK;
}

/*
 * Round a double to IEEE binary16 with round-to-nearest-even, in one rounding
 * step (no detour through float, so no double rounding).  Subnormals are kept;
 * values at or beyond 65520 become infinity; NaN becomes the quiet NaN 0x7e00.
 */
uint16_t oracle_fp16_rne(double x) {
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double ax = fabs(x);
    if (isnan(x)) return 0x7e00u;
    if (ax >= 65520.0) return (uint16_t)(sign | 0x7c00u);
    if (ax < ldexp(1.0, -14)) {
        /* subnormal range: units of 2^-24; 1024 units is the smallest normal */
        double n = nearbyint(ldexp(ax, 24));
        return (uint16_t)(sign | (uint16_t)n);
    }
    int E;
    frexp(ax, &E);          /* ax = m 2^E, m in [0.5, 1) */
    int e = E - 1;          /* ax in [2^e, 2^(e+1)) */
    double n = nearbyint(ldexp(ax, 10 - e)); /* in [1024, 2048] */
    if (n >= 2048.0) { n = 1024.0; e += 1; }
    if (e > 15) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(n - 1024.0));
}

/*
 * Gated RMSNorm to FP16 ([P413] "What changes": gdn_out_norm_kernel writes the
 * FP16 copy y_h that the output projection reads).  The page does not print the
 * formula; the reading used here is the plainest one for a gated RMSNorm: per
 * (token, value head) row of d values,
 *     r   = 1 / sqrt(mean_j o_j^2 + eps)
 *     y_j = fp16( o_j * r * w_j * silu(z_j) ),   silu(z) = z / (1 + e^{-z}),
 * with w of length d shared by all heads, everything in double and one rounding
 * to FP16 at the end.
 *
 * o: [T][n_vh][d] double; z: [T][n_vh][d] float; w: [d] float; y: [T][n_vh][d]
 * binary16 bits.
 */
int oracle_gdn_out_norm(const double* o, const float* z, const float* w,
                        double eps, uint16_t* y, int64_t T, int n_vh, int d, int nthreads) {
    if (T < 0 || n_vh <= 0 || d <= 0) return ORACLE_BAD_ARG;
    const int64_t rows = T * n_vh;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(static) num_threads(nthreads)
    for (int64_t r = 0; r < rows; ++r) {
        const double* orow = o + (size_t)r * d;
        const float* zrow = z + (size_t)r * d;
        double ss = 0.0;
        for (int j = 0; j < d; ++j) ss += orow[j] * orow[j];
        const double rs = 1.0 / sqrt(ss / (double)d + eps);
        for (int j = 0; j < d; ++j) {
            const double zj = (double)zrow[j];
            const double silu = zj / (1.0 + exp(-zj));
            y[(size_t)r * d + j] = oracle_fp16_rne(orow[j] * rs * (double)w[j] * silu);
        }
    }
    return ORACLE_OK;
}

/*
 * Pre-stage: the recurrence's inputs from the layer's projections ("Round 20
 * Track C Audit: gdn_pre Key-Head t >= 3 Vectorized conv_w Fast Path + gdn_scan_r
 * ...", section 1 "Summary of Changes": a 4-tap causal convolution per channel of
 * the packed qkv rows, with the q channels of key head kh at kh*d and its k
 * channels at (n_kh + kh)*d, taps applied to rows t-3 .. t; the stage hands the
 * scan normalised q and k, the convolved v and the gates, and keeps a history).
 *
 * qkv     : [T][Cw] float, Cw = (2 n_kh + n_vh) d: q of the key heads, k of the
 *           key heads, then v of the value heads
 * conv_w  : [Cw][4] float; tap j multiplies row t - 3 + j of the same channel
 * hist_in : [3][Cw] float, rows -3, -2, -1 (the last rows before this call), or
 *           NULL for the start of a sequence (zeros)
 * a, b    : [T][n_vh] float, gate and beta projections; A_log, dt_bias: [n_vh] float
 * act     : 1 applies SiLU to every convolved channel, 0 none
 * eps     : added to the sum of squares in the q and k L2 norms
 * q, k    : [T][n_kh][d] double; v: [T][n_vh][d] double; g, beta: [T][n_vh] double
 * hist_out: [3][Cw] double, the last three rows of (hist_in, qkv), or NULL
 *
 * Per token t and channel c:
 *     x_c  = sum_{j=0..3} conv_w[c][j] X[t-3+j][c]        (X[-3..-1] = hist_in)
 *     u_c  = act ? x_c / (1 + e^{-x_c}) : x_c
 *     q[t][kh] = u_q / sqrt(|u_q|^2 + eps) / sqrt(d);   k[t][kh] = u_k / sqrt(|u_k|^2 + eps)
 *     v[t][h]  = u_v
 *     g[t][h]  = -e^{A_log[h]} softplus(a[t][h] + dt_bias[h]),  softplus(x) = log(1 + e^x)
 *     beta[t][h] = 1 / (1 + e^{-b[t][h]})
 * The pages give neither the activation, the norm's eps, the 1/sqrt(d) on q nor
 * the gate formula; these are the readings this oracle takes (the GDN layer's
 * usual form; the recurrence's tests draw q with norm 1/sqrt(d) and g = -softplus).
 */
static double oracle_softplus(double x) {
    /* log(1 + e^x) = max(x, 0) + log(1 + e^{-|x|}) */
    return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

int oracle_gdn_prestage(const float* qkv, const float* conv_w, const float* hist_in,
                        const float* a, const float* b, const float* A_log, const float* dt_bias,
                        int act, double eps, double* q, double* k, double* v, double* g,
                        double* beta, double* hist_out, int64_t T, int n_kh, int n_vh, int d) {
    if (check_shapes(T, n_kh, n_vh, d) != ORACLE_OK) return ORACLE_BAD_ARG;
    const int64_t Cw = (int64_t)(2 * n_kh + n_vh) * d;
    double* u = (double*)malloc(sizeof(double) * (size_t)Cw);
    if (!u) return ORACLE_NO_MEM;
    for (int64_t t = 0; t < T; ++t) {
        /* convolution and activation of every channel of row t */
        for (int64_t c = 0; c < Cw; ++c) {
            double x = 0.0;
            for (int j = 0; j < 4; ++j) {
                const int64_t r = t - 3 + j;
                double xr;
                if (r >= 0)
                    xr = (double)qkv[r * Cw + c];
                else
                    xr = hist_in ? (double)hist_in[(3 + r) * Cw + c] : 0.0;
                x += (double)conv_w[c * 4 + j] * xr;
            }
            u[c] = act ? x / (1.0 + exp(-x)) : x;
        }
        for (int kh = 0; kh < n_kh; ++kh) {
            const double* uq = u + (int64_t)kh * d;
            const double* uk = u + (int64_t)(n_kh + kh) * d;
            double sq = 0.0, sk = 0.0;
            for (int i = 0; i < d; ++i) {
                sq += uq[i] * uq[i];
                sk += uk[i] * uk[i];
            }
            const double nq = sqrt(sq + eps) * sqrt((double)d), nk = sqrt(sk + eps);
            for (int i = 0; i < d; ++i) {
                q[(t * n_kh + kh) * d + i] = uq[i] / nq;
                k[(t * n_kh + kh) * d + i] = uk[i] / nk;
            }
        }
        for (int h = 0; h < n_vh; ++h) {
            const double* uv = u + (int64_t)(2 * n_kh + h) * d;
            for (int j = 0; j < d; ++j) v[(t * n_vh + h) * d + j] = uv[j];
            const double x = (double)a[t * n_vh + h] + (double)dt_bias[h];
            g[t * n_vh + h] = -exp((double)A_log[h]) * oracle_softplus(x);
            beta[t * n_vh + h] = 1.0 / (1.0 + exp(-(double)b[t * n_vh + h]));
        }
    }
    free(u);
    if (hist_out) {
        /* row -3 + i of the next call is row T - 3 + i of this one */
        for (int i = 0; i < 3; ++i) {
            const int64_t r = T - 3 + i;
            for (int64_t c = 0; c < Cw; ++c) {
                double x;
                if (r >= 0)
                    x = (double)qkv[r * Cw + c];
                else
                    x = hist_in ? (double)hist_in[(3 + r) * Cw + c] : 0.0;
                hist_out[i * Cw + c] = x;
            }
        }
    }
    return ORACLE_OK;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
