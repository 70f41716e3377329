/*
 * ssd_oracle.c -- plain, slow, fp64 CPU oracle for the Mamba-2 SSD forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file: only the tests, the package's smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or constant with the CUDA
 * library under mamba_ssd_chunked_02_gb300/csrc.
 *
 * Pages cited (by title and section):
 *   [P1] "NVIDIA、cuTileでMamba-2フォワードパスを高速化" (ai.newsbites.today),
 *        section "cuTileによるMamba-2フォワードパスの3段階カーネル設計".
 *   [P2] "NVIDIA CUDA Tile로 Mamba-2 순방향 전달 커널 가속화" (devin.kr),
 *        sections "Mamba-2 아키텍처의 핵심 연산" and "세 가지 핵심 커널 구현".
 *   [P3] "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
 *        NVIDIA CUDA Tile" (brifing.si), sections 4, 5, 7, 8, 9 and 11.
 *
 * What is computed.  Per batch b and head h, with state S in R^{P x N}:
 *     a_t = dt[b,t,h] * A[h]                             (A[h] < 0)
 *     S_t = exp(a_t) * S_{t-1} + dt[b,t,h] * x[b,t,h,:] (outer) B[b,t,g,:]
 *     y[b,t,h,:] = S_t . C[b,t,g,:] + D[h] * x[b,t,h,:]
 * with S_{-1} = initial_state[b,h] (or 0) and final_state[b,h] = S_{T-1}.
 * [P2 "핵심 연산"] prints the read-out y_t = c_t^T h_t + D x_t; the pages print
 * no update equation, and the one used is the standard Mamba-2 discretisation
 * (decay exp(dt*A) on the state, dt*x*B^T as input), the plainest reading of
 * the pages' log-space cumulative sum of a_t [P2 "핵심 연산", P3 section 5].
 * Head h reads group g = h / (H/G) of B and C (contiguous head blocks).
 *
 * Three forms are provided:
 *   oracle_ssd_recurrent  -- the definition above, token by token.
 *   oracle_ssd_chunked    -- the pages' four steps in their order and notation:
 *                            chunk-local cumsum of a_t scaled by log2(e) and
 *                            decays by exp2 [P3 section 7]; per-chunk states by
 *                            the jump formula [P3 sections 4, 8]; a sequential
 *                            pass over chunks [P2 "세 가지 핵심 커널 구현"]; the
 *                            three-term output with causal masking applied
 *                            before exponentiation [P3 sections 9, 11].
 *   oracle_ssd_quadratic  -- brute force "attention" view: every decay is the
 *                            explicit sum of a_r between the two tokens.
 *   oracle_ssd_backward   -- gradients of the recurrence: reverse-mode
 *                            differentiation of the token-by-token definition,
 *                            step by step in reverse order.  The pages give no
 *                            method for the backward pass; they only note that
 *                            end-to-end training speed also depends on it [P1
 *                            "開発現場への影響と未確認事項"; P2 "성능 벤치마크
 *                            결과 및 활용"].  This is the chain rule applied to
 *                            the definition above.
 *
 * Inputs are float (the exact values the GPU sees: bf16 and fp32 both widen
 * to float exactly); every operation is done in double.
 *
 * Layouts (row-major, contiguous):
 *   x [b,T,H,P]  dt [b,T,H]  A [H]  B,C [b,T,G,N]  D [H]  init [b,H,P,N]
 *   y [b,T,H,P]  final_state [b,H,P,N]
 *   cum2 [b,H,T] (chunked form), dS and Sprev [b,nc,H,P,N], nc = ceil(T/L).
 *
 * Return value: 0 on success, -1 on an invalid argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define LOG2E_D 1.442695040888963407359924681001892137

static int shape_ok(int64_t Bt, int64_t T, int64_t H, int64_t P, int64_t N, int64_t G) {
    if (Bt <= 0 || T <= 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0) return 0;
    if (H % G != 0) return 0;
    return 1;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Recurrent form (the definition).  `pairs` lists (b,h) pairs to compute as
 * 2*npairs int64 values; pairs == NULL computes all of them.  Only the y rows
 * and final_state slices of the computed pairs are written.
 */
int oracle_ssd_recurrent(int64_t Bt, int64_t T, int64_t H, int64_t P, int64_t N, int64_t G,
                         const float* x, const float* dt, const float* A, const float* B,
                         const float* C, const float* D, const float* init,
                         const int64_t* pairs, int64_t npairs,
                         double* y, double* final_state, int nthreads) {
    if (!shape_ok(Bt, T, H, P, N, G)) return -1;
    if (!x || !dt || !A || !B || !C || !y || !final_state) return -1;
    const int64_t hpg = H / G;
    const int64_t total = pairs ? npairs : Bt * H;
    set_threads(nthreads);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t i = 0; i < total; ++i) {
        const int64_t b = pairs ? pairs[2 * i] : i / H;
        const int64_t h = pairs ? pairs[2 * i + 1] : i % H;
        if (b < 0 || b >= Bt || h < 0 || h >= H) { bad |= 1; continue; }
        const int64_t g = h / hpg;
        double* S = (double*)malloc((size_t)(P * N) * sizeof(double));
        if (!S) { bad |= 1; continue; }
        for (int64_t k = 0; k < P * N; ++k)
            S[k] = init ? (double)init[(b * H + h) * P * N + k] : 0.0;
        const double Ah = (double)A[h];
        const double Dh = D ? (double)D[h] : 0.0;
        for (int64_t t = 0; t < T; ++t) {
            const double dtv = (double)dt[(b * T + t) * H + h];
            const double decay = exp(dtv * Ah);
            const float* xt = x + ((b * T + t) * H + h) * P;
            const float* Bt_ = B + ((b * T + t) * G + g) * N;
            const float* Ct = C + ((b * T + t) * G + g) * N;
            double* yt = y + ((b * T + t) * H + h) * P;
            for (int64_t p = 0; p < P; ++p) {
                const double u = dtv * (double)xt[p];
                double* Sp = S + p * N;
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    Sp[n] = decay * Sp[n] + u * (double)Bt_[n];
                    acc += Sp[n] * (double)Ct[n];
                }
                yt[p] = acc + Dh * (double)xt[p];
            }
        }
        memcpy(final_state + (b * H + h) * P * N, S, (size_t)(P * N) * sizeof(double));
        free(S);
    }
    return bad ? -1 : 0;
}

/*
 * Chunked form: the pages' four steps, in fp64, with chunk length L (a last,
 * shorter chunk is allowed).  Any of cum2, dS, Sprev may be NULL when the
 * caller does not want that intermediate; y and final_state are required.
 */
int oracle_ssd_chunked(int64_t Bt, int64_t T, int64_t H, int64_t P, int64_t N, int64_t G,
                       int64_t L, const float* x, const float* dt, const float* A,
                       const float* B, const float* C, const float* D, const float* init,
                       double* cum2_out, double* dS_out, double* Sprev_out,
                       double* y, double* final_state, int nthreads) {
    if (!shape_ok(Bt, T, H, P, N, G) || L <= 0) return -1;
    if (!x || !dt || !A || !B || !C || !y || !final_state) return -1;
    const int64_t hpg = H / G;
    const int64_t nc = (T + L - 1) / L;
    const int64_t PN = P * N;
    set_threads(nthreads);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t i = 0; i < Bt * H; ++i) {
        const int64_t b = i / H, h = i % H, g = h / hpg;
        const double Ah = (double)A[h];
        const double Dh = D ? (double)D[h] : 0.0;
        double* cum2 = (double*)malloc((size_t)T * sizeof(double));
        double* dS = (double*)malloc((size_t)(nc * PN) * sizeof(double));
        double* Sp = (double*)malloc((size_t)(nc * PN) * sizeof(double));
        double* S = (double*)malloc((size_t)PN * sizeof(double));
        if (!cum2 || !dS || !Sp || !S) { bad |= 1; free(cum2); free(dS); free(Sp); free(S); continue; }

        /* Step 1 -- chunk_cumsum: inclusive cumulative sum of a_t = dt_t*A_h within
         * each chunk (restarting at every chunk start), scaled by log2(e) so that
         * decays are taken with exp2 [P3 section 7; P2 "세 가지 핵심 커널 구현"]. */
        for (int64_t c = 0; c < nc; ++c) {
            double run = 0.0;
            for (int64_t t = c * L; t < T && t < (c + 1) * L; ++t) {
                run += (double)dt[(b * T + t) * H + h] * Ah;
                cum2[t] = LOG2E_D * run;
            }
        }

        /* Step 2 -- per-chunk state by the jump formula [P3 sections 4, 8]:
         * dS_c = sum_{s in chunk c} exp2(cum2_last - cum2_s) * dt_s * x_s B_s^T. */
        for (int64_t c = 0; c < nc; ++c) {
            const int64_t t0 = c * L, t1 = (c + 1) * L < T ? (c + 1) * L : T;
            const double last = cum2[t1 - 1];
            double* d = dS + c * PN;
            for (int64_t k = 0; k < PN; ++k) d[k] = 0.0;
            for (int64_t s = t0; s < t1; ++s) {
                const double w = exp2(last - cum2[s]) * (double)dt[(b * T + s) * H + h];
                const float* xs = x + ((b * T + s) * H + h) * P;
                const float* Bs = B + ((b * T + s) * G + g) * N;
                for (int64_t p = 0; p < P; ++p) {
                    const double u = w * (double)xs[p];
                    for (int64_t n = 0; n < N; ++n) d[p * N + n] += u * (double)Bs[n];
                }
            }
        }

        /* Step 3 -- sequential pass over chunks: the state entering chunk c is
         * Sprev_c; S <- exp2(cum2_last(c)) * S + dS_c; the last S is the final
         * state [P2 "세 가지 핵심 커널 구현", fwd_pass_state]. */
        for (int64_t k = 0; k < PN; ++k)
            S[k] = init ? (double)init[(b * H + h) * PN + k] : 0.0;
        for (int64_t c = 0; c < nc; ++c) {
            const int64_t t1 = (c + 1) * L < T ? (c + 1) * L : T;
            const double chunk_decay = exp2(cum2[t1 - 1]);
            memcpy(Sp + c * PN, S, (size_t)PN * sizeof(double));
            for (int64_t k = 0; k < PN; ++k) S[k] = chunk_decay * S[k] + dS[c * PN + k];
        }
        memcpy(final_state + (b * H + h) * PN, S, (size_t)PN * sizeof(double));

        /* Step 4 -- compute_out: three terms [P3 section 9; P2 "세 가지 핵심 커널 구현"]:
         *   intra-chunk:  sum_{s<=t, same chunk} (C_t.B_s) exp2(cum2_t - cum2_s) dt_s x_s
         *                 (the causal mask s<=t is applied before exp2 [P3 section 11]);
         *   carried:      exp2(cum2_t) * Sprev_c . C_t;
         *   skip:         D_h x_t. */
        for (int64_t c = 0; c < nc; ++c) {
            const int64_t t0 = c * L, t1 = (c + 1) * L < T ? (c + 1) * L : T;
            const double* Sc = Sp + c * PN;
            for (int64_t t = t0; t < t1; ++t) {
                const float* Ct = C + ((b * T + t) * G + g) * N;
                const float* xt = x + ((b * T + t) * H + h) * P;
                double* yt = y + ((b * T + t) * H + h) * P;
                const double carry = exp2(cum2[t]);
                for (int64_t p = 0; p < P; ++p) {
                    double acc = 0.0;
                    for (int64_t n = 0; n < N; ++n) acc += Sc[p * N + n] * (double)Ct[n];
                    yt[p] = carry * acc + Dh * (double)xt[p];
                }
                for (int64_t s = t0; s <= t; ++s) {
                    const float* Bs = B + ((b * T + s) * G + g) * N;
                    const float* xs = x + ((b * T + s) * H + h) * P;
                    double cb = 0.0;
                    for (int64_t n = 0; n < N; ++n) cb += (double)Ct[n] * (double)Bs[n];
                    const double m = cb * exp2(cum2[t] - cum2[s]) * (double)dt[(b * T + s) * H + h];
                    for (int64_t p = 0; p < P; ++p) yt[p] += m * (double)xs[p];
                }
            }
        }

        if (cum2_out)
            for (int64_t t = 0; t < T; ++t) cum2_out[(b * H + h) * T + t] = cum2[t];
        for (int64_t c = 0; c < nc; ++c) {
            const int64_t off = ((b * nc + c) * H + h) * PN;
            if (dS_out) memcpy(dS_out + off, dS + c * PN, (size_t)PN * sizeof(double));
            if (Sprev_out) memcpy(Sprev_out + off, Sp + c * PN, (size_t)PN * sizeof(double));
        }
        free(cum2); free(dS); free(Sp); free(S);
    }
    return bad ? -1 : 0;
}

/*
 * Quadratic (brute-force) form for tiny inputs: every decay between tokens s
 * and t is recomputed as exp of the explicit sum of a_r, r = s+1..t.
 *   y_t = sum_{s<=t} (C_t.B_s) dt_s exp(sum_{r=s+1}^{t} a_r) x_s
 *         + exp(sum_{r=0}^{t} a_r) * init . C_t + D x_t
 *   final = sum_s exp(sum_{r=s+1}^{T-1} a_r) dt_s x_s B_s^T + exp(sum_{r=0}^{T-1} a_r) init
 */
int oracle_ssd_quadratic(int64_t Bt, int64_t T, int64_t H, int64_t P, int64_t N, int64_t G,
                         const float* x, const float* dt, const float* A, const float* B,
                         const float* C, const float* D, const float* init,
                         double* y, double* final_state) {
    if (!shape_ok(Bt, T, H, P, N, G)) return -1;
    if (!x || !dt || !A || !B || !C || !y || !final_state) return -1;
    const int64_t hpg = H / G;
    for (int64_t b = 0; b < Bt; ++b) {
        for (int64_t h = 0; h < H; ++h) {
            const int64_t g = h / hpg;
            const double Ah = (double)A[h];
            const double Dh = D ? (double)D[h] : 0.0;
            const float* S0 = init ? init + (b * H + h) * P * N : NULL;
            for (int64_t t = 0; t <= T; ++t) {
                /* t == T is the final state (no read-out). */
                const int64_t tl = t < T ? t : T - 1;
                double* out = t < T ? y + ((b * T + t) * H + h) * P : NULL;
                double* fin = t == T ? final_state + (b * H + h) * P * N : NULL;
                if (out) for (int64_t p = 0; p < P; ++p) out[p] = Dh * (double)x[((b * T + t) * H + h) * P + p];
                if (fin) for (int64_t k = 0; k < P * N; ++k) fin[k] = 0.0;
                for (int64_t s = 0; s <= tl; ++s) {
                    double e = 0.0;
                    for (int64_t r = s + 1; r <= tl; ++r) e += (double)dt[(b * T + r) * H + h] * Ah;
                    const double w = exp(e) * (double)dt[(b * T + s) * H + h];
                    const float* Bs = B + ((b * T + s) * G + g) * N;
                    const float* xs = x + ((b * T + s) * H + h) * P;
                    if (out) {
                        const float* Ct = C + ((b * T + t) * G + g) * N;
                        double cb = 0.0;
                        for (int64_t n = 0; n < N; ++n) cb += (double)Ct[n] * (double)Bs[n];
                        for (int64_t p = 0; p < P; ++p) out[p] += cb * w * (double)xs[p];
                    }
                    if (fin)
                        for (int64_t p = 0; p < P; ++p)
                            for (int64_t n = 0; n < N; ++n)
                                fin[p * N + n] += w * (double)xs[p] * (double)Bs[n];
                }
                if (S0) {
                    double e = 0.0;
                    for (int64_t r = 0; r <= tl; ++r) e += (double)dt[(b * T + r) * H + h] * Ah;
                    const double decay = exp(e);
                    if (out) {
                        const float* Ct = C + ((b * T + t) * G + g) * N;
                        for (int64_t p = 0; p < P; ++p) {
                            double acc = 0.0;
                            for (int64_t n = 0; n < N; ++n) acc += (double)S0[p * N + n] * (double)Ct[n];
                            out[p] += decay * acc;
                        }
                    }
                    if (fin)
                        for (int64_t k = 0; k < P * N; ++k) fin[k] += decay * (double)S0[k];
                }
            }
        }
    }
    return 0;
}

/*
 * Backward pass of the recurrence (reverse-mode, the chain rule on the
 * definition).  For a scalar loss with dL/dy = dy [b,T,H,P] and
 * dL/dfinal_state = dfin [b,H,P,N] (NULL = 0), per (b,h), with
 * G = dL/dS_t accumulated from the end:
 *     G <- dfin
 *     for t = T-1 .. 0:
 *         G        += dy_t C_t^T                       (read-out of S_t)
 *         dC_t     += S_t^T dy_t                       (summed over the group's heads)
 *         dx_t      = dt_t G B_t + D dy_t
 *         dB_t     += dt_t G^T x_t                     (summed over the group's heads)
 *         ddt_t     = x_t^T G B_t + A e_t <G, S_{t-1}>   (e_t = exp(dt_t A))
 *         dA       += dt_t e_t <G, S_{t-1}>
 *         dD       += dy_t . x_t
 *         G        <- e_t G                            (dL/dS_{t-1})
 *     dinit = G
 * The states S_t are taken from a forward sweep: every K-th state is kept
 * (K ~ sqrt(T)) and the K states of a segment are recomputed from it with the
 * same operations in the same order, so they are the forward sweep's values.
 *
 * `pairs` (2*npairs int64, or NULL = all) restricts the (b,h) pairs; dx, ddt,
 * dinit of other pairs are left untouched and dA, dD, dB, dC then sum the
 * listed pairs only.  Outputs are fully written (dA, dD, dB, dC zeroed first).
 */
int oracle_ssd_backward(int64_t Bt, int64_t T, int64_t H, int64_t P, int64_t N, int64_t G,
                        const float* x, const float* dt, const float* A, const float* B,
                        const float* C, const float* D, const float* init, const float* dy,
                        const float* dfin, const int64_t* pairs, int64_t npairs,
                        double* dx, double* ddt, double* dA, double* dB, double* dC,
                        double* dD, double* dinit, int nthreads) {
    if (!shape_ok(Bt, T, H, P, N, G)) return -1;
    if (!x || !dt || !A || !B || !C || !dy || !dx || !ddt || !dA || !dB || !dC || !dD || !dinit)
        return -1;
    const int64_t hpg = H / G, PN = P * N;
    const int64_t total = pairs ? npairs : Bt * H;
    int64_t K = 1;
    while (K * K < T) ++K;
    const int64_t nseg = (T + K - 1) / K;
    /* Per-pair contributions to the group and head sums, reduced afterwards in a
     * fixed order. */
    double* pdB = (double*)calloc((size_t)(total * T * N), sizeof(double));
    double* pdC = (double*)calloc((size_t)(total * T * N), sizeof(double));
    double* pdA = (double*)calloc((size_t)(total > 0 ? total : 1), sizeof(double));
    double* pdD = (double*)calloc((size_t)(total > 0 ? total : 1), sizeof(double));
    if ((total > 0 && (!pdB || !pdC)) || !pdA || !pdD) { free(pdB); free(pdC); free(pdA); free(pdD); return -1; }
    set_threads(nthreads);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t i = 0; i < total; ++i) {
        const int64_t b = pairs ? pairs[2 * i] : i / H;
        const int64_t h = pairs ? pairs[2 * i + 1] : i % H;
        if (b < 0 || b >= Bt || h < 0 || h >= H) { bad |= 1; continue; }
        const int64_t g = h / hpg;
        const double Ah = (double)A[h];
        const double Dh = D ? (double)D[h] : 0.0;
        double* ck = (double*)malloc((size_t)(nseg * PN) * sizeof(double));   /* S_{sK-1} */
        double* seg = (double*)malloc((size_t)((K + 1) * PN) * sizeof(double));
        double* Gs = (double*)malloc((size_t)PN * sizeof(double));
        if (!ck || !seg || !Gs) { bad |= 1; free(ck); free(seg); free(Gs); continue; }
        /* Forward sweep, keeping the state entering every segment. */
        double* S = seg;
        for (int64_t k = 0; k < PN; ++k) S[k] = init ? (double)init[(b * H + h) * PN + k] : 0.0;
        for (int64_t t = 0; t < T; ++t) {
            if (t % K == 0) memcpy(ck + (t / K) * PN, S, (size_t)PN * sizeof(double));
            const double dtv = (double)dt[(b * T + t) * H + h];
            const double e = exp(dtv * Ah);
            const float* xt = x + ((b * T + t) * H + h) * P;
            const float* Bt_ = B + ((b * T + t) * G + g) * N;
            for (int64_t p = 0; p < P; ++p) {
                const double in = dtv * (double)xt[p];
                for (int64_t n = 0; n < N; ++n) S[p * N + n] = e * S[p * N + n] + in * (double)Bt_[n];
            }
        }
        for (int64_t k = 0; k < PN; ++k) Gs[k] = dfin ? (double)dfin[(b * H + h) * PN + k] : 0.0;
        double sA = 0.0, sD = 0.0;
        double* qB = pdB + i * T * N;
        double* qC = pdC + i * T * N;
        for (int64_t sg = nseg - 1; sg >= 0; --sg) {
            const int64_t t0 = sg * K, t1 = (sg + 1) * K < T ? (sg + 1) * K : T;
            /* seg[j] = S_{t0+j-1}, j = 0 .. t1-t0 (recomputed as in the sweep). */
            memcpy(seg, ck + sg * PN, (size_t)PN * sizeof(double));
            for (int64_t t = t0; t < t1; ++t) {
                const double dtv = (double)dt[(b * T + t) * H + h];
                const double e = exp(dtv * Ah);
                const float* xt = x + ((b * T + t) * H + h) * P;
                const float* Bt_ = B + ((b * T + t) * G + g) * N;
                const double* Sa = seg + (t - t0) * PN;
                double* Sb = seg + (t - t0 + 1) * PN;
                for (int64_t p = 0; p < P; ++p) {
                    const double in = dtv * (double)xt[p];
                    for (int64_t n = 0; n < N; ++n) Sb[p * N + n] = e * Sa[p * N + n] + in * (double)Bt_[n];
                }
            }
            for (int64_t t = t1 - 1; t >= t0; --t) {
                const double dtv = (double)dt[(b * T + t) * H + h];
                const double e = exp(dtv * Ah);
                const float* xt = x + ((b * T + t) * H + h) * P;
                const float* dyt = dy + ((b * T + t) * H + h) * P;
                const float* Bt_ = B + ((b * T + t) * G + g) * N;
                const float* Ct = C + ((b * T + t) * G + g) * N;
                const double* Sprev = seg + (t - t0) * PN;   /* S_{t-1} */
                const double* Scur = seg + (t - t0 + 1) * PN; /* S_t */
                /* G += dy_t C_t^T */
                for (int64_t p = 0; p < P; ++p)
                    for (int64_t n = 0; n < N; ++n) Gs[p * N + n] += (double)dyt[p] * (double)Ct[n];
                /* dC_t += S_t^T dy_t ; dB_t += dt_t G^T x_t */
                for (int64_t n = 0; n < N; ++n) {
                    double ac = 0.0, ab = 0.0;
                    for (int64_t p = 0; p < P; ++p) {
                        ac += Scur[p * N + n] * (double)dyt[p];
                        ab += Gs[p * N + n] * (double)xt[p];
                    }
                    qC[t * N + n] += ac;
                    qB[t * N + n] += dtv * ab;
                }
                /* dx_t = dt_t G B_t + D dy_t ; x^T G B */
                double xgb = 0.0;
                for (int64_t p = 0; p < P; ++p) {
                    double gb = 0.0;
                    for (int64_t n = 0; n < N; ++n) gb += Gs[p * N + n] * (double)Bt_[n];
                    dx[((b * T + t) * H + h) * P + p] = dtv * gb + Dh * (double)dyt[p];
                    xgb += (double)xt[p] * gb;
                }
                /* <G, S_{t-1}> */
                double gs = 0.0;
                for (int64_t k = 0; k < PN; ++k) gs += Gs[k] * Sprev[k];
                ddt[(b * T + t) * H + h] = xgb + Ah * e * gs;
                sA += dtv * e * gs;
                double yx = 0.0;
                for (int64_t p = 0; p < P; ++p) yx += (double)dyt[p] * (double)xt[p];
                sD += yx;
                /* G <- e_t G */
                for (int64_t k = 0; k < PN; ++k) Gs[k] *= e;
            }
        }
        memcpy(dinit + (b * H + h) * PN, Gs, (size_t)PN * sizeof(double));
        pdA[i] = sA;
        pdD[i] = sD;
        free(ck); free(seg); free(Gs);
    }
    if (!bad) {
        for (int64_t k = 0; k < H; ++k) { dA[k] = 0.0; dD[k] = 0.0; }
        for (int64_t k = 0; k < Bt * T * G * N; ++k) { dB[k] = 0.0; dC[k] = 0.0; }
        for (int64_t i = 0; i < total; ++i) {
            const int64_t b = pairs ? pairs[2 * i] : i / H;
            const int64_t h = pairs ? pairs[2 * i + 1] : i % H;
            const int64_t g = h / hpg;
            dA[h] += pdA[i];
            dD[h] += pdD[i];
            for (int64_t t = 0; t < T; ++t)
                for (int64_t n = 0; n < N; ++n) {
                    dB[((b * T + t) * G + g) * N + n] += pdB[(i * T + t) * N + n];
                    dC[((b * T + t) * G + g) * N + n] += pdC[(i * T + t) * N + n];
                }
        }
    }
    free(pdB); free(pdC); free(pdA); free(pdD);
    return bad ? -1 : 0;
}
