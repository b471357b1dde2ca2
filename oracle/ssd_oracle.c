/*
 * ssd_oracle.c -- fp64 CPU oracle for the SSD (structured state-space duality)
 * sequence-mixing forward pass.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the test suite, the
 * smoke check and the CPU-baseline leg of the benchmark may load this file's
 * library.  It shares no code, header or constant with the CUDA path.
 *
 * What it computes (the plain definition, token by token, in fp64):
 *
 *   Structured State Space Duality, "The recurrence as one matrix":
 *     h_t = Abar_t h_{t-1} + Bbar_t x_t ,   y_t = C_t^T h_t .
 *   The same page, same section: the scalar-times-identity case Abar_t = a_t I;
 *   its section "What the duality gives up": the general diagonal case, one
 *   decay per state dimension (also "On Structured State-Space Duality",
 *   abstract, point (i)).
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes of the repository):
 *   - a_t = exp(dt_t * A_h) (scalar) or a_t[n] = exp(dt_t * A_{h,n}) (diagonal);
 *   - Bbar_t x_t is the outer product B_t x_t^T (N x P), no dt factor;
 *   - the state is updated before it is read out, so y_t sees x_t;
 *   - init_state is h_{-1}; it is decayed by a_0 before y_0 is read;
 *   - heads map to B/C groups contiguously: g(h) = h / (H / G);
 *   - y_t gains D_h * x_t when D is given.
 *
 * All inputs arrive as fp32 (bf16 values are exact in fp32) and are upcast
 * exactly to fp64; dt*A is formed in fp64 (exact for fp32 operands) and the
 * exponential is the C library's fp64 exp.
 *
 * Layouts (row-major, contiguous):
 *   x (b,T,H,P)  dt (b,T,H)  A (H) or (H,N)  B,C (b,T,G,N)  D (H)
 *   init_state (b,H,N,P)
 * Outputs are stream-major: stream s = bi*H + h,
 *   y (n_streams, t_end, P)   final_state (n_streams, N, P)
 *
 * The "plant" argument is a test hook: a non-zero value runs a deliberately
 * wrong variant of the recurrence so that the tests can show their pins catch
 * that kind of mistake.  Zero is the oracle.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    PLANT_NONE = 0,
    PLANT_READOUT_BEFORE_UPDATE = 1, /* y_t read from h_{t-1} + B_t x_t^T without decay */
    PLANT_NO_INIT_DECAY = 2,         /* init_state not decayed by a_0 */
    PLANT_DROP_D = 3,                /* skip term dropped */
    PLANT_GROUP_MODULO = 4,          /* g(h) = h mod G instead of h / (H/G) */
    PLANT_DECAY_AFTER_INPUT = 5,     /* h_t = a_t (h_{t-1} + B_t x_t^T) */
    PLANT_SWAP_B_C = 6,              /* C used as input projection, B as output */
    PLANT_DIAG_FIRST_A = 7,          /* diagonal case: A_{h,0} used for every n */
    PLANT_DECAY_OFF_BY_ONE = 8,      /* a_{t-1} used at step t */
    PLANT_TRANSPOSE_STATE = 9        /* readout contracts over the wrong state index */
};

int ssd_oracle_version(void) { return 1; }

int ssd_oracle_fwd(int64_t nb, int64_t T, int64_t H, int64_t P, int64_t N,
                   int64_t G, int a_mode,
                   const float *x, const float *dt, const float *A,
                   const float *B, const float *C, const float *D,
                   const float *init_state,
                   const int64_t *streams, int64_t n_streams, int64_t t_end,
                   double *y, double *final_state, int nthreads, int plant)
{
    if (nb < 0 || T < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0)
        return 1;
    if (a_mode != 0 && a_mode != 1) return 1;
    if (t_end < 0 || t_end > T) return 1;
    if (streams == NULL) n_streams = nb * H;
    const int64_t heads_per_group = H / G;

#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t s = 0; s < n_streams; ++s) {
        const int64_t sid = streams ? streams[s] : s;
        if (sid < 0 || sid >= nb * H) { bad = 1; continue; }
        const int64_t bi = sid / H, h = sid % H;
        int64_t g = h / heads_per_group;
        if (plant == PLANT_GROUP_MODULO) g = h % G;
        const float *Bin = (plant == PLANT_SWAP_B_C) ? C : B;
        const float *Cout = (plant == PLANT_SWAP_B_C) ? B : C;

        double *st = (double *)malloc(sizeof(double) * (size_t)(N * P));
        double *a = (double *)malloc(sizeof(double) * (size_t)N);
        double *a_prev = (double *)malloc(sizeof(double) * (size_t)N);
        if (!st || !a || !a_prev) { free(st); free(a); free(a_prev); bad = 1; continue; }

        for (int64_t i = 0; i < N * P; ++i)
            st[i] = init_state ? (double)init_state[(bi * H + h) * N * P + i] : 0.0;
        for (int64_t n = 0; n < N; ++n) a_prev[n] = 1.0;

        for (int64_t t = 0; t < t_end; ++t) {
            const int64_t tok = bi * T + t;
            const double dtv = (double)dt[tok * H + h];
            for (int64_t n = 0; n < N; ++n) {
                double An;
                if (a_mode == 0) An = (double)A[h];
                else An = (double)A[h * N + ((plant == PLANT_DIAG_FIRST_A) ? 0 : n)];
                a[n] = exp(dtv * An);
            }
            const float *xt = x + (tok * H + h) * P;
            const float *Bt = Bin + (tok * G + g) * N;
            const float *Ct = Cout + (tok * G + g) * N;
            double *yt = y + (s * t_end + t) * P;

            if (plant == PLANT_READOUT_BEFORE_UPDATE) {
                for (int64_t p = 0; p < P; ++p) {
                    double acc = 0.0;
                    for (int64_t n = 0; n < N; ++n) acc += (double)Ct[n] * st[n * P + p];
                    yt[p] = acc;
                }
            }
            for (int64_t n = 0; n < N; ++n) {
                double an = a[n];
                if (plant == PLANT_NO_INIT_DECAY && t == 0) an = 1.0;
                if (plant == PLANT_DECAY_OFF_BY_ONE) an = a_prev[n];
                const double bn = (double)Bt[n];
                double *row = st + n * P;
                if (plant == PLANT_DECAY_AFTER_INPUT) {
                    for (int64_t p = 0; p < P; ++p) row[p] = an * (row[p] + bn * (double)xt[p]);
                } else {
                    for (int64_t p = 0; p < P; ++p) row[p] = an * row[p] + bn * (double)xt[p];
                }
            }
            for (int64_t n = 0; n < N; ++n) a_prev[n] = a[n];
            if (plant != PLANT_READOUT_BEFORE_UPDATE) {
                for (int64_t p = 0; p < P; ++p) {
                    double acc = 0.0;
                    if (plant == PLANT_TRANSPOSE_STATE && N == P) {
                        for (int64_t n = 0; n < N; ++n) acc += (double)Ct[n] * st[p * P + n];
                    } else {
                        for (int64_t n = 0; n < N; ++n) acc += (double)Ct[n] * st[n * P + p];
                    }
                    yt[p] = acc;
                }
            }
            if (D && plant != PLANT_DROP_D) {
                const double dh = (double)D[h];
                for (int64_t p = 0; p < P; ++p) yt[p] += dh * (double)xt[p];
            }
        }
        if (final_state) memcpy(final_state + s * N * P, st, sizeof(double) * (size_t)(N * P));
        free(st);
        free(a);
        free(a_prev);
    }
    return bad ? 1 : 0;
}

/*
 * Backward of the same map, in fp64: the reverse mode of the token recurrence.
 *
 * Given dy (b,T,H,P) and dfinal (b,H,N,P) or NULL, the gradients of the scalar
 *   L = sum_{b,t,h,p} y * dy + sum_{b,h,n,p} final_state * dfinal
 * with respect to x, dt, A, B, C, D and init_state.  Written from the forward
 * definition above (Structured State Space Duality, "The recurrence as one
 * matrix"; the pages do not give a backward, so this is the chain rule applied
 * to it, step by step in reverse):
 *   g       = dL/dh_t, starting from dfinal after the last token;
 *   g      += C_t dy_t^T                     (y_t = C_t^T h_t)
 *   dC_t   += h_t dy_t                        (summed over the heads of the group)
 *   dx_t    = g^T B_t + D dy_t                (h_t gains B_t x_t^T; y_t gains D x_t)
 *   dB_t   += g x_t                           (summed over the heads of the group)
 *   dlog_t  = a_t o rowsum(g o h_{t-1})       (h_t = a_t o h_{t-1} + ..., a_t = exp(dt_t A))
 *   ddt_t   = sum_n A_n dlog_t[n]             (scalar A: A sum_n dlog_t[n])
 *   dA     += dt_t dlog_t                     (scalar A: summed over n)
 *   dD     += dy_t . x_t
 *   g       = a_t o g                         (dL/dh_{t-1})
 * and dinit = g after the first token.  Outputs are fp64 in the input layouts
 * (dx (b,T,H,P), ddt (b,T,H), dA like A, dB and dC (b,T,G,N), dD (H), dinit
 * (b,H,N,P)); dD is written only when D is given.  The whole forward state of a
 * stream is kept (T+1 states), so this is for test sizes.  "plant" selects a
 * deliberately wrong variant for the tests (see PLANT_BWD_*); zero is the oracle.
 */
enum {
    PLANT_BWD_NONE = 0,
    PLANT_BWD_DLOG_NO_DECAY = 1,      /* dlog_t without the a_t factor */
    PLANT_BWD_DECAY_BEFORE_OUTPUT = 2, /* g decayed before C_t dy_t^T is added */
    PLANT_BWD_DX_NO_D = 3,            /* skip term missing from dx */
    PLANT_BWD_DB_USES_H = 4           /* dB_t from h_t instead of the adjoint */
};

int ssd_oracle_bwd(int64_t nb, int64_t T, int64_t H, int64_t P, int64_t N, int64_t G, int a_mode,
                   const float *x, const float *dt, const float *A, const float *B, const float *C,
                   const float *D, const float *init_state, const double *dy, const double *dfinal,
                   double *dx, double *ddt, double *dA, double *dB, double *dC, double *dD,
                   double *dinit, int nthreads, int plant)
{
    if (nb < 0 || T < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0) return 1;
    if (a_mode != 0 && a_mode != 1) return 1;
    const int64_t hpg = H / G, ns = nb * H;
    const int64_t nA = a_mode == 0 ? 1 : N;
    /* per-stream contributions to the gradients shared between streams */
    double *dB_s = (double *)calloc((size_t)(ns * T * N) + 1, sizeof(double));
    double *dC_s = (double *)calloc((size_t)(ns * T * N) + 1, sizeof(double));
    double *dA_s = (double *)calloc((size_t)(ns * nA), sizeof(double));
    double *dD_s = (double *)calloc((size_t)ns + 1, sizeof(double));
    if (!dB_s || !dC_s || !dA_s || !dD_s) { free(dB_s); free(dC_s); free(dA_s); free(dD_s); return 1; }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t s = 0; s < ns; ++s) {
        const int64_t bi = s / H, h = s % H, g = h / hpg;
        double *hs = (double *)malloc(sizeof(double) * (size_t)((T + 1) * N * P));
        double *gr = (double *)malloc(sizeof(double) * (size_t)(N * P));
        double *a = (double *)malloc(sizeof(double) * (size_t)N);
        double *dl = (double *)malloc(sizeof(double) * (size_t)N);
        if (!hs || !gr || !a || !dl) { free(hs); free(gr); free(a); free(dl); bad = 1; continue; }
        /* forward: hs[0] = h_{-1}, hs[t + 1] = h_t */
        for (int64_t i = 0; i < N * P; ++i)
            hs[i] = init_state ? (double)init_state[s * N * P + i] : 0.0;
        for (int64_t t = 0; t < T; ++t) {
            const int64_t tok = bi * T + t;
            const double dtv = (double)dt[tok * H + h];
            const float *xt = x + (tok * H + h) * P;
            const float *Bt = B + (tok * G + g) * N;
            const double *prev = hs + t * N * P;
            double *cur = hs + (t + 1) * N * P;
            for (int64_t n = 0; n < N; ++n) {
                const double an = exp(dtv * (double)(a_mode == 0 ? A[h] : A[h * N + n]));
                for (int64_t p = 0; p < P; ++p) cur[n * P + p] = an * prev[n * P + p] + (double)Bt[n] * (double)xt[p];
            }
        }
        /* reverse */
        for (int64_t i = 0; i < N * P; ++i) gr[i] = dfinal ? dfinal[s * N * P + i] : 0.0;
        for (int64_t t = T - 1; t >= 0; --t) {
            const int64_t tok = bi * T + t;
            const double dtv = (double)dt[tok * H + h];
            const float *xt = x + (tok * H + h) * P;
            const float *Bt = B + (tok * G + g) * N;
            const float *Ct = C + (tok * G + g) * N;
            const double *dyt = dy + (tok * H + h) * P;
            const double *prev = hs + t * N * P;
            const double *cur = hs + (t + 1) * N * P;
            for (int64_t n = 0; n < N; ++n) a[n] = exp(dtv * (double)(a_mode == 0 ? A[h] : A[h * N + n]));
            if (plant == PLANT_BWD_DECAY_BEFORE_OUTPUT)
                for (int64_t n = 0; n < N; ++n)
                    for (int64_t p = 0; p < P; ++p) gr[n * P + p] *= a[n];
            for (int64_t n = 0; n < N; ++n)
                for (int64_t p = 0; p < P; ++p) gr[n * P + p] += (double)Ct[n] * dyt[p];
            for (int64_t n = 0; n < N; ++n) {
                double c = 0.0, b = 0.0, l = 0.0;
                for (int64_t p = 0; p < P; ++p) {
                    c += cur[n * P + p] * dyt[p];
                    b += (plant == PLANT_BWD_DB_USES_H ? cur[n * P + p] : gr[n * P + p]) * (double)xt[p];
                    l += gr[n * P + p] * prev[n * P + p];
                }
                dC_s[(s * T + t) * N + n] = c;
                dB_s[(s * T + t) * N + n] = b;
                dl[n] = plant == PLANT_BWD_DLOG_NO_DECAY ? l : a[n] * l;
            }
            double *dxt = dx + (tok * H + h) * P;
            for (int64_t p = 0; p < P; ++p) {
                double acc = (D && plant != PLANT_BWD_DX_NO_D) ? (double)D[h] * dyt[p] : 0.0;
                for (int64_t n = 0; n < N; ++n) acc += (double)Bt[n] * gr[n * P + p];
                dxt[p] = acc;
            }
            double dd = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                const double An = (double)(a_mode == 0 ? A[h] : A[h * N + n]);
                dd += An * dl[n];
                dA_s[s * nA + (a_mode == 0 ? 0 : n)] += dtv * dl[n];
            }
            ddt[tok * H + h] = dd;
            double xd = 0.0;
            for (int64_t p = 0; p < P; ++p) xd += dyt[p] * (double)xt[p];
            dD_s[s] += xd;
            if (plant != PLANT_BWD_DECAY_BEFORE_OUTPUT)
                for (int64_t n = 0; n < N; ++n)
                    for (int64_t p = 0; p < P; ++p) gr[n * P + p] *= a[n];
        }
        if (dinit) memcpy(dinit + s * N * P, gr, sizeof(double) * (size_t)(N * P));
        free(hs);
        free(gr);
        free(a);
        free(dl);
    }
    /* reductions over the streams that share B/C (heads of a group) and A/D (batch rows) */
    for (int64_t bi = 0; bi < nb; ++bi)
        for (int64_t t = 0; t < T; ++t)
            for (int64_t g = 0; g < G; ++g)
                for (int64_t n = 0; n < N; ++n) {
                    double sb = 0.0, sc = 0.0;
                    for (int64_t h = g * hpg; h < (g + 1) * hpg; ++h) {
                        sb += dB_s[((bi * H + h) * T + t) * N + n];
                        sc += dC_s[((bi * H + h) * T + t) * N + n];
                    }
                    dB[((bi * T + t) * G + g) * N + n] = sb;
                    dC[((bi * T + t) * G + g) * N + n] = sc;
                }
    for (int64_t h = 0; h < H; ++h) {
        for (int64_t k = 0; k < nA; ++k) {
            double sa = 0.0;
            for (int64_t bi = 0; bi < nb; ++bi) sa += dA_s[(bi * H + h) * nA + k];
            dA[h * nA + k] = sa;
        }
        if (D && dD) {
            double sd = 0.0;
            for (int64_t bi = 0; bi < nb; ++bi) sd += dD_s[bi * H + h];
            dD[h] = sd;
        }
    }
    free(dB_s);
    free(dC_s);
    free(dA_s);
    free(dD_s);
    return bad ? 1 : 0;
}

/* Threads an OpenMP parallel region would use with the given request. */
int ssd_oracle_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
    int used = 1;
#pragma omp parallel
    {
#pragma omp single
        used = omp_get_num_threads();
    }
    return used;
#else
    (void)nthreads;
    return 1;
#endif
}
