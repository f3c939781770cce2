/*
 * ssd_oracle.c -- float64 CPU oracle for the Mamba-2 SSD forward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the SSD forward computes.  It shares no code, header,
 * table or constant with the CUDA library; only tests, the smoke check and
 * the benchmark's CPU-baseline leg may load it.
 *
 * What it computes (the definition, token by token, no chunking):
 *   "Mamba-2 SSD for Ascend NPU" README, sections "Usage" and "Implementation"
 *   (public tensors x[B,L,H,P], dt[B,L,H], A[H], B,C[B,L,G,N],
 *   initial_states/final_state[B,H,P,N]; features D, z, dt_bias,
 *   dt_softplus, dt_limit), and the ops-transformer MambaV2 article,
 *   section 1.1 (h(t) = Abar h(t-1) + Bbar x(t), y(t) = C h(t), with Abar, Bbar
 *   from the input-dependent step Delta).  With the Mamba-2 discretisation:
 *
 *     d_t   = clamp(softplus(dt[b,t,h] + dt_bias[h]))     (bias, softplus and
 *             clamp each optional; "Preprocess: softplus / clamp / decay")
 *     a_t   = exp(d_t * A[h])
 *     h_t   = a_t * h_{t-1} + d_t * x_t (outer) B_t        h_t is [P,N]
 *     y_t   = h_t . C_t  (+ D[h] * x_t)  (* silu(z_t))
 *
 *   with group g = h / (H/G) supplying B and C to its H/G heads.
 *
 * Precision: every input is widened exactly from float32 to double and all
 * arithmetic is double, no fast-math.  Inputs stored as bf16/fp16 by a caller
 * are widened to float32 (exact) before they reach this file.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int64_t B, L, H, P, N, G;
    const float *x;        /* [B,L,H,P] */
    const float *dt;       /* [B,L,H]   */
    const float *A;        /* [H]       */
    const float *Bm;       /* [B,L,G,N] */
    const float *Cm;       /* [B,L,G,N] */
    const float *D;        /* [H] or NULL */
    const float *z;        /* [B,L,H,P] or NULL */
    const float *dt_bias;  /* [H] or NULL */
    const float *h0;       /* [B,H,P,N] or NULL */
    int dt_softplus;       /* nonzero: d = softplus(dt + bias) */
    int has_dt_limit;      /* nonzero: clamp d to [dt_min, dt_max] */
    double dt_min, dt_max;
} oracle_problem;

/* softplus(u) = log(1 + e^u), written so that neither branch overflows. */
double oracle_softplus(double u)
{
    if (u > 0.0)
        return u + log1p(exp(-u));
    return log1p(exp(u));
}

/* The processed step d_t for one raw dt value of head h
 * (order: add bias, then softplus, then clamp). */
double oracle_dt_processed(const oracle_problem *p, double raw, int64_t h)
{
    double u = raw;
    if (p->dt_bias)
        u += (double)p->dt_bias[h];
    double d = p->dt_softplus ? oracle_softplus(u) : u;
    if (p->has_dt_limit) {
        if (d < p->dt_min) d = p->dt_min;
        if (d > p->dt_max) d = p->dt_max;
    }
    return d;
}

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Run the recurrence for the (b,h) pairs listed in bh (bh[2i] = b,
 * bh[2i+1] = h).
 *
 *   y            [nbh, L, P]   or NULL
 *   final_state  [nbh, P, N]   or NULL   (state after token L-1)
 *   chunk_states [nbh, c, P, N] or NULL, c = ceil(L/chunk): the state
 *                entering chunk k, i.e. h_{k*chunk-1} (h0 for k = 0).
 *
 * Returns 0 on success, -1 on a bad argument.
 */
int oracle_recurrence(const oracle_problem *p, const int64_t *bh, int64_t nbh,
                      double *y, double *final_state, int64_t chunk,
                      double *chunk_states, int nthreads)
{
    if (!p || !bh || nbh < 0) return -1;
    if (p->B < 0 || p->L < 0 || p->H <= 0 || p->P <= 0 || p->N <= 0 || p->G <= 0) return -1;
    if (p->H % p->G != 0) return -1;
    if (chunk_states && chunk <= 0) return -1;
    const int64_t L = p->L, H = p->H, P = p->P, N = p->N, G = p->G;
    const int64_t heads_per_group = H / G;
    const int64_t nchunks = (chunk > 0) ? (L + chunk - 1) / chunk : 0;
    for (int64_t i = 0; i < nbh; ++i)
        if (bh[2 * i] < 0 || bh[2 * i] >= p->B || bh[2 * i + 1] < 0 || bh[2 * i + 1] >= H)
            return -1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

    int status = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(P * N));
        if (!s) {
#pragma omp atomic write
            status = -1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nbh; ++i) {
            if (!s) continue;
            const int64_t b = bh[2 * i], h = bh[2 * i + 1];
            const int64_t g = h / heads_per_group;
            if (p->h0) {
                const float *h0 = p->h0 + (b * H + h) * P * N;
                for (int64_t e = 0; e < P * N; ++e) s[e] = (double)h0[e];
            } else {
                memset(s, 0, sizeof(double) * (size_t)(P * N));
            }
            if (chunk_states && nchunks > 0)
                memcpy(chunk_states + (i * nchunks) * P * N, s, sizeof(double) * (size_t)(P * N));
            const double Ah = (double)p->A[h];
            const double Dh = p->D ? (double)p->D[h] : 0.0;
            for (int64_t t = 0; t < L; ++t) {
                const double d = oracle_dt_processed(p, (double)p->dt[(b * L + t) * H + h], h);
                const double a = exp(d * Ah);
                const float *xt = p->x + ((b * L + t) * H + h) * P;
                const float *Bt = p->Bm + ((b * L + t) * G + g) * N;
                const float *Ct = p->Cm + ((b * L + t) * G + g) * N;
                const float *zt = p->z ? p->z + ((b * L + t) * H + h) * P : NULL;
                for (int64_t pp = 0; pp < P; ++pp) {
                    const double xv = (double)xt[pp];
                    const double dx = d * xv;
                    double *row = s + pp * N;
                    double acc = 0.0;
                    for (int64_t n = 0; n < N; ++n) {
                        row[n] = a * row[n] + dx * (double)Bt[n];
                        acc += (double)Ct[n] * row[n];
                    }
                    if (p->D) acc += Dh * xv;
                    if (zt) {
                        const double zv = (double)zt[pp];
                        acc *= zv / (1.0 + exp(-zv));
                    }
                    if (y) y[(i * L + t) * P + pp] = acc;
                }
                if (chunk_states && (t + 1) % chunk == 0 && (t + 1) / chunk < nchunks)
                    memcpy(chunk_states + (i * nchunks + (t + 1) / chunk) * P * N, s,
                           sizeof(double) * (size_t)(P * N));
            }
            if (final_state)
                memcpy(final_state + i * P * N, s, sizeof(double) * (size_t)(P * N));
        }
        free(s);
    }
    return status;
}

/*
 * Stage view of the same definition, for checking the chunked steps one at a
 * time (ops-transformer MambaV2 article, sections 4.2-4.4: chunk_cumsum,
 * chunk_state, chunk_state_passing).
 *
 * oracle_chunk_cumsum: for every (b,h,k,i) with token t = k*chunk + i,
 *   dtp[b,h,k,i] = d_t                       (0 past the end, t >= L)
 *   cs [b,h,k,i] = sum_{j<=i} d_{k*chunk+j} * A[h]
 * Past the end the step is zero, so cs keeps its last valid value (the tail
 * rule of the MindSpeed-Ops Mamba-3 notes, "non-integer chunk": pad with
 * zeros and extend the cumulative decay with its last value).
 * Layout of both outputs: [B, H, c, chunk], c = ceil(L/chunk).
 */
int oracle_chunk_cumsum(const oracle_problem *p, int64_t chunk, double *dtp, double *cs)
{
    if (!p || chunk <= 0 || !dtp || !cs) return -1;
    const int64_t B = p->B, L = p->L, H = p->H;
    const int64_t nchunks = (L + chunk - 1) / chunk;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t k = 0; k < nchunks; ++k) {
                double run = 0.0;
                for (int64_t i = 0; i < chunk; ++i) {
                    const int64_t t = k * chunk + i;
                    const int64_t o = ((b * H + h) * nchunks + k) * chunk + i;
                    double d = 0.0;
                    if (t < L) d = oracle_dt_processed(p, (double)p->dt[(b * L + t) * H + h], h);
                    run += d * (double)p->A[h];
                    dtp[o] = d;
                    cs[o] = run;
                }
            }
    return 0;
}

/*
 * oracle_chunk_local_states: the state each chunk produces on its own, i.e.
 * the recurrence run over chunk k alone from a zero state (what the
 * chunk_state step hands to state passing).  Output [nbh, c, P, N].
 */
int oracle_chunk_local_states(const oracle_problem *p, const int64_t *bh, int64_t nbh,
                              int64_t chunk, double *out, int nthreads)
{
    if (!p || !bh || nbh < 0 || chunk <= 0 || !out) return -1;
    if (p->H % p->G != 0) return -1;
    const int64_t L = p->L, H = p->H, P = p->P, N = p->N, G = p->G;
    const int64_t heads_per_group = H / G;
    const int64_t nchunks = (L + chunk - 1) / chunk;
    for (int64_t i = 0; i < nbh; ++i)
        if (bh[2 * i] < 0 || bh[2 * i] >= p->B || bh[2 * i + 1] < 0 || bh[2 * i + 1] >= H)
            return -1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t w = 0; w < nbh * nchunks; ++w) {
        const int64_t i = w / nchunks, k = w % nchunks;
        const int64_t b = bh[2 * i], h = bh[2 * i + 1];
        const int64_t g = h / heads_per_group;
        double *s = out + (i * nchunks + k) * P * N;
        memset(s, 0, sizeof(double) * (size_t)(P * N));
        const double Ah = (double)p->A[h];
        for (int64_t t = k * chunk; t < (k + 1) * chunk && t < L; ++t) {
            const double d = oracle_dt_processed(p, (double)p->dt[(b * L + t) * H + h], h);
            const double a = exp(d * Ah);
            const float *xt = p->x + ((b * L + t) * H + h) * P;
            const float *Bt = p->Bm + ((b * L + t) * G + g) * N;
            for (int64_t pp = 0; pp < P; ++pp) {
                const double dx = d * (double)xt[pp];
                double *row = s + pp * N;
                for (int64_t n = 0; n < N; ++n) row[n] = a * row[n] + dx * (double)Bt[n];
            }
        }
    }
    return 0;
}

/*
 * Backward of the recurrence above (the SSD backward: gradients of
 * L = sum_t dy_t . y_t + <dfinal, final_state> with respect to every input).
 * Written as the adjoint of the token recurrence, in reverse token order:
 *
 *   g        = dfinal                                  (dL/dh_{L-1} via the final state)
 *   for t = L-1 .. 0:
 *     dyp_t  = dy_t * silu(z_t)                        (no gate: dyp_t = dy_t)
 *     dz_t   = dy_t * (h_t . C_t + D x_t) * silu'(z_t)
 *     g     += dyp_t (outer) C_t                       (now dL/dh_t)
 *     dC_t   = sum_p dyp_t[p] h_t[p,:]
 *     dx_t   = d_t (g B_t) + D dyp_t
 *     dB_t   = d_t (g^T x_t)
 *     dd_t   = <g, x_t (outer) B_t> + A a_t <g, h_{t-1}>
 *     dA    += d_t a_t <g, h_{t-1}>,  dD += dyp_t . x_t
 *     ddt_t  = dd_t * softplus'(dt_t + bias) (* 1 inside the dt_limit clamp, 0 outside)
 *     dbias += ddt_t
 *     g      = a_t g                                   (dL/dh_{t-1})
 *   dh0 = g
 *
 * per (b, h) pair listed in bh; dB and dC are this head's contributions (the
 * caller sums the heads of a group), dA, dD and dbias this pair's (summed
 * over b by the caller).  Keeps every h_t of the pair: [L,P,N] doubles.
 * Outputs (nbh leading): dx [L,P], dB, dC [L,N], ddt [L], dA, dD, dbias [1],
 * dz [L,P] (or NULL), dh0 [P,N].
 */
int oracle_backward(const oracle_problem *p, const int64_t *bh, int64_t nbh, const float *dy,
                    const float *dfinal, double *dx, double *dB, double *dC, double *ddt, double *dA,
                    double *dD, double *dbias, double *dz, double *dh0, int nthreads)
{
    if (!p || !bh || nbh < 0 || !dy) return -1;
    if (p->B < 0 || p->L < 0 || p->H <= 0 || p->P <= 0 || p->N <= 0 || p->G <= 0) return -1;
    if (p->H % p->G != 0) return -1;
    const int64_t L = p->L, H = p->H, P = p->P, N = p->N, G = p->G;
    const int64_t heads_per_group = H / G;
    for (int64_t i = 0; i < nbh; ++i)
        if (bh[2 * i] < 0 || bh[2 * i] >= p->B || bh[2 * i + 1] < 0 || bh[2 * i + 1] >= H) return -1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int status = 0;
#pragma omp parallel
    {
        double *hs = (double *)malloc(sizeof(double) * (size_t)((L + 1) * P * N));  /* h_{-1} .. h_{L-1} */
        double *g = (double *)malloc(sizeof(double) * (size_t)(P * N));
        double *dd_raw = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double *av = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        if (!hs || !g || !dd_raw || !av) {
#pragma omp atomic write
            status = -1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nbh; ++i) {
            if (!hs || !g || !dd_raw || !av) continue;
            const int64_t b = bh[2 * i], h = bh[2 * i + 1];
            const int64_t gg = h / heads_per_group;
            const double Ah = (double)p->A[h];
            const double Dh = p->D ? (double)p->D[h] : 0.0;
            /* forward, keeping every state */
            for (int64_t e = 0; e < P * N; ++e)
                hs[e] = p->h0 ? (double)p->h0[(b * H + h) * P * N + e] : 0.0;
            for (int64_t t = 0; t < L; ++t) {
                const double raw = (double)p->dt[(b * L + t) * H + h];
                const double d = oracle_dt_processed(p, raw, h);
                const double a = exp(d * Ah);
                av[t] = a;
                dd_raw[t] = d;
                const float *xt = p->x + ((b * L + t) * H + h) * P;
                const float *Bt = p->Bm + ((b * L + t) * G + gg) * N;
                const double *prev = hs + t * P * N;
                double *cur = hs + (t + 1) * P * N;
                for (int64_t pp = 0; pp < P; ++pp)
                    for (int64_t n = 0; n < N; ++n)
                        cur[pp * N + n] = a * prev[pp * N + n] + d * (double)xt[pp] * (double)Bt[n];
            }
            /* backward */
            for (int64_t e = 0; e < P * N; ++e) g[e] = dfinal ? (double)dfinal[i * P * N + e] : 0.0;
            double sA = 0.0, sD = 0.0, sbias = 0.0;
            for (int64_t t = L - 1; t >= 0; --t) {
                const double d = dd_raw[t], a = av[t];
                const float *xt = p->x + ((b * L + t) * H + h) * P;
                const float *Bt = p->Bm + ((b * L + t) * G + gg) * N;
                const float *Ct = p->Cm + ((b * L + t) * G + gg) * N;
                const float *zt = p->z ? p->z + ((b * L + t) * H + h) * P : NULL;
                const double *ht = hs + (t + 1) * P * N, *hprev = hs + t * P * N;
                const float *dyt = dy + (i * L + t) * P;
                for (int64_t pp = 0; pp < P; ++pp) {
                    double dyp = (double)dyt[pp];
                    if (zt) {
                        const double zv = (double)zt[pp];
                        const double sg = 1.0 / (1.0 + exp(-zv));
                        double ypre = Dh * (double)xt[pp];
                        for (int64_t n = 0; n < N; ++n) ypre += ht[pp * N + n] * (double)Ct[n];
                        if (dz) dz[(i * L + t) * P + pp] = dyp * ypre * sg * (1.0 + zv * (1.0 - sg));
                        dyp *= zv * sg;
                    } else if (dz) {
                        dz[(i * L + t) * P + pp] = 0.0;
                    }
                    sD += dyp * (double)xt[pp];
                    for (int64_t n = 0; n < N; ++n) g[pp * N + n] += dyp * (double)Ct[n];
                    if (dx) dx[(i * L + t) * P + pp] = Dh * dyp;  /* + d (g B)[p] below */
                    if (dC)
                        for (int64_t n = 0; n < N; ++n)
                            dC[(i * L + t) * N + n] = (pp == 0 ? 0.0 : dC[(i * L + t) * N + n]) + dyp * ht[pp * N + n];
                }
                double e_t = 0.0, q_t = 0.0;
                for (int64_t n = 0; n < N; ++n) if (dB) dB[(i * L + t) * N + n] = 0.0;
                for (int64_t pp = 0; pp < P; ++pp) {
                    double gb = 0.0;
                    for (int64_t n = 0; n < N; ++n) {
                        const double gv = g[pp * N + n];
                        gb += gv * (double)Bt[n];
                        q_t += gv * hprev[pp * N + n];
                        if (dB) dB[(i * L + t) * N + n] += d * gv * (double)xt[pp];
                    }
                    e_t += gb * (double)xt[pp];
                    if (dx) dx[(i * L + t) * P + pp] += d * gb;
                }
                const double ddv = e_t + Ah * a * q_t;
                sA += d * a * q_t;
                /* through the clamp and softplus, back to the raw dt */
                double u = (double)p->dt[(b * L + t) * H + h];
                if (p->dt_bias) u += (double)p->dt_bias[h];
                double dpre = p->dt_softplus ? oracle_softplus(u) : u;
                double gr = ddv;
                if (p->has_dt_limit && (dpre < p->dt_min || dpre > p->dt_max)) gr = 0.0;
                if (p->dt_softplus) gr *= 1.0 / (1.0 + exp(-u));
                if (ddt) ddt[i * L + t] = gr;
                sbias += gr;
                for (int64_t e = 0; e < P * N; ++e) g[e] *= a;
            }
            if (dA) dA[i] = sA;
            if (dD) dD[i] = sD;
            if (dbias) dbias[i] = sbias;
            if (dh0) memcpy(dh0 + i * P * N, g, sizeof(double) * (size_t)(P * N));
        }
        free(hs);
        free(g);
        free(dd_raw);
        free(av);
    }
    return status;
}
