/*
 * Float64 CPU oracle for the selective diagonal state-space scan.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call this file:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code with the CUDA library.
 *
 * What it computes follows the page "pssa_kernels.py" (NSC64/pssa-100m: "Fused
 * Triton scan for the PSSA selective diagonal state-space recurrence"):
 *   - its module docstring states the recurrence
 *         h_t = exp(delta_t * A) * h_{t-1} + delta_t * b_t * x_t,
 *         y_t = <h_t, c_t>,
 *     with A (D, DS) negative, delta (B, T, D) positive, b and c (B, T, DS),
 *     and the state carried from h0 to hT;
 *   - its plain loop `scan_reference` fixes that y_t reads the state after the
 *     update at step t, and that hT is the state after the last step;
 *   - its `scan_bwd` kernel fixes the reverse sweep: the adjoint of h_t is
 *     dy_t c_t plus the next step's decay times the next adjoint, and the
 *     gradient of h0 is the first decay times the first adjoint.
 * The checkpoint output follows the chunk-boundary retention of the ruDNN
 * page ("src/kda/chunk.rs", `chunk_kda`): slot j holds the state entering
 * chunk j of length K, so slot 0 is h0.
 *
 * The backward is derived by hand from the forward (chain rule), with
 *     L = sum dy * y + sum ghT * hT,   g_t = dL/dh_t:
 *     g_{T-1} = dy_{T-1} c_{T-1} + ghT,     g_t = dy_t c_t + a_{t+1} g_{t+1}
 *     p_t     = g_t * a_t * h_{t-1}
 *     gdelta  = sum_s (p_t A + g_t b_t x_t)       gx = delta_t sum_s g_t b_t
 *     gb[b,t,s] = sum_d g_t delta_t x_t           gc[b,t,s] = sum_d dy_t h_t
 *     gA[d,s]   = sum_{b,t} p_t delta_t           gh0 = a_0 g_0
 *
 * Layouts (row-major, contiguous, float64):
 *   x, delta, y, dy, gx, gdelta: (B, T, D)   b, c, gb, gc: (B, T, DS)
 *   A, gA: (D, DS)   h0, hT, ghT, gh0: (B, D, DS)   ckpt: (ceil(T/K), B, D, DS)
 *
 * Every (b, d) chain is independent; chains run in parallel with OpenMP. The
 * sums over chains (gb, gc over d; gA over b) use a fixed partition of d into
 * blocks and a fixed summation order, so results do not depend on the number
 * of threads. Build with -ffp-contract=off so that no multiply-add is fused and
 * the result is the same on every host.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int ssm_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Forward scan. h0 may be NULL (zero initial state); hT may be NULL; ckpt is
 * written when K > 0 and ckpt != NULL. Returns 0, or 1 on bad sizes. */
int ssm_oracle_fwd(int64_t B, int64_t T, int64_t D, int64_t DS,
                   const double* x, const double* delta, const double* A,
                   const double* bm, const double* cm, const double* h0,
                   double* y, double* hT, int64_t K, double* ckpt)
{
    if (B < 0 || T < 0 || D < 0 || DS <= 0 || K < 0) return 1;
    const int64_t nck = (K > 0) ? (T + K - 1) / K : 0;
    int64_t chain;
#pragma omp parallel for schedule(dynamic, 4)
    for (chain = 0; chain < B * D; chain++) {
        const int64_t b = chain / D, d = chain % D;
        double* h = (double*)malloc(sizeof(double) * DS);
        for (int64_t s = 0; s < DS; s++)
            h[s] = h0 ? h0[(b * D + d) * DS + s] : 0.0;
        for (int64_t t = 0; t < T; t++) {
            if (K > 0 && ckpt && t % K == 0) {
                const int64_t j = t / K;
                for (int64_t s = 0; s < DS; s++)
                    ckpt[((j * B + b) * D + d) * DS + s] = h[s];
            }
            const double dt = delta[(b * T + t) * D + d];
            const double xt = x[(b * T + t) * D + d];
            double acc = 0.0;
            for (int64_t s = 0; s < DS; s++) {
                const double a = exp(dt * A[d * DS + s]);
                const double u = dt * bm[(b * T + t) * DS + s] * xt;
                h[s] = a * h[s] + u;
                acc += h[s] * cm[(b * T + t) * DS + s];
            }
            y[(b * T + t) * D + d] = acc;
        }
        if (hT)
            for (int64_t s = 0; s < DS; s++) hT[(b * D + d) * DS + s] = h[s];
        free(h);
    }
    (void)nck;
    return 0;
}

/* Backward of the forward above for L = sum dy*y + sum ghT*hT. h0 and ghT may
 * be NULL (zeros). All outputs are overwritten. Returns 0, 1 on bad sizes,
 * 2 if memory runs out. */
int ssm_oracle_bwd(int64_t B, int64_t T, int64_t D, int64_t DS,
                   const double* x, const double* delta, const double* A,
                   const double* bm, const double* cm, const double* h0,
                   const double* dy, const double* ghT,
                   double* gx, double* gdelta, double* gA, double* gb, double* gc,
                   double* gh0)
{
    if (B < 0 || T < 0 || D < 0 || DS <= 0) return 1;
    const int64_t nblk = D < 16 ? D : 16;          /* fixed partition of d */
    const int64_t per_bs = B * T * DS;
    memset(gA, 0, sizeof(double) * D * DS);
    memset(gb, 0, sizeof(double) * per_bs);
    memset(gc, 0, sizeof(double) * per_bs);
    if (nblk == 0) {
        for (int64_t i = 0; i < B * D * DS; i++) gh0[i] = 0.0;
        return 0;
    }
    double* gb_part = (double*)calloc((size_t)(nblk * per_bs) + 1, sizeof(double));
    double* gc_part = (double*)calloc((size_t)(nblk * per_bs) + 1, sizeof(double));
    if (!gb_part || !gc_part) { free(gb_part); free(gc_part); return 2; }
    int failed = 0;
    int64_t blk;
#pragma omp parallel for schedule(dynamic, 1)
    for (blk = 0; blk < nblk; blk++) {
        const int64_t d_lo = D * blk / nblk, d_hi = D * (blk + 1) / nblk;
        double* Hs = (double*)malloc(sizeof(double) * (size_t)((T + 1) * DS)); /* Hs[t+1] = h_t */
        double* g = (double*)malloc(sizeof(double) * DS);
        if (!Hs || !g) { failed = 1; free(Hs); free(g); continue; }
        double* gbp = gb_part + blk * per_bs;
        double* gcp = gc_part + blk * per_bs;
        for (int64_t d = d_lo; d < d_hi; d++) {
            for (int64_t b = 0; b < B; b++) {
                /* forward, keeping the whole state history of this chain */
                for (int64_t s = 0; s < DS; s++)
                    Hs[s] = h0 ? h0[(b * D + d) * DS + s] : 0.0;
                for (int64_t t = 0; t < T; t++) {
                    const double dt = delta[(b * T + t) * D + d];
                    const double xt = x[(b * T + t) * D + d];
                    for (int64_t s = 0; s < DS; s++) {
                        const double a = exp(dt * A[d * DS + s]);
                        Hs[(t + 1) * DS + s] = a * Hs[t * DS + s] + dt * bm[(b * T + t) * DS + s] * xt;
                    }
                }
                /* reverse sweep; g holds the carried part a_{t+1} g_{t+1} on entry */
                for (int64_t s = 0; s < DS; s++)
                    g[s] = ghT ? ghT[(b * D + d) * DS + s] : 0.0;
                for (int64_t t = T - 1; t >= 0; t--) {
                    const double dt = delta[(b * T + t) * D + d];
                    const double xt = x[(b * T + t) * D + d];
                    const double dyt = dy[(b * T + t) * D + d];
                    double q = 0.0, r = 0.0;
                    for (int64_t s = 0; s < DS; s++) {
                        const int64_t bts = (b * T + t) * DS + s;
                        g[s] = dyt * cm[bts] + g[s];                 /* g_t */
                        const double a = exp(dt * A[d * DS + s]);
                        const double p = g[s] * a * Hs[t * DS + s]; /* Hs[t] = h_{t-1} */
                        gA[d * DS + s] += p * dt;
                        r += p * A[d * DS + s];
                        q += g[s] * bm[bts];
                        gbp[bts] += g[s] * dt * xt;
                        gcp[bts] += dyt * Hs[(t + 1) * DS + s];
                        g[s] = a * g[s];                             /* carry to step t-1 */
                    }
                    gx[(b * T + t) * D + d] = dt * q;
                    gdelta[(b * T + t) * D + d] = r + xt * q;
                }
                for (int64_t s = 0; s < DS; s++) gh0[(b * D + d) * DS + s] = g[s];
            }
        }
        free(Hs);
        free(g);
    }
    if (!failed) {
        for (blk = 0; blk < nblk; blk++) {          /* fixed order over blocks */
            const double* gbp = gb_part + blk * per_bs;
            const double* gcp = gc_part + blk * per_bs;
            for (int64_t i = 0; i < per_bs; i++) { gb[i] += gbp[i]; gc[i] += gcp[i]; }
        }
    }
    free(gb_part);
    free(gc_part);
    return failed ? 2 : 0;
}
