/*
 * Selective state-space scan of a Mamba2 layer (the SSD recurrence) in fp64
 * on the CPU: the oracle for the context-parallel SSM path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg use it.  It shares no code with the CUDA library.
 *
 * The axolotl "Sequence Parallelism" page ("Mamba/SSM Hybrid Models") says
 * SSM layers are recurrent: under context parallelism each rank scans its
 * chunk, the final hidden state goes to the next rank, and an additive
 * correction (the SSM is linear in its initial state) accounts for the state
 * the rank did not start from; packed samples reset the state at their
 * boundaries, found from position_ids.  The page gives no formula, so the
 * oracle is the recurrence itself over the WHOLE, unsharded sequence, in
 * token order (the plainest reading of a Mamba2 layer's scan):
 *
 *   for each head h (group g = h / (H / G)) and token t:
 *     if pos[t] == 0 (a packed sample starts): state <- 0
 *     a      = exp(dt[t,h] * A[h])
 *     S[p,n] = a * S[p,n] + dt[t,h] * x[t,h,p] * B[t,g,n]
 *     y[t,h,p] = sum_n S[p,n] * C[t,g,n] + D[h] * x[t,h,p]
 *
 * starting from S = h0[h] (or 0).  Layouts: x, y [T, H, P]; dt [T, H];
 * A, D [H]; B, C [T, G, N]; h0, hT [H, P, N]; row-major doubles.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

int oracle_ssd_scan(const double *x, const double *dt, const double *A, const double *B,
                    const double *C, const double *D, const int32_t *pos, int T, int H, int P,
                    int N, int G, const double *h0, double *y, double *hT)
{
    if (T < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G) return -1;
    int per_group = H / G;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int h = 0; h < H; ++h) {
        double *S = (double *)malloc(sizeof(double) * (size_t)P * N);
        if (!S) {
#pragma omp atomic write
            err = -2;
            continue;
        }
        if (h0)
            memcpy(S, h0 + (size_t)h * P * N, sizeof(double) * (size_t)P * N);
        else
            memset(S, 0, sizeof(double) * (size_t)P * N);
        int g = h / per_group;
        for (int t = 0; t < T; ++t) {
            if (pos && pos[t] == 0) memset(S, 0, sizeof(double) * (size_t)P * N);
            double d = dt[(size_t)t * H + h];
            double a = exp(d * A[h]);
            const double *xt = x + ((size_t)t * H + h) * P;
            const double *Bt = B + ((size_t)t * G + g) * N;
            const double *Ct = C + ((size_t)t * G + g) * N;
            double *yt = y + ((size_t)t * H + h) * P;
            for (int p = 0; p < P; ++p) {
                double *Sp = S + (size_t)p * N;
                double acc = 0.0;
                for (int n = 0; n < N; ++n) {
                    Sp[n] = a * Sp[n] + d * xt[p] * Bt[n];
                    acc += Sp[n] * Ct[n];
                }
                yt[p] = acc + (D ? D[h] : 0.0) * xt[p];
            }
        }
        if (hT) memcpy(hT + (size_t)h * P * N, S, sizeof(double) * (size_t)P * N);
        free(S);
    }
    return err;
}
