/*
 * Float64 CPU oracle in plain C: the Mamba-2 SSD recurrence and the scalar
 * selective scan, written as their definitions (sequential in t).
 *
 * TEST INFRASTRUCTURE ONLY.  The CUDA library never includes, links or calls
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark load it (through oracle/native.py).  It shares no header, helper
 * or constant with the CUDA sources.
 *
 * SSD: "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
 * NVIDIA CUDA Tile", section "Mamba-2 architecture":
 *     h_t = exp(A dt_t) h_{t-1} + x_t (dt_t B_t)^T     (state H x S per head)
 *     y_t = h_t c_t + D x_t                              (inclusive reading)
 * Scan: "Selective-scan CUDA kernels", section "The problem":
 *     h[t] = a[t] h[t-1] + b[t],  h[-1] = 0.
 *
 * Inputs are float32 arrays (bf16 workloads pass bf16-exact values), every
 * operation is in double.  Independent units ((batch, head) pairs for the
 * SSD, rows for the scan) are spread over OpenMP threads; t stays sequential.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/*
 * units[u] = batch * nheads + head selects which (batch, head) pairs are
 * computed.  y_out is [n_units, L, H] and hfinal_out is [n_units, H, S]
 * (either may be NULL).  h0 is float64 [batch, nheads, H, S] so a final
 * state can be fed back unrounded; it may be NULL (zeros).  Returns 0, or -1 on a bad
 * argument, -2 on allocation failure.  threads <= 0 takes the OpenMP default; the count
 * applies to this call only.
 */
int ssm_oracle_ssd(const float *x, const float *dt, const float *A, const float *B,
                   const float *C, const float *D, const double *h0,
                   double *y_out, double *hfinal_out,
                   int64_t batch, int64_t L, int64_t nheads, int64_t H, int64_t S,
                   int64_t ngroups, const int64_t *units, int64_t n_units, int threads)
{
    if (batch < 1 || L < 0 || nheads < 1 || H < 1 || S < 1 || ngroups < 1 ||
        nheads % ngroups != 0 || n_units < 0)
        return -1;
    for (int64_t u = 0; u < n_units; ++u)
        if (units[u] < 0 || units[u] >= batch * nheads)
            return -1;
    const int64_t heads_per_group = nheads / ngroups;
    int failed = 0;
#ifdef _OPENMP
    const int nt = threads > 0 ? threads : omp_get_max_threads();  /* this call only */
#else
    (void)threads;
#endif
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed) num_threads(nt)
    for (int64_t u = 0; u < n_units; ++u) {
        const int64_t bi = units[u] / nheads;
        const int64_t hi = units[u] % nheads;
        const int64_t gi = hi / heads_per_group;
        double *state = (double *)malloc(sizeof(double) * (size_t)(H * S));
        double *bt = (double *)malloc(sizeof(double) * (size_t)S);
        if (!state || !bt) {
            free(state);
            free(bt);
            failed = 1;
            continue;
        }
        for (int64_t i = 0; i < H * S; ++i)
            state[i] = h0 ? h0[(bi * nheads + hi) * H * S + i] : 0.0;
        const double Ah = (double)A[hi], Dh = (double)D[hi];
        for (int64_t t = 0; t < L; ++t) {
            const double dtt = (double)dt[(bi * L + t) * nheads + hi];
            const double decay = exp(Ah * dtt);
            const float *xt = x + ((bi * L + t) * nheads + hi) * H;
            const float *Bt = B + ((bi * L + t) * ngroups + gi) * S;
            const float *Ct = C + ((bi * L + t) * ngroups + gi) * S;
            for (int64_t s = 0; s < S; ++s)
                bt[s] = dtt * (double)Bt[s];
            for (int64_t p = 0; p < H; ++p) {
                double *row = state + p * S;
                const double xp = (double)xt[p];
                double acc = 0.0;
                for (int64_t s = 0; s < S; ++s) {
                    row[s] = decay * row[s] + xp * bt[s];
                    acc += row[s] * (double)Ct[s];
                }
                if (y_out)
                    y_out[(u * L + t) * H + p] = acc + Dh * xp;
            }
        }
        if (hfinal_out)
            memcpy(hfinal_out + u * H * S, state, sizeof(double) * (size_t)(H * S));
        free(state);
        free(bt);
    }
    return failed ? -2 : 0;
}

/*
 * rows_sel[r] picks the rows of the [rows, L] inputs to scan; h_out is
 * [n_sel, L].  Returns 0, or -1 on a bad argument.
 */
int ssm_oracle_linscan(const float *a, const float *b, double *h_out,
                       int64_t rows, int64_t L, const int64_t *rows_sel, int64_t n_sel, int threads)
{
    if (rows < 0 || L < 0 || n_sel < 0)
        return -1;
    for (int64_t r = 0; r < n_sel; ++r)
        if (rows_sel[r] < 0 || rows_sel[r] >= rows)
            return -1;
#ifdef _OPENMP
    const int nt = threads > 0 ? threads : omp_get_max_threads();  /* this call only */
#else
    (void)threads;
#endif
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int64_t r = 0; r < n_sel; ++r) {
        const float *ar = a + rows_sel[r] * L;
        const float *br = b + rows_sel[r] * L;
        double *hr = h_out + r * L;
        double h = 0.0;
        for (int64_t t = 0; t < L; ++t) {
            h = (double)ar[t] * h + (double)br[t];
            hr[t] = h;
        }
    }
    return 0;
}

int ssm_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
