/*
 * TEST INFRASTRUCTURE ONLY -- the fp64 CPU oracle of the Mamba-2 SSD forward.
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may load
 * this file's library. It shares no code with the CUDA path.
 *
 * What it computes: the plain token-by-token recurrence of the Mamba-2 layer,
 * as defined in "Accelerating Mamba-2 with High-Performance Forward Pass
 * Kernels in NVIDIA CUDA Tile", section "Mamba-2 architecture" (the core
 * recurrence and its output equation), which is the same per-token step as
 * "Optimizing Nemotron v3 Super in TensorRT-LLM", section 6.1 "The SSU Math":
 *
 *     alpha_t   = exp(A[h] * dt[b,t,h])
 *     S         = alpha_t * S + dt[b,t,h] * x[b,t,h,:] (outer) B[b,t,g,:]     (P x N)
 *     y[b,t,h,p] = sum_n S[p,n] * C[b,t,g,n] + D[h] * x[b,t,h,p]
 *
 * with the UPDATED state S = h_t in the output (the inclusive reading; the
 * page's shorthand with h_{t-1} contradicts its own first equation, its causal
 * mask i >= j, and the SSU step, all of which use the updated state).
 * Head h reads group g = h / (H / G) (contiguous heads per group, as in the
 * page's fwd_pass_state kernel). S starts at initial_states[b,h] or zero;
 * final_states[b,h] = S after the last token. D absent means zero.
 *
 * Arithmetic is fp64 on the stored input values, upcast exactly (fp32 and
 * bf16 are both exact in fp64). No cumsum, no chunking, no exp2.
 *
 * Layouts (contiguous, row-major):
 *   x  [B, L, H, P]     dt [B, L, H]     A [H]     D [H]
 *   Bm [B, L, G, N]     Cm [B, L, G, N]  h0 [B, H, P, N]
 * Outputs, for the requested (b,h) slabs only:
 *   y_out     [nslab, L, P]   (fp64)
 *   final_out [nslab, P, N]   (fp64)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2 };

/* Exact upcast of one stored element to double. bf16 is the top half of an
 * IEEE binary32, so widening it is a 16-bit shift. */
static double load_elem(const void *base, int dtype, int64_t i) {
    if (dtype == ORC_F64) return ((const double *)base)[i];
    if (dtype == ORC_F32) return (double)((const float *)base)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Returns 0 on success, -1 on a bad argument, -2 on allocation failure. */
int oracle_ssd_recurrence(const void *x, int x_dtype,
                          const void *dt, int dt_dtype,
                          const void *A, int A_dtype,
                          const void *Bm, const void *Cm, int bc_dtype,
                          const void *D, int D_dtype,     /* may be NULL */
                          const void *h0, int h0_dtype,   /* may be NULL */
                          int64_t B, int64_t L, int64_t H, int64_t P,
                          int64_t N, int64_t G,
                          const int64_t *slabs, int64_t nslab, /* flat b*H+h */
                          double *y_out, double *final_out, int nthreads) {
    if (B < 0 || L < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0)
        return -1;
    if (nslab < 0 || (nslab > 0 && (!slabs || !y_out || !final_out)))
        return -1;
    for (int64_t s = 0; s < nslab; ++s)
        if (slabs[s] < 0 || slabs[s] >= B * H) return -1;
    const int64_t heads_per_group = H / G;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
    for (int64_t s = 0; s < nslab; ++s) {
        const int64_t b = slabs[s] / H, h = slabs[s] % H;
        const int64_t g = h / heads_per_group;
        double *S = (double *)malloc(sizeof(double) * (size_t)(P * N));
        double *xv = (double *)malloc(sizeof(double) * (size_t)P);
        double *bv = (double *)malloc(sizeof(double) * (size_t)N);
        double *cv = (double *)malloc(sizeof(double) * (size_t)N);
        if (!S || !xv || !bv || !cv) {
            failed |= 1;
            free(S); free(xv); free(bv); free(cv);
            continue;
        }
        for (int64_t e = 0; e < P * N; ++e)
            S[e] = h0 ? load_elem(h0, h0_dtype, (b * H + h) * P * N + e) : 0.0;
        const double a_h = load_elem(A, A_dtype, h);
        const double d_h = D ? load_elem(D, D_dtype, h) : 0.0;
        double *y = y_out + s * L * P;
        for (int64_t t = 0; t < L; ++t) {
            const double dt_t = load_elem(dt, dt_dtype, (b * L + t) * H + h);
            const double alpha = exp(a_h * dt_t);
            for (int64_t p = 0; p < P; ++p)
                xv[p] = load_elem(x, x_dtype, ((b * L + t) * H + h) * P + p);
            for (int64_t n = 0; n < N; ++n) {
                bv[n] = load_elem(Bm, bc_dtype, ((b * L + t) * G + g) * N + n);
                cv[n] = load_elem(Cm, bc_dtype, ((b * L + t) * G + g) * N + n);
            }
            for (int64_t p = 0; p < P; ++p) {
                double *Sp = S + p * N;
                const double u = dt_t * xv[p];
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    Sp[n] = alpha * Sp[n] + u * bv[n];
                    acc += Sp[n] * cv[n];
                }
                y[t * P + p] = acc + d_h * xv[p];
            }
        }
        memcpy(final_out + s * P * N, S, sizeof(double) * (size_t)(P * N));
        free(S); free(xv); free(bv); free(cv);
    }
    return failed ? -2 : 0;
}

/* Number of threads OpenMP would use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
