/*
 * d3d_oracle_par.c -- all-cores driver of the oracle, for the CPU baseline.
 * TEST INFRASTRUCTURE ONLY (timed next to the CUDA path by the benchmark's
 * CPU legs; never called by the product path).
 *
 * This file adds no arithmetic: it runs the unchanged oracle functions of
 * d3d_oracle.c on disjoint parts of a problem from an OpenMP loop, so that
 * every output is computed by exactly the code, and in exactly the order,
 * that the one-thread oracle uses.
 *   - packed attention: one oracle_packed_attn_sel call per (request, query
 *     head), each over that request's packed rows and that one head;
 *   - verification: one oracle_spec_verify call per request (R = 1 on the
 *     request's slices of every array).
 * Built with -fopenmp into its own library; without OpenMP the pragmas are
 * ignored and the loops run on one thread.
 */
#include <stddef.h>
#include <stdint.h>

#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_packed_attn_sel(const uint16_t *q, const uint16_t *kp, const uint16_t *vp, const uint16_t *kn,
                           const uint16_t *vn, const int32_t *segs, const int32_t *cu_prefix, const int32_t *cu_q,
                           const int32_t *cu_seg, int R, int Hq, int Hkv, int d, double scale, int heads_lo,
                           int heads_hi, int tok_lo, int tok_hi, double *out);
int oracle_spec_verify(const void *target, const void *draft, int dtype, const int32_t *y, const float *u_acc,
                       const float *u_s, int R, int B, int V, double T, int32_t *accept_len, int32_t *out_tokens,
                       int32_t *num_tokens, double *alpha, double *p_out, double *q_out, double *margin_accept,
                       double *margin_sample, int32_t *used_fallback);

/* Threads the parallel loops use (the OpenMP default when n <= 0). */
int oracle_par_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

int oracle_packed_attn_par(const uint16_t *q, const uint16_t *kp, const uint16_t *vp, const uint16_t *kn,
                           const uint16_t *vn, const int32_t *segs, const int32_t *cu_prefix, const int32_t *cu_q,
                           const int32_t *cu_seg, int R, int Hq, int Hkv, int d, double scale, double *out)
{
    int rc = 0;
    const long long n = (long long)R * Hq;
#pragma omp parallel for schedule(dynamic, 1) reduction(min : rc)
    for (long long t = 0; t < n; ++t) {
        const int r = (int)(t / Hq), h = (int)(t % Hq);
        const int e = oracle_packed_attn_sel(q, kp, vp, kn, vn, segs, cu_prefix, cu_q, cu_seg, R, Hq, Hkv, d, scale,
                                             h, h + 1, cu_q[r], cu_q[r + 1], out);
        rc = e < rc ? e : rc;
    }
    return rc;
}

/* The optional outputs (alpha, p, q [R, B-1]; margins, fallback flags [R])
 * may be NULL, as in oracle_spec_verify. */
int oracle_spec_verify_par(const void *target, const void *draft, int dtype, const int32_t *y, const float *u_acc,
                           const float *u_s, int R, int B, int V, double T, int32_t *accept_len,
                           int32_t *out_tokens, int32_t *num_tokens, double *alpha, double *p_out, double *q_out,
                           double *margin_accept, double *margin_sample, int32_t *used_fallback)
{
    const size_t es = dtype == 1 ? 2 : 4; /* bf16 bits or float32 */
    int rc = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(min : rc)
    for (int r = 0; r < R; ++r) {
        const size_t o = (size_t)r * (B - 1);
        const int e = oracle_spec_verify((const char *)target + (size_t)r * B * V * es,
                                         (const char *)draft + o * V * es, dtype, y + o, u_acc + o, u_s + r, 1, B, V,
                                         T, accept_len + r, out_tokens + (size_t)r * B, num_tokens + r,
                                         alpha ? alpha + o : NULL, p_out ? p_out + o : NULL, q_out ? q_out + o : NULL,
                                         margin_accept ? margin_accept + r : NULL,
                                         margin_sample ? margin_sample + r : NULL,
                                         used_fallback ? used_fallback + r : NULL);
        rc = e < rc ? e : rc;
    }
    return rc;
}
