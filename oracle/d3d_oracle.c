/*
 * Oracle for the diffusion-drafted speculative decoding hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, single-threaded CPU
 * statement of what the three steps compute, in double precision.  Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg load it.
 * It shares no code, header, table or helper with the CUDA library, and it
 * never calls it.
 *
 * Sources (pages):
 *   D3D: Decoupled Diffusion Drafting for Asynchronous Speculative Decoding
 *     - "Background / speculative decoding": accept a prefix by rejection
 *       sampling, resample one token from the residual at the first
 *       rejection; output distribution equals the target's.
 *     - "Background / asynchronous drafting and cache hits": one packed
 *       forward pre-drafts successor blocks for several verification
 *       outcomes; a hit is an exact match of the verified prefix with the
 *       beginning of a pre-drafted branch.
 *     - "Core method" and "Method steps" (step 2 and step 4): blocks see the
 *       shared prefix causally, attend bidirectionally inside the block;
 *       N_async = B[(C-1)F+2].
 *   Factorization-Guided Training and Inference for Diffusion-Drafted
 *   Speculative Decoding (DScout)
 *     - "Background / speculative decoding": accept the prefix before the
 *       first rejected token, then add one replacement token, or a bonus
 *       token when everything is accepted.
 *     - "Background / AWL and the acceptance rule":
 *       alpha_j = min(1, P_j(y_j) / Q_j(y_j)).
 *
 * Readings where the pages are silent (listed with reasons in the design
 * notes): scale s = 1/sqrt(d) is an argument; GQA kv head of query head h
 * is h / (Hq/Hkv); acceptance iff u_j < alpha_j; alpha = 1 when
 * Q_j(y_j) <= P_j(y_j) (covers Q_j(y_j) = 0); the inverse CDF takes the
 * smallest token v, in ascending vocabulary order, with C(v) > u * S; if
 * rounding leaves no such v, the last token with nonzero mass; if the
 * residual mass S is 0, the token is drawn from P at that position.
 *
 * Parity pins live in tests/test_oracle_pins.py (closed forms, hand-worked
 * cases, library routines, chi-square losslessness).  Every function here
 * is pinned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_BAD_ARG (-1)
#define OR_NOMEM (-2)

#define OR_CAUSAL 0
#define OR_BIDIR 1

#define OR_F32 0
#define OR_BF16 1

/* bf16 bit pattern -> double (exact). */
static double bf16_value(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double logit_value(const void *base, int dtype, size_t idx)
{
    if (dtype == OR_BF16)
        return bf16_value(((const uint16_t *)base)[idx]);
    return (double)((const float *)base)[idx];
}

/* ------------------------------------------------------------------------
 * Segment table checks.  A segment row is (q_start, len, mode, parent,
 * parent_len), local to its request.  Segments tile the request's packed
 * tokens in order with no gap and no overlap; a parent is an earlier causal
 * segment that itself has no parent; 0 <= parent_len <= len(parent).
 * ---------------------------------------------------------------------- */
int oracle_check_segments(const int32_t *segs, const int32_t *cu_q, const int32_t *cu_seg, int R)
{
    if (R < 0)
        return OR_BAD_ARG;
    if (R == 0)
        return OR_OK;
    if (cu_q[0] != 0 || cu_seg[0] != 0)
        return OR_BAD_ARG;
    for (int r = 0; r < R; ++r) {
        int n_q = cu_q[r + 1] - cu_q[r];
        int s0 = cu_seg[r], s1 = cu_seg[r + 1];
        if (n_q < 0 || s1 < s0)
            return OR_BAD_ARG;
        int next = 0;
        for (int s = s0; s < s1; ++s) {
            const int32_t *g = segs + 5 * (size_t)s;
            if (g[0] != next || g[1] < 1)
                return OR_BAD_ARG;
            if (g[2] != OR_CAUSAL && g[2] != OR_BIDIR)
                return OR_BAD_ARG;
            if (g[3] != -1) {
                int p = g[3];
                if (p < 0 || p >= s - s0)
                    return OR_BAD_ARG;
                const int32_t *pg = segs + 5 * (size_t)(s0 + p);
                if (pg[2] != OR_CAUSAL || pg[3] != -1)
                    return OR_BAD_ARG;
                if (g[4] < 0 || g[4] > pg[1])
                    return OR_BAD_ARG;
            } else if (g[4] != 0) {
                return OR_BAD_ARG;
            }
            next += g[1];
        }
        if (next != n_q)
            return OR_BAD_ARG;
    }
    return OR_OK;
}

/* Visibility of packed key j to packed query i of one request (both local).
 * The prefix is visible to everyone and is not asked here.  A query sees
 * its own segment (up to itself when causal, all of it when bidirectional)
 * and the first parent_len tokens of its parent segment; nothing else. */
static int packed_visible(const int32_t *segs, int nseg, int i, int j)
{
    int s = -1;
    for (int t = 0; t < nseg; ++t) {
        const int32_t *g = segs + 5 * (size_t)t;
        if (i >= g[0] && i < g[0] + g[1]) {
            s = t;
            break;
        }
    }
    if (s < 0)
        return 0;
    const int32_t *g = segs + 5 * (size_t)s;
    if (j >= g[0] && j < g[0] + g[1])
        return g[2] == OR_BIDIR ? 1 : (j <= i);
    if (g[3] >= 0) {
        const int32_t *pg = segs + 5 * (size_t)g[3];
        if (j >= pg[0] && j < pg[0] + g[4])
            return 1;
    }
    return 0;
}

/* Scaled-dot-product attention of one query row over an explicit key list,
 * with max-subtracted softmax, all in double. */
static void attend_row(const uint16_t *qrow, const uint16_t *const *krows, const uint16_t *const *vrows,
                       int nk, int d, double scale, double *score, double *out)
{
    double mx = -INFINITY;
    for (int k = 0; k < nk; ++k) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c)
            acc += bf16_value(qrow[c]) * bf16_value(krows[k][c]);
        score[k] = scale * acc;
        if (score[k] > mx)
            mx = score[k];
    }
    double z = 0.0;
    for (int k = 0; k < nk; ++k) {
        score[k] = exp(score[k] - mx);
        z += score[k];
    }
    for (int c = 0; c < d; ++c)
        out[c] = 0.0;
    for (int k = 0; k < nk; ++k) {
        double w = score[k] / z;
        for (int c = 0; c < d; ++c)
            out[c] += w * bf16_value(vrows[k][c]);
    }
}

/* ------------------------------------------------------------------------
 * Packed drafting attention (visibility predicate form).
 * q [NT, Hq, d], kp/vp [LT, Hkv, d], kn/vn [NT, Hkv, d], bf16 bits,
 * token-major.  Request r owns prefix rows cu_prefix[r] .. cu_prefix[r+1]
 * and packed rows cu_q[r] .. cu_q[r+1], segment rows cu_seg[r] ..
 * cu_seg[r+1].  out [NT, Hq, d] double:
 *   out[q,h] = sum_k softmax_k(scale <Q[q,h], K[k,h/G]>) V[k,h/G]
 * over the visible keys k (whole prefix, plus visible packed keys).
 * Only query heads [heads_lo, heads_hi) of packed rows [tok_lo, tok_hi)
 * (global row indices) are computed; other outputs are left untouched.
 * This selects which outputs to compute (to check or time a sample); it
 * changes nothing in how each output is computed.
 * ---------------------------------------------------------------------- */
int oracle_packed_attn_sel(const uint16_t *q, const uint16_t *kp, const uint16_t *vp,
                           const uint16_t *kn, const uint16_t *vn, const int32_t *segs,
                           const int32_t *cu_prefix, const int32_t *cu_q, const int32_t *cu_seg,
                           int R, int Hq, int Hkv, int d, double scale, int heads_lo, int heads_hi,
                           int tok_lo, int tok_hi, double *out)
{
    if (R < 0 || Hq < 1 || Hkv < 1 || d < 1 || Hq % Hkv)
        return OR_BAD_ARG;
    if (oracle_check_segments(segs, cu_q, cu_seg, R) != OR_OK)
        return OR_BAD_ARG;
    int G = Hq / Hkv;
    int maxk = 0;
    for (int r = 0; r < R; ++r) {
        int nk = (cu_prefix[r + 1] - cu_prefix[r]) + (cu_q[r + 1] - cu_q[r]);
        if (cu_prefix[r + 1] < cu_prefix[r])
            return OR_BAD_ARG;
        if (nk > maxk)
            maxk = nk;
    }
    const uint16_t **krows = malloc(sizeof(*krows) * (size_t)(maxk + 1));
    const uint16_t **vrows = malloc(sizeof(*vrows) * (size_t)(maxk + 1));
    double *score = malloc(sizeof(double) * (size_t)(maxk + 1));
    if (!krows || !vrows || !score) {
        free(krows);
        free(vrows);
        free(score);
        return OR_NOMEM;
    }
    for (int r = 0; r < R; ++r) {
        int L = cu_prefix[r + 1] - cu_prefix[r];
        int N = cu_q[r + 1] - cu_q[r];
        const int32_t *rs = segs + 5 * (size_t)cu_seg[r];
        int nseg = cu_seg[r + 1] - cu_seg[r];
        for (int i = 0; i < N; ++i) {
            size_t qi = (size_t)cu_q[r] + i;
            if ((long)qi < (long)tok_lo || (long)qi >= (long)tok_hi)
                continue;
            for (int h = heads_lo; h < heads_hi; ++h) {
                int hk = h / G;
                int nk = 0;
                for (int k = 0; k < L; ++k) {
                    size_t row = ((size_t)cu_prefix[r] + k) * Hkv + hk;
                    krows[nk] = kp + row * d;
                    vrows[nk] = vp + row * d;
                    ++nk;
                }
                for (int j = 0; j < N; ++j) {
                    if (!packed_visible(rs, nseg, i, j))
                        continue;
                    size_t row = ((size_t)cu_q[r] + j) * Hkv + hk;
                    krows[nk] = kn + row * d;
                    vrows[nk] = vn + row * d;
                    ++nk;
                }
                attend_row(q + (qi * Hq + h) * d, krows, vrows, nk, d, scale, score,
                           out + (qi * Hq + h) * d);
            }
        }
    }
    free(krows);
    free(vrows);
    free(score);
    return OR_OK;
}

int oracle_packed_attn(const uint16_t *q, const uint16_t *kp, const uint16_t *vp, const uint16_t *kn,
                       const uint16_t *vn, const int32_t *segs, const int32_t *cu_prefix,
                       const int32_t *cu_q, const int32_t *cu_seg, int R, int Hq, int Hkv, int d,
                       double scale, double *out)
{
    return oracle_packed_attn_sel(q, kp, vp, kn, vn, segs, cu_prefix, cu_q, cu_seg, R, Hq, Hkv, d, scale,
                                  0, Hq, 0, cu_q[R], out);
}

/* ------------------------------------------------------------------------
 * Explicit dense mask of one request: mask[i][k] for packed query i and key
 * k in [0, L + N) (prefix first, then packed tokens).  Built segment by
 * segment, row block by row block, instead of asking a predicate.
 * ---------------------------------------------------------------------- */
int oracle_dense_mask(const int32_t *segs, int nseg, int L, int N, uint8_t *mask)
{
    memset(mask, 0, (size_t)N * (size_t)(L + N));
    for (int s = 0; s < nseg; ++s) {
        const int32_t *g = segs + 5 * (size_t)s;
        int q0 = g[0], len = g[1];
        if (q0 < 0 || len < 0 || q0 + len > N)
            return OR_BAD_ARG;
        for (int a = 0; a < len; ++a) {
            uint8_t *row = mask + (size_t)(q0 + a) * (size_t)(L + N);
            for (int k = 0; k < L; ++k)
                row[k] = 1;                                    /* shared prefix */
            int own_hi = (g[2] == OR_BIDIR) ? len : a + 1;     /* own block */
            for (int b = 0; b < own_hi; ++b)
                row[L + q0 + b] = 1;
            if (g[3] >= 0) {                                   /* parent's first parent_len tokens */
                if (g[3] >= nseg)
                    return OR_BAD_ARG;
                int p0 = segs[5 * (size_t)g[3]];
                for (int b = 0; b < g[4]; ++b)
                    row[L + p0 + b] = 1;
            }
        }
    }
    return OR_OK;
}

/* Dense masked attention of one request (single request, R = 1 layout):
 * scores over all L + N keys, masked keys get -inf before the softmax. */
int oracle_dense_attn(const uint16_t *q, const uint16_t *kp, const uint16_t *vp, const uint16_t *kn,
                      const uint16_t *vn, const int32_t *segs, int nseg, int L, int N, int Hq, int Hkv,
                      int d, double scale, double *out)
{
    if (Hq < 1 || Hkv < 1 || Hq % Hkv)
        return OR_BAD_ARG;
    int G = Hq / Hkv, nk = L + N;
    uint8_t *mask = malloc((size_t)N * (size_t)nk + 1);
    double *sc = malloc(sizeof(double) * (size_t)nk + 8);
    if (!mask || !sc) {
        free(mask);
        free(sc);
        return OR_NOMEM;
    }
    if (oracle_dense_mask(segs, nseg, L, N, mask) != OR_OK) {
        free(mask);
        free(sc);
        return OR_BAD_ARG;
    }
    for (int i = 0; i < N; ++i)
        for (int h = 0; h < Hq; ++h) {
            int hk = h / G;
            const uint16_t *qr = q + ((size_t)i * Hq + h) * d;
            double mx = -INFINITY;
            for (int k = 0; k < nk; ++k) {
                const uint16_t *kr = (k < L) ? kp + ((size_t)k * Hkv + hk) * d
                                             : kn + ((size_t)(k - L) * Hkv + hk) * d;
                double acc = 0.0;
                for (int c = 0; c < d; ++c)
                    acc += bf16_value(qr[c]) * bf16_value(kr[c]);
                sc[k] = mask[(size_t)i * nk + k] ? scale * acc : -INFINITY;
                if (sc[k] > mx)
                    mx = sc[k];
            }
            double z = 0.0;
            for (int k = 0; k < nk; ++k) {
                sc[k] = mask[(size_t)i * nk + k] ? exp(sc[k] - mx) : 0.0;
                z += sc[k];
            }
            double *o = out + ((size_t)i * Hq + h) * d;
            for (int c = 0; c < d; ++c) {
                double acc = 0.0;
                for (int k = 0; k < nk; ++k) {
                    if (!mask[(size_t)i * nk + k])
                        continue;
                    const uint16_t *vr = (k < L) ? vp + ((size_t)k * Hkv + hk) * d
                                                 : vn + ((size_t)(k - L) * Hkv + hk) * d;
                    acc += sc[k] * bf16_value(vr[c]);
                }
                o[c] = acc / z;
            }
        }
    free(mask);
    free(sc);
    return OR_OK;
}

/* ------------------------------------------------------------------------
 * Verification (speculative sampling), one request at a time.
 * ---------------------------------------------------------------------- */

/* Softmax of one logit row at temperature T, double precision. */
static void softmax_row(const void *base, int dtype, size_t off, int V, double T, double *p)
{
    double mx = -INFINITY;
    for (int v = 0; v < V; ++v) {
        p[v] = logit_value(base, dtype, off + v) / T;
        if (p[v] > mx)
            mx = p[v];
    }
    double z = 0.0;
    for (int v = 0; v < V; ++v) {
        p[v] = exp(p[v] - mx);
        z += p[v];
    }
    for (int v = 0; v < V; ++v)
        p[v] /= z;
}

/* Inverse CDF of the unnormalised mass w over [0, V): smallest v with
 * C(v) = sum_{t<=v} w_t > u * S, S = C(V-1).  If rounding leaves no such
 * v, the last v with w_v > 0.  Returns -1 if S == 0.  *margin gets the
 * distance of u*S to the nearer boundary of the chosen token's CDF step,
 * divided by S. */
static int inverse_cdf(const double *w, int V, double u, double *margin)
{
    double S = 0.0;
    for (int v = 0; v < V; ++v)
        S += w[v];
    if (!(S > 0.0)) {
        *margin = 0.0;
        return -1;
    }
    double target = u * S, c = 0.0;
    for (int v = 0; v < V; ++v) {
        double prev = c;
        c += w[v];
        if (c > target) {
            double lo = target - prev, hi = c - target;
            *margin = (lo < hi ? lo : hi) / S;
            return v;
        }
    }
    for (int v = V - 1; v >= 0; --v)
        if (w[v] > 0.0) {
            *margin = 0.0;
            return v;
        }
    *margin = 0.0;
    return -1;
}

/*
 * target [R, B, V] and draft [R, B-1, V] logits (f32 or bf16 bits), draft
 * tokens y [R, B-1], acceptance uniforms u_acc [R, B-1], sample uniform
 * u_s [R].  Row j (0-based) of the target is the pages' P_{j+1}; row B-1 is
 * P_B, used only for the bonus token.
 * Outputs: accept_len [R] = a; out_tokens [R, B] = y_1..y_a then the
 * resampled or bonus token, rest -1; num_tokens [R] = a + 1 (= tau of the
 * round); alpha/p/q [R, B-1] (may be NULL); margin_accept [R] = smallest
 * |u_j - alpha_j| over the tests that decided a; margin_sample [R] = the
 * inverse-CDF margin (both may be NULL); used_fallback [R] = 1 when the
 * S == 0 rule fired (may be NULL).
 */
int oracle_spec_verify(const void *target, const void *draft, int dtype, const int32_t *y,
                       const float *u_acc, const float *u_s, int R, int B, int V, double T,
                       int32_t *accept_len, int32_t *out_tokens, int32_t *num_tokens, double *alpha,
                       double *p_out, double *q_out, double *margin_accept, double *margin_sample,
                       int32_t *used_fallback)
{
    if (R < 0 || B < 2 || V < 1 || !(T > 0.0) || (dtype != OR_F32 && dtype != OR_BF16))
        return OR_BAD_ARG;
    double *P = malloc(sizeof(double) * (size_t)V);
    double *Q = malloc(sizeof(double) * (size_t)V);
    double *res = malloc(sizeof(double) * (size_t)V);
    double *al = malloc(sizeof(double) * (size_t)B);
    if (!P || !Q || !res || !al) {
        free(P);
        free(Q);
        free(res);
        free(al);
        return OR_NOMEM;
    }
    for (int r = 0; r < R; ++r) {
        /* alpha_j for every draft position */
        for (int j = 0; j < B - 1; ++j) {
            int yj = y[(size_t)r * (B - 1) + j];
            if (yj < 0 || yj >= V) {
                free(P);
                free(Q);
                free(res);
                free(al);
                return OR_BAD_ARG;
            }
            softmax_row(target, dtype, ((size_t)r * B + j) * V, V, T, P);
            softmax_row(draft, dtype, ((size_t)r * (B - 1) + j) * V, V, T, Q);
            double pj = P[yj], qj = Q[yj];
            al[j] = (pj >= qj) ? 1.0 : pj / qj;
            if (alpha)
                alpha[(size_t)r * (B - 1) + j] = al[j];
            if (p_out)
                p_out[(size_t)r * (B - 1) + j] = pj;
            if (q_out)
                q_out[(size_t)r * (B - 1) + j] = qj;
        }
        /* first rejection: accept while u_j < alpha_j */
        int a = 0;
        double mA = INFINITY;
        while (a < B - 1) {
            double u = (double)u_acc[(size_t)r * (B - 1) + a];
            double gap = fabs(u - al[a]);
            if (gap < mA)
                mA = gap;
            if (u < al[a])
                ++a;
            else
                break;
        }
        /* one more token: residual resample at position a+1, or the bonus */
        double mS = 0.0;
        int fb = 0, t;
        if (a < B - 1) {
            softmax_row(target, dtype, ((size_t)r * B + a) * V, V, T, P);
            softmax_row(draft, dtype, ((size_t)r * (B - 1) + a) * V, V, T, Q);
            for (int v = 0; v < V; ++v)
                res[v] = (P[v] > Q[v]) ? P[v] - Q[v] : 0.0;
            t = inverse_cdf(res, V, (double)u_s[r], &mS);
            if (t < 0) {
                fb = 1;
                t = inverse_cdf(P, V, (double)u_s[r], &mS);
            }
        } else {
            softmax_row(target, dtype, ((size_t)r * B + (B - 1)) * V, V, T, P);
            t = inverse_cdf(P, V, (double)u_s[r], &mS);
        }
        accept_len[r] = a;
        num_tokens[r] = a + 1;
        for (int j = 0; j < B; ++j) {
            int32_t tok = -1;
            if (j < a)
                tok = y[(size_t)r * (B - 1) + j];
            else if (j == a)
                tok = t;
            out_tokens[(size_t)r * B + j] = tok;
        }
        if (margin_accept)
            margin_accept[r] = mA;
        if (margin_sample)
            margin_sample[r] = mS;
        if (used_fallback)
            used_fallback[r] = fb;
    }
    free(P);
    free(Q);
    free(res);
    free(al);
    return OR_OK;
}

/*
 * Acceptance-weighted loss weights (DScout, "Background: AWL and the
 * acceptance rule"; "Method steps", fourth step): the weight of draft
 * position k (0-based) is the product of the acceptance probabilities of
 * the drafts before it, w_k = prod_{j<k} alpha_j, so w_0 = 1; it is the
 * probability that verification reaches position k.  alpha [R, Bm1] (as
 * oracle_spec_verify writes it) -> w [R, Bm1].
 */
int oracle_awl_weights(const double *alpha, int R, int Bm1, double *w)
{
    if (R < 0 || Bm1 < 1)
        return OR_BAD_ARG;
    for (int r = 0; r < R; ++r) {
        double prod = 1.0;
        for (int k = 0; k < Bm1; ++k) {
            w[(size_t)r * Bm1 + k] = prod;
            prod *= alpha[(size_t)r * Bm1 + k];
        }
    }
    return OR_OK;
}

/*
 * Per-position acceptance probabilities and the round's expected acceptance
 * length (DScout, "Background: acceptance length tau" and "Background: AWL
 * and the acceptance rule"): with P_j = softmax(target row j / T) and
 * Q_j = softmax(draft row j / T), a draft token y ~ Q_j is accepted with
 * probability a_j = sum_v min(P_j(v), Q_j(v)); the prefix survival is
 * S(k) = a_1 ... a_k and tau = 1 + sum_{k=1}^{B-1} S(k).
 * Outputs: accept_prob [R, B-1] = a, survival [R, B-1] = S, tau [R].
 */
int oracle_accept_probs(const void *target, const void *draft, int dtype, int R, int B, int V, double T,
                        double *accept_prob, double *survival, double *tau)
{
    if (R < 0 || B < 2 || V < 1 || !(T > 0.0) || (dtype != OR_F32 && dtype != OR_BF16))
        return OR_BAD_ARG;
    double *P = malloc(sizeof(double) * (size_t)V);
    double *Q = malloc(sizeof(double) * (size_t)V);
    if (!P || !Q) {
        free(P);
        free(Q);
        return OR_NOMEM;
    }
    for (int r = 0; r < R; ++r) {
        double surv = 1.0, t = 1.0;
        for (int j = 0; j < B - 1; ++j) {
            softmax_row(target, dtype, ((size_t)r * B + j) * V, V, T, P);
            softmax_row(draft, dtype, ((size_t)r * (B - 1) + j) * V, V, T, Q);
            double a = 0.0;
            for (int v = 0; v < V; ++v)
                a += P[v] < Q[v] ? P[v] : Q[v];
            surv *= a;
            t += surv;
            accept_prob[(size_t)r * (B - 1) + j] = a;
            survival[(size_t)r * (B - 1) + j] = surv;
        }
        tau[r] = t;
    }
    free(P);
    free(Q);
    return OR_OK;
}

/*
 * Branch construction for the asynchronous packed pass (D3D, "Background:
 * asynchronous drafting and cache hits" and "Method steps", step 4: for
 * every rejection position, several alternative anchors, plus the
 * all-accept block).  Readings (the pages do not say how the anchors are
 * chosen): the F alternative anchors of rejection position r (0-based draft
 * index r, r = 0..C-2) are the F most likely tokens of the drafter's own
 * distribution Q_r at that position (largest logit first, ties to the
 * lowest index), the drafted token y_r excluded; the all-accept head's last
 * token is the caller's guess of the bonus token (no guess: that head has
 * length 0 and never matches).
 * Outputs, per request (M = (C-1)F + 2 branches, indexed like the segments):
 *   anchors [R, C-1, F];
 *   head_len[r,0] = 0 (the block under verification);
 *   branch k = 1 + r*F + f: head = y_0 .. y_{r-1}, anchor (r, f); len r + 1;
 *   branch M-1: head = y_0 .. y_{B-2}, bonus guess; len B (0 without a guess);
 *   head entries past the length are -1;
 *   segs [R*M, 5] request-local rows: (0, B, causal, -1, 0) for the block
 *   under verification, (k*B, B, bidirectional, 0, r+1) for branch (r, f),
 *   ((M-1)*B, B, bidirectional, 0, B) for the all-accept block;
 *   cu_q[r] = r*M*B, cu_seg[r] = r*M (R+1 entries).
 */
int oracle_build_branches(const void *draft, int dtype, const int32_t *y, const int32_t *bonus_guess, int R,
                          int B, int V, int C, int F, int32_t *anchors, int32_t *heads, int32_t *head_len,
                          int32_t *segs, int32_t *cu_q, int32_t *cu_seg)
{
    if (R < 0 || B < 2 || V < 1 || C < 1 || C > B || F < 0 || (dtype != OR_F32 && dtype != OR_BF16))
        return OR_BAD_ARG;
    if ((C - 1) * F > 0 && F > V - 1)
        return OR_BAD_ARG; /* not enough tokens besides y */
    const int M = (C - 1) * F + 2;
    char *taken = malloc((size_t)V);
    if (!taken)
        return OR_NOMEM;
    for (int r = 0; r < R; ++r) {
        const int32_t *yr = y + (size_t)r * (B - 1);
        for (int j = 0; j < B - 1; ++j)
            if (yr[j] < 0 || yr[j] >= V) {
                free(taken);
                return OR_BAD_ARG;
            }
        /* anchors: repeated maximum over the tokens not yet taken */
        for (int p = 0; p < C - 1; ++p) {
            size_t off = ((size_t)r * (B - 1) + p) * V;
            memset(taken, 0, (size_t)V);
            taken[yr[p]] = 1;
            for (int f = 0; f < F; ++f) {
                int bi = -1;
                double best = 0.0;
                for (int v = 0; v < V; ++v) {
                    if (taken[v])
                        continue;
                    double x = logit_value(draft, dtype, off + v);
                    if (bi < 0 || x > best) {
                        best = x;
                        bi = v;
                    }
                }
                taken[bi] = 1;
                anchors[((size_t)r * (C - 1) + p) * F + f] = bi;
            }
        }
        /* heads */
        int32_t *h = heads + (size_t)r * M * B;
        int32_t *hl = head_len + (size_t)r * M;
        for (int k = 0; k < M; ++k)
            for (int i = 0; i < B; ++i)
                h[(size_t)k * B + i] = -1;
        hl[0] = 0;
        for (int p = 0; p < C - 1; ++p)
            for (int f = 0; f < F; ++f) {
                int k = 1 + p * F + f;
                for (int i = 0; i < p; ++i)
                    h[(size_t)k * B + i] = yr[i];
                h[(size_t)k * B + p] = anchors[((size_t)r * (C - 1) + p) * F + f];
                hl[k] = p + 1;
            }
        if (bonus_guess) {
            for (int i = 0; i < B - 1; ++i)
                h[(size_t)(M - 1) * B + i] = yr[i];
            h[(size_t)(M - 1) * B + B - 1] = bonus_guess[r];
            hl[M - 1] = B;
        } else {
            hl[M - 1] = 0;
        }
        /* segment rows of the packed pass */
        if (segs) {
            int32_t *sg = segs + (size_t)r * M * 5;
            for (int k = 0; k < M; ++k) {
                int32_t row[5];
                if (k == 0) {
                    row[0] = 0, row[1] = B, row[2] = OR_CAUSAL, row[3] = -1, row[4] = 0;
                } else if (k == M - 1) {
                    row[0] = k * B, row[1] = B, row[2] = OR_BIDIR, row[3] = 0, row[4] = B;
                } else {
                    row[0] = k * B, row[1] = B, row[2] = OR_BIDIR, row[3] = 0, row[4] = (k - 1) / F + 1;
                }
                memcpy(sg + (size_t)k * 5, row, sizeof(row));
            }
        }
    }
    if (cu_q && cu_seg)
        for (int r = 0; r <= R; ++r) {
            cu_q[r] = r * M * B;
            cu_seg[r] = r * M;
        }
    free(taken);
    return OR_OK;
}

/*
 * Greedy verification (temperature 0), the decoding setting of the pages'
 * results (D3D, "Experiments": greedy decoding; DScout, "Experiments").
 * The acceptance rule at T = 0 is the limit of the sampling rule: P_j and
 * Q_j become point masses at their argmax, so a draft token is accepted
 * exactly when it is the target's argmax, and the residual (or the bonus
 * distribution) is the point mass at the target's argmax.  Reading: ties go
 * to the lowest token index.
 * Per request r: g_j = argmax_v target[r, j, v] for j = 0..B-1; a = the
 * number of leading positions with y_j == g_j; out_tokens = y_0..y_{a-1},
 * g_a, then -1; num_tokens = a + 1.  accept [R, B-1] (may be NULL) = 1.0
 * where y_j == g_j, else 0.0; argmax [R, B] (may be NULL) = g.  The draft
 * logits are not needed.
 */
int oracle_greedy_verify(const void *target, int dtype, const int32_t *y, int R, int B, int V,
                         int32_t *accept_len, int32_t *out_tokens, int32_t *num_tokens, double *accept,
                         int32_t *argmax)
{
    if (R < 0 || B < 2 || V < 1 || (dtype != OR_F32 && dtype != OR_BF16))
        return OR_BAD_ARG;
    int32_t *g = malloc(sizeof(int32_t) * (size_t)B);
    if (!g)
        return OR_NOMEM;
    for (int r = 0; r < R; ++r) {
        for (int j = 0; j < B; ++j) {
            size_t off = ((size_t)r * B + j) * V;
            double best = logit_value(target, dtype, off);
            int bi = 0;
            for (int v = 1; v < V; ++v) {
                double x = logit_value(target, dtype, off + v);
                if (x > best) { /* strict: an equal value later in the row never wins */
                    best = x;
                    bi = v;
                }
            }
            g[j] = bi;
            if (argmax)
                argmax[(size_t)r * B + j] = bi;
        }
        int a = 0;
        for (int j = 0; j < B - 1; ++j) {
            int yj = y[(size_t)r * (B - 1) + j];
            if (yj < 0 || yj >= V) {
                free(g);
                return OR_BAD_ARG;
            }
            if (accept)
                accept[(size_t)r * (B - 1) + j] = (yj == g[j]) ? 1.0 : 0.0;
        }
        while (a < B - 1 && y[(size_t)r * (B - 1) + a] == g[a])
            ++a;
        accept_len[r] = a;
        num_tokens[r] = a + 1;
        for (int j = 0; j < B; ++j)
            out_tokens[(size_t)r * B + j] = j < a ? y[(size_t)r * (B - 1) + j] : (j == a ? g[a] : -1);
    }
    free(g);
    return OR_OK;
}

/* ------------------------------------------------------------------------
 * Branch cache-hit match: the smallest branch index k whose head has the
 * verified prefix's length and equals it token for token; -1 on a miss.
 * ---------------------------------------------------------------------- */
int oracle_branch_match(const int32_t *verified, const int32_t *verified_len, const int32_t *heads,
                        const int32_t *head_len, int R, int M, int B, int32_t *branch)
{
    if (R < 0 || M < 0 || B < 1)
        return OR_BAD_ARG;
    for (int r = 0; r < R; ++r) {
        int n = verified_len[r], hit = -1;
        if (n < 0 || n > B)
            return OR_BAD_ARG;
        for (int k = 0; k < M && hit < 0; ++k) {
            if (head_len[(size_t)r * M + k] != n)
                continue;
            int same = 1;
            for (int i = 0; i < n; ++i)
                if (heads[((size_t)r * M + k) * B + i] != verified[(size_t)r * B + i]) {
                    same = 0;
                    break;
                }
            if (same)
                hit = k;
        }
        branch[r] = hit;
    }
    return OR_OK;
}
