// Speculative-sampling verification over the vocabulary.
//
// [D3D] "Background: speculative decoding"; [DScout] "Background:
// speculative decoding" and "Background: AWL and the acceptance rule":
// alpha_j = min(1, P_j(y_j)/Q_j(y_j)), accept while u_j < alpha_j, then
// resample from norm(max(0, P - Q)) at the first rejection or draw a bonus
// token from P_B when every draft is accepted.
//
// Two launches, both streaming HBM with 16-byte vector loads:
//   1. verify_stats_kernel: one CTA per (logit row, 8192-entry chunk) computes
//      the chunk's softmax statistics (max and sum of exp2, log2 domain).  The
//      last CTA of a request (atomic ticket) merges the chunk statistics per
//      row, forms p_j, q_j, alpha_j, runs the first-rejection scan and writes
//      a, the accepted tokens, and which row pair the sample needs.
//   2. verify_sample_kernel: one CTA per chunk of that row pair sums the
//      residual (or P_B) mass of its chunk; the last CTA finds the chunk where
//      the CDF crosses u*S and scans it in vocabulary order for the token.
// The second pass re-reads one row pair, normally still resident in L2.
#include <math.h>

#include <mutex>

#include "d3d_common.cuh"

namespace d3d {
namespace {

constexpr int kVThreads = 256;
constexpr int kVWarps = kVThreads / 32;
constexpr int kVChunk = 8192;
constexpr int kVPer = kVChunk / kVThreads;  // 32 logits per thread
constexpr int kMaxB = 256;
constexpr int kMaxChunks = 1024;  // vocabulary up to 8M entries
constexpr unsigned kFull = 0xffffffffu;

struct ReqInfo {
    int32_t a;     // accepted drafts
    int32_t mode;  // 0: residual at target/draft row a; 1: bonus from target row B-1
    int32_t row;   // target row the sample uses (and draft row when mode == 0)
    int32_t pad;
    float mP, rZP, mQ, rZQ;  // log2-domain row max and 1 / normaliser of that target / draft row
};

struct VerifyLayout {
    size_t cnt1, cnt2, part1, info, part2, total;
    int nch;
};

__host__ __device__ inline VerifyLayout verify_layout(int R, int B, int V)
{
    VerifyLayout L;
    L.nch = (V + kVChunk - 1) / kVChunk;
    size_t o = sizeof(WsHeader);
    L.cnt1 = o;
    o = align_up(o + sizeof(int) * (size_t)R, kWsAlign);
    L.cnt2 = o;
    o = align_up(o + sizeof(int) * (size_t)R, kWsAlign);
    L.part1 = o;
    o = align_up(o + sizeof(float2) * (size_t)R * (size_t)(2 * B - 1) * (size_t)L.nch, kWsAlign);
    L.info = o;
    o = align_up(o + sizeof(ReqInfo) * (size_t)R, kWsAlign);
    L.part2 = o;
    o = align_up(o + sizeof(float2) * (size_t)R * (size_t)L.nch, kWsAlign);
    L.total = o;
    return L;
}

// ---- logit access (float32 or bf16 bit patterns) -------------------------
template <typename T> struct Logit;

template <> struct Logit<float> {
    __device__ static float at(const float *p, size_t i) { return __ldg(p + i); }
    __device__ static void load8(const float *p, float (&v)[8])
    {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
        v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
    }
};

template <> struct Logit<uint16_t> {
    __device__ static float at(const uint16_t *p, size_t i) { return bf16_bits_to_float(__ldg(p + i)); }
    __device__ static void load8(const uint16_t *p, float (&v)[8])
    {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
        v[0] = __uint_as_float(u.x << 16), v[1] = __uint_as_float(u.x & 0xffff0000u);
        v[2] = __uint_as_float(u.y << 16), v[3] = __uint_as_float(u.y & 0xffff0000u);
        v[4] = __uint_as_float(u.z << 16), v[5] = __uint_as_float(u.z & 0xffff0000u);
        v[6] = __uint_as_float(u.w << 16), v[7] = __uint_as_float(u.w & 0xffff0000u);
    }
};

template <typename T> __device__ inline bool aligned16(const T *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Scaled logits x*c of one chunk [v0, v1) in a strided (coalesced) ownership:
// slot 8k+e of thread t holds position v0 + 2048k + 8t + e, whichever load
// path a row takes, so two rows loaded this way line up slot by slot.
// Positions past v1 read as -inf.
template <typename T>
__device__ inline void load_chunk_strided(const T *row, int v0, int v1, float c, float (&x)[kVPer])
{
    const int tid = threadIdx.x;
    if (v1 - v0 == kVChunk && aligned16(row + v0)) {
#pragma unroll
        for (int k = 0; k < kVPer / 8; ++k) {
            float t[8];
            Logit<T>::load8(row + v0 + k * kVThreads * 8 + tid * 8, t);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                x[k * 8 + e] = t[e] * c;
        }
    } else {
#pragma unroll
        for (int k = 0; k < kVPer / 8; ++k) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int v = v0 + k * kVThreads * 8 + tid * 8 + e;
                x[k * 8 + e] = v < v1 ? Logit<T>::at(row, v) * c : -INFINITY;
            }
        }
    }
}

// Scaled logits of thread-contiguous positions v0 + tid*kVPer + k (vocabulary
// order inside a thread), -inf past v1.  Used for the ordered scan.
template <typename T>
__device__ inline void load_chunk_contig(const T *row, int v0, int v1, float c, float (&x)[kVPer])
{
    const int base = v0 + threadIdx.x * kVPer;
    if (base + kVPer <= v1 && aligned16(row + base)) {
#pragma unroll
        for (int k = 0; k < kVPer / 8; ++k) {
            float t[8];
            Logit<T>::load8(row + base + k * 8, t);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                x[k * 8 + e] = t[e] * c;
        }
    } else {
#pragma unroll
        for (int k = 0; k < kVPer; ++k) {
            const int v = base + k;
            x[k] = v < v1 ? Logit<T>::at(row, v) * c : -INFINITY;
        }
    }
}

// 2^x with the hardware approximation (relative error about 2^-22, far
// inside the 1e-5 tolerance on probabilities); -inf gives 0.
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// (max, sum of exp2(x - max)) merge; an empty side has max = -inf, sum = 0.
__device__ inline void ms_merge(float &m, float &z, float m2, float z2)
{
    const float M = fmaxf(m, m2);
    if (M == -INFINITY) {
        m = M;
        z = 0.f;
        return;
    }
    z = z * fast_exp2(m - M) + z2 * fast_exp2(m2 - M);
    m = M;
}

// Block-wide (max, sum) merge; the result is valid in thread 0.
__device__ inline void block_ms(float &m, float &z, float *red)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float m2 = __shfl_xor_sync(kFull, m, o), z2 = __shfl_xor_sync(kFull, z, o);
        ms_merge(m, z, m2, z2);
    }
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        red[w] = m;
        red[kVWarps + w] = z;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        m = red[0];
        z = red[kVWarps];
        for (int i = 1; i < kVWarps; ++i)
            ms_merge(m, z, red[i], red[kVWarps + i]);
    }
}

// Block-wide sums of two values; the result is valid in thread 0.
__device__ inline void block_sum2(float &a, float &b, float *red)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        a += __shfl_xor_sync(kFull, a, o);
        b += __shfl_xor_sync(kFull, b, o);
    }
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        red[w] = a;
        red[kVWarps + w] = b;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        a = red[0];
        b = red[kVWarps];
        for (int i = 1; i < kVWarps; ++i) {
            a += red[i];
            b += red[kVWarps + i];
        }
    }
}

// Block-wide exclusive scan of one value per thread, in thread order.
__device__ inline float block_exclusive_scan(float v, float *red)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(kFull, inc, o);
        if (lane >= o)
            inc += t;
    }
    if (lane == 31)
        red[w] = inc;
    __syncthreads();
    float base = 0.f;
    for (int i = 0; i < w; ++i)
        base += red[i];
    return base + inc - v;
}

// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kVThreads)
    verify_stats_kernel(const T *__restrict__ target, const T *__restrict__ draft, const int32_t *__restrict__ y,
                        const float *__restrict__ u_acc, int R, int B, int V, float c,
                        int32_t *__restrict__ accept_len, int32_t *__restrict__ out_tokens,
                        int32_t *__restrict__ num_tokens, float *__restrict__ alpha_out,
                        float *__restrict__ p_out, float *__restrict__ q_out, unsigned char *__restrict__ ws)
{
    const VerifyLayout L = verify_layout(R, B, V);
    const int rows = 2 * B - 1;
    const int chunk = blockIdx.x % L.nch;
    const int rowg = blockIdx.x / L.nch;
    const int r = rowg / rows, j = rowg % rows;
    const T *row = (j < B) ? target + ((size_t)r * B + j) * V : draft + ((size_t)r * (B - 1) + (j - B)) * V;
    const int v0 = chunk * kVChunk, v1 = min(V, v0 + kVChunk);

    float x[kVPer];
    load_chunk_strided<T>(row, v0, v1, c, x);
    float m = -INFINITY, z = 0.f;
#pragma unroll
    for (int k = 0; k < kVPer; ++k)
        m = fmaxf(m, x[k]);
    if (m != -INFINITY) {
#pragma unroll
        for (int k = 0; k < kVPer; ++k)
            z += fast_exp2(x[k] - m);
    }
    __shared__ float red[2 * kVWarps];
    __shared__ int s_last;
    block_ms(m, z, red);

    float2 *part = reinterpret_cast<float2 *>(ws + L.part1);
    int *cnt = reinterpret_cast<int *>(ws + L.cnt1);
    if (threadIdx.x == 0) {
        part[(size_t)rowg * L.nch + chunk] = make_float2(m, z);
        __threadfence();
        const int prev = atomicAdd(&cnt[r], 1);
        s_last = (prev == rows * L.nch - 1);
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();

    // ---- last CTA of request r: row statistics, alpha, first-rejection scan
    __shared__ float s_m[2 * kMaxB], s_z[2 * kMaxB];
    __shared__ int s_a;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float2 *pr = part + (size_t)r * rows * L.nch;
    for (int jj = warp; jj < rows; jj += kVWarps) {
        float mm = -INFINITY, zz = 0.f;
        for (int cc = lane; cc < L.nch; cc += 32) {
            const float2 t = __ldcg(&pr[(size_t)jj * L.nch + cc]);
            ms_merge(mm, zz, t.x, t.y);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float m2 = __shfl_xor_sync(kFull, mm, o), z2 = __shfl_xor_sync(kFull, zz, o);
            ms_merge(mm, zz, m2, z2);
        }
        if (lane == 0) {
            s_m[jj] = mm;
            s_z[jj] = zz;
        }
    }
    __syncthreads();
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    if (threadIdx.x == 0)
        s_a = B - 1;
    __syncthreads();
    // alpha_j and the acceptance test of every position in parallel; the
    // first rejection is the smallest rejected position
    for (int jj = threadIdx.x; jj < B - 1; jj += kVThreads) {
        const int yy = y[(size_t)r * (B - 1) + jj];
        const float uj = u_acc[(size_t)r * (B - 1) + jj];
        float p = 0.f, q = 0.f, al = 0.f;
        if (yy < 0 || yy >= V) {
            record_status(status, D3D_ERR_DEVICE_INPUT);
        } else {
            const float xt = Logit<T>::at(target + ((size_t)r * B + jj) * V, yy) * c;
            const float xd = Logit<T>::at(draft + ((size_t)r * (B - 1) + jj) * V, yy) * c;
            p = fast_exp2(xt - s_m[jj]) / s_z[jj];
            q = fast_exp2(xd - s_m[B + jj]) / s_z[B + jj];
            al = (p >= q) ? 1.f : p / q;
        }
        if (!(uj < al))
            atomicMin(&s_a, jj);
        const size_t o = (size_t)r * (B - 1) + jj;
        if (alpha_out)
            alpha_out[o] = al;
        if (p_out)
            p_out[o] = p;
        if (q_out)
            q_out[o] = q;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const int a = s_a;
        ReqInfo inf;
        inf.a = a;
        inf.mode = (a < B - 1) ? 0 : 1;
        inf.row = (a < B - 1) ? a : B - 1;
        inf.pad = 0;
        inf.mP = s_m[inf.row];
        inf.rZP = __frcp_rn(s_z[inf.row]);
        inf.mQ = (a < B - 1) ? s_m[B + a] : 0.f;
        inf.rZQ = (a < B - 1) ? __frcp_rn(s_z[B + a]) : 1.f;
        reinterpret_cast<ReqInfo *>(ws + L.info)[r] = inf;
        accept_len[r] = a;
        num_tokens[r] = a + 1;
        cnt[r] = 0;  // ready for the next call
    }
    __syncthreads();
    const int a = s_a;
    for (int jj = threadIdx.x; jj < B; jj += kVThreads)
        if (jj != a)
            out_tokens[(size_t)r * B + jj] = (jj < a) ? y[(size_t)r * (B - 1) + jj] : -1;
}

// Mass of position v of the sampled distribution: the residual
// max(0, P - Q) (kind 0) or P itself (kind 1); xp/xq are scaled logits.
__device__ inline float sample_mass(int kind, float xp, float xq, const ReqInfo &inf)
{
    const float P = fast_exp2(xp - inf.mP) * inf.rZP;
    if (kind != 0)
        return P;
    const float Q = fast_exp2(xq - inf.mQ) * inf.rZQ;
    return fmaxf(P - Q, 0.f);
}

template <typename T>
__global__ void __launch_bounds__(kVThreads)
    verify_sample_kernel(const T *__restrict__ target, const T *__restrict__ draft, const float *__restrict__ u_s,
                         int R, int B, int V, float c, int32_t *__restrict__ out_tokens,
                         unsigned char *__restrict__ ws)
{
    const VerifyLayout L = verify_layout(R, B, V);
    const int chunk = blockIdx.x % L.nch;
    const int r = blockIdx.x / L.nch;
    const ReqInfo inf = reinterpret_cast<const ReqInfo *>(ws + L.info)[r];
    const T *prow = target + ((size_t)r * B + inf.row) * V;
    const T *qrow = draft + ((size_t)r * (B - 1) + (inf.mode == 0 ? inf.row : 0)) * V;
    const int v0 = chunk * kVChunk, v1 = min(V, v0 + kVChunk);

    float xp[kVPer], xq[kVPer];
    load_chunk_strided<T>(prow, v0, v1, c, xp);
    if (inf.mode == 0)
        load_chunk_strided<T>(qrow, v0, v1, c, xq);
    float s_res = 0.f, s_p = 0.f;
#pragma unroll
    for (int k = 0; k < kVPer; ++k) {
        const float P = fast_exp2(xp[k] - inf.mP) * inf.rZP;
        s_p += P;
        s_res += (inf.mode == 0) ? fmaxf(P - fast_exp2(xq[k] - inf.mQ) * inf.rZQ, 0.f) : P;
    }
    __shared__ float red[2 * kVWarps];
    __shared__ int s_last;
    block_sum2(s_res, s_p, red);
    float2 *part = reinterpret_cast<float2 *>(ws + L.part2);
    int *cnt = reinterpret_cast<int *>(ws + L.cnt2);
    if (threadIdx.x == 0) {
        part[(size_t)r * L.nch + chunk] = make_float2(s_res, s_p);
        __threadfence();
        const int prev = atomicAdd(&cnt[r], 1);
        s_last = (prev == L.nch - 1);
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();

    // ---- last CTA: crossing chunk, then the ordered scan inside it
    __shared__ int s_kind, s_chunk, s_takelast, s_cand, s_lastpos;
    __shared__ float s_prefix, s_target;
    __shared__ float2 s_sums[kMaxChunks];
    const float2 *pr = part + (size_t)r * L.nch;
    for (int cc = threadIdx.x; cc < L.nch; cc += kVThreads)
        s_sums[cc] = __ldcg(&pr[cc]);
    __syncthreads();
    if (threadIdx.x == 0) {
        float S_res = 0.f, S_p = 0.f;
        for (int cc = 0; cc < L.nch; ++cc) {
            S_res += s_sums[cc].x;
            S_p += s_sums[cc].y;
        }
        // residual unless it has no mass left in fp32 (then P at that row)
        const int kind = (inf.mode == 0 && S_res > 0.f) ? 0 : 1;
        const float S = kind == 0 ? S_res : S_p;
        const float tgt = u_s[r] * S;
        float run = 0.f;
        int ch = -1;
        for (int cc = 0; cc < L.nch; ++cc) {
            const float2 t = s_sums[cc];
            const float sc = kind == 0 ? t.x : t.y;
            if (run + sc > tgt) {
                ch = cc;
                break;
            }
            run += sc;
        }
        int takelast = 0;
        if (ch < 0) {  // rounding left u*S at or past the end: last chunk with mass
            takelast = 1;
            for (int cc = L.nch - 1; cc >= 0 && ch < 0; --cc) {
                const float2 t = s_sums[cc];
                if ((kind == 0 ? t.x : t.y) > 0.f)
                    ch = cc;
            }
        }
        s_kind = kind;
        s_chunk = ch;
        s_takelast = takelast;
        s_prefix = run;
        s_target = tgt;
        s_cand = kVThreads;
        s_lastpos = -1;
        cnt[r] = 0;  // ready for the next call
    }
    __syncthreads();
    const int ch = s_chunk;
    if (ch < 0) {  // no mass anywhere: cannot happen for a finite softmax row
        if (threadIdx.x == 0) {
            record_status(reinterpret_cast<int32_t *>(ws), D3D_ERR_DEVICE_INPUT);
            out_tokens[(size_t)r * B + inf.a] = 0;
        }
        return;
    }
    const int kind = s_kind;
    const int c0 = ch * kVChunk, c1 = min(V, c0 + kVChunk);
    load_chunk_contig<T>(prow, c0, c1, c, xp);
    if (kind == 0)
        load_chunk_contig<T>(qrow, c0, c1, c, xq);
    float w[kVPer], tot = 0.f;
    int lastpos = -1;
#pragma unroll
    for (int k = 0; k < kVPer; ++k) {
        w[k] = (c0 + threadIdx.x * kVPer + k < c1) ? sample_mass(kind, xp[k], kind == 0 ? xq[k] : 0.f, inf) : 0.f;
        tot += w[k];
        if (w[k] > 0.f)
            lastpos = c0 + threadIdx.x * kVPer + k;
    }
    const float excl = block_exclusive_scan(tot, red);
    const float base = s_prefix + excl;
    if (!s_takelast && base + tot > s_target)
        atomicMin(&s_cand, (int)threadIdx.x);
    atomicMax(&s_lastpos, lastpos);
    __syncthreads();
    int tok = -1;
    if (!s_takelast && (int)threadIdx.x == s_cand) {
        float cum = base;
        for (int k = 0; k < kVPer; ++k) {
            cum += w[k];
            if (cum > s_target) {
                tok = c0 + threadIdx.x * kVPer + k;
                break;
            }
        }
        if (tok < 0)
            tok = lastpos;  // rounding between the two summation orders
        out_tokens[(size_t)r * B + inf.a] = tok;
    }
    if ((s_takelast || s_cand == kVThreads) && threadIdx.x == 0)
        out_tokens[(size_t)r * B + inf.a] = s_lastpos;
}

template <typename T>
int launch_verify(const void *target, const void *draft, const int32_t *y, const float *u_acc, const float *u_s,
                  int R, int B, int V, float c, int32_t *accept_len, int32_t *out_tokens, int32_t *num_tokens,
                  float *alpha, float *p, float *q, unsigned char *ws, cudaStream_t stream)
{
    const VerifyLayout L = verify_layout(R, B, V);
    const size_t n1 = (size_t)R * (size_t)(2 * B - 1) * (size_t)L.nch;
    const size_t n2 = (size_t)R * (size_t)L.nch;
    if (n1 > 0x7fffffffull)
        return D3D_ERR_UNSUPPORTED;
    verify_stats_kernel<T><<<(unsigned)n1, kVThreads, 0, stream>>>(
        static_cast<const T *>(target), static_cast<const T *>(draft), y, u_acc, R, B, V, c, accept_len,
        out_tokens, num_tokens, alpha, p, q, ws);
    verify_sample_kernel<T><<<(unsigned)n2, kVThreads, 0, stream>>>(
        static_cast<const T *>(target), static_cast<const T *>(draft), u_s, R, B, V, c, out_tokens, ws);
    return cuda_status(cudaGetLastError());
}

}  // namespace
}  // namespace d3d

extern "C" {

size_t d3d_spec_verify_workspace_size(int R, int B, int V)
{
    if (R < 0 || B < 2 || V < 1 || B > d3d::kMaxB || V > d3d::kMaxChunks * d3d::kVChunk)
        return 0;
    return d3d::verify_layout(R, B, V).total;
}

int d3d_spec_verify(const void *target_logits, const void *draft_logits, int logits_dtype,
                    const int32_t *draft_tokens, const float *u_accept, const float *u_sample, int R, int B,
                    int V, float temperature, int32_t *accept_len, int32_t *out_tokens, int32_t *num_tokens,
                    float *alpha, float *p_draft, float *q_draft, void *ws, size_t ws_bytes,
                    cudaStream_t stream)
{
    if (R < 0 || B < 2 || V < 1 || !(temperature > 0.f) || !isfinite(temperature))
        return D3D_ERR_INVALID_ARG;
    if (logits_dtype != D3D_DTYPE_F32 && logits_dtype != D3D_DTYPE_BF16)
        return D3D_ERR_INVALID_ARG;
    if (B > d3d::kMaxB || V > d3d::kMaxChunks * d3d::kVChunk)
        return D3D_ERR_UNSUPPORTED;
    if (R == 0)
        return D3D_OK;
    if (!target_logits || !draft_logits || !draft_tokens || !u_accept || !u_sample || !accept_len ||
        !out_tokens || !num_tokens)
        return D3D_ERR_INVALID_ARG;
    if (!d3d::ws_ok(ws, ws_bytes, d3d::verify_layout(R, B, V).total))
        return D3D_ERR_WORKSPACE;
    const float c = (float)(1.4426950408889634 / (double)temperature);  // log2(e) / T
    unsigned char *w = static_cast<unsigned char *>(ws);
    if (logits_dtype == D3D_DTYPE_BF16)
        return d3d::launch_verify<uint16_t>(target_logits, draft_logits, draft_tokens, u_accept, u_sample, R, B, V,
                                            c, accept_len, out_tokens, num_tokens, alpha, p_draft, q_draft, w,
                                            stream);
    return d3d::launch_verify<float>(target_logits, draft_logits, draft_tokens, u_accept, u_sample, R, B, V, c,
                                     accept_len, out_tokens, num_tokens, alpha, p_draft, q_draft, w, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Verification without a caller workspace.
//
// For callers that cannot allocate device memory, the scratch the two
// verification kernels need lives in one fixed, file-scope device array.
// Every device that loads this library holds it until the process exits.
// ---------------------------------------------------------------------------
namespace d3d {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;  // 2 MiB
constexpr int kNoAllocMaxDevices = 64;

std::mutex g_noalloc_mu;
void *g_noalloc_addr[kNoAllocMaxDevices];

}  // namespace
}  // namespace d3d

static __device__ __align__(256) unsigned char d3d_noalloc_verify_scratch[d3d::kNoAllocScratchBytes];

namespace d3d {
namespace {

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device, with that device current, and cached.
int noalloc_scratch(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return D3D_ERR_CUDA;
    }
    if (dev < 0 || dev >= kNoAllocMaxDevices)
        return D3D_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, d3d_noalloc_verify_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return D3D_ERR_CUDA;
        }
        g_noalloc_addr[dev] = ptr;
    }
    *out = g_noalloc_addr[dev];
    return D3D_OK;
}

}  // namespace
}  // namespace d3d

extern "C" int d3d_spec_verify_noalloc(const void *target_logits, const void *draft_logits, int logits_dtype,
                                       const int32_t *draft_tokens, const float *u_accept, const float *u_sample,
                                       int R, int B, int V, float temperature, int32_t *accept_len,
                                       int32_t *out_tokens, int32_t *num_tokens, float *alpha, float *p_draft,
                                       float *q_draft, cudaStream_t stream)
{
    if (R < 0 || B < 2 || V < 1 || !(temperature > 0.f) || !isfinite(temperature))
        return D3D_ERR_INVALID_ARG;
    if (logits_dtype != D3D_DTYPE_F32 && logits_dtype != D3D_DTYPE_BF16)
        return D3D_ERR_INVALID_ARG;
    if (B > d3d::kMaxB || V > d3d::kMaxChunks * d3d::kVChunk)
        return D3D_ERR_UNSUPPORTED;
    if (R == 0)
        return D3D_OK;
    if (!target_logits || !draft_logits || !draft_tokens || !u_accept || !u_sample || !accept_len ||
        !out_tokens || !num_tokens)
        return D3D_ERR_INVALID_ARG;
    const d3d::VerifyLayout L = d3d::verify_layout(R, B, V);
    if (L.total > d3d::kNoAllocScratchBytes)
        return D3D_ERR_UNSUPPORTED;  // needs more scratch than the fixed array holds
    void *scratch = nullptr;
    const int rc = d3d::noalloc_scratch(&scratch);
    if (rc != D3D_OK)
        return rc;
    // the array keeps the previous call's contents: zero the status word and
    // the two per-request tickets, which must start at zero
    if (cudaMemsetAsync(scratch, 0, L.part1, stream) != cudaSuccess)
        return D3D_ERR_CUDA;
    const float c = (float)(1.4426950408889634 / (double)temperature);
    unsigned char *w = static_cast<unsigned char *>(scratch);
    if (logits_dtype == D3D_DTYPE_BF16)
        return d3d::launch_verify<uint16_t>(target_logits, draft_logits, draft_tokens, u_accept, u_sample, R, B, V,
                                            c, accept_len, out_tokens, num_tokens, alpha, p_draft, q_draft, w,
                                            stream);
    return d3d::launch_verify<float>(target_logits, draft_logits, draft_tokens, u_accept, u_sample, R, B, V, c,
                                     accept_len, out_tokens, num_tokens, alpha, p_draft, q_draft, w, stream);
}
