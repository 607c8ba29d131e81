// Speculative-sampling verification over the vocabulary.
//
// [D3D] "Background: speculative decoding"; [DScout] "Background:
// speculative decoding" and "Background: AWL and the acceptance rule":
// alpha_j = min(1, P_j(y_j)/Q_j(y_j)), accept while u_j < alpha_j, then
// resample from norm(max(0, P - Q)) at the first rejection or draw a bonus
// token from P_B when every draft is accepted.
//
// One cooperative kernel (all CTAs resident, guaranteed by the launch) in
// three phases.  A phase waits only for the previous phase of the same
// request, through per-request counters (bounded spins); phase A waits for
// nothing, so every wait ends even when CTAs loop over several items:
//   A. one work item per (logit row, 8192-entry chunk): 16-byte vector loads,
//      the chunk's softmax statistics (max and sum of exp2, log2 domain) and,
//      for rows that are evaluated at a draft token, that token's logit when
//      it lies in the chunk.  One record per item.
//   B+C. one item per (request, chunk): the CTA combines its request's records
//      in shared memory (every such CTA does, which costs L2 reads instead of
//      a barrier), forms p_j, q_j, alpha_j, runs the first-rejection scan,
//      picks the row pair the sample needs, and computes its chunk's residual
//      max(0, P - Q) (or P_B) mass, keeping the per-entry masses in registers.
//      The chunk-0 CTA writes the per-request outputs.
//   D. every item reads its request's chunk sums; the one chunk holding the
//      crossing C(v) > u*S scans its registers in vocabulary order and writes
//      the sampled token.  The request's last phase-D item resets its counters.
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
constexpr int kVBlocksPerSm = 2;  // register budget for four resident CTAs per SM
constexpr uint64_t kBarrierTimeoutNs = 250ull * 1000ull * 1000ull;
constexpr int kStagedRecords = 2048;  // chunk records the finalising CTA stages in shared memory (32 KB)
constexpr unsigned kFull = 0xffffffffu;

// What the sample of one request uses.
struct Sel {
    int32_t a;     // accepted drafts
    int32_t mode;  // 0: residual at target/draft row a; 1: bonus from target row B-1
    int32_t row;   // target row the sample uses (and draft row when mode == 0)
    float mP, rZP, mQ, rZQ;  // log2-domain row max and 1 / normaliser of that target / draft row
};

struct VerifyLayout {
    size_t bar, part1, part2, total;  // bar: per-request counters
    int nch;
};

__host__ __device__ inline VerifyLayout verify_layout(int R, int B, int V)
{
    VerifyLayout L;
    L.nch = (V + kVChunk - 1) / kVChunk;
    size_t o = sizeof(WsHeader);
    L.bar = o;  // per request: phase-A items done, phase-C items done, phase-D items done
    o = align_up(o + 3 * sizeof(int) * (size_t)R, kWsAlign);
    L.part1 = o;  // per (row, chunk): max, sum, scaled logit of the row's draft token if in the chunk
    o = align_up(o + sizeof(float4) * (size_t)R * (size_t)(2 * B - 1) * (size_t)L.nch, kWsAlign);
    L.part2 = o;  // per (request, chunk): residual mass, P mass
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

// Wait (thread 0 spins, bounded) until *cnt reaches `target`, then make the
// producers' writes visible to the whole CTA.  Returns false if the wait ran
// out (the status word is then set).
__device__ bool wait_count(const int *cnt, int target, int32_t *status)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        if (*reinterpret_cast<const volatile int *>(cnt) < target) {
            uint64_t t0;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
            while (*reinterpret_cast<const volatile int *>(cnt) < target) {
                uint64_t t1;
                asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
                if (t1 - t0 > kBarrierTimeoutNs) {
                    record_status(status, D3D_ERR_DEVICE_TIMEOUT);
                    ok = 0;
                    break;
                }
            }
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// Signal one finished item: its writes first, then the count (no return value).
__device__ inline void signal_count(int *cnt)
{
    __threadfence();
    asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(cnt) : "memory");
}

// Phase B for request r, done by one CTA: combine the records, alpha_j, the
// first rejection, the sample's row pair.  With write_outputs the CTA also
// writes accept_len, num_tokens, alpha/p/q and the accepted tokens.
template <typename T>
__device__ void select_request(int r, int B, int V, int nch, const float4 *__restrict__ part1,
                               const int32_t *__restrict__ y, const float *__restrict__ u_acc, bool write_outputs,
                               int32_t *__restrict__ accept_len, int32_t *__restrict__ out_tokens,
                               int32_t *__restrict__ num_tokens, float *__restrict__ alpha_out,
                               float *__restrict__ p_out, float *__restrict__ q_out, int32_t *status, Sel &sel,
                               float4 *s_part)
{
    __shared__ float s_m[2 * kMaxB], s_z[2 * kMaxB], s_u[kMaxB];
    __shared__ int s_y[kMaxB], s_a;
    const int rows = 2 * B - 1;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float4 *pr = part1 + (size_t)r * rows * nch;
    const int nrec = rows * nch;
    const bool staged = nrec <= kStagedRecords;
    if (staged)
        for (int i = threadIdx.x; i < nrec; i += kVThreads)
            s_part[i] = __ldcg(&pr[i]);
    for (int jj = threadIdx.x; jj < B - 1; jj += kVThreads) {
        s_y[jj] = y[(size_t)r * (B - 1) + jj];
        s_u[jj] = u_acc[(size_t)r * (B - 1) + jj];
    }
    if (threadIdx.x == 0)
        s_a = B - 1;
    __syncthreads();
    for (int jj = warp; jj < rows; jj += kVWarps) {
        // row max over the chunk records, then the rescaled sums
        float mm = -INFINITY, zz = 0.f;
        for (int cc = lane; cc < nch; cc += 32) {
            const float4 t = staged ? s_part[jj * nch + cc] : __ldcg(&pr[(size_t)jj * nch + cc]);
            ms_merge(mm, zz, t.x, t.y);
        }
        float M = mm;
#pragma unroll
        for (int o = 16; o; o >>= 1)
            M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
        float zs = (mm == -INFINITY) ? 0.f : zz * fast_exp2(mm - M);
#pragma unroll
        for (int o = 16; o; o >>= 1)
            zs += __shfl_xor_sync(kFull, zs, o);
        if (lane == 0) {
            s_m[jj] = M;
            s_z[jj] = zs;
        }
    }
    __syncthreads();
    // alpha_j and the acceptance test of every position in parallel; the first
    // rejection is the smallest rejected position
    for (int jj = threadIdx.x; jj < B - 1; jj += kVThreads) {
        const int yv = s_y[jj];
        float p = 0.f, q = 0.f, al = 0.f;
        if (yv < 0 || yv >= V) {
            if (write_outputs)
                record_status(status, D3D_ERR_DEVICE_INPUT);
        } else {
            const int ch = yv / kVChunk;
            const size_t it = (size_t)jj * nch + ch, id = (size_t)(B + jj) * nch + ch;
            const float xt = staged ? s_part[it].z : __ldcg(&pr[it]).z;
            const float xd = staged ? s_part[id].z : __ldcg(&pr[id]).z;
            p = fast_exp2(xt - s_m[jj]) / s_z[jj];
            q = fast_exp2(xd - s_m[B + jj]) / s_z[B + jj];
            al = (p >= q) ? 1.f : p / q;
        }
        if (!(s_u[jj] < al))
            atomicMin(&s_a, jj);
        if (write_outputs) {
            const size_t o = (size_t)r * (B - 1) + jj;
            if (alpha_out)
                alpha_out[o] = al;
            if (p_out)
                p_out[o] = p;
            if (q_out)
                q_out[o] = q;
        }
    }
    __syncthreads();
    const int a = s_a;
    sel.a = a;
    sel.mode = (a < B - 1) ? 0 : 1;
    sel.row = (a < B - 1) ? a : B - 1;
    sel.mP = s_m[sel.row];
    sel.rZP = __frcp_rn(s_z[sel.row]);
    sel.mQ = (a < B - 1) ? s_m[B + a] : 0.f;
    sel.rZQ = (a < B - 1) ? __frcp_rn(s_z[B + a]) : 1.f;
    if (write_outputs) {
        if (threadIdx.x == 0) {
            accept_len[r] = a;
            num_tokens[r] = a + 1;
        }
        for (int jj = threadIdx.x; jj < B; jj += kVThreads)
            if (jj != a)
                out_tokens[(size_t)r * B + jj] = (jj < a) ? s_y[jj] : -1;
    }
    __syncthreads();  // the shared arrays are reused by the next call
}

// Mass of position v of the sampled distribution: the residual
// max(0, P - Q) (kind 0) or P itself (kind 1); xp/xq are scaled logits.
__device__ inline float sample_mass(int kind, float xp, float xq, const Sel &sel)
{
    const float P = fast_exp2(xp - sel.mP) * sel.rZP;
    if (kind != 0)
        return P;
    const float Q = fast_exp2(xq - sel.mQ) * sel.rZQ;
    return fmaxf(P - Q, 0.f);
}

// Per-entry masses of one chunk [c0, c1) in thread-contiguous order
// (positions c0 + tid*kVPer + k), and their sums.
template <typename T>
__device__ inline void chunk_masses(const T *prow, const T *qrow, int kind, int c0, int c1, float c,
                                    const Sel &sel, float (&w)[kVPer], float &s_kind, float &s_p)
{
    float xp[kVPer], xq[kVPer];
    load_chunk_contig<T>(prow, c0, c1, c, xp);
    if (kind == 0)
        load_chunk_contig<T>(qrow, c0, c1, c, xq);
    s_kind = 0.f;
    s_p = 0.f;
#pragma unroll
    for (int k = 0; k < kVPer; ++k) {
        const bool in = c0 + (int)threadIdx.x * kVPer + k < c1;
        const float P = in ? fast_exp2(xp[k] - sel.mP) * sel.rZP : 0.f;
        w[k] = in ? (kind == 0 ? fmaxf(P - fast_exp2(xq[k] - sel.mQ) * sel.rZQ, 0.f) : P) : 0.f;
        s_kind += w[k];
        s_p += P;
    }
}

template <typename T>
__global__ void __launch_bounds__(kVThreads, kVBlocksPerSm)
    verify_kernel(const T *__restrict__ target, const T *__restrict__ draft, const int32_t *__restrict__ y,
                  const float *__restrict__ u_acc, const float *__restrict__ u_s, int R, int B, int V, float c,
                  int32_t *__restrict__ accept_len, int32_t *__restrict__ out_tokens,
                  int32_t *__restrict__ num_tokens, float *__restrict__ alpha_out, float *__restrict__ p_out,
                  float *__restrict__ q_out, unsigned char *__restrict__ ws)
{
    extern __shared__ float4 s_part[];  // request records when staged; chunk sums in phase D
    __shared__ float red[2 * kVWarps];
    __shared__ float s_xy;
    const VerifyLayout L = verify_layout(R, B, V);
    const int rows = 2 * B - 1, nch = L.nch;
    const long long nA = (long long)R * rows * nch;
    const int nC = R * nch;
    float4 *part1 = reinterpret_cast<float4 *>(ws + L.part1);
    float2 *part2 = reinterpret_cast<float2 *>(ws + L.part2);
    int *bar = reinterpret_cast<int *>(ws + L.bar);
    int32_t *status = reinterpret_cast<int32_t *>(ws);

    // ---- phase A: per (row, chunk) statistics; the next item's loads are in
    // flight while the current item is reduced
    auto item_row = [&](long long item, int &v0, int &v1, int &yy) -> const T * {
        const int chunk = (int)(item % nch);
        const int rowg = (int)(item / nch);
        const int r = rowg / rows, j = rowg % rows;
        v0 = chunk * kVChunk;
        v1 = min(V, v0 + kVChunk);
        // the draft token this row is evaluated at (none for the bonus row P_B)
        const int yj = (j < B - 1) ? j : (j >= B ? j - B : -1);
        yy = (yj >= 0) ? __ldg(y + (size_t)r * (B - 1) + yj) : -1;
        return (j < B) ? target + ((size_t)r * B + j) * V : draft + ((size_t)r * (B - 1) + (j - B)) * V;
    };
    float xc[kVPer];
    int v0c = 0, v1c = 0, yyc = -1;
    long long item = blockIdx.x;
    if (item < nA)
        load_chunk_strided<T>(item_row(item, v0c, v1c, yyc), v0c, v1c, c, xc);
    while (item < nA) {
        const long long next = item + gridDim.x;
        float xn[kVPer];
        int v0n = 0, v1n = 0, yyn = -1;
        if (next < nA)
            load_chunk_strided<T>(item_row(next, v0n, v1n, yyn), v0n, v1n, c, xn);
        const int r = (int)(item / nch) / rows;
        if (yyc >= v0c && yyc < v1c) {  // the thread holding x[yy] keeps it for the record
            const int rel = yyc - v0c;
            if ((int)threadIdx.x == (rel % (kVThreads * 8)) / 8) {
                const int slot = (rel / (kVThreads * 8)) * 8 + rel % 8;
                float xv = 0.f;
#pragma unroll
                for (int k = 0; k < kVPer; ++k)
                    xv = (k == slot) ? xc[k] : xv;
                s_xy = xv;
            }
        }
        float m = -INFINITY, z = 0.f;
#pragma unroll
        for (int k = 0; k < kVPer; ++k)
            m = fmaxf(m, xc[k]);
        if (m != -INFINITY) {
#pragma unroll
            for (int k = 0; k < kVPer; ++k)
                z += fast_exp2(xc[k] - m);
        }
        block_ms(m, z, red);  // has a __syncthreads: s_xy is visible to thread 0 after it
        if (threadIdx.x == 0) {
            part1[item] = make_float4(m, z, (yyc >= v0c && yyc < v1c) ? s_xy : 0.f, 0.f);
            signal_count(bar + 3 * r);
        }
        __syncthreads();  // red and s_xy are reused by the next item
        if (next < nA) {
#pragma unroll
            for (int k = 0; k < kVPer; ++k)
                xc[k] = xn[k];
        }
        v0c = v0n, v1c = v1n, yyc = yyn;
        item = next;
    }

    // ---- phase B+C: the request's selection, then this chunk's masses
    const bool keep = nC <= (int)gridDim.x;  // at most one item per CTA: masses stay in registers
    float w[kVPer];
    Sel sel;
#pragma unroll
    for (int k = 0; k < kVPer; ++k)
        w[k] = 0.f;
    sel.a = 0, sel.mode = 1, sel.row = 0, sel.mP = 0.f, sel.rZP = 0.f, sel.mQ = 0.f, sel.rZQ = 0.f;
    for (int item = blockIdx.x; item < nC; item += gridDim.x) {
        const int r = item / nch, chunk = item % nch;
        if (!wait_count(bar + 3 * r, rows * nch, status))
            return;
        select_request<T>(r, B, V, nch, part1, y, u_acc, chunk == 0, accept_len, out_tokens, num_tokens, alpha_out,
                          p_out, q_out, status, sel, s_part);
        const T *prow = target + ((size_t)r * B + sel.row) * V;
        const T *qrow = draft + ((size_t)r * (B - 1) + (sel.mode == 0 ? sel.row : 0)) * V;
        const int c0 = chunk * kVChunk, c1 = min(V, c0 + kVChunk);
        float s_kind, s_p;
        chunk_masses<T>(prow, qrow, sel.mode == 0 ? 0 : 1, c0, c1, c, sel, w, s_kind, s_p);
        block_sum2(s_kind, s_p, red);
        if (threadIdx.x == 0) {
            part2[item] = make_float2(s_kind, s_p);
            signal_count(bar + 3 * r + 1);
        }
        __syncthreads();
    }

    // ---- phase D: the chunk holding the crossing scans its masses
    __shared__ int s_kind_used, s_owner, s_takelast, s_cand, s_lastpos;
    __shared__ float s_prefix, s_target;
    for (int item = blockIdx.x; item < nC; item += gridDim.x) {
        const int r = item / nch, chunk = item % nch;
        if (!wait_count(bar + 3 * r + 1, nch, status))
            return;
        if (!keep)  // every phase-C item of r waited for r's phase A, so the records are complete
            select_request<T>(r, B, V, nch, part1, y, u_acc, false, accept_len, out_tokens, num_tokens, alpha_out,
                              p_out, q_out, status, sel, s_part);
        float2 *s_sums = reinterpret_cast<float2 *>(s_part);  // the records are no longer needed
        for (int cc = threadIdx.x; cc < nch; cc += kVThreads)
            s_sums[cc] = __ldcg(part2 + (size_t)r * nch + cc);
        __syncthreads();
        if (threadIdx.x == 0) {
            const float2 *pr = s_sums;
            float S_res = 0.f, S_p = 0.f;
            for (int cc = 0; cc < nch; ++cc) {
                const float2 t = pr[cc];
                S_res += t.x;
                S_p += t.y;
            }
            // residual unless it has no mass left in fp32 (then P at that row)
            const int kind = (sel.mode == 0 && S_res > 0.f) ? 0 : 1;
            const float S = kind == 0 ? S_res : S_p;
            const float tgt = u_s[r] * S;
            float run = 0.f;
            int owner = -1;
            for (int cc = 0; cc < nch; ++cc) {
                const float2 t = pr[cc];
                const float sc = kind == 0 ? t.x : t.y;
                if (run + sc > tgt) {
                    owner = cc;
                    break;
                }
                run += sc;
            }
            int takelast = 0;
            if (owner < 0) {  // rounding left u*S at or past the end: last chunk with mass
                takelast = 1;
                for (int cc = nch - 1; cc >= 0 && owner < 0; --cc) {
                    const float2 t = pr[cc];
                    if ((kind == 0 ? t.x : t.y) > 0.f)
                        owner = cc;
                }
            }
            s_kind_used = kind;
            s_owner = owner;
            s_takelast = takelast;
            s_prefix = run;
            s_target = tgt;
            s_cand = kVThreads;
            s_lastpos = -1;
        }
        __syncthreads();
        const int owner = s_owner;
        if (owner == chunk) {
            const int kind = s_kind_used;
            const int c0 = chunk * kVChunk, c1 = min(V, c0 + kVChunk);
            if (!keep || kind != (sel.mode == 0 ? 0 : 1)) {  // masses not in registers (or the fallback kind)
                const T *prow = target + ((size_t)r * B + sel.row) * V;
                const T *qrow = draft + ((size_t)r * (B - 1) + (sel.mode == 0 ? sel.row : 0)) * V;
                float a1, a2;
                chunk_masses<T>(prow, qrow, kind, c0, c1, c, sel, w, a1, a2);
            }
            float tot = 0.f;
            int lastpos = -1;
#pragma unroll
            for (int k = 0; k < kVPer; ++k) {
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
            if (!s_takelast && (int)threadIdx.x == s_cand) {
                int tok = -1;
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
                out_tokens[(size_t)r * B + sel.a] = tok;
            }
            if ((s_takelast || s_cand == kVThreads) && threadIdx.x == 0)
                out_tokens[(size_t)r * B + sel.a] = s_lastpos;
        } else if (owner < 0 && chunk == 0 && threadIdx.x == 0) {
            // no mass anywhere: cannot happen for a finite softmax row
            record_status(status, D3D_ERR_DEVICE_INPUT);
            out_tokens[(size_t)r * B + sel.a] = 0;
        }
        // the request's last phase-D item resets its counters for the next call
        // (every phase-A and phase-C signal of the request has arrived by now)
        if (threadIdx.x == 0 && atomicAdd(bar + 3 * r + 2, 1) == nch - 1) {
            bar[3 * r] = 0;
            bar[3 * r + 1] = 0;
            bar[3 * r + 2] = 0;
        }
        __syncthreads();
    }
}

template <typename T>
int launch_verify(const void *target, const void *draft, const int32_t *y, const float *u_acc, const float *u_s,
                  int R, int B, int V, float c, int32_t *accept_len, int32_t *out_tokens, int32_t *num_tokens,
                  float *alpha, float *p, float *q, unsigned char *ws, cudaStream_t stream)
{
    const VerifyLayout L = verify_layout(R, B, V);
    const long long nA = (long long)R * (2 * B - 1) * L.nch;
    if (nA > 0x7fffffffLL)
        return D3D_ERR_UNSUPPORTED;
    const int nrec = (2 * B - 1) * L.nch;
    // dynamic shared memory: the request's records when they are staged, and
    // at least the request's chunk sums (phase D)
    size_t dyn = nrec <= kStagedRecords ? sizeof(float4) * (size_t)nrec : 0;
    if (dyn < sizeof(float2) * (size_t)L.nch)
        dyn = sizeof(float2) * (size_t)L.nch;
    // every CTA must be resident (grid-wide barriers): at most the occupancy
    // limit, and no more than there are phase-A items
    int dev = 0, nsm = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_kernel<T>, kVThreads, dyn) != cudaSuccess ||
        per_sm < 1)
        return D3D_ERR_CUDA;
    const long long cap = (long long)nsm * per_sm;
    const unsigned grid = (unsigned)(nA < cap ? nA : cap);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kVThreads);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, verify_kernel<T>, static_cast<const T *>(target),
                                             static_cast<const T *>(draft), y, u_acc, u_s, R, B, V, c, accept_len,
                                             out_tokens, num_tokens, alpha, p, q, ws);
    return cuda_status(e);
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
