// Per-position acceptance probabilities, prefix survivals and the expected
// acceptance length of a verification round.
//
// [DScout] "Background: AWL and the acceptance rule": a draft token y ~ Q_j is
// accepted with probability min(1, P_j(y)/Q_j(y)), so position j accepts with
// probability a_j = sum_v min(P_j(v), Q_j(v)).  [DScout] "Background:
// acceptance length tau": S(k) = a_1 ... a_k survives k positions and
// tau = 1 + sum_{k=1}^{B-1} S(k).  P_j = softmax(target row j / T),
// Q_j = softmax(draft row j / T), in fp32.
//
// Two shapes.  Vocabulary slices (when each request's rows split over the
// SMs with the 2(B-1) rows of a slice resident in one CTA's shared memory):
// one cooperative launch, one CTA per (request, slice); the CTA copies its
// slice of every target and draft row once (bulk copies), stores each row's
// slice (max, sum of exponentials), waits for the request's other slices,
// merges the statistics into the softmax normalisers and sums min(P, Q) over
// its slice from shared memory; the CTA that counts the request's last slice
// adds the slice sums of each row in a fixed order and writes a_j, S(k) and
// tau.  The logits are read once.  Otherwise two launches over the logits,
// both streaming 8192-entry chunks of a row pair (target row j, draft row j)
// per CTA: the first stores each chunk's (max, sum of exponentials) of both
// rows; the second merges its row's chunk statistics, sums min(P, Q) over its
// chunk, and the CTA that counts a request's last chunk adds the chunk sums
// of each row in a fixed order (deterministic) and writes a_j, S(k) and tau.
// No CTA of the two-launch shape waits for another.
#include <math.h>

#include <mutex>

#include "d3d_common.cuh"
#include "sm100_ptx.cuh"

namespace d3d {
namespace {

constexpr int kAThreads = 256;
constexpr int kAChunk = 8192;
constexpr int kAPer = kAChunk / kAThreads;  // 32 entries per thread and item

struct AArgs {
    const void *target, *draft;
    int R, B, V;
    float c;  // log2(e) / T
    float *accept_prob, *survival, *tau;
    unsigned char *ws;
};

struct ALayout {
    size_t cnt, stats, part, total;
    int nch;
};

constexpr int kACnt = 4;  // counters per request

// chunk: 8192 entries (two launches) or the slice width (one launch)
__host__ __device__ inline ALayout accept_layout(int R, int B, int V, int chunk = kAChunk)
{
    ALayout L;
    L.nch = (V + chunk - 1) / chunk;
    const size_t items = (size_t)R * (size_t)(B - 1) * (size_t)L.nch;
    size_t o = sizeof(WsHeader);
    L.cnt = o;  // per request: slices done, waiters past them, min-sums done (the two launches use the last)
    o = align_up(o + sizeof(int) * kACnt * (size_t)R, kWsAlign);
    L.stats = o;  // per item: (max, sum) of the target chunk, then of the draft chunk (log2 units)
    o = align_up(o + sizeof(float4) * items, kWsAlign);
    L.part = o;  // per item: sum over the chunk of min(P, Q)
    o = align_up(o + sizeof(float) * items, kWsAlign);
    L.total = o;
    return L;
}

// This thread's entries of chunk [v0, v1) of a row, scaled by c (-inf past v1).
template <typename T>
__device__ __forceinline__ void load_chunk(const T *row, int v0, int v1, bool vec, float c, float (&x)[kAPer])
{
    if (vec) {
#pragma unroll
        for (int g = 0; g < kAPer / 8; ++g) {
            const int p = v0 + g * (8 * kAThreads) + 8 * (int)threadIdx.x;
            float t[8];
            if (p < v1) {
                load_logits8(row + p, t);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    t[e] = -INFINITY;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e)
                x[8 * g + e] = t[e] * c;
        }
    } else {
#pragma unroll
        for (int q = 0; q < kAPer; ++q) {
            const int p = v0 + q * kAThreads + (int)threadIdx.x;
            x[q] = p < v1 ? load_logit(row, p) * c : -INFINITY;
        }
    }
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Block-wide max of a and b (every thread gets both).
__device__ __forceinline__ float2 block_max2(float a, float b, float2 *s)
{
    a = warp_max(a), b = warp_max(b);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0)
        s[w] = make_float2(a, b);
    __syncthreads();
    float2 r = s[0];
#pragma unroll
    for (int i = 1; i < kAThreads / 32; ++i)
        r = make_float2(fmaxf(r.x, s[i].x), fmaxf(r.y, s[i].y));
    __syncthreads();
    return r;
}

// Block-wide sums of a and b (every thread gets both; fixed order).
__device__ __forceinline__ float2 block_sum2(float a, float b, float2 *s)
{
    a = warp_sum(a), b = warp_sum(b);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0)
        s[w] = make_float2(a, b);
    __syncthreads();
    float2 r = s[0];
#pragma unroll
    for (int i = 1; i < kAThreads / 32; ++i)
        r = make_float2(r.x + s[i].x, r.y + s[i].y);
    __syncthreads();
    return r;
}

// Item it = (request, position j, chunk) of target row (r, j) and draft row (r, j).
template <typename T>
__device__ __forceinline__ void item_rows(const AArgs &a, long long it, int nch, const T *&tr, const T *&dr, int &v0,
                                          int &v1)
{
    const int c = (int)(it % nch);
    const long long rj = it / nch;  // r * (B-1) + j
    const int r = (int)(rj / (a.B - 1)), j = (int)(rj % (a.B - 1));
    tr = static_cast<const T *>(a.target) + ((long long)r * a.B + j) * a.V;
    dr = static_cast<const T *>(a.draft) + rj * a.V;
    v0 = c * kAChunk;
    v1 = min(a.V, v0 + kAChunk);
}

template <typename T> __global__ void __launch_bounds__(kAThreads) accept_stats_kernel(const AArgs a)
{
    __shared__ float2 s_r[kAThreads / 32];
    const ALayout L = accept_layout(a.R, a.B, a.V);
    const long long n_items = (long long)a.R * (a.B - 1) * L.nch;
    float4 *stats = reinterpret_cast<float4 *>(a.ws + L.stats);
    const bool vec = a.V % 8 == 0 && (reinterpret_cast<uintptr_t>(a.target) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(a.draft) & 15) == 0;
    for (long long it = blockIdx.x; it < n_items; it += gridDim.x) {
        const T *tr, *dr;
        int v0, v1;
        item_rows<T>(a, it, L.nch, tr, dr, v0, v1);
        float x[kAPer], z[kAPer];
        load_chunk<T>(tr, v0, v1, vec, a.c, x);
        load_chunk<T>(dr, v0, v1, vec, a.c, z);
        float mx = -INFINITY, mz = -INFINITY;
#pragma unroll
        for (int q = 0; q < kAPer; ++q)
            mx = fmaxf(mx, x[q]), mz = fmaxf(mz, z[q]);
        const float2 m = block_max2(mx, mz, s_r);
        float sx = 0.f, sz = 0.f;
#pragma unroll
        for (int q = 0; q < kAPer; ++q) {
            sx += exp2f(x[q] - m.x);
            sz += exp2f(z[q] - m.y);
        }
        const float2 zs = block_sum2(sx, sz, s_r);
        if (threadIdx.x == 0)
            stats[it] = make_float4(m.x, zs.x, m.y, zs.y);
    }
    // the second launch reads these statistics once this grid has finished
    __threadfence();
    if (threadIdx.x == 0)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename T> __global__ void __launch_bounds__(kAThreads) accept_min_kernel(const AArgs a)
{
    __shared__ float2 s_r[kAThreads / 32];
    __shared__ float4 s_norm;
    __shared__ int s_last;
    __shared__ float s_a[256];
    // every statistic of the first launch is visible after this
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const ALayout L = accept_layout(a.R, a.B, a.V);
    const int nch = L.nch, B = a.B;
    const long long n_items = (long long)a.R * (B - 1) * nch;
    int *cnt = reinterpret_cast<int *>(a.ws + L.cnt);
    const float4 *stats = reinterpret_cast<const float4 *>(a.ws + L.stats);
    float *part = reinterpret_cast<float *>(a.ws + L.part);
    const bool vec = a.V % 8 == 0 && (reinterpret_cast<uintptr_t>(a.target) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(a.draft) & 15) == 0;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (long long it = blockIdx.x; it < n_items; it += gridDim.x) {
        const long long rj = it / nch;
        const int r = (int)(rj / (B - 1));
        // the row pair's softmax normalisers from its chunks' statistics
        if (w == 0) {
            float mx = -INFINITY, mz = -INFINITY;
            for (int k = lane; k < nch; k += 32) {
                const float4 st = __ldcg(stats + rj * nch + k);
                mx = fmaxf(mx, st.x), mz = fmaxf(mz, st.z);
            }
            mx = warp_max(mx), mz = warp_max(mz);
            float zx = 0.f, zz = 0.f;
            for (int k = lane; k < nch; k += 32) {
                const float4 st = __ldcg(stats + rj * nch + k);
                zx += st.y * exp2f(st.x - mx);
                zz += st.w * exp2f(st.z - mz);
            }
            zx = warp_sum(zx), zz = warp_sum(zz);
            if (lane == 0)
                s_norm = make_float4(mx, 1.f / zx, mz, 1.f / zz);
        }
        const T *tr, *dr;
        int v0, v1;
        item_rows<T>(a, it, nch, tr, dr, v0, v1);
        float x[kAPer], z[kAPer];
        load_chunk<T>(tr, v0, v1, vec, a.c, x);
        load_chunk<T>(dr, v0, v1, vec, a.c, z);
        __syncthreads();
        const float4 nm = s_norm;
        float sm = 0.f;
#pragma unroll
        for (int q = 0; q < kAPer; ++q)
            sm += fminf(exp2f(x[q] - nm.x) * nm.y, exp2f(z[q] - nm.z) * nm.w);
        const float2 tot = block_sum2(sm, 0.f, s_r);
        if (threadIdx.x == 0) {
            part[it] = tot.x;
            __threadfence();  // the chunk sum is visible before the count says so
            s_last = atomicAdd(cnt + kACnt * r + 2, 1) == (B - 1) * nch - 1;
        }
        __syncthreads();
        if (!s_last)
            continue;
        // ---- the request's last chunk: a_j (fixed order), then S(k) and tau
        __threadfence();
        for (int j = w; j < B - 1; j += kAThreads / 32) {
            // every lane adds its chunks in order, then a fixed shuffle tree
            float aj = 0.f;
            for (int k = lane; k < nch; k += 32)
                aj += __ldcg(part + ((long long)r * (B - 1) + j) * nch + k);
            aj = warp_sum(aj);
            if (lane == 0)
                s_a[j] = fminf(aj, 1.f);  // a probability: rounding may carry the sum past 1
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            float surv = 1.f, t = 1.f;
            for (int j = 0; j < B - 1; ++j) {
                surv *= s_a[j];
                t += surv;
                a.accept_prob[(long long)r * (B - 1) + j] = s_a[j];
                if (a.survival)
                    a.survival[(long long)r * (B - 1) + j] = surv;
            }
            if (a.tau)
                a.tau[r] = t;
            cnt[kACnt * r + 2] = 0;  // every chunk of the request has been counted: ready for the next call
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Vocabulary-slice shape: one CTA per (request, slice), every row of the slice
// resident in shared memory, the CTAs of a request resident together.
// ---------------------------------------------------------------------------
constexpr int kASliceThreads = 512;
constexpr int kASliceWarps = kASliceThreads / 32;
constexpr int kASliceGrain = 64;            // slice widths: multiples of 64 entries (16-byte aligned)
constexpr int kASliceMaxUnits = 256;        // units one launch may hold (bounds the workspace)
constexpr int kASliceSmemMax = 219 * 1024;  // dynamic shared memory of a slice CTA
constexpr uint64_t kAWaitNs = 250ull * 1000ull * 1000ull;

__device__ __forceinline__ float a_ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// One 16-byte vector (vi) of a row slice in shared memory as floats: 8 bf16
// or 4 fp32 entries.
template <typename T> struct AVec;
template <> struct AVec<uint16_t> {
    static constexpr int kN = 8;
    static __device__ __forceinline__ void get(const uint16_t *row, int vi, float (&x)[8])
    {
        const uint4 u = reinterpret_cast<const uint4 *>(row)[vi];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            x[2 * e] = __uint_as_float(w[e] << 16);
            x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
        }
    }
};
template <> struct AVec<float> {
    static constexpr int kN = 4;
    static __device__ __forceinline__ void get(const float *row, int vi, float (&x)[4])
    {
        const float4 u = reinterpret_cast<const float4 *>(row)[vi];
        x[0] = u.x, x[1] = u.y, x[2] = u.z, x[3] = u.w;
    }
};

// (scaled max, sum of exp2) of a row slice of n entries in shared memory (n
// a multiple of the vector width), by one warp
template <typename T>
__device__ __forceinline__ float2 a_row_stats(const T *row, int n, float c)
{
    constexpr int kN = AVec<T>::kN;
    const int lane = threadIdx.x & 31, nv = n / kN;
    float mr = -INFINITY;
    for (int vi = lane; vi < nv; vi += 32) {
        float x[kN];
        AVec<T>::get(row, vi, x);
#pragma unroll
        for (int e = 0; e < kN; ++e)
            mr = fmaxf(mr, x[e]);
    }
    mr = warp_max(mr);
    const float m = (mr == -INFINITY) ? -INFINITY : mr * c;
    const float nm = (mr == -INFINITY) ? 0.f : -m;
    float za = 0.f, zb = 0.f;
    for (int vi = lane; vi < nv; vi += 32) {
        float x[kN];
        AVec<T>::get(row, vi, x);
#pragma unroll
        for (int e = 0; e < kN; e += 2) {
            float a0, a1;
            sm100::ffma2(a0, a1, x[e], x[e + 1], c, c, nm, nm);
            sm100::fadd2(za, zb, za, zb, a_ex2(a0), a_ex2(a1));
        }
    }
    return make_float2(m, warp_sum(za + zb));
}

template <typename T>
__global__ void __launch_bounds__(kASliceThreads, 1) accept_slice_kernel(const AArgs a, int W, int nS)
{
    const int r = (int)blockIdx.x / nS, s = (int)blockIdx.x % nS;
    const int B = a.B, V = a.V, nb = B - 1, nrows = 2 * nb;
    const int v0 = s * W, v1 = min(V, v0 + W), n = v1 - v0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float c = a.c;
    const ALayout L = accept_layout(a.R, B, V, W);  // chunks = slices
    int *cnt = reinterpret_cast<int *>(a.ws + L.cnt) + kACnt * r;
    float4 *stats = reinterpret_cast<float4 *>(a.ws + L.stats);
    float *part = reinterpret_cast<float *>(a.ws + L.part);
    int32_t *status = reinterpret_cast<int32_t *>(a.ws);
    extern __shared__ __align__(128) unsigned char s_acc[];
    const T *rows = reinterpret_cast<const T *>(s_acc);
    const uint32_t rows_s = sm100::smem_u32(s_acc);
    const uint32_t bars_s = rows_s + (uint32_t)nrows * (uint32_t)W * (uint32_t)sizeof(T);
    auto row_of = [&](int i) { return rows + (size_t)i * W; };
    __shared__ volatile int s_abort;
    __shared__ int s_ok, s_last;
    __shared__ float s_a[256];

    // row i: target row j = i (i < nb) or draft row j = i - nb; thread i issues its copy
    const uint32_t row_bytes = (uint32_t)n * (uint32_t)sizeof(T);
    for (int i = threadIdx.x; i < nrows; i += kASliceThreads) {
        const uint32_t b = bars_s + 8u * (uint32_t)i;
        sm100::mbar_init(b, 1);
        sm100::fence_barrier_init();
        const T *src = i < nb ? static_cast<const T *>(a.target) + ((size_t)r * B + i) * V + v0
                              : static_cast<const T *>(a.draft) + ((size_t)r * nb + (i - nb)) * V + v0;
        sm100::mbar_arrive_expect_tx(b, row_bytes);
        sm100::bulk_load(rows_s + (uint32_t)i * (uint32_t)W * (uint32_t)sizeof(T), src, row_bytes, b);
    }
    if (threadIdx.x == 0)
        s_abort = 0;
    __syncthreads();
    auto wait_row = [&](int i) -> bool {
        const uint32_t b = bars_s + 8u * (uint32_t)i;
        bool ok = sm100::mbar_try_wait(b, 0);
        if (!ok) {
            const uint64_t t0 = sm100::global_ns();
            while (!(ok = sm100::mbar_try_wait_sleep(b, 0))) {
                if (s_abort || sm100::global_ns() - t0 > kAWaitNs) {
                    record_status(status, D3D_ERR_DEVICE_TIMEOUT);
                    s_abort = 1;
                    break;
                }
            }
        }
        return __all_sync(0xffffffffu, ok);
    };
    // the slice's statistics of each row pair (warp per position)
    for (int j = warp; j < nb; j += kASliceWarps) {
        if (!wait_row(j) || !wait_row(nb + j))
            break;
        const float2 px = a_row_stats<T>(row_of(j), n, c);
        const float2 pz = a_row_stats<T>(row_of(nb + j), n, c);
        if (lane == 0) {
            stats[((size_t)r * nb + j) * nS + s] = make_float4(px.x, px.y, pz.x, pz.y);
            __threadfence();  // before thread 0's signal, for the other CTAs
        }
    }
    __syncthreads();
    if (s_abort) {  // wait out the copies in flight (bounded), then leave
        if (threadIdx.x == 0)
            for (int i = 0; i < nrows; ++i) {
                const uint64_t t0 = sm100::global_ns();
                while (!sm100::mbar_try_wait_sleep(bars_s + 8u * (uint32_t)i, 0))
                    if (sm100::global_ns() - t0 > kAWaitNs)
                        break;
            }
        __syncthreads();
        return;
    }
    // every slice of the request has its statistics (release add, bounded acquire poll)
    if (threadIdx.x == 0) {
        asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(cnt) : "memory");
        int ok = 1;
        const uint64_t t0 = sm100::global_ns();
        for (;;) {
            int v;
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
            if (v >= nS)
                break;
            if (sm100::global_ns() - t0 > kAWaitNs) {
                record_status(status, D3D_ERR_DEVICE_TIMEOUT);
                ok = 0;
                break;
            }
        }
        s_ok = ok;
        if (ok && atomicAdd(cnt + 1, 1) == nS - 1) {  // the last waiter past resets the pair
            cnt[0] = 0;
            cnt[1] = 0;
        }
    }
    __syncthreads();
    if (!s_ok)
        return;
    // the row pair's normalisers from every slice, then min(P, Q) over this slice
    for (int j = warp; j < nb; j += kASliceWarps) {
        const float4 *st = stats + ((size_t)r * nb + j) * nS;
        float mx = -INFINITY, mz = -INFINITY;
        for (int k = lane; k < nS; k += 32) {
            const float4 t = __ldcg(st + k);
            mx = fmaxf(mx, t.x), mz = fmaxf(mz, t.z);
        }
        mx = warp_max(mx), mz = warp_max(mz);
        float zx = 0.f, zz = 0.f;
        for (int k = lane; k < nS; k += 32) {
            const float4 t = __ldcg(st + k);
            zx += t.x == -INFINITY ? 0.f : t.y * a_ex2(t.x - mx);
            zz += t.z == -INFINITY ? 0.f : t.w * a_ex2(t.z - mz);
        }
        const float rzx = 1.f / warp_sum(zx), rzz = 1.f / warp_sum(zz);
        const T *tx = row_of(j), *tz = row_of(nb + j);
        constexpr int kN = AVec<T>::kN;
        float sm = 0.f;
        for (int vi = lane; vi < n / kN; vi += 32) {
            float x[kN], z[kN];
            AVec<T>::get(tx, vi, x);
            AVec<T>::get(tz, vi, z);
#pragma unroll
            for (int e = 0; e < kN; ++e)
                sm += fminf(a_ex2(x[e] * c - mx) * rzx, a_ex2(z[e] * c - mz) * rzz);
        }
        sm = warp_sum(sm);
        if (lane == 0) {
            part[((size_t)r * nb + j) * nS + s] = sm;
            __threadfence();  // the slice sum is visible before the count says so
        }
    }
    __syncthreads();
    if (threadIdx.x == 0)
        s_last = atomicAdd(cnt + 2, 1) == nS - 1;
    __syncthreads();
    if (!s_last)
        return;
    // ---- the request's last slice: a_j (fixed order), then S(k) and tau
    __threadfence();
    for (int j = warp; j < nb; j += kASliceWarps) {
        float aj = 0.f;
        for (int k = lane; k < nS; k += 32)
            aj += __ldcg(part + ((size_t)r * nb + j) * nS + k);
        aj = warp_sum(aj);
        if (lane == 0)
            s_a[j] = fminf(aj, 1.f);  // a probability: rounding may carry the sum past 1
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float surv = 1.f, t = 1.f;
        for (int j = 0; j < nb; ++j) {
            surv *= s_a[j];
            t += surv;
            a.accept_prob[(size_t)r * nb + j] = s_a[j];
            if (a.survival)
                a.survival[(size_t)r * nb + j] = surv;
        }
        if (a.tau)
            a.tau[r] = t;
        cnt[2] = 0;
    }
}

// Slice width for R requests over `units` CTAs (0 when a request gets none).
inline int a_slice_width(int R, int V, int units)
{
    const int per = units / R;
    if (per < 1)
        return 0;
    const long long w = ((long long)V + per - 1) / per;
    return (int)((w + kASliceGrain - 1) / kASliceGrain * kASliceGrain);
}

template <typename T> bool a_slice_plan(const AArgs &a, size_t ws_bytes, int &W, int &nS, size_t &dyn)
{
    if ((size_t)a.V * sizeof(T) % 16 != 0 || (reinterpret_cast<uintptr_t>(a.target) & 15) != 0 ||
        (reinterpret_cast<uintptr_t>(a.draft) & 15) != 0 || a.B - 1 > 256)
        return false;
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    W = a_slice_width(a.R, a.V, nsm < kASliceMaxUnits ? nsm : kASliceMaxUnits);
    if (W <= 0)
        return false;
    nS = (a.V + W - 1) / W;
    const int nrows = 2 * (a.B - 1);
    dyn = (size_t)nrows * (size_t)W * sizeof(T) + (size_t)nrows * 8;
    if (dyn > (size_t)kASliceSmemMax || accept_layout(a.R, a.B, a.V, W).total > ws_bytes)
        return false;
    return set_max_dyn_smem<accept_slice_kernel<T>>(kASliceSmemMax) == cudaSuccess;
}

template <typename T> int launch_accept_slice(const AArgs &a, int W, int nS, size_t dyn, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.R * nS));
    cfg.blockDim = dim3(kASliceThreads);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // the CTAs of a request wait on one another
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, accept_slice_kernel<T>, a, W, nS));
}

template <typename T> int launch_accept(const AArgs &a, cudaStream_t stream, size_t ws_bytes)
{
    int W = 0, nS = 0;
    size_t dyn = 0;
    if (a_slice_plan<T>(a, ws_bytes, W, nS, dyn))
        return launch_accept_slice<T>(a, W, nS, dyn, stream);
    cudaGetLastError();
    const ALayout L = accept_layout(a.R, a.B, a.V);
    const long long n_items = (long long)a.R * (a.B - 1) * L.nch;
    int dev = 0, nsm = 0, per_a = 0, per_b = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_a, accept_stats_kernel<T>, kAThreads, 0) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_b, accept_min_kernel<T>, kAThreads, 0) != cudaSuccess ||
        per_a < 1 || per_b < 1)
        return D3D_ERR_CUDA;
    const long long cap_a = (long long)nsm * per_a, cap_b = (long long)nsm * per_b;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kAThreads);
    cfg.stream = stream;
    cfg.gridDim = dim3((unsigned)(n_items < cap_a ? n_items : cap_a));
    cudaError_t e = cudaLaunchKernelEx(&cfg, accept_stats_kernel<T>, a);
    if (e != cudaSuccess)
        return D3D_ERR_CUDA;
    // the second launch starts as the first one's CTAs finish (programmatic
    // dependent launch) and waits for all of them before reading
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)(n_items < cap_b ? n_items : cap_b));
    e = cudaLaunchKernelEx(&cfg, accept_min_kernel<T>, a);
    return cuda_status(e);
}

}  // namespace
}  // namespace d3d

extern "C" {

size_t d3d_accept_probs_workspace_size(int R, int B, int V)
{
    if (R < 0 || B < 2 || V < 1 || B > 257)
        return 0;
    // the two launches' chunks, or the finest slices a launch may take
    const size_t chunked = d3d::accept_layout(R, B, V).total;
    const int W = d3d::a_slice_width(R, V, d3d::kASliceMaxUnits);
    const size_t sliced = W > 0 ? d3d::accept_layout(R, B, V, W).total : 0;
    return chunked > sliced ? chunked : sliced;
}

int d3d_accept_probs(const void *target_logits, const void *draft_logits, int logits_dtype, int R, int B, int V,
                     float temperature, float *accept_prob, float *survival, float *tau, void *ws, size_t ws_bytes,
                     cudaStream_t stream)
{
    if (R < 0 || B < 2 || V < 1 || !(temperature > 0.f) || !isfinite(temperature))
        return D3D_ERR_INVALID_ARG;
    if (logits_dtype != D3D_DTYPE_F32 && logits_dtype != D3D_DTYPE_BF16)
        return D3D_ERR_INVALID_ARG;
    if (B > 257)
        return D3D_ERR_UNSUPPORTED;
    if (R == 0)
        return D3D_OK;
    if (!target_logits || !draft_logits || !accept_prob)
        return D3D_ERR_INVALID_ARG;
    if (!d3d::ws_ok(ws, ws_bytes, d3d::accept_layout(R, B, V).total))
        return D3D_ERR_WORKSPACE;
    d3d::AArgs a;
    a.target = target_logits;
    a.draft = draft_logits;
    a.R = R, a.B = B, a.V = V;
    a.c = (float)(1.4426950408889634 / (double)temperature);
    a.accept_prob = accept_prob, a.survival = survival, a.tau = tau;
    a.ws = static_cast<unsigned char *>(ws);
    return logits_dtype == D3D_DTYPE_BF16 ? d3d::launch_accept<uint16_t>(a, stream, ws_bytes)
                                          : d3d::launch_accept<float>(a, stream, ws_bytes);
}

}  // extern "C"
