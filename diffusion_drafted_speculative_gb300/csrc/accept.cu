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
// Two launches over the logits, both streaming 8192-entry chunks of a row
// pair (target row j, draft row j) per CTA: the first stores each chunk's
// (max, sum of exponentials) of both rows; the second merges its row's chunk
// statistics into the softmax normalisers, sums min(P, Q) over its chunk, and
// the CTA that counts a request's last chunk adds the chunk sums of each row
// in a fixed order (deterministic) and writes a_j, S(k) and tau.  No CTA waits
// for another.
#include <math.h>

#include "d3d_common.cuh"

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

__host__ __device__ inline ALayout accept_layout(int R, int B, int V)
{
    ALayout L;
    L.nch = (V + kAChunk - 1) / kAChunk;
    const size_t items = (size_t)R * (size_t)(B - 1) * (size_t)L.nch;
    size_t o = sizeof(WsHeader);
    L.cnt = o;
    o = align_up(o + sizeof(int) * (size_t)R, kWsAlign);
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
            s_last = atomicAdd(cnt + r, 1) == (B - 1) * nch - 1;
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
            cnt[r] = 0;  // every chunk of the request has been counted: ready for the next call
        }
        __syncthreads();
    }
}

template <typename T> int launch_accept(const AArgs &a, cudaStream_t stream)
{
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
    return d3d::accept_layout(R, B, V).total;
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
    return logits_dtype == D3D_DTYPE_BF16 ? d3d::launch_accept<uint16_t>(a, stream)
                                          : d3d::launch_accept<float>(a, stream);
}

}  // extern "C"
