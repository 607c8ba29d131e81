// Greedy verification (temperature 0): the decoding setting of the pages'
// results ([D3D] "Experiments"; [DScout] "Experiments").  At temperature 0
// the speculative-sampling rule ([D3D] "Background: speculative decoding")
// keeps a draft token exactly when it is the target's most likely token and
// adds the target's most likely token after the accepted prefix.  Ties go to
// the lowest token index.
//
// One pass over the target logits only (the draft logits are not needed):
// a work item is 8192 entries of one target row; its CTA reduces them to the
// (largest value, lowest index) pair and stores it in the workspace.  The
// CTA that completes the last item of a request (a per-request counter)
// reduces the request's pairs to the argmax of every row, finds the accepted
// prefix and writes the outputs, then the fused branch match.  No CTA ever
// waits for another, so the launch needs no co-residency.
#pragma once

#include <math.h>

#include "verify_body.cuh"

namespace d3d {
namespace {

constexpr int kGThreads = 256;
constexpr int kGChunk = kVChunkMin;         // entries per item: the records fit the sampling layout
constexpr int kGPer = kGChunk / kGThreads;  // 32 entries per thread and item
static_assert(kGPer % 8 == 0, "whole 8-entry groups per thread");

// Larger value first, then the lower index.
__device__ __forceinline__ bool ahead(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

__device__ __forceinline__ void warp_best(float &v, int &i)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_down_sync(0xffffffffu, v, o);
        const int oi = __shfl_down_sync(0xffffffffu, i, o);
        if (ahead(ov, oi, v, i))
            v = ov, i = oi;
    }
}

// (largest value, lowest index) over entries [v0, v1) of row `row`,
// returned to thread 0.  Entries equal to NaN never win; an empty or all-NaN
// range reports index INT_MAX.
template <typename T>
__device__ void chunk_best(const T *row, int v0, int v1, bool vec, float *s_v, int *s_i, float &bv, int &bi)
{
    bv = -INFINITY;
    bi = INT_MAX;
    if (vec) {  // 16-byte aligned groups of 8 entries (V % 8 == 0)
        float x[kGPer];
#pragma unroll
        for (int g = 0; g < kGPer / 8; ++g) {
            const int p = v0 + g * (8 * kGThreads) + 8 * (int)threadIdx.x;
            float t[8];
            if (p < v1) {
                Logit<T>::load8(row + p, t);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    t[e] = -INFINITY;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e)
                x[8 * g + e] = t[e];
        }
#pragma unroll
        for (int g = 0; g < kGPer / 8; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int p = v0 + g * (8 * kGThreads) + 8 * (int)threadIdx.x + e;
                if (p < v1 && ahead(x[8 * g + e], p, bv, bi))
                    bv = x[8 * g + e], bi = p;
            }
    } else {
        for (int p = v0 + (int)threadIdx.x; p < v1; p += kGThreads) {
            const float x = Logit<T>::at(row, (size_t)p);
            if (ahead(x, p, bv, bi))
                bv = x, bi = p;
        }
    }
    warp_best(bv, bi);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0)
        s_v[w] = bv, s_i[w] = bi;
    __syncthreads();
    if (w == 0) {
        bv = lane < kGThreads / 32 ? s_v[lane] : -INFINITY;
        bi = lane < kGThreads / 32 ? s_i[lane] : INT_MAX;
        warp_best(bv, bi);
    }
    __syncthreads();  // s_v / s_i are reused by the next item
}

template <typename T>
__global__ void __launch_bounds__(kGThreads) greedy_kernel(const VArgs a)
{
    __shared__ float s_v[kGThreads / 32];
    __shared__ int s_i[kGThreads / 32];
    __shared__ int32_t s_y[kMaxB];
    __shared__ int32_t s_g[kMaxB];
    __shared__ int s_last;
    if (threadIdx.x == 0)
        sm100::pdl_trigger();  // an independent kernel launched after this one may start
    const int R = a.R, B = a.B, V = a.V;
    const VerifyLayout L = verify_layout(R, B, V, kGChunk);
    const int nch = L.nch;
    const long long n_items = (long long)R * B * nch;
    int *bar = reinterpret_cast<int *>(a.ws + L.bar);
    Rec *rec = reinterpret_cast<Rec *>(a.ws + L.rec);
    int32_t *status = reinterpret_cast<int32_t *>(a.ws);
    const T *tgt = static_cast<const T *>(a.target);
    const bool vec = V % 8 == 0 && (reinterpret_cast<uintptr_t>(tgt) & 15) == 0;

    for (long long it = blockIdx.x; it < n_items; it += gridDim.x) {
        const int c = (int)(it % nch);
        const long long rj = it / nch;
        const int r = (int)(rj / B);
        const int v0 = c * kGChunk, v1 = min(V, v0 + kGChunk);
        float bv;
        int bi;
        chunk_best<T>(tgt + rj * (long long)V, v0, v1, vec, s_v, s_i, bv, bi);
        if (threadIdx.x == 0) {
            float2 *dst = reinterpret_cast<float2 *>(rec + it);
            *dst = make_float2(bv, __int_as_float(bi));
            __threadfence();  // the pair is visible before the count says so
            s_last = atomicAdd(bar + kBarInts * r, 1) == B * nch - 1;
        }
        __syncthreads();
        if (!s_last)
            continue;
        // ---- the request's last item: argmax of every row, then the round's outputs
        __threadfence();
        const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
        for (int j = w; j < B; j += kGThreads / 32) {
            float v = -INFINITY;
            int i = INT_MAX;
            for (int k = lane; k < nch; k += 32) {
                const float2 p = __ldcg(reinterpret_cast<const float2 *>(rec + ((long long)r * B + j) * nch + k));
                if (ahead(p.x, __float_as_int(p.y), v, i))
                    v = p.x, i = __float_as_int(p.y);
            }
            warp_best(v, i);
            if (lane == 0)
                s_g[j] = i == INT_MAX ? 0 : i;
        }
        for (int j = threadIdx.x; j < B - 1; j += kGThreads)
            s_y[j] = __ldg(a.y + (long long)r * (B - 1) + j);
        __syncthreads();
        if (threadIdx.x == 0) {
            int acc = 0;
            bool prefix = true;
            for (int j = 0; j < B - 1; ++j) {
                const int yj = s_y[j];
                const bool bad = yj < 0 || yj >= V;
                if (bad)
                    record_status(status, D3D_ERR_DEVICE_INPUT);  // treated as rejected
                const bool ok = !bad && yj == s_g[j];
                if (a.alpha)
                    a.alpha[(long long)r * (B - 1) + j] = ok ? 1.f : 0.f;
                if (a.p)
                    a.p[(long long)r * (B - 1) + j] = ok ? 1.f : 0.f;
                if (a.awl)  // the product of the acceptance indicators before j
                    a.awl[(long long)r * (B - 1) + j] = prefix ? 1.f : 0.f;
                prefix = prefix && ok;
                acc += prefix ? 1 : 0;
            }
            a.accept_len[r] = acc;
            a.num_tokens[r] = acc + 1;
            for (int j = 0; j < B; ++j)
                a.out_tokens[(long long)r * B + j] = j < acc ? s_y[j] : (j == acc ? s_g[acc] : -1);
            s_v[0] = __int_as_float(acc);
            bar[kBarInts * r] = 0;  // every item of the request has been counted: ready for the next call
        }
        __syncthreads();
        if (a.M > 0 && w == 0) {
            const int acc = __float_as_int(s_v[0]);
            match_request(r, acc, s_g[acc], s_y, B, a.M, a.heads, a.head_len, a.branch);
        } else if (a.branch && a.M == 0 && threadIdx.x == 0) {
            a.branch[r] = -1;
        }
        __syncthreads();
    }
    // launched as the programmatic dependent of an independent kernel:
    // finish only after it has finished
    sm100::pdl_wait();
}

// Launch of the greedy verification (see above); the workspace is the
// sampling launch's (counters at L.bar, one 8-byte pair per item in the
// 32-byte record slots).
template <typename T> int launch_greedy(const VArgs &a, int sm_limit, int flags, cudaStream_t stream)
{
    const VerifyLayout L = verify_layout(a.R, a.B, a.V, kGChunk);
    const long long n_items = (long long)a.R * a.B * L.nch;
    int dev = 0, nsm = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, greedy_kernel<T>, kGThreads, 0) != cudaSuccess ||
        per_sm < 1)
        return D3D_ERR_CUDA;
    long long cap = (long long)(sm_limit > 0 && sm_limit < nsm ? sm_limit : nsm) * per_sm;
    const unsigned grid = (unsigned)(n_items < cap ? n_items : cap);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    unsigned na = 0;
    if (flags & D3D_VERIFY_AFTER_INDEPENDENT) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = na ? attr : nullptr;
    cfg.numAttrs = na;
    return cuda_status(cudaLaunchKernelEx(&cfg, greedy_kernel<T>, a));
}

}  // namespace
}  // namespace d3d
