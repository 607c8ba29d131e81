// Branch construction for the asynchronous packed pass.
//
// [D3D] "Background: asynchronous drafting and cache hits" and "Method
// steps" (step 4): one packed pass drafts, for every rejection position, a
// block from each of several alternative anchors, plus the all-accept block;
// a branch hypothesises the accepted drafts before its position.  The pages
// do not say how the anchors are chosen; here they are the F most likely
// tokens of the drafter's own distribution Q at that position (largest
// logit first, ties to the lowest index), the drafted token excluded: the
// target's correction there is never the drafted token.
//
// One pass over draft rows 0..C-2: a work item is 8192 entries of one row;
// its CTA keeps each thread's F best (value, index) pairs, merges them into
// the chunk's F best and stores them.  The CTA that counts a request's last
// item merges the chunks' lists of every row and writes the request's
// anchors, branch heads and lengths, and the packed pass's segment rows.
// No CTA waits for another.
#include <limits.h>
#include <math.h>

#include "d3d_common.cuh"
#include "sm100_ptx.cuh"

namespace d3d {
namespace {

constexpr int kBThreads = 256;
constexpr int kBChunk = 8192;              // entries per item
constexpr int kBPer = kBChunk / kBThreads;  // 32 entries per thread and item
constexpr int kMaxF = 8;

struct BArgs {
    const void *draft;
    const int32_t *y, *bonus;
    int R, B, V, C, F;
    int32_t *anchors, *heads, *head_len;
    d3d_segment_t *segs;
    int32_t *cu_q, *cu_seg;
    unsigned char *ws;
};

struct BLayout {
    size_t cnt, rec, total;
    int nch;
};

__host__ __device__ inline BLayout branch_layout(int R, int V, int C, int F)
{
    BLayout L;
    L.nch = (V + kBChunk - 1) / kBChunk;
    size_t o = sizeof(WsHeader);
    L.cnt = o;
    o = align_up(o + sizeof(int) * (size_t)R, kWsAlign);
    L.rec = o;  // F (value, index) pairs per (request, row, chunk)
    const long long rows = (long long)R * (C > 1 ? C - 1 : 0);
    o = align_up(o + sizeof(float2) * (size_t)F * (size_t)rows * (size_t)L.nch, kWsAlign);
    L.total = o;
    return L;
}

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

// Insert (x, v) into the sorted list (bv, bi) of length kF (best first):
// the carried pair swaps into every slot it is ahead of, so the list stays
// sorted and its last pair drops out.
template <int kF> __device__ __forceinline__ void keep_best(float (&bv)[kF], int (&bi)[kF], float x, int v)
{
    if (!ahead(x, v, bv[kF - 1], bi[kF - 1]))  // behind the list's last pair
        return;
#pragma unroll
    for (int t = 0; t < kF; ++t) {
        if (ahead(x, v, bv[t], bi[t])) {
            const float tx = bv[t];
            const int tv = bi[t];
            bv[t] = x, bi[t] = v;
            x = tx, v = tv;
        }
    }
}

// kF rounds of a block-wide best over each thread's sorted list: the kF best
// pairs of the block, to the shared out arrays.  Indices are distinct, so
// exactly one thread's list moves on per round.
template <int kF>
__device__ __forceinline__ void block_top(const float (&bv)[kF], const int (&bi)[kF], float *s_v, int *s_i,
                                          float *out_v, int *out_i)
{
    int head = 0;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int f = 0; f < kF; ++f) {
        float hv = -INFINITY;
        int hi = INT_MAX;
#pragma unroll
        for (int t = 0; t < kF; ++t)
            if (t == head)
                hv = bv[t], hi = bi[t];
        float v = hv;
        int i = hi;
        warp_best(v, i);
        if (lane == 0)
            s_v[w] = v, s_i[w] = i;
        __syncthreads();
        if (w == 0) {
            v = lane < kBThreads / 32 ? s_v[lane] : -INFINITY;
            i = lane < kBThreads / 32 ? s_i[lane] : INT_MAX;
            warp_best(v, i);
            if (lane == 0)
                s_v[kBThreads / 32] = v, s_i[kBThreads / 32] = i;
        }
        __syncthreads();
        const int win = s_i[kBThreads / 32];
        if (threadIdx.x == 0)
            out_v[f] = s_v[kBThreads / 32], out_i[f] = win;
        if (win != INT_MAX && hi == win)
            ++head;
        __syncthreads();
    }
}

// Heads, lengths and segment rows of request r once its anchors are known.
__device__ void write_request(const BArgs &a, int r, const int32_t *s_y, const int32_t *s_anc)
{
    const int B = a.B, C = a.C, F = a.F, M = (C - 1) * F + 2;
    int32_t *h = a.heads + (long long)r * M * B;
    for (int e = threadIdx.x; e < M * B; e += kBThreads) {
        const int k = e / B, i = e % B;
        int32_t t = -1;
        if (k >= 1 && k < M - 1) {
            const int p = (k - 1) / F;
            t = i < p ? s_y[i] : (i == p ? s_anc[k - 1] : -1);
        } else if (k == M - 1 && a.bonus) {
            t = i < B - 1 ? s_y[i] : __ldg(a.bonus + r);
        }
        h[e] = t;
    }
    for (int k = threadIdx.x; k < M; k += kBThreads) {
        const int len = k == 0 ? 0 : (k < M - 1 ? (k - 1) / F + 1 : (a.bonus ? B : 0));
        a.head_len[(long long)r * M + k] = len;
        if (a.segs) {
            d3d_segment_t sg;
            sg.q_start = k * B;
            sg.len = B;
            sg.mode = k == 0 ? D3D_SEG_CAUSAL : D3D_SEG_BIDIR;
            sg.parent = k == 0 ? -1 : 0;
            sg.parent_len = k == 0 ? 0 : (k < M - 1 ? (k - 1) / F + 1 : B);
            a.segs[(long long)r * M + k] = sg;
        }
    }
    if (a.cu_q && threadIdx.x == 0) {
        a.cu_q[r] = r * M * B;
        a.cu_seg[r] = r * M;
        if (r == a.R - 1) {
            a.cu_q[a.R] = a.R * M * B;
            a.cu_seg[a.R] = a.R * M;
        }
    }
}

template <typename T, int kF>
__global__ void __launch_bounds__(kBThreads, 2) branch_build_kernel(const BArgs a)
{
    __shared__ float s_v[kBThreads / 32 + 1];
    __shared__ int s_i[kBThreads / 32 + 1];
    __shared__ float s_ov[kMaxF];
    __shared__ int s_oi[kMaxF];
    __shared__ int32_t s_y[256];
    __shared__ int32_t s_anc[256 * kMaxF];
    __shared__ int s_last;
    const int R = a.R, B = a.B, V = a.V, C = a.C, F = a.F;
    const int P = C - 1;  // rejection positions with anchors
    const BLayout L = branch_layout(R, V, C, F);
    const int nch = L.nch;
    int *cnt = reinterpret_cast<int *>(a.ws + L.cnt);
    float2 *rec = reinterpret_cast<float2 *>(a.ws + L.rec);
    int32_t *status = reinterpret_cast<int32_t *>(a.ws);
    const T *dr = static_cast<const T *>(a.draft);
    const bool vec = V % 8 == 0 && (reinterpret_cast<uintptr_t>(dr) & 15) == 0;
    const long long n_items = F > 0 ? (long long)R * P * nch : 0;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (n_items == 0) {  // no anchors to choose (C == 1 or F == 0): heads and rows only
        for (int r = blockIdx.x; r < R; r += gridDim.x) {
            for (int j = threadIdx.x; j < B - 1; j += kBThreads)
                s_y[j] = __ldg(a.y + (long long)r * (B - 1) + j);
            __syncthreads();
            write_request(a, r, s_y, s_anc);
            __syncthreads();
        }
        return;
    }
    // the outputs the request's last CTA writes, touched now (their address
    // translations are then at hand when the last CTA stores to them)
    if (threadIdx.x < 6) {
        const int o = (int)threadIdx.x;
        const void *ptr = o == 0 ? (const void *)a.anchors : o == 1 ? (const void *)a.heads
                        : o == 2 ? (const void *)a.head_len : o == 3 ? (const void *)a.segs
                        : o == 4 ? (const void *)a.cu_q : (const void *)a.cu_seg;
        if (ptr != nullptr)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
    }
    for (long long it = blockIdx.x; it < n_items; it += gridDim.x) {
        const int c = (int)(it % nch);
        const long long rp = it / nch;  // request * P + position
        const int r = (int)(rp / P), p = (int)(rp % P);
        int yv = __ldg(a.y + (long long)r * (B - 1) + p);
        if (yv < 0 || yv >= V) {
            if (threadIdx.x == 0 && c == 0)
                record_status(status, D3D_ERR_DEVICE_INPUT);
            yv = -1;  // nothing to exclude
        }
        const T *row = dr + ((long long)r * (B - 1) + p) * V;
        const int v0 = c * kBChunk, v1 = min(V, v0 + kBChunk);
        float bv[kF];
        int bi[kF];
#pragma unroll
        for (int t = 0; t < kF; ++t)
            bv[t] = -INFINITY, bi[t] = INT_MAX;
        if (vec) {  // 16-byte loads of 8 entries (V % 8 == 0, aligned rows), all in flight before the compares
            float x[kBPer / 8][8];
#pragma unroll
            for (int g = 0; g < kBPer / 8; ++g) {
                const int v = v0 + g * (8 * kBThreads) + 8 * (int)threadIdx.x;
                if (v < v1) {
                    load_logits8(row + v, x[g]);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        x[g][e] = -INFINITY;
                }
            }
#pragma unroll
            for (int g = 0; g < kBPer / 8; ++g) {
                const int v = v0 + g * (8 * kBThreads) + 8 * (int)threadIdx.x;
                if (v < v1) {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (v + e != yv)
                            keep_best<kF>(bv, bi, x[g][e], v + e);
                }
            }
        } else {
#pragma unroll 4
            for (int q = 0; q < kBPer; ++q) {
                const int v = v0 + q * kBThreads + (int)threadIdx.x;
                if (v < v1 && v != yv)
                    keep_best<kF>(bv, bi, load_logit(row, v), v);
            }
        }
        block_top<kF>(bv, bi, s_v, s_i, s_ov, s_oi);
        if (threadIdx.x == 0) {
            float2 *dst = rec + (rp * nch + c) * F;
            for (int f = 0; f < F; ++f)
                dst[f] = make_float2(s_ov[f], __int_as_float(s_oi[f]));
            __threadfence();  // the list is visible before the count says so
            s_last = atomicAdd(cnt + r, 1) == P * nch - 1;
        }
        __syncthreads();
        if (!s_last)
            continue;
        // ---- the request's last item: merge every row's chunk lists
        __threadfence();
        for (int j = threadIdx.x; j < B - 1; j += kBThreads)  // in flight while the lists merge
            s_y[j] = __ldg(a.y + (long long)r * (B - 1) + j);
        constexpr int kCache = 8;  // list entries each lane holds (rows of up to 256 entries)
        constexpr int kW = kBThreads / 32;
        const int n = nch * F;
        const bool cached = n <= 32 * kCache;
        // warp w merges rows w, w + kW, w + 2 kW, ... in that order, the lists
        // of two rows loaded together (one L2 round trip for both)
        for (int pp0 = w; pp0 < P; pp0 += 2 * kW) {
            float cvv[2][kCache];
            int civ[2][kCache];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int pp = pp0 + h * kW;
                const float2 *lst = rec + ((long long)r * P + pp) * nch * F;
#pragma unroll
                for (int t = 0; t < kCache; ++t) {  // one pass over the row's lists
                    const int k = lane + 32 * t;
                    const float2 e = (cached && pp < P && k < n) ? __ldcg(lst + k)
                                                                 : make_float2(-INFINITY, __int_as_float(INT_MAX));
                    cvv[h][t] = e.x, civ[h][t] = __float_as_int(e.y);
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int pp = pp0 + h * kW;
                if (pp >= P)
                    break;
                const float2 *lst = rec + ((long long)r * P + pp) * nch * F;
                float(&cv)[kCache] = cvv[h];
                int(&ci)[kCache] = civ[h];
                for (int f = 0; f < F; ++f) {
                    float v = -INFINITY;
                    int i = INT_MAX;
                    if (cached) {
#pragma unroll
                        for (int t = 0; t < kCache; ++t)
                            if (ahead(cv[t], ci[t], v, i))
                                v = cv[t], i = ci[t];
                    } else {  // long rows: read the lists again, skipping the pairs already taken
                        for (int k = lane; k < n; k += 32) {
                            const float2 e = __ldcg(lst + k);
                            const int ei = __float_as_int(e.y);
                            bool used = false;
                            for (int t = 0; t < f; ++t)
                                used = used || s_anc[pp * F + t] == ei;
                            if (!used && ahead(e.x, ei, v, i))
                                v = e.x, i = ei;
                        }
                    }
                    warp_best(v, i);
                    i = __shfl_sync(0xffffffffu, i, 0);
                    if (lane == 0)
                        s_anc[pp * F + f] = i;
                    if (cached) {  // the winner leaves its lane's cache (indices are distinct)
#pragma unroll
                        for (int t = 0; t < kCache; ++t)
                            if (ci[t] == i)
                                cv[t] = -INFINITY, ci[t] = INT_MAX;
                    }
                    __syncwarp();
                }
            }
        }
        __syncthreads();
        for (int e = threadIdx.x; e < P * F; e += kBThreads)
            a.anchors[(long long)r * P * F + e] = s_anc[e];
        write_request(a, r, s_y, s_anc);
        if (threadIdx.x == 0)
            cnt[r] = 0;  // every item of the request has been counted: ready for the next call
        __syncthreads();
    }
}

template <typename T, int kF> int launch_branches_f(const BArgs &a, cudaStream_t stream)
{
    const BLayout L = branch_layout(a.R, a.V, a.C, a.F);
    const long long n_items = a.F > 0 ? (long long)a.R * (a.C - 1) * L.nch : 0;
    int dev = 0, nsm = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, branch_build_kernel<T, kF>, kBThreads, 0) !=
            cudaSuccess ||
        per_sm < 1)
        return D3D_ERR_CUDA;
    const long long want = n_items > 0 ? n_items : a.R;
    const long long cap = (long long)nsm * per_sm;
    const unsigned grid = (unsigned)(want < cap ? want : cap);
    branch_build_kernel<T, kF><<<grid, kBThreads, 0, stream>>>(a);
    return cuda_status(cudaGetLastError());
}

// the list length is a compile-time constant of the kernel (registers only)
template <typename T> int launch_branches(const BArgs &a, cudaStream_t stream)
{
    switch (a.F) {
    case 0:  // no anchors: the kernel writes heads and rows only
    case 1: return launch_branches_f<T, 1>(a, stream);
    case 2: return launch_branches_f<T, 2>(a, stream);
    case 3: return launch_branches_f<T, 3>(a, stream);
    case 4: return launch_branches_f<T, 4>(a, stream);
    case 5: return launch_branches_f<T, 5>(a, stream);
    case 6: return launch_branches_f<T, 6>(a, stream);
    case 7: return launch_branches_f<T, 7>(a, stream);
    default: return launch_branches_f<T, 8>(a, stream);
    }
}

}  // namespace
}  // namespace d3d

extern "C" {

size_t d3d_build_branches_workspace_size(int R, int B, int V, int C, int F)
{
    if (R < 0 || B < 2 || V < 1 || C < 1 || C > B || F < 0 || F > d3d::kMaxF)
        return 0;
    return d3d::branch_layout(R, V, C, F).total;
}

int d3d_build_branches(const void *draft_logits, int logits_dtype, const int32_t *draft_tokens,
                       const int32_t *bonus_guess, int R, int B, int V, int C, int F, int32_t *anchors,
                       int32_t *heads, int32_t *head_len, d3d_segment_t *segs, int32_t *cu_q, int32_t *cu_seg,
                       void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (R < 0 || B < 2 || V < 1 || C < 1 || C > B || F < 0)
        return D3D_ERR_INVALID_ARG;
    if (logits_dtype != D3D_DTYPE_F32 && logits_dtype != D3D_DTYPE_BF16)
        return D3D_ERR_INVALID_ARG;
    const bool any_anchor = C > 1 && F > 0;
    if (any_anchor && F > V - 1)  // fewer tokens than anchors besides the drafted one
        return D3D_ERR_INVALID_ARG;
    if (F > d3d::kMaxF || B > 256 || (long long)(C - 1) * F > 256)
        return D3D_ERR_UNSUPPORTED;
    if ((long long)R * ((long long)(C - 1) * F + 2) * B > 0x7fffffffLL)
        return D3D_ERR_UNSUPPORTED;
    if ((cu_q == nullptr) != (cu_seg == nullptr))
        return D3D_ERR_INVALID_ARG;
    if (R == 0)
        return D3D_OK;
    if (!draft_tokens || !heads || !head_len || (any_anchor && (!draft_logits || !anchors)))
        return D3D_ERR_INVALID_ARG;
    const d3d::BLayout L = d3d::branch_layout(R, V, C, F);
    if (!d3d::ws_ok(ws, ws_bytes, L.total))
        return D3D_ERR_WORKSPACE;
    d3d::BArgs a;
    a.draft = draft_logits;
    a.y = draft_tokens;
    a.bonus = bonus_guess;
    a.R = R, a.B = B, a.V = V, a.C = C, a.F = F;
    a.anchors = anchors, a.heads = heads, a.head_len = head_len;
    a.segs = segs, a.cu_q = cu_q, a.cu_seg = cu_seg;
    a.ws = static_cast<unsigned char *>(ws);
    return logits_dtype == D3D_DTYPE_BF16 ? d3d::launch_branches<uint16_t>(a, stream)
                                          : d3d::launch_branches<float>(a, stream);
}

}  // extern "C"
