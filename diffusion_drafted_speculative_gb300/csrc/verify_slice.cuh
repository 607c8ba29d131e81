// Speculative-sampling verification over vocabulary slices: one CTA per
// (request, slice of the vocabulary), every row of the request's slice
// resident in its shared memory.
//
// The same rule as verify_body.cuh ([D3D] "Background: speculative
// decoding"; [DScout] "Background: speculative decoding", "Background:
// acceptance length tau", "Background: AWL and the acceptance rule"), laid
// out for a launch that holds one unit per CTA (a request whose rows split
// over the SMs the launch may use):
//   1. the CTA copies its slice of the B target rows and B-1 draft rows into
//      shared memory (one bulk copy per row, one mbarrier per row); each warp
//      takes a position j as soon as its two rows have landed: the slice's
//      (max, sum of exp2) of both rows and, in the slice holding y_j, both
//      scaled logits at y_j, written as the (j, slice) record;
//   2. after every slice of the request has signalled, each CTA combines the
//      records (select_request: p_j, q_j, alpha_j, the first rejection a and
//      the row the sample uses; slice 0 writes the per-request outputs);
//   3. each CTA sums its slice's masses of the sampled distribution (the
//      residual max(0, P - Q) at row a, or P at row B-1) from shared memory;
//   4. after every slice has signalled its sums, each CTA takes the same
//      decision (decide_request); the slice holding the crossing scans its
//      masses in vocabulary order and writes the token, then runs the fused
//      branch match.
// No row is read from global memory twice.  Two hand-offs between CTAs
// (release adds and bounded acquire polls on the per-request counters of
// the workspace); every CTA of the launch is resident (cooperative launch).
#pragma once

#include "verify_body.cuh"

namespace d3d {
namespace {

constexpr int kSliceThreads = 512;
constexpr int kSliceWarps = kSliceThreads / 32;
constexpr int kSliceGrain = 64;      // slice widths are multiples of 64 entries (16-byte aligned rows)
constexpr int kSliceMaxUnits = 256;  // units one launch may hold (bounds the workspace)

// Shared-memory carve-up of a slice CTA: the 2B-1 rows of W entries, then
// the request's records (staged for select_request when they are few, and
// reused for the slice sums of the decision), then one mbarrier per row.
template <typename T> struct SliceLayout {
    size_t rows, recs, bars, total;
    __host__ __device__ SliceLayout(int B, int W, int nS)
    {
        rows = 0;
        recs = (size_t)(2 * B - 1) * (size_t)W * sizeof(T);
        const size_t nrec = (size_t)B * (size_t)nS;
        size_t rec_bytes = nrec <= (size_t)kStagedRecords ? nrec * sizeof(Rec) : 0;
        if (rec_bytes < (size_t)nS * sizeof(float2))
            rec_bytes = (size_t)nS * sizeof(float2);
        bars = align_up(recs + rec_bytes, 16);
        total = bars + (size_t)(2 * B - 1) * 8;
    }
};

// max(a, b, c) in one instruction; a NaN operand is ignored
__device__ __forceinline__ float slice_fmax3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Raw logits of one 16-byte vector of a row in shared memory, as floats;
// at() reads one entry.
template <typename T> struct SliceVec;
template <> struct SliceVec<uint16_t> {
    static constexpr int kN = 8;
    static __device__ __forceinline__ float at(const uint16_t *row, int i) { return bf16_bits_to_float(row[i]); }
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
template <> struct SliceVec<float> {
    static constexpr int kN = 4;
    static __device__ __forceinline__ float at(const float *row, int i) { return row[i]; }
    static __device__ __forceinline__ void get(const float *row, int vi, float (&x)[4])
    {
        const float4 u = reinterpret_cast<const float4 *>(row)[vi];
        x[0] = u.x, x[1] = u.y, x[2] = u.z, x[3] = u.w;
    }
};

// (max, sum of exp2) of the scaled row c * x over n entries in shared
// memory, by one warp: m = c * max(x) (-inf for an empty or all -inf row), z
// = sum of exp2(c * x - m); every lane returns the same pair.
template <typename T>
__device__ __forceinline__ void slice_row_stats(const T *row, int n, float c, float &m, float &z)
{
    constexpr int kN = SliceVec<T>::kN;
    const int lane = threadIdx.x & 31, nv = n / kN;
    float mr = -INFINITY;
    for (int vi = lane; vi < nv; vi += 32) {
        float x[kN];
        SliceVec<T>::get(row, vi, x);
#pragma unroll
        for (int e = 0; e < kN; e += 2)
            mr = slice_fmax3(mr, x[e], x[e + 1]);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1)
        mr = fmaxf(mr, __shfl_xor_sync(kFull, mr, o));
    m = (mr == -INFINITY) ? -INFINITY : mr * c;
    const float nm = (mr == -INFINITY) ? 0.f : -m;
    float za = 0.f, zb = 0.f;
    for (int vi = lane; vi < nv; vi += 32) {
        float x[kN];
        SliceVec<T>::get(row, vi, x);
#pragma unroll
        for (int e = 0; e < kN; e += 2) {
            float a0, a1;
            sm100::ffma2(a0, a1, x[e], x[e + 1], c, c, nm, nm);
            sm100::fadd2(za, zb, za, zb, fast_exp2(a0), fast_exp2(a1));
        }
    }
    z = za + zb;
#pragma unroll
    for (int o = 16; o; o >>= 1)
        z += __shfl_xor_sync(kFull, z, o);
}


// Mass of entry i of the slice in the sampled distribution: P(v) =
// exp2(c x_t - mP) / ZP, and max(0, P - Q) for the residual (kind 0).
__device__ __forceinline__ float slice_mass(int kind, float xt, float xd, float c, const Sel &sel, float &P)
{
    P = fast_exp2(xt * c - sel.mP) * sel.rZP;
    return kind == 0 ? fmaxf(P - fast_exp2(xd * c - sel.mQ) * sel.rZQ, 0.f) : P;
}

template <typename T>
__device__ __forceinline__ void verify_slice_body(const VArgs &a, int W, int nS)
{
    const int r = (int)blockIdx.x / nS, s = (int)blockIdx.x % nS;
    const int B = a.B, V = a.V, M = a.M;
    const int nrows = 2 * B - 1;
    const int v0 = s * W, v1 = min(V, v0 + W), n = v1 - v0;  // n >= 1: nS = ceil(V / W)
    const float c = a.c;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kN = SliceVec<T>::kN;
    const T *__restrict__ target = static_cast<const T *>(a.target);
    const T *__restrict__ draft = static_cast<const T *>(a.draft);
    unsigned char *__restrict__ ws = a.ws;
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    const VerifyLayout L = verify_layout(a.R, B, V, W);  // chunks = slices
    Rec *rec = reinterpret_cast<Rec *>(ws + L.rec);
    float2 *part2 = reinterpret_cast<float2 *>(ws + L.part2);
    int *bar = reinterpret_cast<int *>(ws + L.bar) + kBarInts * r;

    extern __shared__ __align__(128) unsigned char s_slice[];
    const SliceLayout<T> SL(B, W, nS);
    T *rows = reinterpret_cast<T *>(s_slice);
    Rec *s_rec = reinterpret_cast<Rec *>(s_slice + SL.recs);
    const uint32_t rows_s = sm100::smem_u32(s_slice), bars_s = sm100::smem_u32(s_slice + SL.bars);
    auto row_of = [&](int i) { return rows + (size_t)i * W; };
    __shared__ float red[2 * kSliceWarps];
    __shared__ int32_t s_y[kMaxB];
    __shared__ float s_u[kMaxB], s_us;
    __shared__ volatile int s_abort;
    __shared__ Decision s_dec;
    __shared__ int s_cand, s_lastpos;

    // a kernel launched after this one as an independent programmatic
    // dependent (the round's drafting attention) may start at once
    if (threadIdx.x == 0)
        sm100::pdl_trigger();
    // ---- 1. the slice's rows into shared memory (rows are 16-byte aligned and
    // the slice is a multiple of 16 bytes: checked by the host): thread i
    // initialises row i's mbarrier and issues its bulk copy, before anything
    // else, so that the copies are in flight while the request's inputs load
    const uint32_t row_bytes = (uint32_t)n * (uint32_t)sizeof(T);
    for (int i = threadIdx.x; i < nrows; i += kSliceThreads) {
        const uint32_t b = bars_s + 8u * (uint32_t)i;
        sm100::mbar_init(b, 1);
        sm100::fence_barrier_init();
        if (a.fault == 2 && blockIdx.x == 0 && i == 0)
            continue;  // injected fault: this row's copy never arrives
        const T *src = (i < B) ? target + ((size_t)r * B + i) * V + v0
                               : draft + ((size_t)r * (B - 1) + (i - B)) * V + v0;
        sm100::mbar_arrive_expect_tx(b, row_bytes);
        sm100::bulk_load(rows_s + (uint32_t)i * (uint32_t)W * (uint32_t)sizeof(T), src, row_bytes, b);
    }
    if (threadIdx.x == 0)
        s_abort = 0;
    // the branch heads of the fused match go to L2 now (read once the token is known)
    if (a.branch != nullptr) {
        const int32_t *h = a.heads + (size_t)r * M * B;
        for (int o = (int)threadIdx.x * 32; o < M * B; o += kSliceThreads * 32)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(h + o));
        if (threadIdx.x == 0 && M > 0)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a.head_len + (size_t)r * M));
    }
    load_request_inputs<kSliceThreads>(r, B, a.y, a.u_acc, a.u_s, s_y, s_u, &s_us);
    __syncthreads();
    // bounded wait for row i (the whole warp); false when it or another wait ran out
    auto wait_row = [&](int i) -> bool {
        const uint32_t b = bars_s + 8u * (uint32_t)i;
        bool ok = sm100::mbar_try_wait(b, 0);
        if (!ok) {
            const uint64_t t0 = sm100::global_ns();
            while (!(ok = sm100::mbar_try_wait_sleep(b, 0))) {
                if (s_abort || sm100::global_ns() - t0 > kBarrierTimeoutNs) {
                    record_status(status, D3D_ERR_DEVICE_TIMEOUT);
                    s_abort = 1;
                    break;
                }
            }
        }
        return __all_sync(kFull, ok);
    };
    // warp w: positions j = w, w + 16, ...: both rows' statistics and, in the
    // slice holding y_j, both scaled logits at y_j
    for (int j = warp; j < B; j += kSliceWarps) {
        if (!wait_row(j))
            break;
        float mP, zP, mQ = -INFINITY, zQ = 0.f, xP = 0.f, xQ = 0.f;
        slice_row_stats<T>(row_of(j), n, c, mP, zP);
        const int yv = (j < B - 1) ? s_y[j] : -1;
        const bool has_y = yv >= v0 && yv < v1;
        if (has_y)
            xP = SliceVec<T>::at(row_of(j), yv - v0) * c;
        if (j < B - 1) {
            if (!wait_row(B + j))
                break;
            slice_row_stats<T>(row_of(B + j), n, c, mQ, zQ);
            if (has_y)
                xQ = SliceVec<T>::at(row_of(B + j), yv - v0) * c;
        }
        if (lane == 0 && dbg_ok(r < a.R && s < nS && ((size_t)r * B + j) * nS + s < (size_t)a.R * B * nS, status)) {
            float4 *dst = reinterpret_cast<float4 *>(rec + ((size_t)r * B + j) * nS + s);
            dst[0] = make_float4(mP, zP, mQ, zQ);
            dst[1] = make_float4(xP, xQ, 0.f, 0.f);
            __threadfence();  // the record before thread 0's signal, for the other CTAs
        }
    }
    __syncthreads();
    if (s_abort) {
        // copies may still be in flight: wait them out (bounded) before leaving;
        // the request's other CTAs give up their waits for this one
        if (threadIdx.x == 0)
            for (int i = 0; i < nrows; ++i) {
                const uint64_t t0 = sm100::global_ns();
                while (!sm100::mbar_try_wait_sleep(bars_s + 8u * (uint32_t)i, 0))
                    if (sm100::global_ns() - t0 > kBarrierTimeoutNs)
                        break;
            }
        __syncthreads();
        return;
    }
    if (threadIdx.x == 0)
        signal_count(bar + 0);

    // ---- 2. the request's selection from every slice's records
    if (!wait_count(bar + 0, nS, status))
        return;
    if (threadIdx.x == 0 && atomicAdd(bar + 1, 1) == nS - 1) {  // the last waiter past resets the phase-1 pair
        bar[0] = 0;
        bar[1] = 0;
    }
    Sel sel;
    select_request<kSliceThreads>(r, B, V, nS, W, rec, s_y, s_u, s == 0, a.accept_len, a.out_tokens,
                                  a.num_tokens, a.alpha, a.p, a.q, a.awl, status, sel, s_rec);

    // ---- 3. this slice's masses of the sampled distribution (kind from the
    // selection; the decision may fall back to P when the residual has no mass)
    const T *rowt = row_of(sel.row);
    const T *rowd = row_of(sel.mode == 0 ? B + sel.row : sel.row);  // the draft row is read for kind 0 only
    {
        float sk = 0.f, sp = 0.f;
        for (int vi = threadIdx.x; vi < n / kN; vi += kSliceThreads) {
            float xt[kN], xd[kN];
            SliceVec<T>::get(rowt, vi, xt);
            SliceVec<T>::get(rowd, vi, xd);
#pragma unroll
            for (int e = 0; e < kN; ++e) {
                float P;
                sk += slice_mass(sel.mode, xt[e], xd[e], c, sel, P);
                sp += P;
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            sk += __shfl_xor_sync(kFull, sk, o);
            sp += __shfl_xor_sync(kFull, sp, o);
        }
        if (lane == 0) {
            red[warp] = sk;
            red[kSliceWarps + warp] = sp;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            float tk = 0.f, tp = 0.f;
            for (int w2 = 0; w2 < kSliceWarps; ++w2) {
                tk += red[w2];
                tp += red[kSliceWarps + w2];
            }
            part2[(size_t)r * nS + s] = make_float2(tk, tp);
            signal_count(bar + 2);
        }
    }

    // ---- 4. the decision, then the ordered scan in the slice that holds it
    if (!wait_count(bar + 2, nS, status))
        return;
    if (threadIdx.x == 0 && atomicAdd(bar + 3, 1) == nS - 1) {
        bar[2] = 0;
        bar[3] = 0;
    }
    decide_request<kSliceThreads>(part2 + (size_t)r * nS, nS, sel.mode, s_us, reinterpret_cast<float2 *>(s_rec),
                                  &s_dec);
    int32_t *out_tok = a.out_tokens + (size_t)r * B + sel.a;
    if (s_dec.owner == s) {
        // thread t: the contiguous run [t * per, t * per + per) of the slice
        const int kind = s_dec.kind;
        const int per = (n + kSliceThreads - 1) / kSliceThreads;
        const int i0 = min(n, (int)threadIdx.x * per), i1 = min(n, i0 + per);
        float run = 0.f;
        int lastpos = -1;
        for (int i = i0; i < i1; ++i) {
            float P;
            const float wv = slice_mass(kind, SliceVec<T>::at(rowt, i), SliceVec<T>::at(rowd, i), c, sel, P);
            run += wv;
            if (wv > 0.f)
                lastpos = v0 + i;
        }
        // exclusive scan of the runs over the CTA (thread order = vocabulary order)
        float incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(kFull, incl, o);
            if (lane >= o)
                incl += t;
        }
        if (threadIdx.x == 0) {
            s_cand = 0x7fffffff;
            s_lastpos = -1;
        }
        if (lane == 31)
            red[warp] = incl;
        __syncthreads();
        float before = 0.f;
        for (int w2 = 0; w2 < warp; ++w2)
            before += red[w2];
        const float excl = before + incl - run;
        const float target = s_dec.rem;
        const bool takelast = s_dec.takelast != 0;
        if (!takelast && i0 < i1 && excl + run > target)
            atomicMin(&s_cand, (int)threadIdx.x);
        atomicMax(&s_lastpos, lastpos);
        __syncthreads();
        const int cand = s_cand;
        if (!takelast && cand == (int)threadIdx.x) {
            int tok = -1, last = -1;
            float cum = excl;
            for (int i = i0; i < i1; ++i) {
                float P;
                const float wv =
                    slice_mass(kind, SliceVec<T>::at(rowt, i), SliceVec<T>::at(rowd, i), c, sel, P);
                cum += wv;
                if (wv > 0.f)
                    last = v0 + i;
                if (cum > target) {
                    tok = v0 + i;
                    break;
                }
            }
            // rounding between the two summation orders: the run's last position with mass
            if (tok < 0)
                tok = last >= 0 ? last : s_lastpos;
            if (dbg_ok(tok >= v0 && tok < v1, status))
                *out_tok = tok;
        }
        if ((takelast || cand == 0x7fffffff) && threadIdx.x == 0 && dbg_ok(s_lastpos >= v0 && s_lastpos < v1, status))
            *out_tok = s_lastpos;
        __syncthreads();
        if (a.branch != nullptr && threadIdx.x < 32) {
            const int tok = *reinterpret_cast<volatile const int32_t *>(out_tok);
            match_request(r, sel.a, tok, s_y, B, M, a.heads, a.head_len, a.branch);
        }
    } else if (s_dec.owner < 0 && s == 0) {
        // no mass anywhere: cannot happen for a finite softmax row
        if (threadIdx.x == 0) {
            record_status(status, D3D_ERR_DEVICE_INPUT);
            *out_tok = 0;
        }
        __syncthreads();
        if (a.branch != nullptr && threadIdx.x < 32)
            match_request(r, sel.a, 0, s_y, B, M, a.heads, a.head_len, a.branch);
    }
}

template <typename T>
__global__ void __launch_bounds__(kSliceThreads, 1) verify_slice_kernel(const VArgs a, int W, int nS)
{
    verify_slice_body<T>(a, W, nS);
    // launched as the programmatic dependent of an independent kernel: finish
    // only after it has finished
    sm100::pdl_wait();
}

}  // namespace
}  // namespace d3d
