// Device code of the speculative-sampling verification (and the host helpers
// a launch needs), shared by the verification's own launch and the fused
// round launch.
#pragma once
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
//   A. one work item per (request, position j, 8192-entry chunk): the chunk of
//      target row j and, for j < B-1, of draft row j, with 16-byte vector
//      loads; the chunk's softmax statistics of both rows (max and sum of
//      exp2, log2 domain) and the two logits at the draft token y_j when it
//      lies in the chunk.  One record per item.
//   B. every CTA that goes on combines its request's records in shared memory
//      (each does it redundantly, which costs L2 reads instead of a hand-off),
//      forms p_j, q_j, alpha_j, runs the first-rejection scan and picks the
//      row pair the sample uses.  One CTA writes the per-request outputs.
//   C. the items of that row pair compute their chunk's residual max(0, P - Q)
//      (or P_B) mass.  When every item has its own CTA, phase A's
//      exponentials are still in registers and a per-thread scale turns them
//      into probabilities: no reload and no exponential.  Otherwise the
//      chunk is reloaded.
//   D. the chunk holding the crossing C(v) > u*S scans its masses in
//      vocabulary order and writes the sampled token.
#include <math.h>

#include "d3d_common.cuh"
#include "sm100_ptx.cuh"

namespace d3d {
namespace {

constexpr int kVPer = 32;  // logits per thread and row of an item
// Thread count NT of a CTA: 256 for a launch over the whole device (two CTAs
// per SM), 512 when the launch is limited to some SMs (one CTA fills an SM).
// A chunk is NT * 32 vocabulary entries.
template <int NT> struct VCfg {
    static constexpr int kWarps = NT / 32;
    static constexpr int kChunk = NT * kVPer;
    static constexpr int kGroup = NT * 8;  // positions covered by one 8-wide slot group
};
constexpr int kNTDevice = 256;
constexpr int kNTLimited = 512;
constexpr int kVChunkMin = kNTDevice * kVPer;  // the workspace is sized for the smaller chunk
constexpr int kMaxB = 256;
constexpr int kMaxChunks = 1024;  // vocabulary up to 8M entries (in the smaller chunks)
constexpr uint64_t kBarrierTimeoutNs = 250ull * 1000ull * 1000ull;
constexpr int kStagedRecords = 1024;  // item records staged in shared memory (32 KB)
constexpr unsigned kFull = 0xffffffffu;

// Statistics of one (request, position, chunk) item.  Target row: mP, zP and
// the scaled logit at the draft token xP; draft row likewise.  An absent row
// (the bonus row has no draft row) has m = -inf, z = 0.
struct Rec {
    float mP, zP, mQ, zQ;
    float xP, xQ, pad0, pad1;
};

// What the sample of one request uses.
struct Sel {
    int32_t a;     // accepted drafts
    int32_t mode;  // 0: residual at target/draft row a; 1: bonus from target row B-1
    int32_t row;   // position whose rows the sample uses
    float mP, rZP, mQ, rZQ;  // log2-domain row max and 1 / normaliser of that target / draft row
};

struct VerifyLayout {
    size_t bar, rec, part2, total;
    int nch;
};

// Per-request counters: phase-A items done, waiters that passed the phase-A
// wait, phase-C items done, phase-D items done.
constexpr int kBarInts = 4;

__host__ __device__ inline VerifyLayout verify_layout(int R, int B, int V, int chunk)
{
    VerifyLayout L;
    L.nch = (V + chunk - 1) / chunk;
    size_t o = sizeof(WsHeader);
    L.bar = o;
    o = align_up(o + kBarInts * sizeof(int) * (size_t)R, kWsAlign);
    L.rec = o;  // per (request, position, chunk)
    o = align_up(o + sizeof(Rec) * (size_t)R * (size_t)B * (size_t)L.nch, kWsAlign);
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

// Vocabulary position of slot i (0..kVPer) of this thread in chunk v0: slot
// 8g+e holds v0 + g*(8 NT) + 8*tid + e, so each 8-slot group is one
// coalesced 16-byte load per thread.
template <int NT>
__device__ __forceinline__ int slot_pos(int v0, int i)
{
    return v0 + (i >> 3) * VCfg<NT>::kGroup + (int)threadIdx.x * 8 + (i & 7);
}

// Scaled logits x*c of one chunk [v0, v1) in slot order; positions past v1
// read as -inf.
template <typename T, int NT>
__device__ inline void load_chunk(const T *row, int v0, int v1, float c, float (&x)[kVPer])
{
    if (v1 - v0 == VCfg<NT>::kChunk && aligned16(row + v0)) {
#pragma unroll
        for (int g = 0; g < kVPer / 8; ++g) {
            float t[8];
            Logit<T>::load8(row + slot_pos<NT>(v0, 8 * g), t);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                x[8 * g + e] = t[e] * c;
        }
    } else {
#pragma unroll
        for (int i = 0; i < kVPer; ++i) {
            const int v = slot_pos<NT>(v0, i);
            x[i] = v < v1 ? Logit<T>::at(row, v) * c : -INFINITY;
        }
    }
}

// One row chunk's 16-byte loads, issued ahead of use (phase A prefetches
// the next item while it reduces the current one).  bf16 rows only: an f32
// row chunk would need twice the registers, so f32 rows load at use.
template <typename T, int NT> struct RawChunk {
    __device__ void issue(const T *, int, int) {}
    __device__ void take(const T *row, int v0, int v1, float c, float (&x)[kVPer]) { load_chunk<T, NT>(row, v0, v1, c, x); }
};

// The 512-thread launch streams bf16 rows through its shared-memory ring; its
// fallback for rows off the 16-byte grid loads at use, keeping registers free.
template <> struct RawChunk<uint16_t, kNTLimited> {
    __device__ void issue(const uint16_t *, int, int) {}
    __device__ void take(const uint16_t *row, int v0, int v1, float c, float (&x)[kVPer])
    {
        load_chunk<uint16_t, kNTLimited>(row, v0, v1, c, x);
    }
};

template <int NT> struct RawChunk<uint16_t, NT> {
    uint4 u[kVPer / 8];
    bool ok;
    __device__ void issue(const uint16_t *row, int v0, int v1)
    {
        ok = v1 - v0 == VCfg<NT>::kChunk && aligned16(row + v0);
        if (ok) {
#pragma unroll
            for (int g = 0; g < kVPer / 8; ++g)
                u[g] = __ldg(reinterpret_cast<const uint4 *>(row + slot_pos<NT>(v0, 8 * g)));
        }
    }
    __device__ void take(const uint16_t *row, int v0, int v1, float c, float (&x)[kVPer])
    {
        if (!ok) {
            load_chunk<uint16_t, NT>(row, v0, v1, c, x);
            return;
        }
#pragma unroll
        for (int g = 0; g < kVPer / 8; ++g) {
            const uint32_t w[4] = {u[g].x, u[g].y, u[g].z, u[g].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[8 * g + 2 * e] = __uint_as_float(w[e] << 16) * c;
                x[8 * g + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u) * c;
            }
        }
    }
};

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

// Per-thread max and exponentials of one row chunk, in place: x[i] becomes
// exp2(x[i] - m) with m this thread's max (0 everywhere when m = -inf).
__device__ inline void thread_exp(float (&x)[kVPer], float &m, float &z)
{
    m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kVPer; ++i)
        m = fmaxf(m, x[i]);
    z = 0.f;
    const float mm = (m == -INFINITY) ? 0.f : m;
#pragma unroll
    for (int i = 0; i < kVPer; ++i) {
        x[i] = fast_exp2(x[i] - mm);
        z += x[i];
    }
}

// The same on raw (unscaled) logits with the scale c > 0 folded into the
// exponent: x[i] becomes exp2(c*x[i] - m) with m = c * max(raw) this thread's
// scaled max, by one fused multiply-add per pair of entries.
__device__ inline void thread_exp_scaled(float (&x)[kVPer], float c, float &m, float &z)
{
    float m4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
    for (int i = 4; i < kVPer; i += 4)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            m4[e] = fmaxf(m4[e], x[i + e]);
    const float mr = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
    m = (mr == -INFINITY) ? -INFINITY : mr * c;
    const float nm = (mr == -INFINITY) ? 0.f : -m;
    float za = 0.f, zb = 0.f;
#pragma unroll
    for (int i = 0; i < kVPer; i += 2) {
        float a0, a1;
        sm100::ffma2(a0, a1, x[i], x[i + 1], c, c, nm, nm);
        x[i] = fast_exp2(a0);
        x[i + 1] = fast_exp2(a1);
        sm100::fadd2(za, zb, za, zb, x[i], x[i + 1]);
    }
    z = za + zb;
}

// Block-wide merge of two (max, sum) pairs; the result is valid in thread 0.
// Warps reduce by shuffles; warp 0 then merges the per-warp pairs by a
// shuffle tree (log2 of the warp count steps instead of a serial loop).
template <int NT>
__device__ inline void block_ms2(float &m1, float &z1, float &m2, float &z2, float *red)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float a = __shfl_xor_sync(kFull, m1, o), b = __shfl_xor_sync(kFull, z1, o);
        const float c = __shfl_xor_sync(kFull, m2, o), d = __shfl_xor_sync(kFull, z2, o);
        ms_merge(m1, z1, a, b);
        ms_merge(m2, z2, c, d);
    }
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        red[4 * w + 0] = m1;
        red[4 * w + 1] = z1;
        red[4 * w + 2] = m2;
        red[4 * w + 3] = z2;
    }
    __syncthreads();
    if (w == 0) {
        constexpr int kW = VCfg<NT>::kWarps;
        m1 = lane < kW ? red[4 * lane + 0] : -INFINITY;
        z1 = lane < kW ? red[4 * lane + 1] : 0.f;
        m2 = lane < kW ? red[4 * lane + 2] : -INFINITY;
        z2 = lane < kW ? red[4 * lane + 3] : 0.f;
#pragma unroll
        for (int o = kW / 2; o; o >>= 1) {
            const float a = __shfl_xor_sync(kFull, m1, o), b = __shfl_xor_sync(kFull, z1, o);
            const float c = __shfl_xor_sync(kFull, m2, o), d = __shfl_xor_sync(kFull, z2, o);
            ms_merge(m1, z1, a, b);
            ms_merge(m2, z2, c, d);
        }
    }
}

// Block-wide sums of two values; the result is valid in thread 0.
template <int NT>
__device__ inline void block_sum2(float &a, float &b, float *red)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        a += __shfl_xor_sync(kFull, a, o);
        b += __shfl_xor_sync(kFull, b, o);
    }
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        red[2 * w] = a;
        red[2 * w + 1] = b;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        a = red[0];
        b = red[1];
        for (int i = 1; i < VCfg<NT>::kWarps; ++i) {
            a += red[2 * i];
            b += red[2 * i + 1];
        }
    }
}

// Block-wide exclusive scan of the four per-thread group sums g[0..3] in
// vocabulary order (group-major, then thread): returns each group's prefix.
template <int NT>
__device__ inline float4 block_group_scan(float4 g, float *red)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float4 inc = g;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float a = __shfl_up_sync(kFull, inc.x, o), b = __shfl_up_sync(kFull, inc.y, o);
        const float c = __shfl_up_sync(kFull, inc.z, o), d = __shfl_up_sync(kFull, inc.w, o);
        if (lane >= o)
            inc.x += a, inc.y += b, inc.z += c, inc.w += d;
    }
    if (lane == 31) {
        red[4 * w + 0] = inc.x;
        red[4 * w + 1] = inc.y;
        red[4 * w + 2] = inc.z;
        red[4 * w + 3] = inc.w;
    }
    __syncthreads();
    float tot[4] = {0.f, 0.f, 0.f, 0.f}, before[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = 0; i < VCfg<NT>::kWarps; ++i) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float t = red[4 * i + q];
            tot[q] += t;
            if (i < w)
                before[q] += t;
        }
    }
    float4 r;
    r.x = before[0] + inc.x - g.x;
    r.y = tot[0] + before[1] + inc.y - g.y;
    r.z = tot[0] + tot[1] + before[2] + inc.z - g.z;
    r.w = tot[0] + tot[1] + tot[2] + before[3] + inc.w - g.w;
    return r;
}

// fp32 pairs (hi + lo, |lo| <= ulp(hi)) for the sample's magnitude-S sums:
// error-free transformations (Knuth's TwoSum, Dekker's product with an FMA),
// about 2^-44 relative instead of fp32's 2^-24.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// (h, l) += (h2, l2)
__device__ __forceinline__ void df_add(float &h, float &l, float h2, float l2)
{
    float s, e;
    two_sum(h, h2, s, e);
    e = __fadd_rn(e, __fadd_rn(l, l2));
    h = __fadd_rn(s, e);
    l = __fsub_rn(e, __fsub_rn(h, s));
}

// (th, tl) = u * (h, l)
__device__ __forceinline__ void df_mul(float u, float h, float l, float &th, float &tl)
{
    const float p = __fmul_rn(u, h);
    const float e = __fadd_rn(__fmaf_rn(u, h, -p), __fmul_rn(u, l));
    th = __fadd_rn(p, e);
    tl = __fsub_rn(e, __fsub_rn(th, p));
}

// (ah, al) > (bh, bl)
__device__ __forceinline__ bool df_gt(float ah, float al, float bh, float bl)
{
    return __fadd_rn(__fsub_rn(ah, bh), __fsub_rn(al, bl)) > 0.f;
}

__device__ __forceinline__ int load_acquire(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Wait (thread 0 spins with acquire loads, bounded) until *cnt reaches
// `target`; the barrier after it passes the producers' writes on to the whole
// CTA.  Returns false if the wait ran out (the status word is then set).
__device__ bool wait_count(const int *cnt, int target, int32_t *status)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        if (load_acquire(cnt) < target) {
            uint64_t t0;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
            while (load_acquire(cnt) < target) {
                uint64_t t1;
                asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
                if (t1 - t0 > kBarrierTimeoutNs) {
                    record_status(status, D3D_ERR_DEVICE_TIMEOUT);
                    ok = 0;
                    break;
                }
            }
        }
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// Signal one finished item (no return value).  The release orders the
// calling thread's earlier writes (the item's record) before the count.
__device__ inline void signal_count(int *cnt)
{
    asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(cnt) : "memory");
}

// Draft tokens, acceptance uniforms and the sample uniform of request r into
// shared memory (issued before the selection's wait, which they do not
// depend on).
template <int NT>
__device__ inline void load_request_inputs(int r, int B, const int32_t *__restrict__ y,
                                           const float *__restrict__ u_acc, const float *__restrict__ u_s,
                                           int32_t *s_y, float *s_u, float *s_us)
{
    for (int jj = threadIdx.x; jj < B - 1; jj += NT) {
        s_y[jj] = __ldg(y + (size_t)r * (B - 1) + jj);
        s_u[jj] = __ldg(u_acc + (size_t)r * (B - 1) + jj);
    }
    if (threadIdx.x == 0)
        *s_us = __ldg(u_s + r);
}

// Phase B for request r: combine the records, alpha_j, the first rejection,
// the sample's row pair.  s_y / s_u hold the request's draft tokens and
// uniforms.  With write_outputs the CTA also writes accept_len, num_tokens,
// alpha/p/q and the accepted tokens.
template <int NT>
__device__ void select_request(int r, int B, int V, int nch, int chunk_w, const Rec *__restrict__ rec,
                               const int32_t *s_y, const float *s_u, bool write_outputs,
                               int32_t *__restrict__ accept_len, int32_t *__restrict__ out_tokens,
                               int32_t *__restrict__ num_tokens, float *__restrict__ alpha_out,
                               float *__restrict__ p_out, float *__restrict__ q_out, float *__restrict__ awl_out,
                               int32_t *status, Sel &sel,
                               Rec *s_rec)
{
    __shared__ float s_mp[kMaxB], s_zp[kMaxB], s_mq[kMaxB], s_zq[kMaxB], s_al[kMaxB];
    __shared__ int s_a;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const Rec *pr = rec + (size_t)r * B * nch;
    const int nrec = B * nch;
    const bool staged = nrec <= kStagedRecords;
    if (staged) {
        const float4 *src = reinterpret_cast<const float4 *>(pr);
        float4 *dst = reinterpret_cast<float4 *>(s_rec);
        for (int i = threadIdx.x; i < 2 * nrec; i += NT)
            dst[i] = __ldcg(src + i);
    }
    if (threadIdx.x == 0)
        s_a = B - 1;
    __syncthreads();
    // records written by other CTAs of this launch: L2 reads when not staged
    auto rec_at = [&](int i) -> Rec {
        if (staged)
            return s_rec[i];
        const float4 a = __ldcg(reinterpret_cast<const float4 *>(pr + i));
        const float4 b = __ldcg(reinterpret_cast<const float4 *>(pr + i) + 1);
        return Rec{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    };
    // one warp per position: the row statistics over the chunk records, then
    // p_j, q_j, alpha_j and the acceptance test
    for (int jj = warp; jj < B; jj += VCfg<NT>::kWarps) {
        float mp = -INFINITY, zp = 0.f, mq = -INFINITY, zq = 0.f;
        for (int cc = lane; cc < nch; cc += 32) {
            const Rec t = rec_at(jj * nch + cc);
            ms_merge(mp, zp, t.mP, t.zP);
            ms_merge(mq, zq, t.mQ, t.zQ);
        }
        float MP = mp, MQ = mq;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            MP = fmaxf(MP, __shfl_xor_sync(kFull, MP, o));
            MQ = fmaxf(MQ, __shfl_xor_sync(kFull, MQ, o));
        }
        float sp = (mp == -INFINITY) ? 0.f : zp * fast_exp2(mp - MP);
        float sq = (mq == -INFINITY) ? 0.f : zq * fast_exp2(mq - MQ);
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            sp += __shfl_xor_sync(kFull, sp, o);
            sq += __shfl_xor_sync(kFull, sq, o);
        }
        if (lane == 0) {
            s_mp[jj] = MP, s_zp[jj] = sp, s_mq[jj] = MQ, s_zq[jj] = sq;
            if (jj < B - 1) {
                const int yv = s_y[jj];
                float p = 0.f, q = 0.f, al = 0.f;
                if (yv < 0 || yv >= V) {
                    if (write_outputs)
                        record_status(status, D3D_ERR_DEVICE_INPUT);
                } else {
                    const Rec t = rec_at(jj * nch + yv / chunk_w);
                    p = fast_exp2(t.xP - MP) / sp;
                    q = fast_exp2(t.xQ - MQ) / sq;
                    al = (p >= q) ? 1.f : p / q;
                }
                if (!(s_u[jj] < al))
                    atomicMin(&s_a, jj);
                s_al[jj] = al;
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
        }
    }
    __syncthreads();
    const int a = s_a;
    sel.a = a;
    sel.mode = (a < B - 1) ? 0 : 1;
    sel.row = (a < B - 1) ? a : B - 1;
    sel.mP = s_mp[sel.row];
    sel.rZP = __frcp_rn(s_zp[sel.row]);
    sel.mQ = (a < B - 1) ? s_mq[a] : 0.f;
    sel.rZQ = (a < B - 1) ? __frcp_rn(s_zq[a]) : 1.f;
    if (write_outputs) {
        if (threadIdx.x == 0) {
            accept_len[r] = a;
            num_tokens[r] = a + 1;
            if (awl_out) {
                // [DScout] "Background: AWL and the acceptance rule": the weight of
                // position k is the product of the acceptance probabilities of the
                // drafts before it (the probability that verification reaches k)
                float w = 1.f;
                for (int jj = 0; jj < B - 1; ++jj) {
                    awl_out[(size_t)r * (B - 1) + jj] = w;
                    w *= s_al[jj];
                }
            }
        }
        for (int jj = threadIdx.x; jj < B; jj += NT)
            if (jj != a)
                out_tokens[(size_t)r * B + jj] = (jj < a) ? s_y[jj] : -1;
    }
    __syncthreads();  // the shared arrays are reused by the next call
}

// Per-slot masses w of the sampled distribution in chunk [c0, c1): the
// residual max(0, P - Q) (kind 0) or P (kind 1), reloading the chunk; and
// the sums of w and of P.
template <typename T, int NT>
__device__ inline void chunk_masses(const T *prow, const T *qrow, int kind, int c0, int c1, float c,
                                    const Sel &sel, float (&w)[kVPer], float &s_kind, float &s_p)
{
    float xp[kVPer];
    load_chunk<T, NT>(prow, c0, c1, c, xp);
    if (kind == 0)
        load_chunk<T, NT>(qrow, c0, c1, c, w);
    s_kind = 0.f;
    s_p = 0.f;
#pragma unroll
    for (int i = 0; i < kVPer; ++i) {
        const float P = fast_exp2(xp[i] - sel.mP) * sel.rZP;
        w[i] = (kind == 0) ? fmaxf(P - fast_exp2(w[i] - sel.mQ) * sel.rZQ, 0.f) : P;
        s_kind += w[i];
        s_p += P;
    }
}

// The same from exponentials kept since phase A: eP/eQ = exp2(x - m_t) with
// m_t this thread's max of the row chunk; w may alias eQ.
__device__ inline void kept_masses(int kind, const float (&eP)[kVPer], float (&eQ)[kVPer], float mtP, float mtQ,
                                   const Sel &sel, float &s_kind, float &s_p)
{
    const float sP = (mtP == -INFINITY) ? 0.f : fast_exp2(mtP - sel.mP) * sel.rZP;
    const float sQ = (kind != 0 || mtQ == -INFINITY) ? 0.f : fast_exp2(mtQ - sel.mQ) * sel.rZQ;
    s_kind = 0.f;
    s_p = 0.f;
#pragma unroll
    for (int i = 0; i < kVPer; ++i) {
        const float P = eP[i] * sP;
        eQ[i] = fmaxf(P - eQ[i] * sQ, 0.f);
        s_kind += eQ[i];
        s_p += P;
    }
}

// Phase D of request r in the chunk [c0, c1) that holds the crossing: the
// ordered scan of the slot masses w (slot order is group-major vocabulary
// order) for the first position whose in-chunk cumulative mass passes
// `target` (the sample's target minus the masses of the earlier chunks);
// writes the sampled token.
template <int NT>
__device__ void scan_owner(const float (&w)[kVPer], int c0, float target, bool takelast, int32_t *out_tok,
                           float *red)
{
    __shared__ int s_cand, s_lastpos;
    if (threadIdx.x == 0) {
        s_cand = 0x7fffffff;
        s_lastpos = -1;
    }
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f);
    int lastpos = -1;
#pragma unroll
    for (int i = 0; i < kVPer; ++i) {
        const int q = i >> 3;
        if (q == 0) g.x += w[i];
        else if (q == 1) g.y += w[i];
        else if (q == 2) g.z += w[i];
        else g.w += w[i];
        if (w[i] > 0.f)
            lastpos = max(lastpos, slot_pos<NT>(c0, i));
    }
    const float4 ex = block_group_scan<NT>(g, red);  // has a __syncthreads (s_cand initialised)
    const float gs[4] = {g.x, g.y, g.z, g.w}, bs[4] = {ex.x, ex.y, ex.z, ex.w};
    if (!takelast) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (bs[q] + gs[q] > target) {
                atomicMin(&s_cand, q * NT + (int)threadIdx.x);
                break;
            }
    }
    atomicMax(&s_lastpos, lastpos);
    __syncthreads();
    const int cand = s_cand;
    if (!takelast && cand != 0x7fffffff && (cand % NT) == (int)threadIdx.x) {
        const int q = cand / NT;
        int tok = -1, last = -1;
        float cum = bs[q];
#pragma unroll
        for (int i = 0; i < kVPer; ++i) {
            if ((i >> 3) == q && tok < 0) {
                cum += w[i];
                if (w[i] > 0.f)
                    last = slot_pos<NT>(c0, i);
                if (cum > target)
                    tok = slot_pos<NT>(c0, i);
            }
        }
        // rounding between the two summation orders: the group's last position with mass
        if (tok < 0)
            tok = last >= 0 ? last : s_lastpos;
        *out_tok = tok;
    }
    if ((takelast || cand == 0x7fffffff) && threadIdx.x == 0)
        *out_tok = s_lastpos;
    __syncthreads();
}

// The phase-D decision of one request: which chunk holds the sample's
// crossing and where.  From the request's chunk sums part2_r[cc] = (residual
// mass, P mass), by warp 0 (every thread of the CTA calls it; the result is
// in *dec after the final barrier): the total S of the residual (or of P when
// the residual has no mass left in fp32, or for the bonus row), the target
// u*S, the first chunk whose inclusive sum passes it and the target's offset
// into that chunk.  Sums and the product are kept as fp32 pairs (df_add /
// df_mul), so that magnitude-S quantities carry no 2^-24 S rounding; the
// owner chunk then scans against an offset on its own scale.  When rounding
// leaves the target at or past the end, the last chunk with mass owns it and
// takes its last position with mass.
struct Decision {
    int kind;      // 0: residual max(0, P - Q); 1: P
    int owner;     // chunk holding the crossing (-1: no mass anywhere)
    int takelast;  // take the owner's last position with mass
    float rem;     // target minus the masses of the chunks before the owner
};

template <int NT>
__device__ void decide_request(const float2 *__restrict__ part2_r, int nch, int mode, float us, float2 *s_sums,
                               Decision *dec)
{
    for (int cc = threadIdx.x; cc < nch; cc += NT)
        s_sums[cc] = __ldcg(part2_r + cc);
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int per = (nch + 31) >> 5;  // consecutive chunks per lane
        const int c_lo = min(nch, lane * per), c_hi = min(nch, c_lo + per);
        float rh = 0.f, rl = 0.f, ph = 0.f, pl = 0.f;  // this lane's residual and P masses
        for (int cc = c_lo; cc < c_hi; ++cc) {
            df_add(rh, rl, s_sums[cc].x, 0.f);
            df_add(ph, pl, s_sums[cc].y, 0.f);
        }
        // inclusive scan over the lanes (chunk order) of both masses
        float irh = rh, irl = rl, iph = ph, ipl = pl;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float a = __shfl_up_sync(kFull, irh, o), b = __shfl_up_sync(kFull, irl, o);
            const float c2 = __shfl_up_sync(kFull, iph, o), d = __shfl_up_sync(kFull, ipl, o);
            if (lane >= o) {
                df_add(irh, irl, a, b);
                df_add(iph, ipl, c2, d);
            }
        }
        // residual unless it has no mass left in fp32 (then P at that row)
        const float Srh = __shfl_sync(kFull, irh, 31);
        const int kind = (mode == 0 && Srh > 0.f) ? 0 : 1;
        const float inh = kind == 0 ? irh : iph, inl = kind == 0 ? irl : ipl;
        const float Sh = __shfl_sync(kFull, inh, 31), Sl = __shfl_sync(kFull, inl, 31);
        float th, tl;
        df_mul(us, Sh, Sl, th, tl);
        float exh = __shfl_up_sync(kFull, inh, 1), exl = __shfl_up_sync(kFull, inl, 1);
        if (lane == 0)
            exh = exl = 0.f;
        auto mass = [&](int cc) { return kind == 0 ? s_sums[cc].x : s_sums[cc].y; };
        // the first lane whose inclusive sum passes the target holds the crossing
        const unsigned bal = __ballot_sync(kFull, c_lo < c_hi && df_gt(inh, inl, th, tl));
        int owner = -1, takelast = 0;
        float rem = 0.f;
        if (bal) {
            const int L = __ffs(bal) - 1;
            if (lane == L) {
                float runh = exh, runl = exl;
                int last_mass = -1;
                for (int cc = c_lo; cc < c_hi; ++cc) {
                    float nh = runh, nl = runl;
                    df_add(nh, nl, mass(cc), 0.f);
                    if (mass(cc) > 0.f)
                        last_mass = cc;
                    if (df_gt(nh, nl, th, tl)) {
                        owner = cc;
                        break;
                    }
                    runh = nh, runl = nl;
                }
                if (owner < 0) {  // the two summation orders disagree in the last bits
                    owner = last_mass;
                    takelast = 1;
                }
                rem = (th - runh) + (tl - runl);
            }
            owner = __shfl_sync(kFull, owner, L);
            takelast = __shfl_sync(kFull, takelast, L);
            rem = __shfl_sync(kFull, rem, L);
        } else {  // rounding left u*S at or past the end: last chunk with mass
            takelast = 1;
            int lastc = -1;
            for (int cc = c_lo; cc < c_hi; ++cc)
                if (mass(cc) > 0.f)
                    lastc = cc;
            const unsigned b2 = __ballot_sync(kFull, lastc >= 0);
            owner = b2 ? __shfl_sync(kFull, lastc, 31 - __clz(b2)) : -1;
        }
        if (lane == 0) {
            dec->kind = kind;
            dec->owner = owner;
            dec->takelast = takelast;
            dec->rem = rem;
        }
    }
    __syncthreads();
}

// Branch cache-hit match of request r fused after its sample ([D3D]
// "Background: asynchronous drafting and cache hits"): the verified tokens are
// y_0..y_{a-1} (shared memory) and the sampled token; the smallest head index
// of equal length and equal tokens wins, -1 on a miss.  Run by warp 0.
__device__ void match_request(int r, int a, int tok, const int32_t *s_y, int B, int M,
                              const int32_t *__restrict__ heads, const int32_t *__restrict__ head_len,
                              int32_t *__restrict__ branch)
{
    const int lane = threadIdx.x & 31, n = a + 1;
    int hit = -1;
    for (int k0 = 0; k0 < M && hit < 0; k0 += 32) {
        const int k = k0 + lane;
        bool same = false;
        if (k < M && __ldg(head_len + (size_t)r * M + k) == n) {
            const int32_t *h = heads + ((size_t)r * M + k) * B;
            same = true;
            for (int i = 0; i < n && same; ++i)
                same = __ldg(h + i) == (i < a ? s_y[i] : tok);
        }
        const unsigned ballot = __ballot_sync(0xffffffffu, same);
        if (ballot)
            hit = k0 + __ffs(ballot) - 1;
    }
    if (lane == 0)
        branch[r] = hit;
}

// Arguments of one verification launch (device pointers; logits typed by
// the launch's T).
struct VArgs {
    const void *target, *draft;
    const int32_t *y;
    const float *u_acc, *u_s;
    int R, B, V, M;
    float c;  // log2(e) / temperature
    int32_t *accept_len, *out_tokens, *num_tokens;
    float *alpha, *p, *q, *awl;
    const int32_t *heads, *head_len;
    int32_t *branch;
    unsigned char *ws;
    int ring;  // > 0: phase A streams items through this many shared-memory slots (bf16 rows, bulk copies)
    int fault;  // 2: CTA 0 never issues the copies of its first ring item (failure-detection hook)
};

// Phase-A ring of the SM-limited launch: per slot, the target row's and the
// draft row's chunk as bf16, then one mbarrier per slot.
constexpr int kRingSlots = 3;
template <int NT> struct Ring {
    static constexpr uint32_t kRowBytes = VCfg<NT>::kChunk * 2;
    static constexpr uint32_t kSlotBytes = 2 * kRowBytes;
    static constexpr size_t bytes(int slots) { return (size_t)slots * kSlotBytes + (size_t)slots * 8; }
};

// The verification of CTA vb of vgrid (all vgrid CTAs resident: they wait on
// one another).  A kernel of its own, or the verification part of a fused
// round launch.
template <typename T, int NT>
__device__ __forceinline__ void verify_body(unsigned vb, unsigned vgrid, const VArgs &a)
{
    const T *__restrict__ target = static_cast<const T *>(a.target);
    const T *__restrict__ draft = static_cast<const T *>(a.draft);
    const int32_t *__restrict__ y = a.y;
    const float *__restrict__ u_acc = a.u_acc;
    const float *__restrict__ u_s = a.u_s;
    const int R = a.R, B = a.B, V = a.V, M = a.M;
    const float c = a.c;
    int32_t *__restrict__ accept_len = a.accept_len;
    int32_t *__restrict__ out_tokens = a.out_tokens;
    int32_t *__restrict__ num_tokens = a.num_tokens;
    float *__restrict__ alpha_out = a.alpha;
    float *__restrict__ p_out = a.p;
    float *__restrict__ q_out = a.q;
    float *__restrict__ awl_out = a.awl;
    const int32_t *__restrict__ heads = a.heads;
    const int32_t *__restrict__ head_len = a.head_len;
    int32_t *__restrict__ branch = a.branch;
    unsigned char *__restrict__ ws = a.ws;
    extern __shared__ float4 s_dyn[];  // request records when staged; chunk sums in phase D
    using C = VCfg<NT>;
    __shared__ float red[4 * C::kWarps];
    __shared__ float s_xy[2];
    __shared__ int32_t s_y[kMaxB];
    __shared__ float s_u[kMaxB], s_us;
    const VerifyLayout L = verify_layout(R, B, V, C::kChunk);
    const int nch = L.nch;
    const long long nA = (long long)R * B * nch;
    const int nC = R * nch;
    Rec *rec = reinterpret_cast<Rec *>(ws + L.rec);
    float2 *part2 = reinterpret_cast<float2 *>(ws + L.part2);
    int *bar = reinterpret_cast<int *>(ws + L.bar);
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    Rec *s_rec = reinterpret_cast<Rec *>(s_dyn);
    // a kernel launched after this one as an independent programmatic
    // dependent may start now
    if (threadIdx.x == 0)
        sm100::pdl_trigger();
    // one phase-A item per CTA: its exponentials stay in registers for phase C
    const bool keep = nA <= (long long)vgrid;

    // ---- phase A: per (request, position, chunk) statistics of the row pair;
    // the next item's loads are in flight while the current one is reduced
    float eP[kVPer], eQ[kVPer];
    float mtP = -INFINITY, mtQ = -INFINITY;
    auto target_row = [&](long long it, int &v0, int &v1, int &j) -> const T * {
        const int chunk = (int)(it % nch);
        const int rj = (int)(it / nch);
        j = rj % B;
        v0 = chunk * C::kChunk;
        v1 = min(V, v0 + C::kChunk);
        return target + (size_t)rj * V;
    };
    auto draft_row = [&](long long it) -> const T * {
        const int rj = (int)(it / nch);
        return draft + ((size_t)(rj / B) * (B - 1) + (rj % B)) * V;  // valid only when j < B - 1
    };
    RawChunk<T, NT> rawP, rawQ;
    // ring path: each slot's two row chunks arrive by bulk copies, issued
    // kRingSlots items ahead (the host enables it for bf16 rows whose chunks
    // are 16-byte aligned, with the ring's shared memory)
    // (compiled for the 512-thread launch only; the 256-thread one keeps its registers)
    const int nring = (NT == kNTLimited) ? a.ring : 0;
    const int nring1 = nring > 0 ? nring : 1;  // divisor for the ring's slot arithmetic (used only with a ring)
    uint8_t *ring = reinterpret_cast<uint8_t *>(s_dyn);  // reused for the staged records after phase A
    const uint32_t ring_s = sm100::smem_u32(ring), ring_bar = ring_s + (uint32_t)nring * Ring<NT>::kSlotBytes;
    auto ring_issue = [&](long long it, int slot) {
        if (a.fault == 2 && vb == 0 && it == 0)
            return;  // injected fault: this slot's copies never arrive
        int v0, v1, j;
        const T *rp = target_row(it, v0, v1, j);
        const uint32_t row_bytes = (uint32_t)(v1 - v0) * 2u;
        const uint32_t bar = ring_bar + 8u * (uint32_t)slot, dst = ring_s + (uint32_t)slot * Ring<NT>::kSlotBytes;
        sm100::mbar_arrive_expect_tx(bar, j < B - 1 ? 2u * row_bytes : row_bytes);
        sm100::bulk_load(dst, rp + v0, row_bytes, bar);
        if (j < B - 1)
            sm100::bulk_load(dst + Ring<NT>::kRowBytes, draft_row(it) + v0, row_bytes, bar);
    };
    // slot values in the thread's slot order, raw (unscaled); -inf past v1
    auto ring_take = [&](int slot, int row, int v0, int v1, float (&x)[kVPer]) {
        const uint8_t *src = ring + (size_t)slot * Ring<NT>::kSlotBytes + (size_t)row * Ring<NT>::kRowBytes;
        const bool full = v1 - v0 == C::kChunk;
#pragma unroll
        for (int g = 0; g < kVPer / 8; ++g) {
            const int off = g * C::kGroup + 8 * (int)threadIdx.x;
            const uint4 u = *reinterpret_cast<const uint4 *>(src + 2 * off);
            const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[8 * g + 2 * e] = __uint_as_float(wv[e] << 16);
                x[8 * g + 2 * e + 1] = __uint_as_float(wv[e] & 0xffff0000u);
            }
        }
        if (!full) {
#pragma unroll
            for (int i = 0; i < kVPer; ++i)
                x[i] = slot_pos<NT>(v0, i) < v1 ? x[i] : -INFINITY;
        }
    };
    if (nring > 0) {
        if (threadIdx.x == 0) {
            for (int sl = 0; sl < nring; ++sl)
                sm100::mbar_init(ring_bar + 8u * (uint32_t)sl, 1);
            sm100::fence_barrier_init();
        }
        __syncthreads();
        if (threadIdx.x == 0)
            for (int sl = 0; sl < nring && (long long)vb + (long long)sl * vgrid < nA; ++sl)
                ring_issue((long long)vb + (long long)sl * vgrid, sl);
    } else if ((long long)vb < nA) {
        int v0, v1, j;
        const T *rp = target_row(vb, v0, v1, j);
        rawP.issue(rp, v0, v1);
        if (j < B - 1)
            rawQ.issue(draft_row(vb), v0, v1);
    }
    // a ring slot whose copies did not land in time stops the CTA's phase A:
    // no further copies are issued, the copies in flight are waited out, and
    // the CTA leaves (the request's other CTAs then give up waiting for its
    // records; the status word holds the timeout)
    __shared__ volatile int s_ring_abort;
    if (threadIdx.x == 0)
        s_ring_abort = 0;
    __syncthreads();
    int k_item = 0;  // this CTA's item count
    for (long long item = vb; item < nA; item += vgrid, ++k_item) {
        int v0, v1, j;
        const T *rowP = target_row(item, v0, v1, j);
        const int r = (int)(item / nch) / B;
        const int yv = (j < B - 1) ? __ldg(y + (size_t)r * (B - 1) + j) : -1;
        if (NT == kNTLimited && nring > 0) {
            const int slot = k_item % nring1;
            const uint32_t bar = ring_bar + 8u * (uint32_t)slot;
            const uint32_t parity = (uint32_t)(k_item / nring1) & 1u;
            if (!sm100::mbar_try_wait(bar, parity)) {  // bounded wait for the slot's copies
                const uint64_t t0 = sm100::global_ns();
                while (!sm100::mbar_try_wait_sleep(bar, parity))
                    if (s_ring_abort || sm100::global_ns() - t0 > kBarrierTimeoutNs) {
                        record_status(reinterpret_cast<int32_t *>(ws), D3D_ERR_DEVICE_TIMEOUT);
                        s_ring_abort = 1;
                        break;
                    }
            }
            ring_take(slot, 0, v0, v1, eP);
            if (j < B - 1) {
                ring_take(slot, 1, v0, v1, eQ);
            } else {
#pragma unroll
                for (int i = 0; i < kVPer; ++i)
                    eQ[i] = -INFINITY;
            }
        } else {
            rawP.take(rowP, v0, v1, 1.f, eP);  // raw logits: the scale goes into the exponent
            if (j < B - 1) {
                rawQ.take(draft_row(item), v0, v1, 1.f, eQ);
            } else {
#pragma unroll
                for (int i = 0; i < kVPer; ++i)
                    eQ[i] = -INFINITY;
            }
            const long long next = item + vgrid;
            if (next < nA) {
                int nv0, nv1, nj;
                const T *np = target_row(next, nv0, nv1, nj);
                rawP.issue(np, nv0, nv1);
                if (nj < B - 1)
                    rawQ.issue(draft_row(next), nv0, nv1);
            }
        }
        if (yv >= v0 && yv < v1) {  // the thread holding position y keeps both logits for the record
            const int rel = yv - v0;
            if ((int)threadIdx.x == (rel % C::kGroup) / 8) {
                const int slot = (rel / C::kGroup) * 8 + rel % 8;
                float xp = 0.f, xq = 0.f;
#pragma unroll
                for (int i = 0; i < kVPer; ++i) {
                    xp = (i == slot) ? eP[i] : xp;
                    xq = (i == slot) ? eQ[i] : xq;
                }
                s_xy[0] = xp * c;
                s_xy[1] = xq * c;
            }
        }
        float zP, zQ;
        thread_exp_scaled(eP, c, mtP, zP);
        thread_exp_scaled(eQ, c, mtQ, zQ);
        float m1 = mtP, z1 = zP, m2 = mtQ, z2 = zQ;
        block_ms2<NT>(m1, z1, m2, z2, red);  // has a __syncthreads: s_xy is visible to thread 0 after it
        const bool has = yv >= v0 && yv < v1;
        const float xyP = (threadIdx.x == 0 && has) ? s_xy[0] : 0.f, xyQ = (threadIdx.x == 0 && has) ? s_xy[1] : 0.f;
        __syncthreads();  // red and s_xy are reused by the next item; the slot has been read
        if (nring > 0 && s_ring_abort) {
            // this item and the next nring - 1 have copies issued that may still
            // be in flight: wait for each (bounded) before the CTA leaves
            if (threadIdx.x == 0) {
                for (int jj = k_item; jj < k_item + nring; ++jj) {
                    if ((long long)vb + (long long)jj * vgrid >= nA)
                        break;
                    const uint32_t b2 = ring_bar + 8u * (uint32_t)(jj % nring1);
                    const uint32_t par = (uint32_t)(jj / nring1) & 1u;
                    const uint64_t t0 = sm100::global_ns();
                    while (!sm100::mbar_try_wait_sleep(b2, par))
                        if (sm100::global_ns() - t0 > kBarrierTimeoutNs)
                            break;
                }
            }
            __syncthreads();
            return;
        }
        // the record and its signal after the barrier: the release's wait
        // overlaps the next item's loads and exponentials in the other warps
        if (threadIdx.x == 0 && dbg_ok(item < nA, reinterpret_cast<int32_t *>(ws))) {
            float4 *dst = reinterpret_cast<float4 *>(rec + item);
            dst[0] = make_float4(m1, z1, m2, z2);
            dst[1] = make_float4(xyP, xyQ, 0.f, 0.f);
            signal_count(bar + kBarInts * r);
        }
        if (nring > 0 && threadIdx.x == 0) {
            const long long nxt = item + (long long)nring * vgrid;
            if (nxt < nA)
                ring_issue(nxt, k_item % nring1);
        }
    }

    __shared__ Decision s_dec;
    // phase D decision for request r from its chunk sums (the records are no
    // longer needed: their shared memory holds the sums)
    auto decide = [&](int r, const Sel &sel) {
        decide_request<NT>(part2 + (size_t)r * nch, nch, sel.mode, s_us, reinterpret_cast<float2 *>(s_dyn), &s_dec);
    };
    // The match of request r once its sampled token is written (the writer is a
    // thread of this CTA, and a barrier separates the write from this read).
    auto fused_match = [&](int r, int a) {
        if (branch != nullptr && threadIdx.x < 32) {
            const int tok = *reinterpret_cast<volatile const int32_t *>(out_tokens + (size_t)r * B + a);
            match_request(r, a, tok, s_y, B, M, heads, head_len, branch);
        }
    };
    // The request's last phase-D item resets the phase-C/D counters (every
    // phase-C signal has arrived and every phase-D waiter has passed).
    auto finish_d = [&](int r) {
        if (threadIdx.x == 0 && atomicAdd(bar + kBarInts * r + 3, 1) == nch - 1) {
            bar[kBarInts * r + 2] = 0;
            bar[kBarInts * r + 3] = 0;
        }
    };
    // Count a waiter past the phase-A wait; the last one resets the phase-A
    // counters (no waiter reads them any more).
    auto passed_a = [&](int r, int waiters) {
        if (threadIdx.x == 0 && atomicAdd(bar + kBarInts * r + 1, 1) == waiters - 1) {
            bar[kBarInts * r + 0] = 0;
            bar[kBarInts * r + 1] = 0;
        }
    };

    Sel sel;
    if (keep) {
        // ---- B, C, D on the CTA's own item
        if ((long long)vb >= nA)
            return;
        const int item = vb;
        const int chunk = item % nch, rj = item / nch;
        const int r = rj / B, j = rj % B;
        load_request_inputs<NT>(r, B, y, u_acc, u_s, s_y, s_u, &s_us);
        if (!wait_count(bar + kBarInts * r, B * nch, status))
            return;
        select_request<NT>(r, B, V, nch, C::kChunk, rec, s_y, s_u, j == 0 && chunk == 0, accept_len, out_tokens, num_tokens,
                       alpha_out, p_out, q_out, awl_out, status, sel, s_rec);
        if (j != sel.row) {
            passed_a(r, B * nch);  // counted once the CTA's work is done: off the critical path
            return;
        }
        const int c0 = chunk * C::kChunk;
        float s_kind, s_p;
        kept_masses(sel.mode == 0 ? 0 : 1, eP, eQ, mtP, mtQ, sel, s_kind, s_p);  // eQ now holds the masses
        block_sum2<NT>(s_kind, s_p, red);
        if (threadIdx.x == 0) {
            part2[(size_t)r * nch + chunk] = make_float2(s_kind, s_p);
            signal_count(bar + kBarInts * r + 2);
        }
        if (!wait_count(bar + kBarInts * r + 2, nch, status))
            return;
        decide(r, sel);
        if (s_dec.owner == chunk) {
            if (s_dec.kind != sel.mode) {  // residual without mass in fp32: P at that row
                float a1, a2;
                kept_masses(1, eP, eQ, mtP, mtQ, sel, a1, a2);
            }
            scan_owner<NT>(eQ, c0, s_dec.rem, s_dec.takelast != 0, out_tokens + (size_t)r * B + sel.a, red);
            fused_match(r, sel.a);
        } else if (s_dec.owner < 0 && chunk == 0) {
            // no mass anywhere: cannot happen for a finite softmax row
            if (threadIdx.x == 0) {
                record_status(status, D3D_ERR_DEVICE_INPUT);
                out_tokens[(size_t)r * B + sel.a] = 0;
            }
            __syncthreads();
            fused_match(r, sel.a);
        }
        finish_d(r);
        passed_a(r, B * nch);
        return;
    }

    // ---- phase C: the request's selection, then this chunk's masses from a
    // reload.  With at most one C item per CTA, the CTA's D item is the same
    // (request, chunk): it keeps the selection and the masses.
    const bool cd_same = nC <= (int)vgrid;
    float w[kVPer];
    for (int item = vb; item < nC; item += vgrid) {
        const int r = item / nch, chunk = item % nch;
        load_request_inputs<NT>(r, B, y, u_acc, u_s, s_y, s_u, &s_us);
        if (!wait_count(bar + kBarInts * r, B * nch, status))
            return;
        passed_a(r, nch);
        select_request<NT>(r, B, V, nch, C::kChunk, rec, s_y, s_u, chunk == 0, accept_len, out_tokens, num_tokens, alpha_out,
                       p_out, q_out, awl_out, status, sel, s_rec);
        const T *prow = target + ((size_t)r * B + sel.row) * V;
        const T *qrow = draft + ((size_t)r * (B - 1) + (sel.mode == 0 ? sel.row : 0)) * V;
        const int c0 = chunk * C::kChunk, c1 = min(V, c0 + C::kChunk);
        float s_kind, s_p;
        chunk_masses<T, NT>(prow, qrow, sel.mode == 0 ? 0 : 1, c0, c1, c, sel, w, s_kind, s_p);
        block_sum2<NT>(s_kind, s_p, red);
        if (threadIdx.x == 0) {
            part2[item] = make_float2(s_kind, s_p);
            signal_count(bar + kBarInts * r + 2);
        }
        __syncthreads();
    }

    // ---- phase D: the chunk holding the crossing reloads its masses and scans
    for (int item = vb; item < nC; item += vgrid) {
        const int r = item / nch, chunk = item % nch;
        load_request_inputs<NT>(r, B, y, u_acc, u_s, s_y, s_u, &s_us);
        if (!wait_count(bar + kBarInts * r + 2, nch, status))
            return;
        // every phase-C item of r waited for r's phase A, so the records are complete
        if (!cd_same)
            select_request<NT>(r, B, V, nch, C::kChunk, rec, s_y, s_u, false, accept_len, out_tokens, num_tokens, alpha_out,
                               p_out, q_out, awl_out, status, sel, s_rec);
        decide(r, sel);
        if (s_dec.owner == chunk) {
            const int c0 = chunk * C::kChunk, c1 = min(V, c0 + C::kChunk);
            if (!cd_same || s_dec.kind != sel.mode) {  // masses not kept (or the fallback kind)
                const T *prow = target + ((size_t)r * B + sel.row) * V;
                const T *qrow = draft + ((size_t)r * (B - 1) + (sel.mode == 0 ? sel.row : 0)) * V;
                float a1, a2;
                chunk_masses<T, NT>(prow, qrow, s_dec.kind, c0, c1, c, sel, w, a1, a2);
            }
            scan_owner<NT>(w, c0, s_dec.rem, s_dec.takelast != 0, out_tokens + (size_t)r * B + sel.a, red);
            fused_match(r, sel.a);
        } else if (s_dec.owner < 0 && chunk == 0) {
            if (threadIdx.x == 0) {
                record_status(status, D3D_ERR_DEVICE_INPUT);
                out_tokens[(size_t)r * B + sel.a] = 0;
            }
            __syncthreads();
            fused_match(r, sel.a);
        }
        finish_d(r);
        __syncthreads();
    }
}


template <typename T, int NT>
__global__ void __launch_bounds__(NT, NT == kNTDevice ? 2 : 1) verify_kernel(const VArgs a)
{
    verify_body<T, NT>(blockIdx.x, gridDim.x, a);
    // launched as the programmatic dependent of an independent kernel (the
    // drafting attention of the round): finish only after it has finished
    sm100::pdl_wait();
}

// Dynamic shared memory of a verification CTA: the request's records when
// they are staged, and at least the request's chunk sums (phase D).
inline size_t verify_dyn_smem(int B, int nch)
{
    const int nrec = B * nch;
    size_t dyn = nrec <= kStagedRecords ? sizeof(Rec) * (size_t)nrec : 0;
    if (dyn < sizeof(float2) * (size_t)nch)
        dyn = sizeof(float2) * (size_t)nch;
    return dyn;
}

// Host-side checks of d3d_spec_verify's arguments (everything but the
// workspace size and the SM limit) and the kernel arguments they give.
// Returns D3D_OK, a status, or 1 when there is nothing to do (R == 0).
inline int verify_prepare(const void *target_logits, const void *draft_logits, int logits_dtype,
                          const int32_t *draft_tokens, const float *u_accept, const float *u_sample, int R, int B,
                          int V, float temperature, int32_t *accept_len, int32_t *out_tokens, int32_t *num_tokens,
                          float *alpha, float *p_draft, float *q_draft, float *awl_weight, const int32_t *heads,
                          const int32_t *head_len, int M, int32_t *branch, VArgs &a)
{
    // temperature 0: greedy verification (no draft logits, no uniforms)
    const bool greedy = temperature == 0.f;
    if (R < 0 || B < 2 || V < 1 || !(temperature >= 0.f) || !isfinite(temperature) || M < 0)
        return D3D_ERR_INVALID_ARG;
    if (greedy && q_draft != nullptr)
        return D3D_ERR_INVALID_ARG;
    if (branch != nullptr && M > 0 && (!heads || !head_len))
        return D3D_ERR_INVALID_ARG;
    if (logits_dtype != D3D_DTYPE_F32 && logits_dtype != D3D_DTYPE_BF16)
        return D3D_ERR_INVALID_ARG;
    if (B > kMaxB || V > kMaxChunks * kVChunkMin)
        return D3D_ERR_UNSUPPORTED;
    if (R == 0)
        return 1;
    if (!target_logits || !draft_tokens || !accept_len || !out_tokens || !num_tokens)
        return D3D_ERR_INVALID_ARG;
    if (!greedy && (!draft_logits || !u_accept || !u_sample))
        return D3D_ERR_INVALID_ARG;
    a.target = target_logits;
    a.draft = draft_logits;
    a.y = draft_tokens;
    a.u_acc = u_accept;
    a.u_s = u_sample;
    a.R = R, a.B = B, a.V = V, a.M = branch ? M : 0;
    a.c = greedy ? 0.f : (float)(1.4426950408889634 / (double)temperature);  // log2(e) / T
    a.accept_len = accept_len, a.out_tokens = out_tokens, a.num_tokens = num_tokens;
    a.alpha = alpha, a.p = p_draft, a.q = q_draft, a.awl = awl_weight;
    a.heads = heads, a.head_len = head_len, a.branch = branch;
    a.ws = nullptr;
    a.ring = 0;
    a.fault = fault_mode();
    return D3D_OK;
}

// Whether a launch of NT-thread CTAs may stream phase A through the ring:
// bf16 rows whose chunks start and end on 16-byte boundaries.
template <typename T, int NT> inline bool ring_fits(const VArgs &a)
{
    return NT == kNTLimited && sizeof(T) == 2 && a.V % 8 == 0 &&
           (reinterpret_cast<uintptr_t>(a.target) % 16) == 0 && (reinterpret_cast<uintptr_t>(a.draft) % 16) == 0;
}

}  // namespace
}  // namespace d3d
