// Packed drafting attention on the 5th-generation tensor cores (sm_103a).
//
// [D3D] "Core method", "Method steps" steps 2 and 4; [DScout] "Background:
// block-diffusion drafter".  See attn_common.cuh for the visibility rule.
//
// Work unit (one CTA): request r, KV head hk, a 128-row query tile and one
// KV split.  The 128 rows are (packed token, query head of hk's group)
// pairs, token-major, so one KV tile serves all G query heads of the group.
// A unit's key list is every 128-key tile of the request's prefix followed
// by the packed-key tiles that its rows can see (computed from the segment
// table at CTA start); the list is cut into `S` contiguous splits.
//
// Roles (192 threads):
//   warps 0-3  softmax: thread i owns TMEM lane i = query row i.  Reads S
//              from TMEM, applies the visibility mask, keeps the running max
//              (rescaling O in TMEM only when the max grows by > 2^8) and the
//              row sum, writes P (bf16) to shared memory in the 128-byte
//              swizzled K-major layout, and finally normalises O.
//   warp 4     TMA producer: Q once, then K and V tiles into 3- and 2-deep
//              rings (3-D tensor maps over [rows, heads, head_dim]).
//   warp 5     MMA issuer (one thread): S = Q K^T into one of two TMEM
//              buffers, O += P V into TMEM; tcgen05.commit releases ring
//              slots and signals the softmax warps.  Also owns TMEM.
// With S > 1 splits each thread writes its row's partial (O, max, sum) to the
// workspace; the thread that completes a row's last split (per-row atomic
// ticket) merges the partials and writes the output row.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <mutex>

#include "attn_common.cuh"
#include "sm100_ptx.cuh"

namespace d3d {
namespace {

using namespace sm100;

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per KV tile
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kThreads = 192;
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxPackedTiles = 64;  // packed keys per request <= 8192
constexpr float kRescaleLog2 = 8.f;  // rescale O only when the max grows by more than 2^8
constexpr uint32_t kBlockBytes = kBN * 128;  // one 128-row x 128-byte swizzled block (16 KB)

// barrier indices
enum {
    B_Q = 0,
    B_KF = 1,                       // 3
    B_KE = B_KF + kKStages,         // 3
    B_VF = B_KE + kKStages,         // 2
    B_VE = B_VF + kVStages,         // 2
    B_SF = B_VE + kVStages,         // 2
    B_SE = B_SF + 2,                // 2
    B_PR = B_SE + 2,
    B_PF = B_PR + 1,
    B_DONE = B_PF + 1,
    B_COUNT = B_DONE + 1
};

template <int D> struct Layout {
    static constexpr uint32_t kQBytes = kBM * D * 2;
    static constexpr uint32_t kKBytes = kBN * D * 2;
    static constexpr uint32_t kVBytes = kBN * D * 2;
    static constexpr uint32_t kPBytes = kBM * kBN * 2;
    static constexpr uint32_t q = 0;
    static constexpr uint32_t k = q + kQBytes;
    static constexpr uint32_t v = k + kKStages * kKBytes;
    static constexpr uint32_t p = v + kVStages * kVBytes;
    static constexpr uint32_t bars = p + kPBytes;
    static constexpr uint32_t misc = bars + B_COUNT * 8;
    static constexpr uint32_t total = misc + 64;
    static constexpr uint32_t alloc = total + 1024;  // room to align the base to 1024 bytes
};

struct AttnParams {
    const d3d_segment_t *segs;
    const int32_t *cu_prefix, *cu_q, *cu_seg;
    uint16_t *out;
    unsigned char *ws;
    int Hq, Hkv, G, TQ, MT, S;
    int max_q, max_prefix, total_q, total_prefix, total_segs;
    float scale_log2;
    unsigned long long off_cnt, off_opart, off_ml;
    int fault;
};

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// k-th set bit (0-based) of the 64-bit mask (m0 | m1 << 32); k < popcount.
__device__ __forceinline__ int nth_set_bit(uint32_t m0, uint32_t m1, int k)
{
    const int c0 = __popc(m0);
    uint32_t m = m0;
    int off = 0;
    if (k >= c0) {
        m = m1;
        k -= c0;
        off = 32;
    }
    for (int i = 0; i < k; ++i)
        m &= m - 1;
    return off + __ffs(m) - 1;
}

// Wait that ignores the abort flag (used to drain in-flight copies / MMAs).
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, int32_t *status)
{
    if (mbar_try_wait(bar, parity))
        return;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWaitTimeoutNs) {
            record_status(status, D3D_ERR_DEVICE_TIMEOUT);
            return;
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kp,
                   const __grid_constant__ CUtensorMap tm_vp, const __grid_constant__ CUtensorMap tm_kn,
                   const __grid_constant__ CUtensorMap tm_vn, const AttnParams p)
{
    using Lay = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- unit: ((r * Hkv + hk) * MT + mt) * S + sp
    unsigned u = blockIdx.x;
    const int sp = (int)(u % (unsigned)p.S);
    u /= (unsigned)p.S;
    const int mt = (int)(u % (unsigned)p.MT);
    u /= (unsigned)p.MT;
    const int hk = (int)(u % (unsigned)p.Hkv);
    const int r = (int)(u / (unsigned)p.Hkv);
    const unsigned tile_id = blockIdx.x / (unsigned)p.S;  // (r, hk, mt)
    int32_t *status = reinterpret_cast<int32_t *>(p.ws);

    ReqBounds b;
    if (!request_bounds(p.cu_prefix, p.cu_q, p.cu_seg, r, p.max_q, p.max_prefix, p.total_q, p.total_prefix,
                        p.total_segs, b)) {
        if (tid == 0)
            record_status(status, D3D_ERR_DEVICE_INPUT);
        return;
    }
    const int tq0 = mt * p.TQ;
    if (tq0 >= b.n_q)
        return;

    // ---- shared memory carve-up (1024-byte aligned base for the swizzled tiles)
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (sbase - raw);
    const uint32_t sQ = sbase + Lay::q, sK = sbase + Lay::k, sV = sbase + Lay::v, sP = sbase + Lay::p;
    auto bar = [&](int i) -> uint32_t { return sbase + Lay::bars + 8u * (uint32_t)i; };
    uint32_t *misc = reinterpret_cast<uint32_t *>(gbase + Lay::misc);
    volatile uint32_t *tmem_slot = misc + 0;
    volatile uint32_t *abort_flag = misc + 1;
    uint32_t *mask = misc + 2;  // 2 words: packed tiles visible to some row

    if (tid == 0) {
        mbar_init(bar(B_Q), 1);
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(bar(B_KF + i), 1);
            mbar_init(bar(B_KE + i), 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(bar(B_VF + i), 1);
            mbar_init(bar(B_VE + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_SF + i), 1);
            mbar_init(bar(B_SE + i), 128);
        }
        mbar_init(bar(B_PR), 128);
        mbar_init(bar(B_PF), 1);
        mbar_init(bar(B_DONE), 1);
        *abort_flag = 0u;
        mask[0] = mask[1] = 0u;
        fence_barrier_init();
    }
    if (warp == kTmaWarp && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_kp);
        prefetch_tmap(&tm_vp);
        prefetch_tmap(&tm_kn);
        prefetch_tmap(&tm_vn);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
        tmem_relinquish();
    }
    __syncthreads();

    // ---- rows: visibility intervals and the packed tiles they need
    RowVis vis;
    vis.own_lo = vis.own_hi = vis.par_lo = vis.par_hi = 0;
    bool row_valid = false, row_bad = false;
    int token = 0;
    if (warp < 4) {
        token = tq0 + tid / p.G;
        row_valid = token < b.n_q;
        if (row_valid) {
            if (!row_visibility(p.segs, b.s0, b.s1, b.n_q, token, vis)) {
                row_bad = true;
                vis.own_lo = vis.own_hi = vis.par_lo = vis.par_hi = 0;
            }
            auto mark = [&](int lo, int hi) {
                if (lo >= hi)
                    return;
                for (int t = lo / kBN; t <= (hi - 1) / kBN && t < kMaxPackedTiles; ++t)
                    atomicOr(&mask[t >> 5], 1u << (t & 31));
            };
            mark(vis.own_lo, vis.own_hi);
            mark(vis.par_lo, vis.par_hi);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t m0 = mask[0], m1 = mask[1];
    const int nP = (b.L + kBN - 1) / kBN;
    const int T = nP + __popc(m0) + __popc(m1);
    const int t_begin = (int)(((long long)T * sp) / p.S);
    const int n = (int)(((long long)T * (sp + 1)) / p.S) - t_begin;
    // tile i of this split: prefix tile index, or packed tile index (is_prefix false)
    auto tile_of = [&](int i, bool &is_prefix) -> int {
        const int g = t_begin + i;
        is_prefix = g < nP;
        return is_prefix ? g : nth_set_bit(m0, m1, g - nP);
    };

    const uint32_t tS0 = tmem, tO = tmem + 256u;

    if (warp == kTmaWarp) {
        // =================== TMA producer ===================
        if (lane == 0 && n > 0) {
            int k_cnt[kKStages] = {0, 0, 0}, v_cnt[kVStages] = {0, 0};
            bool ok = true;
            mbar_arrive_expect_tx(bar(B_Q), Lay::kQBytes);
            for (int cb = 0; cb < D / 64; ++cb)
                tma_load_3d(sQ + cb * kBlockBytes, &tm_q, bar(B_Q), cb * 64, hk * p.G, b.q0 + tq0);
            auto issue_k = [&](int j) -> bool {
                const int s = j % kKStages;
                if (j >= kKStages && !wait_bar(bar(B_KE + s), ((j - kKStages) / kKStages) & 1, abort_flag, status))
                    return false;
                if (p.fault == 1 && j == 0)
                    return true;  // injected fault: this tile never arrives
                bool pre;
                const int t = tile_of(j, pre);
                const CUtensorMap *m = pre ? &tm_kp : &tm_kn;
                const int row = pre ? b.p0 + t * kBN : b.q0 + t * kBN;
                mbar_arrive_expect_tx(bar(B_KF + s), Lay::kKBytes);
                for (int cb = 0; cb < D / 64; ++cb)
                    tma_load_3d(sK + s * Lay::kKBytes + cb * kBlockBytes, m, bar(B_KF + s), cb * 64, hk, row);
                ++k_cnt[s];
                return true;
            };
            auto issue_v = [&](int j) -> bool {
                const int s = j % kVStages;
                if (j >= kVStages && !wait_bar(bar(B_VE + s), ((j - kVStages) / kVStages) & 1, abort_flag, status))
                    return false;
                bool pre;
                const int t = tile_of(j, pre);
                const CUtensorMap *m = pre ? &tm_vp : &tm_vn;
                const int row = pre ? b.p0 + t * kBN : b.q0 + t * kBN;
                mbar_arrive_expect_tx(bar(B_VF + s), Lay::kVBytes);
                for (int cb = 0; cb < D / 64; ++cb)
                    tma_load_3d(sV + s * Lay::kVBytes + cb * kBlockBytes, m, bar(B_VF + s), cb * 64, hk, row);
                ++v_cnt[s];
                return true;
            };
            ok = issue_k(0);
            for (int j = 0; j < n && ok; ++j) {
                if (j + 1 < n)
                    ok = issue_k(j + 1);
                if (ok)
                    ok = issue_v(j);
            }
            // every copy this thread started must land before the CTA exits
            wait_drain(bar(B_Q), 0, status);
            for (int s = 0; s < kKStages; ++s)
                if (k_cnt[s] > 0)
                    wait_drain(bar(B_KF + s), (k_cnt[s] - 1) & 1, status);
            for (int s = 0; s < kVStages; ++s)
                if (v_cnt[s] > 0)
                    wait_drain(bar(B_VF + s), (v_cnt[s] - 1) & 1, status);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // =================== MMA issuer ===================
        if (lane == 0 && n > 0) {
            constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, 0, 0);
            constexpr uint32_t idO = idesc_bf16_f32(kBM, D, 0, 1);
            auto pv = [&](int i) -> bool {
                if (!wait_bar(bar(B_PR), i & 1, abort_flag, status))
                    return false;
                const int vs = i % kVStages;
                if (!wait_bar(bar(B_VF + vs), (i / kVStages) & 1, abort_flag, status))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    // A = P (K-major, 64 keys per swizzled block); B = V (MN-major:
                    // 16 keys = two 8-row groups = 2048 bytes; next 64 d-columns +16 KB)
                    const uint64_t a = sdesc_sw128(sP + (kk / 4) * kBlockBytes + (kk % 4) * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(sV + vs * Lay::kVBytes + kk * 2048, kBlockBytes, 1024);
                    mma_bf16_ss(tO, a, bd, idO, (i > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar(B_VE + vs));
                mma_commit(bar(B_PF));
                return true;
            };
            bool ok = wait_bar(bar(B_Q), 0, abort_flag, status);
            for (int j = 0; j < n && ok; ++j) {
                const int ks = j % kKStages;
                ok = wait_bar(bar(B_KF + ks), (j / kKStages) & 1, abort_flag, status);
                if (ok && j >= 2)
                    ok = wait_bar(bar(B_SE + (j & 1)), ((j - 2) / 2) & 1, abort_flag, status);
                if (!ok)
                    break;
                tc_fence_after();
                const uint32_t tS = tS0 + (uint32_t)(j & 1) * 128u;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * kBlockBytes + (kk % 4) * 32;
                    const uint64_t a = sdesc_sw128(sQ + off, 16, 1024);
                    const uint64_t bd = sdesc_sw128(sK + ks * Lay::kKBytes + off, 16, 1024);
                    mma_bf16_ss(tS, a, bd, idS, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(B_SF + (j & 1)));
                mma_commit(bar(B_KE + ks));
                if (j >= 1)
                    ok = pv(j - 1);
            }
            if (ok)
                pv(n - 1);
            // all MMAs this thread issued must finish before TMEM is released
            mma_commit(bar(B_DONE));
            wait_drain(bar(B_DONE), 0, status);
        }
        __syncwarp();
    } else {
        // =================== softmax warps ===================
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const int row = tid;
        float m_ref = -INFINITY, l = 0.f;
        bool aborted = false;
        for (int j = 0; j < n; ++j) {
            bool ok = wait_bar(bar(B_SF + (j & 1)), (j / 2) & 1, abort_flag, status);
            if (!__all_sync(0xffffffffu, ok)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            float s[kBN];
            const uint32_t tS = tS0 + (uint32_t)(j & 1) * 128u + lane_off;
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c)
                tmem_ld32(tS + c * 32, *reinterpret_cast<float(*)[32]>(&s[c * 32]));
            tc_fence_before();
            mbar_arrive(bar(B_SE + (j & 1)));

            bool pre;
            const int t = tile_of(j, pre);
            if (pre) {
                const int valid = b.L - t * kBN;
                if (valid < kBN) {
#pragma unroll
                    for (int c = 0; c < kBN; ++c)
                        if (c >= valid)
                            s[c] = -INFINITY;
                }
            } else {
                const int kb = t * kBN;
#pragma unroll
                for (int c = 0; c < kBN; ++c)
                    if (!vis_has(vis, kb + c))
                        s[c] = -INFINITY;
            }
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < kBN; ++c)
                mx = fmaxf(mx, s[c]);
            mx *= p.scale_log2;
            float factor = 1.f;
            if (mx > m_ref + kRescaleLog2) {
                factor = ex2(m_ref - mx);  // 0 when m_ref = -inf
                m_ref = mx;
            }
            const float msub = (m_ref == -INFINITY) ? 0.f : m_ref;
            float rs = 0.f;
#pragma unroll
            for (int c = 0; c < kBN; ++c) {
                s[c] = ex2(fmaf(s[c], p.scale_log2, -msub));
                rs += s[c];
            }
            l = l * factor + rs;

            if (j >= 1) {  // P buffer free and O final for the previous tile
                ok = wait_bar(bar(B_PF), (j - 1) & 1, abort_flag, status);
                if (!__all_sync(0xffffffffu, ok)) {
                    aborted = true;
                    break;
                }
                if (__any_sync(0xffffffffu, factor != 1.f)) {
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        tmem_ld32(tO + lane_off + c * 32, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] *= factor;
                        tmem_st32(tO + lane_off + c * 32, o);
                    }
                    tmem_wait_st();
                }
            }
            // P row -> shared memory, 128-byte swizzle: chunk ch of row i at (ch ^ (i & 7))
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const float *q8 = &s[cb * 64 + ch * 8];
                    const uint32_t addr = sP + cb * kBlockBytes + row * 128 + (((uint32_t)ch ^ (row & 7)) << 4);
                    st_shared_v4(addr, pack_bf16x2(q8[0], q8[1]), pack_bf16x2(q8[2], q8[3]),
                                 pack_bf16x2(q8[4], q8[5]), pack_bf16x2(q8[6], q8[7]));
                }
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(bar(B_PR));
        }

        // ---- epilogue
        if (!aborted) {
            bool have_o = n > 0;
            if (have_o) {
                const bool ok = wait_bar(bar(B_PF), (n - 1) & 1, abort_flag, status);
                if (!__all_sync(0xffffffffu, ok))
                    aborted = true;
            }
            if (!aborted) {
                tc_fence_after();
                uint16_t *orow = p.out + ((size_t)(b.q0 + token) * p.Hq + hk * p.G + (row % p.G)) * D;
                if (p.S == 1) {
                    const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        tmem_ld32(tO + lane_off + c * 32, o);
                        if (row_valid) {
                            uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                uint4 w;
                                const float sc = row_bad ? 0.f : inv;
                                w.x = pack_bf16x2(o[q4 * 8 + 0] * sc, o[q4 * 8 + 1] * sc);
                                w.y = pack_bf16x2(o[q4 * 8 + 2] * sc, o[q4 * 8 + 3] * sc);
                                w.z = pack_bf16x2(o[q4 * 8 + 4] * sc, o[q4 * 8 + 5] * sc);
                                w.w = pack_bf16x2(o[q4 * 8 + 6] * sc, o[q4 * 8 + 7] * sc);
                                dst[q4] = w;
                            }
                        }
                    }
                } else {
                    // partial of this split, then the per-row ticket
                    const size_t pidx = (size_t)tile_id * p.S + sp;
                    float *opart = reinterpret_cast<float *>(p.ws + p.off_opart) + (pidx * kBM + row) * D;
                    float2 *ml = reinterpret_cast<float2 *>(p.ws + p.off_ml) + pidx * kBM + row;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        if (have_o) {
                            tmem_ld32(tO + lane_off + c * 32, o);
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                o[e] = 0.f;
                        }
                        float4 *dst = reinterpret_cast<float4 *>(opart + c * 32);
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            dst[q4] = make_float4(o[q4 * 4], o[q4 * 4 + 1], o[q4 * 4 + 2], o[q4 * 4 + 3]);
                    }
                    *ml = make_float2(m_ref, l);
                    __threadfence();
                    int *cnt = reinterpret_cast<int *>(p.ws + p.off_cnt) + (size_t)tile_id * kBM + row;
                    const int prev = atomicAdd(cnt, 1);
                    if (prev == p.S - 1) {
                        __threadfence();
                        *cnt = 0;  // ready for the next call
                        float M = -INFINITY;
                        for (int s2 = 0; s2 < p.S; ++s2)
                            M = fmaxf(M, __ldcg(reinterpret_cast<float2 *>(p.ws + p.off_ml) +
                                                ((size_t)tile_id * p.S + s2) * kBM + row)
                                             .x);
                        float Lsum = 0.f;
                        float acc[D];
#pragma unroll
                        for (int e = 0; e < D; ++e)
                            acc[e] = 0.f;
                        if (M != -INFINITY) {
                            for (int s2 = 0; s2 < p.S; ++s2) {
                                const size_t q2 = ((size_t)tile_id * p.S + s2) * kBM + row;
                                const float2 mls = __ldcg(reinterpret_cast<float2 *>(p.ws + p.off_ml) + q2);
                                const float wgt = ex2(mls.x - M);
                                Lsum += mls.y * wgt;
                                const float4 *src = reinterpret_cast<const float4 *>(
                                    reinterpret_cast<float *>(p.ws + p.off_opart) + q2 * D);
#pragma unroll
                                for (int e4 = 0; e4 < D / 4; ++e4) {
                                    const float4 v = __ldcg(src + e4);
                                    acc[e4 * 4 + 0] += wgt * v.x;
                                    acc[e4 * 4 + 1] += wgt * v.y;
                                    acc[e4 * 4 + 2] += wgt * v.z;
                                    acc[e4 * 4 + 3] += wgt * v.w;
                                }
                            }
                        }
                        if (row_valid) {
                            const float sc = (row_bad || !(Lsum > 0.f)) ? 0.f : 1.f / Lsum;
                            uint4 *dst = reinterpret_cast<uint4 *>(orow);
#pragma unroll
                            for (int q8 = 0; q8 < D / 8; ++q8) {
                                uint4 w;
                                w.x = pack_bf16x2(acc[q8 * 8 + 0] * sc, acc[q8 * 8 + 1] * sc);
                                w.y = pack_bf16x2(acc[q8 * 8 + 2] * sc, acc[q8 * 8 + 3] * sc);
                                w.z = pack_bf16x2(acc[q8 * 8 + 4] * sc, acc[q8 * 8 + 5] * sc);
                                w.w = pack_bf16x2(acc[q8 * 8 + 6] * sc, acc[q8 * 8 + 7] * sc);
                                dst[q8] = w;
                            }
                        }
                    }
                }
                if (row_valid && row_bad)
                    record_status(status, D3D_ERR_DEVICE_INPUT);
            }
        }
    }

    // ---- teardown: every role is done (all waits are bounded); release TMEM
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
struct AttnPlan {
    int G, TQ, MT, S;
    long long units;
    size_t off_cnt, off_opart, off_ml, total;
};

int num_sms()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 152;
    }
    return n;
}

// Split count: minimise (waves of one-CTA-per-SM units) x (tiles per unit +
// a fixed per-unit cost), where the per-unit cost covers the prologue, the
// pipeline fill and, with splits, the merge.
AttnPlan make_plan(int R, int Hq, int Hkv, int d, int max_q, int max_prefix, int nsm)
{
    AttnPlan pl{};
    pl.G = Hq / Hkv;
    pl.TQ = kBM / pl.G;
    pl.MT = (max_q + pl.TQ - 1) / pl.TQ;
    const long long base = (long long)R * Hkv * pl.MT;
    const int tiles = (max_prefix + kBN - 1) / kBN + 2;
    double best = 1e300;
    pl.S = 1;
    for (int S = 1; S <= 32 && S <= tiles; ++S) {
        const double waves = (double)((base * S + nsm - 1) / nsm);
        const double cost = waves * (double)((tiles + S - 1) / S + 2 + (S > 1 ? 1 : 0));
        if (cost < best - 1e-9) {
            best = cost;
            pl.S = S;
        }
    }
    pl.units = base * pl.S;
    size_t o = sizeof(WsHeader);
    pl.off_cnt = o;
    if (pl.S > 1) {
        o = align_up(o + sizeof(int) * (size_t)base * kBM, kWsAlign);
        pl.off_opart = o;
        o = align_up(o + sizeof(float) * (size_t)base * pl.S * kBM * d, kWsAlign);
        pl.off_ml = o;
        o = align_up(o + sizeof(float2) * (size_t)base * pl.S * kBM, kWsAlign);
    } else {
        pl.off_opart = pl.off_ml = o;
    }
    pl.total = o;
    return pl;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        else
            cudaGetLastError();
    });
    return fn;
}

// 3-D map over a [rows, heads, d] bf16 tensor; box = 64 x box_h x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *ptr, int d, int heads, long long rows, int box_h, int box_rows)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_h, (cuuint32_t)box_rows};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int g_fault_mode = 0;

template <int D>
int launch_attn(const CUtensorMap (&maps)[5], const AttnParams &prm, long long units, cudaStream_t stream)
{
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)Layout<D>::alloc);
    });
    if (attr_err != cudaSuccess)
        return D3D_ERR_CUDA;
    attn_tc_kernel<D><<<(unsigned)units, kThreads, Layout<D>::alloc, stream>>>(maps[0], maps[1], maps[2], maps[3],
                                                                               maps[4], prm);
    return cuda_status(cudaGetLastError());
}

}  // namespace
}  // namespace d3d

extern "C" {

size_t d3d_packed_draft_attn_workspace_size(int R, int Hq, int Hkv, int d, int max_q, int max_prefix)
{
    if (R < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || max_q < 0 || max_prefix < 0 || (d != 64 && d != 128) ||
        d3d::kBM % (Hq / Hkv) != 0)
        return 0;
    return d3d::make_plan(R, Hq, Hkv, d, max_q, max_prefix, d3d::num_sms()).total;
}

void d3d_debug_inject_fault(int mode) { d3d::g_fault_mode = mode; }

int d3d_packed_draft_attn(const void *q, const void *k_prefix, const void *v_prefix, const void *k_packed,
                          const void *v_packed, const d3d_segment_t *segs, const int32_t *cu_prefix,
                          const int32_t *cu_q, const int32_t *cu_seg, int R, int Hq, int Hkv, int d, int max_q,
                          int max_prefix, int total_q, int total_prefix, int total_segs, float scale, void *out,
                          void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (R < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || max_q < 0 || max_prefix < 0 || total_q < 0 ||
        total_prefix < 0 || total_segs < 0 || !(scale > 0.f) || !isfinite(scale))
        return D3D_ERR_INVALID_ARG;
    if (d != 64 && d != 128)
        return D3D_ERR_UNSUPPORTED;
    if (d3d::kBM % (Hq / Hkv) != 0 || max_q > d3d::kMaxPackedTiles * d3d::kBN)
        return D3D_ERR_UNSUPPORTED;
    if (R == 0 || max_q == 0)
        return D3D_OK;
    if (!q || !k_packed || !v_packed || !segs || !cu_prefix || !cu_q || !cu_seg || !out ||
        (total_prefix > 0 && (!k_prefix || !v_prefix)) || total_q < 1)
        return D3D_ERR_INVALID_ARG;
    const void *aligned_ptrs[4] = {q, k_packed, v_packed, out};
    for (const void *ptr : aligned_ptrs)
        if (reinterpret_cast<uintptr_t>(ptr) % 16)
            return D3D_ERR_INVALID_ARG;
    if (total_prefix > 0 && (reinterpret_cast<uintptr_t>(k_prefix) % 16 || reinterpret_cast<uintptr_t>(v_prefix) % 16))
        return D3D_ERR_INVALID_ARG;
    const d3d::AttnPlan pl = d3d::make_plan(R, Hq, Hkv, d, max_q, max_prefix, d3d::num_sms());
    if (!d3d::ws_ok(ws, ws_bytes, pl.total))
        return D3D_ERR_WORKSPACE;
    if (pl.units > 0x7fffffffLL)
        return D3D_ERR_UNSUPPORTED;

    CUtensorMap maps[5];
    const bool have_prefix = total_prefix > 0;
    if (!d3d::make_map(&maps[0], q, d, Hq, total_q, pl.G, pl.TQ) ||
        !d3d::make_map(&maps[3], k_packed, d, Hkv, total_q, 1, d3d::kBN) ||
        !d3d::make_map(&maps[4], v_packed, d, Hkv, total_q, 1, d3d::kBN))
        return D3D_ERR_CUDA;
    if (have_prefix) {
        if (!d3d::make_map(&maps[1], k_prefix, d, Hkv, total_prefix, 1, d3d::kBN) ||
            !d3d::make_map(&maps[2], v_prefix, d, Hkv, total_prefix, 1, d3d::kBN))
            return D3D_ERR_CUDA;
    } else {  // no prefix rows anywhere: the prefix maps are never used
        maps[1] = maps[3];
        maps[2] = maps[4];
    }

    d3d::AttnParams prm;
    prm.segs = segs;
    prm.cu_prefix = cu_prefix;
    prm.cu_q = cu_q;
    prm.cu_seg = cu_seg;
    prm.out = static_cast<uint16_t *>(out);
    prm.ws = static_cast<unsigned char *>(ws);
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.G = pl.G;
    prm.TQ = pl.TQ;
    prm.MT = pl.MT;
    prm.S = pl.S;
    prm.max_q = max_q;
    prm.max_prefix = max_prefix;
    prm.total_q = total_q;
    prm.total_prefix = total_prefix;
    prm.total_segs = total_segs;
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.off_cnt = pl.off_cnt;
    prm.off_opart = pl.off_opart;
    prm.off_ml = pl.off_ml;
    prm.fault = d3d::g_fault_mode;
    if (d == 64)
        return d3d::launch_attn<64>(maps, prm, pl.units, stream);
    return d3d::launch_attn<128>(maps, prm, pl.units, stream);
}

}  // extern "C"
