// Packed drafting attention on the 5th-generation tensor cores (sm_103a).
//
// [D3D] "Core method", "Method steps" steps 2 and 4; [DScout] "Background:
// block-diffusion drafter".  See attn_common.cuh for the visibility rule.
//
// Work unit (one CTA): request r, KV head hk, a pair of 128-row query tiles
// and one KV split.  A query tile's 128 rows are (packed token, query head of
// hk's group) pairs, token-major, so one K/V tile serves all G query heads
// of the group and both query tiles of the pair.  A unit's key list is every
// 128-key tile of the request's prefix followed by the packed-key tiles its
// rows can see.  Splits cut the prefix tiles; the last split also takes the
// packed tiles, so every other split knows its tiles without the visibility
// mask and starts loading at once.
//
// Roles (320 threads):
//   warps 0-3 / 4-7  softmax warpgroup of query tile 0 / 1: thread i owns
//              TMEM lane i = row i.  Reads S (one tcgen05.ld of 128 columns),
//              masks it, keeps the running max (rescaling O in TMEM only when
//              the max grows by more than 2^8) and the row sum, and writes P
//              as bf16 pairs back over the first 64 columns of S.
//   warp 8     TMA producer: Q tiles once, then K and V tiles into 3- and
//              2-deep rings (3-D tensor maps, 128-byte swizzle).
//   warp 9     MMA issuer (one thread), owner of TMEM.  Per key tile j it
//              issues PV_0(j), S_0(j+1), PV_1(j), S_1(j+1): O_t += P_t V_j
//              with P read from TMEM, S_t = Q_t K^T into TMEM.  While one
//              warpgroup computes its softmax the tensor core works for the
//              other.  S_t(j+1) overwrites P_t(j) only after PV_t(j), which
//              the tensor core executes first (MMAs of one thread run in
//              issue order), and the commit that signals S_t(j+1) also
//              guarantees PV_t(j) is complete, so O_t is stable for the
//              softmax's rescale.
// TMEM: tile t uses columns [256t, 256t+128) for S/P and [256t+128, +D) for O.
// With several splits, a warpgroup takes a per-tile ticket when it has
// finished its key tiles; all but the last write their partial (O divided by
// its row sum, bf16, row-fastest layout, plus max and sum) to the workspace,
// and the last waits for those stores and merges them with its own O, which
// is still in TMEM.
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
constexpr int kTiles = 2;  // query tiles per CTA
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kSoftmaxThreads = kTiles * 128;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxPackedTiles = 64;  // packed keys per request <= 8192
constexpr float kRescaleLog2 = 8.f;  // rescale O only when the max grows by more than 2^8
constexpr uint32_t kBlockBytes = kBN * 128;  // one 128-row x 128-byte swizzled block (16 KB)
constexpr int kStagedSegs = 80;  // segment rows staged in shared memory (more: searched in global memory)
constexpr int kMergeUnroll = 3;  // other splits' partial loads issued together in the merge
constexpr int kMaxSplits = 32;

// barrier indices
enum {
    B_Q = 0,
    B_KF = 1,                   // kKStages
    B_KE = B_KF + kKStages,     // kKStages
    B_VF = B_KE + kKStages,     // kVStages
    B_VE = B_VF + kVStages,     // kVStages
    B_SF = B_VE + kVStages,     // kTiles: S_t(j) in TMEM
    B_PR = B_SF + kTiles,       // kTiles: P_t(j) in TMEM (128 arrivals)
    B_OD = B_PR + kTiles,       // kTiles: O_t final
    B_TK = B_OD + kTiles,       // kTiles: split ticket of the tile taken
    B_RDY = B_TK + kTiles,      // kTiles: merger saw every other split's partial
    B_MASK = B_RDY + kTiles,    // visibility mask complete (256 arrivals)
    B_DONE = B_MASK + 1,        // every MMA of the CTA complete
    B_COUNT = B_DONE + 1
};

template <int D> struct Layout {
    static constexpr uint32_t kQBytes = kBM * D * 2;
    static constexpr uint32_t kKBytes = kBN * D * 2;
    static constexpr uint32_t kVBytes = kBN * D * 2;
    static constexpr uint32_t q = 0;
    static constexpr uint32_t k = q + kTiles * kQBytes;
    static constexpr uint32_t v = k + kKStages * kKBytes;
    static constexpr uint32_t bars = v + kVStages * kVBytes;
    static constexpr uint32_t misc = bars + B_COUNT * 8;
    static constexpr uint32_t segs = misc + 64;  // staged segment table of the request
    static constexpr uint32_t total = segs + kStagedSegs * sizeof(d3d_segment_t);
    static constexpr uint32_t alloc = total + 1024;  // room to align the base to 1024 bytes
};

struct AttnParams {
    const d3d_segment_t *segs;
    const int32_t *cu_prefix, *cu_q, *cu_seg;
    uint16_t *out;
    unsigned char *ws;
    int Hq, Hkv, G, TQ, MT, MP, S, PK;
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

// Bits [lo, hi) of a 32-bit word, clipped to [0, 32).
__device__ __forceinline__ uint32_t range_bits(int lo, int hi)
{
    lo = max(lo, 0);
    hi = min(hi, 32);
    if (lo >= hi)
        return 0u;
    const uint32_t upto_hi = (hi == 32) ? 0xffffffffu : ((1u << hi) - 1u);
    return upto_hi & ~((1u << lo) - 1u);
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

// First prefix tile of split sp: the prefix tiles are cut as if the packed
// tiles (estimated PK of them) were part of the list, then clamped.
__device__ __forceinline__ int split_prefix_begin(int sp, int S, int nP, int PK)
{
    if (sp >= S)
        return nP;
    const long long b = ((long long)(nP + PK) * sp) / S;
    return (int)(b < nP ? b : nP);
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

    // ---- unit: ((r * Hkv + hk) * MP + mp) * S + sp
    unsigned u = blockIdx.x;
    const int sp = (int)(u % (unsigned)p.S);
    u /= (unsigned)p.S;
    const int mp = (int)(u % (unsigned)p.MP);
    u /= (unsigned)p.MP;
    const int hk = (int)(u % (unsigned)p.Hkv);
    const int r = (int)(u / (unsigned)p.Hkv);
    const unsigned pair_id = blockIdx.x / (unsigned)p.S;  // (r, hk, mp)
    int32_t *status = reinterpret_cast<int32_t *>(p.ws);

    ReqBounds b;
    if (!request_bounds(p.cu_prefix, p.cu_q, p.cu_seg, r, p.max_q, p.max_prefix, p.total_q, p.total_prefix,
                        p.total_segs, b)) {
        if (tid == 0)
            record_status(status, D3D_ERR_DEVICE_INPUT);
        return;
    }
    bool tile_valid[kTiles];
    for (int t = 0; t < kTiles; ++t)
        tile_valid[t] = (2 * mp + t) < p.MT && (2 * mp + t) * p.TQ < b.n_q;
    if (!tile_valid[0])
        return;
    const int ntiles = tile_valid[1] ? 2 : 1;

    // ---- this split's tiles: prefix tiles [pb, pe), then (last split only) packed tiles
    const int nP = (b.L + kBN - 1) / kBN;
    const int pb = split_prefix_begin(sp, p.S, nP, p.PK);
    const int pe = (sp == p.S - 1) ? nP : split_prefix_begin(sp + 1, p.S, nP, p.PK);
    const int n_pre = pe - pb;
    const bool last_split = sp == p.S - 1;

    // ---- shared memory carve-up (1024-byte aligned base for the swizzled tiles)
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (sbase - raw);
    const uint32_t sQ = sbase + Lay::q, sK = sbase + Lay::k, sV = sbase + Lay::v;
    auto bar = [&](int i) -> uint32_t { return sbase + Lay::bars + 8u * (uint32_t)i; };
    uint32_t *misc = reinterpret_cast<uint32_t *>(gbase + Lay::misc);
    volatile uint32_t *tmem_slot = misc + 0;
    volatile uint32_t *abort_flag = misc + 1;
    uint32_t *mask = misc + 2;  // 2 words: packed tiles visible to some row of the pair
    volatile int *ticket = reinterpret_cast<volatile int *>(misc + 4);  // 2 words: split tickets
    volatile int *ready_flag = reinterpret_cast<volatile int *>(misc + 6);  // 2 words: merger may go

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
        for (int t = 0; t < kTiles; ++t) {
            mbar_init(bar(B_SF + t), 1);
            mbar_init(bar(B_PR + t), 128);
            mbar_init(bar(B_OD + t), 1);
        }
        for (int t = 0; t < kTiles; ++t) {
            mbar_init(bar(B_TK + t), 1);
            mbar_init(bar(B_RDY + t), 1);
        }
        mbar_init(bar(B_MASK), kSoftmaxThreads);
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // number of packed tiles of the pair; waits for the mask on first use
    int npk_cache = -1;
    uint32_t mk0 = 0, mk1 = 0;
    auto npk = [&]() -> int {
        if (npk_cache < 0) {
            if (!wait_bar(bar(B_MASK), 0, abort_flag, status))
                return -1;
            mk0 = *(volatile uint32_t *)&mask[0];
            mk1 = *(volatile uint32_t *)&mask[1];
            npk_cache = __popc(mk0) + __popc(mk1);
        }
        return npk_cache;
    };
    // does tile j of this split exist (-1: gave up waiting)
    auto exists = [&](int j) -> int {
        if (j < n_pre)
            return 1;
        if (!last_split)
            return 0;
        const int c = npk();
        return c < 0 ? -1 : (j - n_pre < c ? 1 : 0);
    };
    // global K/V row and map of tile j (call only when it exists)
    auto tile_row = [&](int j, bool &pre) -> int {
        pre = j < n_pre;
        return pre ? b.p0 + (pb + j) * kBN : b.q0 + nth_set_bit(mk0, mk1, j - n_pre) * kBN;
    };

    if (warp == kTmaWarp) {
        // =================== TMA producer ===================
        if (lane == 0) {
            int k_cnt[kKStages] = {0, 0, 0}, v_cnt[kVStages] = {0, 0};
            mbar_arrive_expect_tx(bar(B_Q), Lay::kQBytes * ntiles);
            for (int t = 0; t < ntiles; ++t)
                for (int cb = 0; cb < D / 64; ++cb)
                    tma_load_3d(sQ + t * Lay::kQBytes + cb * kBlockBytes, &tm_q, bar(B_Q), cb * 64, hk * p.G,
                                b.q0 + (2 * mp + t) * p.TQ);
            auto issue = [&](int j, bool is_k) -> bool {
                const int ns = is_k ? kKStages : kVStages;
                const int s = j % ns;
                const int empty = is_k ? B_KE : B_VE, full = is_k ? B_KF : B_VF;
                if (j >= ns && !wait_bar(bar(empty + s), ((j - ns) / ns) & 1, abort_flag, status))
                    return false;
                if (p.fault == 1 && is_k && j == 0)
                    return true;  // injected fault: this tile never arrives
                bool pre;
                const int row = tile_row(j, pre);
                const CUtensorMap *m = is_k ? (pre ? &tm_kp : &tm_kn) : (pre ? &tm_vp : &tm_vn);
                const uint32_t dst = (is_k ? sK : sV) + s * Lay::kKBytes;
                mbar_arrive_expect_tx(bar(full + s), Lay::kKBytes);
                for (int cb = 0; cb < D / 64; ++cb)
                    tma_load_3d(dst + cb * kBlockBytes, m, bar(full + s), cb * 64, hk, row);
                ++(is_k ? k_cnt[s] : v_cnt[s]);
                return true;
            };
            int more = exists(0);
            bool ok = more >= 0;
            if (more == 1)
                ok = issue(0, true);
            for (int j = 0; ok && more == 1; ++j) {
                const int next = exists(j + 1);
                if (next < 0)
                    break;
                if (next == 1)
                    ok = issue(j + 1, true);
                if (ok)
                    ok = issue(j, false);
                more = next;
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
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, 0, 0);
            constexpr uint32_t idO = idesc_bf16_f32(kBM, D, 0, 1);
            auto issue_s = [&](int t, int j) {
                const int ks = j % kKStages;
                const uint32_t tS = tmem + (uint32_t)t * 256u;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * kBlockBytes + (kk % 4) * 32;
                    const uint64_t a = sdesc_sw128(sQ + t * Lay::kQBytes + off, 16, 1024);
                    const uint64_t bd = sdesc_sw128(sK + ks * Lay::kKBytes + off, 16, 1024);
                    mma_bf16_ss(tS, a, bd, idS, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(B_SF + t));
            };
            auto issue_pv = [&](int t, int j) {
                const int vs = j % kVStages;
                const uint32_t tP = tmem + (uint32_t)t * 256u, tO = tP + 128u;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    // A = P_t in TMEM (8 columns of bf16 pairs per 16 keys); B = V
                    // MN-major: 16 keys = two 8-row groups = 2048 bytes, the next 64
                    // head-dim columns are 16 KB further
                    const uint64_t bd = sdesc_sw128(sV + vs * Lay::kVBytes + kk * 2048, kBlockBytes, 1024);
                    mma_bf16_ts(tO, tP + kk * 8, bd, idO, (j > 0 || kk > 0) ? 1u : 0u);
                }
            };
            int more = exists(0);
            bool ok = more >= 0 && wait_bar(bar(B_Q), 0, abort_flag, status);
            if (ok && more == 1) {
                ok = wait_bar(bar(B_KF), 0, abort_flag, status);
                if (ok) {
                    tc_fence_after();
                    for (int t = 0; t < ntiles; ++t)
                        issue_s(t, 0);
                    mma_commit(bar(B_KE));
                }
            }
            for (int j = 0; ok && more == 1; ++j) {
                const int next = exists(j + 1);
                if (next < 0)
                    break;
                ok = wait_bar(bar(B_VF + j % kVStages), (j / kVStages) & 1, abort_flag, status);
                if (ok && next == 1)
                    ok = wait_bar(bar(B_KF + (j + 1) % kKStages), ((j + 1) / kKStages) & 1, abort_flag, status);
                for (int t = 0; ok && t < ntiles; ++t) {
                    ok = wait_bar(bar(B_PR + t), j & 1, abort_flag, status);
                    if (!ok)
                        break;
                    tc_fence_after();
                    issue_pv(t, j);
                    if (next == 1)
                        issue_s(t, j + 1);
                    else
                        mma_commit(bar(B_OD + t));
                }
                if (!ok)
                    break;
                mma_commit(bar(B_VE + j % kVStages));
                if (next == 1)
                    mma_commit(bar(B_KE + (j + 1) % kKStages));
                more = next;
            }
            // all MMAs this thread issued must finish before TMEM is released
            mma_commit(bar(B_DONE));
            wait_drain(bar(B_DONE), 0, status);
        }
        __syncwarp();
    } else {
        // =================== softmax warpgroups ===================
        const int t = warp >> 2;  // query tile of this warpgroup
        const int row = tid & 127;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + (uint32_t)t * 256u + lane_off, tO = tS + 128u;
        const int token = (2 * mp + t) * p.TQ + row / p.G;
        const bool row_valid = tile_valid[t] && token < b.n_q;
        bool row_bad = false;
        RowVis vis;
        vis.own_lo = vis.own_hi = vis.par_lo = vis.par_hi = 0;
        // only the last split visits packed keys; it searches a shared-memory copy of
        // the request's segment table when the table is small enough
        const d3d_segment_t *seg_base = p.segs;
        int seg_lo = b.s0, seg_hi = b.s1;
        const int n_seg = b.s1 - b.s0;
        if (last_split && n_seg <= kStagedSegs) {
            d3d_segment_t *staged = reinterpret_cast<d3d_segment_t *>(gbase + Lay::segs);
            const int32_t *src = reinterpret_cast<const int32_t *>(p.segs + b.s0);
            int32_t *dst = reinterpret_cast<int32_t *>(staged);
            for (int i = tid; i < n_seg * 5; i += kSoftmaxThreads)
                dst[i] = src[i];
            asm volatile("bar.sync 1, %0;" ::"n"(kSoftmaxThreads) : "memory");
            seg_base = staged;
            seg_lo = 0;
            seg_hi = n_seg;
        }
        if (row_valid && last_split) {
            if (!row_visibility(seg_base, seg_lo, seg_hi, b.n_q, token, vis)) {
                row_bad = true;
                vis.own_lo = vis.own_hi = vis.par_lo = vis.par_hi = 0;
            }
            auto mark = [&](int lo, int hi) {
                if (lo >= hi)
                    return;
                for (int k = lo / kBN; k <= (hi - 1) / kBN && k < kMaxPackedTiles; ++k)
                    atomicOr(&mask[k >> 5], 1u << (k & 31));
            };
            mark(vis.own_lo, vis.own_hi);
            mark(vis.par_lo, vis.par_hi);
        }
        mbar_arrive(bar(B_MASK));

        // split ticket of this query tile, taken before the last key tile so the
        // atomic's round trip overlaps that tile's work
        const size_t tile_id = (size_t)pair_id * kTiles + t;
        const size_t n_tiles = (size_t)(gridDim.x / p.S) * kTiles;
        int *tk_cnt = reinterpret_cast<int *>(p.ws + p.off_cnt) + tile_id;
        int *wr_cnt = reinterpret_cast<int *>(p.ws + p.off_cnt) + n_tiles + tile_id;
        int my_ticket = -1;
        float m_ref = -INFINITY, l = 0.f;
        bool aborted = false;
        int n_done = 0;
        if (tile_valid[t]) {
            for (int j = 0;; ++j) {
                const int ex = exists(j);
                if (!__all_sync(0xffffffffu, ex >= 0)) {
                    aborted = true;
                    break;
                }
                if (ex == 0)
                    break;
                if (p.S > 1 && row == 0 && my_ticket < 0 && exists(j + 1) == 0)
                    my_ticket = atomicAdd(tk_cnt, 1);
                bool ok = wait_bar(bar(B_SF + t), j & 1, abort_flag, status);
                if (!__all_sync(0xffffffffu, ok)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
                float s[kBN];
                tmem_ld128(tS, s);
                bool pre;
                const int krow = tile_row(j, pre);
                if (pre) {
                    const int valid = b.L - (pb + j) * kBN;
                    if (valid < kBN) {
#pragma unroll
                        for (int c = 0; c < kBN; ++c)
                            if (c >= valid)
                                s[c] = -INFINITY;
                    }
                } else {
                    // this row's visible keys in the tile as a 128-bit mask: two
                    // half-open intervals cut into four 32-key words
                    const int kb = krow - b.q0;
                    uint32_t wbits[4];
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const int base = kb + 32 * w;
                        wbits[w] = range_bits(vis.own_lo - base, vis.own_hi - base) |
                                   range_bits(vis.par_lo - base, vis.par_hi - base);
                    }
#pragma unroll
                    for (int c = 0; c < kBN; ++c)
                        s[c] = ((wbits[c >> 5] >> (c & 31)) & 1u) ? s[c] : -INFINITY;
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
                uint32_t pk[kBN / 2];
#pragma unroll
                for (int c = 0; c < kBN / 2; ++c) {
                    const float e0 = ex2(fmaf(s[2 * c], p.scale_log2, -msub));
                    const float e1 = ex2(fmaf(s[2 * c + 1], p.scale_log2, -msub));
                    rs += e0 + e1;
                    pk[c] = pack_bf16x2(e0, e1);
                }
                l = l * factor + rs;
                // O_t is stable here: PV_t(j-1) completed before S_t(j) was signalled
                if (j > 0 && __any_sync(0xffffffffu, factor != 1.f)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        tmem_ld32(tO + c * 32, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] *= factor;
                        tmem_st32(tO + c * 32, o);
                    }
                }
                tmem_st64(tS, pk);  // P over the first 64 columns of S
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(B_PR + t));
                n_done = j + 1;
            }
        }

        // ---- epilogue
        if (tile_valid[t] && !aborted) {
            const bool have_o = n_done > 0;
            if (have_o) {
                const bool ok = wait_bar(bar(B_OD + t), 0, abort_flag, status);
                if (!__all_sync(0xffffffffu, ok))
                    aborted = true;
            }
            if (!aborted) {
                tc_fence_after();
                uint16_t *orow = p.out + ((size_t)(b.q0 + token) * p.Hq + hk * p.G + (row % p.G)) * D;
                if (p.S == 1) {
                    const float inv = (l > 0.f && !row_bad) ? 1.f / l : 0.f;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        tmem_ld32(tO + c * 32, o);
                        if (row_valid) {
                            uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                uint4 w;
                                w.x = pack_bf16x2(o[q4 * 8 + 0] * inv, o[q4 * 8 + 1] * inv);
                                w.y = pack_bf16x2(o[q4 * 8 + 2] * inv, o[q4 * 8 + 3] * inv);
                                w.z = pack_bf16x2(o[q4 * 8 + 4] * inv, o[q4 * 8 + 5] * inv);
                                w.w = pack_bf16x2(o[q4 * 8 + 6] * inv, o[q4 * 8 + 7] * inv);
                                dst[q4] = w;
                            }
                        }
                    }
                } else {
                    // Ticket first: the warpgroup that finishes this query tile's key
                    // tiles last merges; the others write their partial normalised by
                    // its row sum, as bf16 (16-byte chunk c8 of row i of partial q at
                    // ((q * D/8 + c8) * 128 + i)), with (max, sum) beside it.
                    uint4 *opart = reinterpret_cast<uint4 *>(p.ws + p.off_opart);
                    float2 *mls = reinterpret_cast<float2 *>(p.ws + p.off_ml);
                    if (row == 0) {
                        ticket[t] = (my_ticket >= 0) ? my_ticket : atomicAdd(tk_cnt, 1);
                        mbar_arrive(bar(B_TK + t));
                    }
                    const bool got = wait_bar(bar(B_TK + t), 0, abort_flag, status);
                    if (__all_sync(0xffffffffu, got)) {
                        const bool is_last = ticket[t] == p.S - 1;
                        if (!is_last) {
                            const size_t pidx = tile_id * p.S + sp;
                            const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
                            for (int c = 0; c < D / 32; ++c) {
                                float o[32];
                                if (have_o) {
                                    tmem_ld32(tO + c * 32, o);
                                } else {
#pragma unroll
                                    for (int e = 0; e < 32; ++e)
                                        o[e] = 0.f;
                                }
#pragma unroll
                                for (int q4 = 0; q4 < 4; ++q4) {
                                    uint4 w;
                                    w.x = pack_bf16x2(o[q4 * 8 + 0] * inv, o[q4 * 8 + 1] * inv);
                                    w.y = pack_bf16x2(o[q4 * 8 + 2] * inv, o[q4 * 8 + 3] * inv);
                                    w.z = pack_bf16x2(o[q4 * 8 + 4] * inv, o[q4 * 8 + 5] * inv);
                                    w.w = pack_bf16x2(o[q4 * 8 + 6] * inv, o[q4 * 8 + 7] * inv);
                                    opart[(pidx * (D / 8) + c * 4 + q4) * kBM + row] = w;
                                }
                            }
                            // a negative sum marks a row whose descriptors failed the
                            // check (only the last split, which visits packed keys, checks)
                            mls[pidx * kBM + row] = make_float2(m_ref, row_bad ? -1.f : l);
                            __threadfence();
                            __syncwarp();
                            if (lane == 0)
                                atomicAdd(wr_cnt, 32);
                        } else {
                            // every other split holds a ticket, so it is past its key
                            // tiles and only has stores left: wait (bounded) for them
                            if (row == 0) {
                                // one poller; it also resets both counters for the next call
                                const int need = (p.S - 1) * kBM;
                                const uint64_t t0 = global_ns();
                                int ok_all = 1;
                                while (*reinterpret_cast<volatile int *>(wr_cnt) < need) {
                                    if (global_ns() - t0 > kWaitTimeoutNs) {
                                        record_status(status, D3D_ERR_DEVICE_TIMEOUT);
                                        ok_all = 0;
                                        break;
                                    }
                                }
                                if (ok_all) {
                                    *wr_cnt = 0;
                                    *tk_cnt = 0;
                                }
                                ready_flag[t] = ok_all;
                                mbar_arrive(bar(B_RDY + t));
                            }
                            const bool rel = wait_bar(bar(B_RDY + t), 0, abort_flag, status);
                            const int ready = __all_sync(0xffffffffu, rel) ? ready_flag[t] : 0;
                            if (ready) {
                                __threadfence();
                                float2 mlv[kMaxSplits];
                                float M = m_ref;
                                for (int s2 = 0; s2 < p.S; ++s2) {
                                    mlv[s2] = (s2 == sp) ? make_float2(m_ref, l)
                                                         : __ldcg(mls + (tile_id * p.S + s2) * kBM + row);
                                    M = fmaxf(M, mlv[s2].x);
                                }
                                float Lsum = 0.f;
                                bool bad = row_bad;
                                for (int s2 = 0; s2 < p.S; ++s2) {
                                    bad = bad || mlv[s2].y < 0.f;
                                    const float w = (M == -INFINITY) ? 0.f : ex2(mlv[s2].x - M);
                                    Lsum += w * fmaxf(mlv[s2].y, 0.f);
                                    // own O is unnormalised; the others were divided by their sum
                                    mlv[s2].x = (s2 == sp) ? w : w * fmaxf(mlv[s2].y, 0.f);
                                }
                                const float sc = (bad || !(Lsum > 0.f)) ? 0.f : 1.f / Lsum;
                                const uint4 *pa = nullptr, *pb = nullptr;  // the other splits (fast path)
                                float wa = 0.f, wb = 0.f;
                                if (p.S <= 3) {
                                    // the other splits: (1, 2), (0, 2) or (0, 1); only one when S = 2
                                    const int oa = (sp == 0) ? 1 : 0, ob = (p.S < 3) ? -1 : ((sp == 2) ? 1 : 2);
                                    pa = opart + ((tile_id * p.S + oa) * (D / 8)) * kBM + row;
                                    wa = mlv[oa].x;
                                    if (ob >= 0) {
                                        pb = opart + ((tile_id * p.S + ob) * (D / 8)) * kBM + row;
                                        wb = mlv[ob].x;
                                    }
                                }
                                if (p.S <= 3 && sc != 0.f) {
                                    // software-pipelined: chunk c+1's loads are in flight while
                                    // chunk c is accumulated
                                    uint4 cur[2][4], nxt[2][4];
#pragma unroll
                                    for (int q4 = 0; q4 < 4; ++q4) {
                                        cur[0][q4] = __ldcg(pa + (size_t)q4 * kBM);
                                        cur[1][q4] = pb ? __ldcg(pb + (size_t)q4 * kBM) : make_uint4(0, 0, 0, 0);
                                    }
#pragma unroll
                                    for (int c = 0; c < D / 32; ++c) {
                                        if (c + 1 < D / 32) {
#pragma unroll
                                            for (int q4 = 0; q4 < 4; ++q4) {
                                                nxt[0][q4] = __ldcg(pa + (size_t)((c + 1) * 4 + q4) * kBM);
                                                nxt[1][q4] = pb ? __ldcg(pb + (size_t)((c + 1) * 4 + q4) * kBM)
                                                                : make_uint4(0, 0, 0, 0);
                                            }
                                        }
                                        float acc[32];
                                        if (have_o) {
                                            tmem_ld32(tO + c * 32, acc);
                                        } else {
#pragma unroll
                                            for (int e = 0; e < 32; ++e)
                                                acc[e] = 0.f;
                                        }
                                        const float wown = mlv[sp].x;
#pragma unroll
                                        for (int q4 = 0; q4 < 4; ++q4) {
                                            const uint32_t da[4] = {cur[0][q4].x, cur[0][q4].y, cur[0][q4].z, cur[0][q4].w};
                                            const uint32_t db[4] = {cur[1][q4].x, cur[1][q4].y, cur[1][q4].z, cur[1][q4].w};
#pragma unroll
                                            for (int e = 0; e < 4; ++e) {
                                                float &lo = acc[q4 * 8 + 2 * e], &hi = acc[q4 * 8 + 2 * e + 1];
                                                lo = lo * wown + wa * __uint_as_float(da[e] << 16) +
                                                     wb * __uint_as_float(db[e] << 16);
                                                hi = hi * wown + wa * __uint_as_float(da[e] & 0xffff0000u) +
                                                     wb * __uint_as_float(db[e] & 0xffff0000u);
                                            }
                                        }
                                        if (row_valid) {
                                            uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                                            for (int q4 = 0; q4 < 4; ++q4) {
                                                uint4 w;
                                                w.x = pack_bf16x2(acc[q4 * 8 + 0] * sc, acc[q4 * 8 + 1] * sc);
                                                w.y = pack_bf16x2(acc[q4 * 8 + 2] * sc, acc[q4 * 8 + 3] * sc);
                                                w.z = pack_bf16x2(acc[q4 * 8 + 4] * sc, acc[q4 * 8 + 5] * sc);
                                                w.w = pack_bf16x2(acc[q4 * 8 + 6] * sc, acc[q4 * 8 + 7] * sc);
                                                dst[q4] = w;
                                            }
                                        }
#pragma unroll
                                        for (int q4 = 0; q4 < 4; ++q4) {
                                            cur[0][q4] = nxt[0][q4];
                                            cur[1][q4] = nxt[1][q4];
                                        }
                                    }
                                } else
                                {
                                for (int c = 0; c < D / 32; ++c) {
                                    float acc[32];
                                    if (have_o) {
                                        tmem_ld32(tO + c * 32, acc);
                                    } else {
#pragma unroll
                                        for (int e = 0; e < 32; ++e)
                                            acc[e] = 0.f;
                                    }
                                    const float wown = mlv[sp].x;
#pragma unroll
                                    for (int e = 0; e < 32; ++e)
                                        acc[e] *= wown;
                                    for (int s0 = 0; sc != 0.f && s0 < p.S; s0 += kMergeUnroll) {
                                        uint4 v[kMergeUnroll][4];
#pragma unroll
                                        for (int u = 0; u < kMergeUnroll; ++u) {
                                            const int s2 = s0 + u;
                                            if (s2 < p.S && s2 != sp) {
                                                const size_t q2 = tile_id * p.S + s2;
#pragma unroll
                                                for (int q4 = 0; q4 < 4; ++q4)
                                                    v[u][q4] = __ldcg(opart + (q2 * (D / 8) + c * 4 + q4) * kBM + row);
                                            }
                                        }
#pragma unroll
                                        for (int u = 0; u < kMergeUnroll; ++u) {
                                            const int s2 = s0 + u;
                                            if (s2 < p.S && s2 != sp) {
                                                const float wgt = mlv[s2].x;
#pragma unroll
                                                for (int q4 = 0; q4 < 4; ++q4) {
                                                    const uint32_t wd[4] = {v[u][q4].x, v[u][q4].y, v[u][q4].z, v[u][q4].w};
#pragma unroll
                                                    for (int e = 0; e < 4; ++e) {
                                                        acc[q4 * 8 + 2 * e] += wgt * __uint_as_float(wd[e] << 16);
                                                        acc[q4 * 8 + 2 * e + 1] += wgt * __uint_as_float(wd[e] & 0xffff0000u);
                                                    }
                                                }
                                            }
                                        }
                                    }
                                    if (row_valid) {
                                        uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                                        for (int q4 = 0; q4 < 4; ++q4) {
                                            uint4 w;
                                            w.x = pack_bf16x2(acc[q4 * 8 + 0] * sc, acc[q4 * 8 + 1] * sc);
                                            w.y = pack_bf16x2(acc[q4 * 8 + 2] * sc, acc[q4 * 8 + 3] * sc);
                                            w.z = pack_bf16x2(acc[q4 * 8 + 4] * sc, acc[q4 * 8 + 5] * sc);
                                            w.w = pack_bf16x2(acc[q4 * 8 + 6] * sc, acc[q4 * 8 + 7] * sc);
                                            dst[q4] = w;
                                        }
                                    }
                                }
                                }
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
    int G, TQ, MT, MP, S, PK;
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
// a fixed per-unit cost for the prologue and pipeline fill, one more for the
// merge when splitting).
AttnPlan make_plan(int R, int Hq, int Hkv, int d, int max_q, int max_prefix, int nsm)
{
    AttnPlan pl{};
    pl.G = Hq / Hkv;
    pl.TQ = kBM / pl.G;
    pl.MT = (max_q + pl.TQ - 1) / pl.TQ;
    pl.MP = (pl.MT + kTiles - 1) / kTiles;
    pl.PK = (max_q + kBN - 1) / kBN < 2 ? (max_q + kBN - 1) / kBN : 2;
    const long long base = (long long)R * Hkv * pl.MP;
    const int tiles = (max_prefix + kBN - 1) / kBN + pl.PK;
    double best = 1e300;
    pl.S = 1;
    for (int S = 1; S <= kMaxSplits && S <= tiles; ++S) {
        const double waves = (double)((base * S + nsm - 1) / nsm);
        const double cost = waves * (double)((tiles + S - 1) / S + 3 + (S > 1 ? 1 : 0));
        if (cost < best - 1e-9) {
            best = cost;
            pl.S = S;
        }
    }
    pl.units = base * pl.S;
    const size_t rows = (size_t)base * kTiles * kBM;
    size_t o = sizeof(WsHeader);
    pl.off_cnt = o;
    if (pl.S > 1) {
        const size_t tiles_total = (size_t)base * kTiles;
        o = align_up(o + sizeof(int) * 2 * tiles_total, kWsAlign);  // split tickets, rows written
        pl.off_opart = o;
        o = align_up(o + sizeof(uint16_t) * rows * pl.S * d, kWsAlign);  // bf16 partials
        pl.off_ml = o;
        o = align_up(o + sizeof(float2) * rows * pl.S, kWsAlign);
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
    if (!d3d::make_map(&maps[0], q, d, Hq, total_q, pl.G, pl.TQ) ||
        !d3d::make_map(&maps[3], k_packed, d, Hkv, total_q, 1, d3d::kBN) ||
        !d3d::make_map(&maps[4], v_packed, d, Hkv, total_q, 1, d3d::kBN))
        return D3D_ERR_CUDA;
    if (total_prefix > 0) {
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
    prm.MP = pl.MP;
    prm.S = pl.S;
    prm.PK = pl.PK;
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
