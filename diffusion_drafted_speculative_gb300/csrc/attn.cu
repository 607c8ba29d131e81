// Packed drafting attention on the 5th-generation tensor cores (sm_103a).
//
// [D3D] "Core method", "Method steps" steps 2 and 4; [DScout] "Background:
// block-diffusion drafter".  See attn_common.cuh for the visibility rule.
//
// Work unit (one CTA, which holds one SM): request r, KV head hk, one 128-row
// query tile and one key split.  A query tile's 128 rows are (packed token,
// query head of hk's group) pairs, token-major, so one K/V tile serves all G
// query heads of the group.  A unit's key list is every 128-key tile of the request's prefix
// followed by the packed-key tiles its rows can see.  Splits cut the prefix
// tiles; the last split also takes the packed tiles, so every other split
// knows its tiles without the visibility mask and starts loading at once.
//
// Roles (320 threads with two softmax warpgroups; the count kWG is a build
// option, 2 or 4):
//   warps 0..4kWG-1  softmax warpgroups: warpgroup w takes key columns
//              [w*128/kWG, (w+1)*128/kWG) of every key tile; thread i of any
//              warpgroup owns TMEM lane i = query row i.  Per tile: one
//              tcgen05.ld of its S columns, the mask, its part of the row max,
//              published in shared memory (mbarrier, bounded wait) to form the
//              row max, a rescale of its part of O in TMEM only when the max
//              grows by more than 2^8, the exponentials (arguments and sums in
//              packed f32x2 arithmetic), its part of the row sum, and P as
//              bf16 pairs written over the first half of the S buffer.  Once
//              at the start each thread also copies its half of its Q row into
//              TMEM (bf16 pairs, the A operand of S), so the S MMAs read only
//              K from shared memory.
//   warp 4kWG  TMA producer: the Q tile once, then K and V tiles into 3- and
//              2-deep rings (3-D tensor maps, 128-byte swizzle), in the order
//              the tensor core consumes them.
//   warp 4kWG+1  MMA issuer (one thread), owner of TMEM.  S(k) = Q K_k^T (Q from
//              TMEM, K from shared memory) goes to TMEM buffer k % 2; once
//              P(k) is written it issues O += P(k) V_k
//              (P read from TMEM) and S(k+2) into the buffer P(k) came from.
//              The tensor core thus computes PV(k-1) and S(k+1) while the
//              softmax works on tile k; MMAs of one thread run in issue order,
//              so S(k+2) never overwrites P(k) before PV(k) has read it.
// TMEM: S buffers in columns [0, 128) and [128, 256), O in [256, 256 + D),
// Q in [256 + D, 256 + 3D/2).  At the end the parts' row sums add up (every part keeps the same running
// max) and each thread normalises and stores its D/kWG columns of the row.
//
// With S > 1 splits the S CTAs of a query tile run as one thread-block
// cluster.  Each CTA writes its combined partial (O divided by its row sum,
// bf16) into its own shared memory, in the K ring that nothing reads any
// more, with the rows' (max, sum).  After a cluster barrier every CTA
// combines its share of the head-dim columns (split sp takes a contiguous
// range of 8-column units) from all splits through distributed shared
// memory, in a fixed order, and stores it; a second cluster barrier keeps
// every CTA resident until its shared memory has been read.  No global
// scratch is used.
//
// The same body, instantiated with kDuo, is the CTA-pair kernel
// (attn_duo_kernel): query tiles 2j and 2j+1 run as a cluster of two whose
// even CTA issues cta_group::2 MMAs for both (each CTA's 128 rows in its own
// TMEM, half of every K and V tile in each CTA's shared memory); the odd
// CTA's softmax warps arrive on the even CTA's barriers and the MMA commits
// arrive on both.  It is selected only through d3d_debug_force_attn_kernel
// (measured slower than the one-tile kernel on every workload here).
// The two-tile kernel (two query tiles per CTA) follows the one-tile body.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <mutex>

#include "attn_common.cuh"
#include "sm100_ptx.cuh"
#include "verify_body.cuh"

namespace d3d {
namespace {

using namespace sm100;

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per KV tile
#ifndef D3D_ATTN_WG
#define D3D_ATTN_WG 2
#endif
static_assert(D3D_ATTN_WG == 2 || D3D_ATTN_WG == 4, "two or four softmax warpgroups");
constexpr int kWG = D3D_ATTN_WG;  // softmax warpgroups: each takes 1/kWG of every key tile's columns
constexpr int kPart = kBN / kWG;  // keys per softmax thread and tile (64 with two warpgroups)
constexpr int kKStages = 3;
constexpr int kVStages = 2;
// a CTA pair's stages hold half tiles: deeper rings in the same room
constexpr int kDuoKStages = 4;
constexpr int kDuoVStages = 3;
constexpr int kMaxKStages = kDuoKStages;
constexpr int kMaxVStages = kDuoVStages;
constexpr int kSoftmaxThreads = kWG * 128;
constexpr int kTmaWarp = kWG * 4;
constexpr int kMmaWarp = kTmaWarp + 1;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxPackedTiles = 64;  // packed keys per request <= 8192
constexpr float kRescaleLog2 = 8.f;  // rescale O only when the max grows by more than 2^8
constexpr uint32_t kBlockBytes = kBN * 128;  // one 128-row x 128-byte swizzled block (16 KB)
constexpr int kStagedSegs = 80;  // segment rows staged in shared memory (more: searched in global memory)
constexpr int kMaxSplits = 8;  // key splits of a query tile: one thread-block cluster

// barrier indices
enum {
    B_Q = 0,
    B_KF = 1,                   // K stages
    B_KE = B_KF + kMaxKStages,  // K stages
    B_VF = B_KE + kMaxKStages,  // V stages
    B_VE = B_VF + kMaxVStages,  // V stages
    B_SF = B_VE + kMaxVStages,  // 2: S(k) in TMEM buffer k % 2
    B_PR = B_SF + 2,            // 2: P(k) in TMEM buffer k % 2 (one arrival per softmax warp)
    B_MX = B_PR + 2,            // 2: both halves' row maxima of tile k published (one per softmax warp)
    B_OW = B_MX + 2,            // one completion per PV (O written)
    B_MASK = B_OW + 1,          // visibility mask complete (256 arrivals)
    B_DONE = B_MASK + 1,        // every MMA of the CTA complete
    B_QT = B_DONE + 1,          // Q copied into TMEM (one arrival per softmax warp)
    B_COUNT = B_QT + 1
};

// kDuo: one CTA of a pair (attn_duo_kernel), whose K stages hold half of a
// tile's keys and V stages half of its head-dim columns
template <int D, bool kDuo = false> struct Layout {
    static constexpr int kKS = kDuo ? kDuoKStages : kKStages;
    static constexpr int kVS = kDuo ? kDuoVStages : kVStages;
    static constexpr uint32_t kQBytes = kBM * D * 2;
    static constexpr uint32_t kKRows = kDuo ? kBN / 2 : kBN;  // keys of a K stage
    static constexpr uint32_t kKBlock = kKRows * 128;         // one 64-column block of a K stage
    static constexpr uint32_t kKBytes = kKRows * D * 2;
    static constexpr uint32_t kVBytes = kBN * (kDuo ? D / 2 : D) * 2;
    static constexpr uint32_t q = 0;
    static constexpr uint32_t k = q + kQBytes;
    static constexpr uint32_t v = k + kKS * kKBytes;
    static constexpr uint32_t bars = v + kVS * kVBytes;
    static constexpr uint32_t misc = bars + B_COUNT * 8;
    static constexpr uint32_t mx = misc + 64;  // [2 buffers][kWG][kBM] row maxima of a tile's column parts
    static constexpr uint32_t ml = q;  // per warpgroup and row: (max, sum, tiles done), over Q after the last MMA
    static constexpr uint32_t segs = mx + 2 * kWG * kBM * 4;  // staged segment table of the request
    static constexpr uint32_t total = segs + kStagedSegs * sizeof(d3d_segment_t);
    static constexpr uint32_t alloc = total + 1024;  // room to align the base to 1024 bytes
};

struct AttnParams {
    const d3d_segment_t *segs;
    const int32_t *cu_prefix, *cu_q, *cu_seg;
    uint16_t *out;
    unsigned char *ws;
    int Hq, Hkv, G, TQ, MT, S, PK;
    int max_q, max_prefix, total_q, total_prefix, total_segs;
    float scale_log2;
    int fault;
    // one request whose offsets the contract fixes (cu_*[0] = 0, cu_*[1] = the
    // totals, within max_q / max_prefix): the kernel takes them from here and
    // checks the device arrays against them in its epilogue
    int one_request;
    // the launch may start before the kernel ahead of it has finished, whose
    // output it may read: it waits for that kernel before its first read
    int wait_first;
};

// The bounds of request r: for a single request the documented offsets
// (known on the host), otherwise from the device arrays (ok = false when they
// lie).  For a single request `ok` only says the host values are usable; the
// arrays are compared with them later (one_request_matches).
__device__ __forceinline__ bool kernel_bounds(const AttnParams &p, const ReqRaw &braw, ReqBounds &b)
{
    if (p.one_request) {
        b.q0 = 0, b.n_q = p.total_q, b.p0 = 0, b.L = p.total_prefix, b.s0 = 0, b.s1 = p.total_segs;
        return true;
    }
    return check_bounds(braw, p.max_q, p.max_prefix, p.total_q, p.total_prefix, p.total_segs, b);
}
__device__ __forceinline__ bool one_request_matches(const AttnParams &p, const ReqRaw &w)
{
    return w.q0 == 0 && w.q1 == p.total_q && w.p0 == 0 && w.p1 == p.total_prefix && w.s0 == 0 &&
           w.s1 == p.total_segs;
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction (sm_100 family); a NaN operand is ignored
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
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
    while (!mbar_try_wait_sleep(bar, parity)) {
        if (global_ns() - t0 > kWaitTimeoutNs) {
            record_status(status, D3D_ERR_DEVICE_TIMEOUT);
            return;
        }
    }
}

// Work of the last key split beyond its prefix tiles, in prefix tiles: the
// packed tiles (estimated PK of them) cost about two each (their masks), and
// the rows' visibility from the segment table about one more.
__host__ __device__ __forceinline__ int packed_tile_weight(int PK) { return PK > 0 ? 2 * PK + 1 : 0; }

// First prefix tile of split sp: the prefix tiles are cut as if the last
// split's extra work were part of the list, then clamped.
__device__ __forceinline__ int split_prefix_begin(int sp, int S, int nP, int PK)
{
    if (sp >= S)
        return nP;
    const long long b = ((long long)(nP + packed_tile_weight(PK)) * sp) / S;
    return (int)(b < nP ? b : nP);
}

// Shared-memory exchange area of the split combine (in the K ring, free once
// every MMA is done): the CTA's partial O normalised by its row sum as bf16,
// 16-byte unit u (head-dim columns 8u..8u+7) of row i at (u * 128 + i) * 16,
// then (max, sum) per row.
template <int D> struct Xchg {
    static constexpr uint32_t kPartBytes = (D / 8) * kBM * 16;
    static __device__ uint32_t part(uint32_t sK) { return sK; }
    static __device__ uint32_t ml(uint32_t sK) { return sK + kPartBytes; }
};
static_assert(Xchg<128>::kPartBytes + kBM * 8 <= kKStages * kBN * 128 * 2, "exchange fits the K ring");
static_assert(Xchg<64>::kPartBytes + kBM * 8 <= kKStages * kBN * 64 * 2, "exchange fits the K ring");

__device__ __forceinline__ uint4 pack8(const float *a, float sc)
{
    uint4 w;
    w.x = pack_bf16x2(a[0] * sc, a[1] * sc);
    w.y = pack_bf16x2(a[2] * sc, a[3] * sc);
    w.z = pack_bf16x2(a[4] * sc, a[5] * sc);
    w.w = pack_bf16x2(a[6] * sc, a[7] * sc);
    return w;
}

// Output staging.  A thread owns a row of the output tile, so storing its
// 16-byte units straight to global memory makes every warp store touch 32
// rows 256 or 512 bytes apart.  Instead the units go to shared memory first,
// in the 128-byte-swizzled layout of a query tile (column block c / 8 of unit
// c, row i at 128 i within it, unit position (c mod 8) xor (i mod 8): the 8
// threads of a quarter-warp writing one unit of 8 consecutive rows, or reading
// 8 consecutive units of one row, hit distinct banks), and after a barrier of
// the writing threads consecutive threads copy consecutive units of a row out,
// so each warp stores whole runs of the rows it covers.
__device__ __forceinline__ uint32_t stage_addr(uint32_t tile, int i, int c)
{
    return tile + (uint32_t)(c >> 3) * kBlockBytes + (uint32_t)i * 128u + ((uint32_t)((c & 7) ^ (i & 7)) << 4);
}

// Units [c0, c1) of staged rows [0, n_rows) to global memory by the n_thr
// threads (index it) that staged them; row i lives in staged tile i / 128 (at
// stage + (i / 128) * tile_bytes) and goes to row_ptr(i), or nowhere when that
// is null.
template <typename RowPtr>
__device__ __forceinline__ void store_staged(uint32_t stage, uint32_t tile_bytes, int n_rows, int c0, int c1, int it,
                                             int n_thr, RowPtr row_ptr)
{
    const int w = c1 - c0;
    if (w <= 0)
        return;
    for (int idx = it; idx < n_rows * w; idx += n_thr) {
        const int i = idx / w, c = c0 + idx % w;
        uint16_t *dst = row_ptr(i);
        if (dst != nullptr)
            *reinterpret_cast<uint4 *>(dst + 8 * c) =
                smem_ld_v4(stage_addr(stage + (uint32_t)(i >> 7) * tile_bytes, i & 127, c));
    }
}

// The output units of the S CTAs of a cluster: CTA sp takes the contiguous
// range [sp * U / S, (sp + 1) * U / S) of the U = D / 8 units of every row.
__device__ __forceinline__ int split_unit_begin(int sp, int S, int units) { return sp * units / S; }

// Split combine of one query row over the S CTAs of the cluster: the
// (max, sum) of every split and this thread's units of the CTA's range
// (u = u0 + kWG*k + w: its warpgroups take turns), read through distributed
// shared memory in split order; stages those output units at `stage`.
template <int D, int S>
__device__ __forceinline__ void cluster_merge(int sp, int w, uint32_t part, uint32_t ml, int row, uint32_t stage)
{
    constexpr int kUnits = D / 8;
    constexpr int kMine = ((kUnits + S - 1) / S + kWG - 1) / kWG;
    const int u0 = split_unit_begin(sp, S, kUnits), u1 = split_unit_begin(sp + 1, S, kUnits);
    float ms[S], ls[S];
#pragma unroll
    for (int s2 = 0; s2 < S; ++s2) {
        const float2 v = dsmem_ld_f2(dsmem_addr(ml + (uint32_t)row * 8u, (uint32_t)s2));
        ms[s2] = v.x;
        ls[s2] = v.y;
    }
    float M = -INFINITY;
    bool bad = false;
#pragma unroll
    for (int s2 = 0; s2 < S; ++s2) {
        M = fmaxf(M, ms[s2]);
        bad = bad || ls[s2] < 0.f;
    }
    float coef[S], Lsum = 0.f;
#pragma unroll
    for (int s2 = 0; s2 < S; ++s2) {
        const float wt = (M == -INFINITY) ? 0.f : ex2(ms[s2] - M);
        coef[s2] = wt * fmaxf(ls[s2], 0.f);  // every partial was divided by its own sum
        Lsum += coef[s2];
    }
    const float sc = (bad || !(Lsum > 0.f)) ? 0.f : 1.f / Lsum;
    uint4 rem[kMine][S];
#pragma unroll
    for (int k = 0; k < kMine; ++k) {
        const int u = u0 + kWG * k + w;
#pragma unroll
        for (int s2 = 0; s2 < S; ++s2) {
            rem[k][s2] = make_uint4(0, 0, 0, 0);
            if (u < u1)
                rem[k][s2] = dsmem_ld_v4(dsmem_addr(part + ((uint32_t)u * kBM + (uint32_t)row) * 16u, (uint32_t)s2));
        }
    }
#pragma unroll
    for (int k = 0; k < kMine; ++k) {
        const int u = u0 + kWG * k + w;
        if (u >= u1)
            break;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s2 = 0; s2 < S; ++s2) {
            const float cw = coef[s2];
            const uint32_t wd[4] = {rem[k][s2].x, rem[k][s2].y, rem[k][s2].z, rem[k][s2].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[2 * e] += cw * __uint_as_float(wd[e] << 16);
                acc[2 * e + 1] += cw * __uint_as_float(wd[e] & 0xffff0000u);
            }
        }
        smem_st_v4(stage_addr(stage, row, u), pack8(acc, sc));
    }
}

// The attention of work unit `unit` (see the top of this file).  Threads past
// the kThreads roles (a fused round launch has more) only pass the CTA's
// barriers.  The tensor maps live in the kernel's parameter space.
template <int D, bool kDuo>
__device__ __forceinline__ void attn_body(unsigned unit, const CUtensorMap *tm_q, const CUtensorMap *tm_kp,
                                          const CUtensorMap *tm_vp, const CUtensorMap *tm_kn,
                                          const CUtensorMap *tm_vn, const CUtensorMap *tm_o,
                                          const AttnParams &p)
{
    using Lay = Layout<D, kDuo>;
    static_assert(!kDuo || D == 128, "a CTA pair splits the head dimension into two 64-column blocks");
    extern __shared__ uint8_t smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- unit: ((r * Hkv + hk) * MT + mt) * S + sp
    unsigned u = unit;
    const int sp = (int)(u % (unsigned)p.S);
    u /= (unsigned)p.S;
    const int mt = (int)(u % (unsigned)p.MT);
    u /= (unsigned)p.MT;
    const int hk = (int)(u % (unsigned)p.Hkv);
    const int r = (int)(u / (unsigned)p.Hkv);
    int32_t *status = reinterpret_cast<int32_t *>(p.ws);
    // CTA pair (kDuo): query tiles mt = 2j (rank 0, which issues the MMAs)
    // and 2j + 1 (rank 1) of one request and KV head, one key list
    const uint32_t crank = kDuo ? cluster_ctarank() : 0u;
    const uint32_t peer = crank ^ 1u;
    // a kernel launched after this one as an independent programmatic
    // dependent (the verification of the same round) may start now
    if (tid == 0)
        pdl_trigger();

    // the request's offsets: loaded now, checked once the setup below is done
    // (the setup does not depend on them and hides their latency)
    // (after a kernel whose output this one may read, nothing is read before
    // it has finished: the offsets load after the setup then)
    ReqRaw braw{};
    if (!p.wait_first)
        braw = load_bounds(p.cu_prefix, p.cu_q, p.cu_seg, r);

    // ---- shared memory carve-up (1024-byte aligned base for the swizzled tiles)
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (sbase - raw);
    const uint32_t sQ = sbase + Lay::q, sK = sbase + Lay::k, sV = sbase + Lay::v;
    auto bar = [&](int i) -> uint32_t { return sbase + Lay::bars + 8u * (uint32_t)i; };
    uint32_t *misc = reinterpret_cast<uint32_t *>(gbase + Lay::misc);
    volatile uint32_t *tmem_slot = misc + 0;
    volatile uint32_t *abort_flag = misc + 1;
    uint32_t *mask = misc + 2;  // 2 words: packed tiles visible to some row of the tile
    float4 *s_ml = reinterpret_cast<float4 *>(gbase + Lay::ml);  // [kWG][kBM]: max, sum, tiles done
    float *s_mx = reinterpret_cast<float *>(gbase + Lay::mx);     // [2][kWG][kBM]

    if (tid == 0) {
        mbar_init(bar(B_Q), 1);
        for (int i = 0; i < Lay::kKS; ++i) {
            mbar_init(bar(B_KF + i), 1);
            mbar_init(bar(B_KE + i), 1);
        }
        for (int i = 0; i < Lay::kVS; ++i) {
            mbar_init(bar(B_VF + i), 1);
            mbar_init(bar(B_VE + i), 1);
        }
        // a pair's MMA-issuing CTA counts both CTAs' softmax warps; both
        // CTAs' masks count the first warpgroups' warps of both
        constexpr uint32_t kIssuerArrivals = (kDuo ? 2 : 1) * kSoftmaxThreads / 32;
        for (int b2 = 0; b2 < 2; ++b2) {
            mbar_init(bar(B_SF + b2), 1);
            mbar_init(bar(B_PR + b2), kIssuerArrivals);
            mbar_init(bar(B_MX + b2), kSoftmaxThreads / 32);
        }
        mbar_init(bar(B_OW), 1);
        mbar_init(bar(B_MASK), kDuo ? 2 * 4 : kSoftmaxThreads);
        mbar_init(bar(B_DONE), 1);
        mbar_init(bar(B_QT), kIssuerArrivals);
        *abort_flag = 0u;
        mask[0] = mask[1] = 0u;
        fence_barrier_init();
    }
    if (warp == kTmaWarp && lane == 0) {
        prefetch_tmap(tm_q);
        prefetch_tmap(tm_kp);
        prefetch_tmap(tm_vp);
        prefetch_tmap(tm_kn);
        prefetch_tmap(tm_vn);
        prefetch_tmap(tm_o);
    }
    if (warp == kMmaWarp) {
        if constexpr (kDuo) {
            tmem_alloc_pair(smem_u32(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (kDuo) {  // both CTAs' barriers are initialised before either signals the other's
        cluster_arrive();
        cluster_wait();
    }
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // the offsets are used only from here on (the empty asm keeps the compiler
    // from moving their first use, and so the wait for the loads, above the
    // barrier).  Early exits are uniform over the CTAs of a cluster (same r
    // and tile) and come before any copy or cluster barrier; every exit first
    // waits for a kernel this launch overlaps (programmatic dependent launch):
    // the stream moves on only when both have finished.
    if (p.wait_first) {  // the kernel ahead has finished and its writes are visible after this
        pdl_wait();
        braw = load_bounds(p.cu_prefix, p.cu_q, p.cu_seg, r);
    }
    if (!p.one_request)  // a single request's bounds come from the host: nothing to wait for here
        asm volatile("" : "+r"(braw.q0), "+r"(braw.q1), "+r"(braw.p0), "+r"(braw.p1), "+r"(braw.s0), "+r"(braw.s1));
    ReqBounds b;
    const bool bounds_ok = kernel_bounds(p, braw, b);
    // a pair leaves together: only when its first tile is past the request
    // (the second CTA of a pair with one tile in the request has no valid row)
    if (!bounds_ok || (kDuo ? (mt & ~1) : mt) * p.TQ >= b.n_q) {
        if (!bounds_ok && tid == 0 && sp == 0 && crank == 0)
            record_status(status, D3D_ERR_DEVICE_INPUT);
        if (warp == kMmaWarp) {
            if constexpr (kDuo)
                tmem_dealloc_pair(tmem, kTmemCols);
            else
                tmem_dealloc(tmem, kTmemCols);
        }
        pdl_wait();
        return;
    }

    // ---- this split's key list: prefix tiles [pb, pe), then (last split only) packed tiles
    const int nP = (b.L + kBN - 1) / kBN;
    const int pb = split_prefix_begin(sp, p.S, nP, p.PK);
    const int pe = (sp == p.S - 1) ? nP : split_prefix_begin(sp + 1, p.S, nP, p.PK);
    const int n_pre = pe - pb;
    const bool last_split = sp == p.S - 1;

    // number of packed tiles of the query tile; waits for the mask on first use
    // (called by whole warps: the vote keeps the answer warp-uniform)
    int npk_cache = -1;
    uint32_t mk0 = 0, mk1 = 0;
    auto npk = [&]() -> int {
        if (npk_cache < 0) {
            const bool okm = kDuo ? wait_bar_cluster(bar(B_MASK), 0, abort_flag, status)
                                  : wait_bar(bar(B_MASK), 0, abort_flag, status);
            if (!__all_sync(0xffffffffu, okm))
                return -1;
            mk0 = *(volatile uint32_t *)&mask[0];
            mk1 = *(volatile uint32_t *)&mask[1];
            npk_cache = __popc(mk0) + __popc(mk1);
        }
        return npk_cache;
    };
    // does list tile k of this split exist (-1: gave up waiting)
    auto exists = [&](int k) -> int {
        if (k < n_pre)
            return 1;
        if (!last_split)
            return 0;
        const int c = npk();
        return c < 0 ? -1 : (k - n_pre < c ? 1 : 0);
    };
    // global K/V row of list tile k (call only when it exists)
    auto tile_row = [&](int k, bool &pre) -> int {
        pre = k < n_pre;
        return pre ? b.p0 + (pb + k) * kBN : b.q0 + nth_set_bit(mk0, mk1, k - n_pre) * kBN;
    };

    // what a softmax thread hands to the split combine after the role code
    bool mg_on = false;  // a softmax thread that reached the epilogue
    // output row of staged row i of the query tile, or null beyond the request
    auto out_row = [&](int i) -> uint16_t * {
        const int tok = mt * p.TQ + i / p.G;
        if (tok >= b.n_q || !dbg_ok(b.q0 + tok < p.total_q && hk * p.G + (i % p.G) < p.Hq, status))
            return nullptr;
        return p.out + ((size_t)(b.q0 + tok) * p.Hq + hk * p.G + (i % p.G)) * D;
    };

    if (warp == kTmaWarp) {
        // =================== TMA producer ===================
        // The whole warp runs the loop (warp-uniform control flow: every value
        // the copies need stays warp-uniform); one elected lane issues.
        // Issue order = the tensor core's consumption order: K0, K1, then
        // V(k), K(k+2) for k = 0, 1, ...
        const bool leader = elect_one();
        int nk = 0, nv = 0;     // K / V tiles handled, in list order
        bool skipped0 = false;  // the injected fault left K tile 0 unissued
        if (leader) {
            mbar_arrive_expect_tx(bar(B_Q), Lay::kQBytes);
            for (int cb = 0; cb < D / 64; ++cb)
                tma_load_3d(sQ + cb * kBlockBytes, tm_q, bar(B_Q), cb * 64, hk * p.G, b.q0 + mt * p.TQ);
        }
        __syncwarp();
        auto issue = [&](int k, bool is_k) -> bool {
            const int ns = is_k ? Lay::kKS : Lay::kVS;
            const int s = k % ns;
            const int empty = is_k ? B_KE : B_VE, full = is_k ? B_KF : B_VF;
            if (k >= ns && !__all_sync(0xffffffffu, wait_bar(bar(empty + s), ((k - ns) / ns) & 1, abort_flag, status)))
                return false;
            ++(is_k ? nk : nv);
            if (p.fault == 1 && is_k && k == 0) {
                skipped0 = true;  // injected fault: this tile never arrives
                return true;
            }
            bool pre;
            int row = tile_row(k, pre);
            // debug build: the tile's first row lies in the request's prefix or
            // packed rows (else the copy reads row 0 and the status says so)
            if (!dbg_ok(pre ? (row >= b.p0 && row < b.p0 + b.L) : (row >= b.q0 && row < b.q0 + b.n_q), status))
                row = 0;
            const CUtensorMap *m = is_k ? (pre ? tm_kp : tm_kn) : (pre ? tm_vp : tm_vn);
            const uint32_t dst = is_k ? sK + s * Lay::kKBytes : sV + s * Lay::kVBytes;
            if (leader) {
                if constexpr (kDuo) {
                    // this CTA's half (keys [64 crank, +64) of K, head-dim columns
                    // [64 crank, +64) of V), counted on the issuing CTA's barrier,
                    // which expects both halves
                    const uint32_t fb = dsmem_addr(bar(full + s), 0u);
                    if (crank == 0)
                        mbar_arrive_expect_tx(bar(full + s), 2u * (is_k ? Lay::kKBytes : Lay::kVBytes));
                    if (is_k) {
                        for (int cb = 0; cb < D / 64; ++cb)
                            tma_load_3d_pair(dst + cb * Lay::kKBlock, m, fb, cb * 64, hk, row + (int)crank * (kBN / 2));
                    } else {
                        tma_load_3d_pair(dst, m, fb, (int)crank * 64, hk, row);
                    }
                } else {
                    mbar_arrive_expect_tx(bar(full + s), Lay::kKBytes);
                    for (int cb = 0; cb < D / 64; ++cb)
                        tma_load_3d(dst + cb * kBlockBytes, m, bar(full + s), cb * 64, hk, row);
                }
            }
            __syncwarp();
            return true;
        };
        bool ok = true;
        for (int k = 0; ok && k < 2; ++k) {
            const int e = exists(k);
            ok = e >= 0;
            if (e == 1)
                ok = issue(k, true);
        }
        for (int k = 0; ok; ++k) {
            const int e = exists(k);
            if (e != 1)
                break;
            ok = issue(k, false);
            const int e2 = ok ? exists(k + 2) : -1;
            if (e2 < 0)
                break;
            if (e2 == 1)
                ok = issue(k + 2, true);
        }
        // every copy this warp started must land before the CTA exits: the
        // last phase of each stage (tiles s, s + ns, ... of the n handled)
        auto issued = [](int n, int s, int ns) { return n > s ? (n - 1 - s) / ns + 1 : 0; };
        wait_drain(bar(B_Q), 0, status);
        // (a pair's K/V copies are counted on the issuing CTA's barriers: it
        // drains both halves, and the other CTA stays until the cluster
        // barrier at the end)
        for (int s = 0; crank == 0 && s < Lay::kKS; ++s) {
            const int c = issued(nk, s, Lay::kKS) - ((s == 0 && skipped0) ? 1 : 0);
            if (c > 0)
                wait_drain(bar(B_KF + s), (c - 1) & 1, status);
        }
        for (int s = 0; crank == 0 && s < Lay::kVS; ++s) {
            const int c = issued(nv, s, Lay::kVS);
            if (c > 0)
                wait_drain(bar(B_VF + s), (c - 1) & 1, status);
        }
        __syncwarp();
    } else if (warp == kMmaWarp && crank == 0) {
        // =================== MMA issuer ===================
        // The whole warp runs the loop and waits (warp-uniform control flow,
        // so the descriptors stay warp-uniform); one elected lane issues the
        // MMAs and their commits.  A pair's MMAs span both CTAs (M = 256: each
        // CTA's 128 rows of Q, P, S and O in its own TMEM) and read K and V
        // from both CTAs' halves; their commits arrive on both CTAs' barriers.
        const bool leader = elect_one();
        constexpr uint32_t kM = kDuo ? 2 * kBM : kBM;
        constexpr uint32_t idS = idesc_bf16_f32(kM, kBN, 0, 0);
        constexpr uint32_t idO = idesc_bf16_f32(kM, D, 0, 1);
        auto wait_all = [&](uint32_t bar_addr, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, wait_bar(bar_addr, parity, abort_flag, status));
        };
        // a barrier both CTAs' softmax warps arrive on (TMEM hand-offs: the
        // tcgen05 fences order them)
        auto wait_all_pair = [&](uint32_t bar_addr, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, wait_bar(bar_addr, parity, abort_flag, status));
        };
        auto mma_ts = [&](uint32_t d_tmem, uint32_t a_tmem, uint64_t bd, uint32_t idesc, uint32_t acc) {
            if constexpr (kDuo)
                mma_bf16_ts_pair(d_tmem, a_tmem, bd, idesc, acc);
            else
                mma_bf16_ts(d_tmem, a_tmem, bd, idesc, acc);
        };
        auto commit = [&](uint32_t b_addr) {
            if constexpr (kDuo)
                mma_commit_pair(b_addr);
            else
                mma_commit(b_addr);
        };
        // S(k) = Q K_k^T into TMEM buffer k % 2, then release the K stage
        auto issue_s = [&](int k) {
            const int ks = k % Lay::kKS;
            const uint32_t tS = tmem + (uint32_t)(k & 1) * kBN;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * Lay::kKBlock + (kk % 4) * 32;
                    const uint64_t bd = sdesc_sw128(sK + ks * Lay::kKBytes + off, 16, 1024);
                    mma_ts(tS, tmem + 2u * kBN + D + (uint32_t)(kk * 8), bd, idS, kk > 0 ? 1u : 0u);
                }
                commit(bar(B_SF + (k & 1)));
                commit(bar(B_KE + ks));
            }
            __syncwarp();
        };
        // O += P(k) V_k with P read from buffer k % 2, then release the V stage
        auto issue_pv = [&](int k) {
            const int vs = k % Lay::kVS;
            const uint32_t tP = tmem + (uint32_t)(k & 1) * kBN, tO = tmem + 2u * kBN;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    // A = P in TMEM (8 columns of bf16 pairs per 16 keys); B = V
                    // MN-major: 16 keys = two 8-row groups = 2048 bytes, the next 64
                    // head-dim columns are 16 KB further
                    const uint64_t bd = sdesc_sw128(sV + vs * Lay::kVBytes + kk * 2048, kBlockBytes, 1024);
                    mma_ts(tO, tP + kk * 8, bd, idO, (k > 0 || kk > 0) ? 1u : 0u);
                }
                commit(bar(B_OW));
                commit(bar(B_VE + vs));
            }
            __syncwarp();
        };
        bool ok = wait_all_pair(bar(B_QT), 0);
        for (int k = 0; ok && k < 2; ++k) {
            const int e = exists(k);
            ok = e >= 0;
            if (e == 1) {
                ok = wait_all(bar(B_KF + k % Lay::kKS), (k / Lay::kKS) & 1);
                if (ok) {
                    tc_fence_after();
                    issue_s(k);
                }
            }
        }
        // per tile k: PV(k) once P(k) is written, then S(k+2) into the buffer
        // PV(k) has just read; the tensor core computes these while the softmax
        // works on tile k+1.  S(k+2) is attempted after every PV (its own K wait
        // returns at once when the CTA aborts); only then does a failure end
        // the loop, and no MMA is issued without its data.
        for (int k = 0; ok; ++k) {
            const int e = exists(k);
            if (e != 1) {
                ok = e >= 0;
                break;
            }
            ok = wait_all(bar(B_VF + k % Lay::kVS), (k / Lay::kVS) & 1) &&
                 wait_all_pair(bar(B_PR + (k & 1)), (k >> 1) & 1);
            if (!ok)
                break;
            tc_fence_after();
            issue_pv(k);
            const int e2 = exists(k + 2);
            ok = e2 >= 0;
            if (e2 == 1) {
                ok = wait_all(bar(B_KF + (k + 2) % Lay::kKS), ((k + 2) / Lay::kKS) & 1);
                if (ok)
                    issue_s(k + 2);
            }
        }
        // every MMA is complete when B_DONE fires: O final, and the Q and K/V
        // buffers free; TMEM is released only after it
        if (leader)
            commit(bar(B_DONE));
        __syncwarp();
        wait_drain(bar(B_DONE), 0, status);
        __syncwarp();
    } else if (warp < kTmaWarp) {
        // =================== softmax warpgroups ===================
        const int w = warp >> 2;  // warpgroup: key columns [32w, 32w + 32) of every tile
        const int row = tid & 127;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS0 = tmem + lane_off, tO = tmem + 2u * kBN + lane_off;
        const int token = mt * p.TQ + row / p.G;
        const bool row_valid = token < b.n_q;
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
        uint32_t mw0 = 0u, mw1 = 0u;  // (pair) packed tiles this thread's row sees
        if (row_valid && last_split) {
            if (!row_visibility(seg_base, seg_lo, seg_hi, b.n_q, token, vis)) {
                row_bad = true;
                vis.own_lo = vis.own_hi = vis.par_lo = vis.par_hi = 0;
            }
            if (w == 0) {
                auto mark = [&](int lo, int hi) {
                    if (lo >= hi)
                        return;
                    for (int k = lo / kBN; k <= (hi - 1) / kBN && k < kMaxPackedTiles; ++k) {
                        if constexpr (kDuo) {
                            if (k < 32)
                                mw0 |= 1u << k;
                            else
                                mw1 |= 1u << (k - 32);
                        } else
                            atomicOr(&mask[k >> 5], 1u << (k & 31));
                    }
                };
                mark(vis.own_lo, vis.own_hi);
                mark(vis.par_lo, vis.par_hi);
            }
        }
        if constexpr (kDuo) {
            // the pair's key list covers the rows of both tiles: each first-
            // warpgroup warp ors its rows' tiles into both CTAs' masks, then
            // arrives on both CTAs' mask barriers
            if (w == 0) {
                mw0 = __reduce_or_sync(0xffffffffu, mw0);
                mw1 = __reduce_or_sync(0xffffffffu, mw1);
                if (lane == 0) {
                    if (mw0 != 0u) {
                        atomicOr(&mask[0], mw0);
                        red_or_cluster(dsmem_addr(smem_u32(&mask[0]), peer), mw0);
                    }
                    if (mw1 != 0u) {
                        atomicOr(&mask[1], mw1);
                        red_or_cluster(dsmem_addr(smem_u32(&mask[1]), peer), mw1);
                    }
                    mbar_arrive(bar(B_MASK));
                    mbar_arrive_cluster(dsmem_addr(bar(B_MASK), peer));
                }
            }
        } else {
            mbar_arrive(bar(B_MASK));
        }

        // Q into TMEM as the A operand of S = Q K^T: this thread's row, its
        // warpgroup's half of the head dimension, as bf16 pairs per column
        {
            const bool okq = wait_bar(bar(B_Q), 0, abort_flag, status);
            if (__all_sync(0xffffffffu, okq)) {
                constexpr int kChunks = D / 8 / kWG;  // 16-byte chunks of the row per thread
                uint32_t qv[kChunks * 4];
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    const int gc = w * kChunks + c;
                    const uint4 u = smem_ld_v4(sQ + (uint32_t)(gc / 8) * kBlockBytes + (uint32_t)row * 128u +
                                               ((uint32_t)((gc % 8) ^ (row & 7)) << 4));
                    qv[4 * c] = u.x, qv[4 * c + 1] = u.y, qv[4 * c + 2] = u.z, qv[4 * c + 3] = u.w;
                }
                const uint32_t tQ = tmem + lane_off + 2u * kBN + D + (uint32_t)(w * kChunks * 4);
                if constexpr (kChunks * 4 == 32)
                    tmem_st32u(tQ, qv);
                else
                    tmem_st16(tQ, qv);
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (kDuo && crank != 0)
                    mbar_arrive_remote(dsmem_addr(bar(B_QT), 0u));
                else
                    mbar_arrive(bar(B_QT));
            }
        }

        float m_ref = -INFINITY, l = 0.f;  // l: this thread's column part of the row sum
        bool aborted = false;
        int n_done = 0;
        for (int k = 0;; ++k) {
            const int ex = exists(k);
            if (!__all_sync(0xffffffffu, ex >= 0)) {
                aborted = true;
                break;
            }
            if (ex == 0)
                break;
            const int bf = k & 1;
            const uint32_t tS = tS0 + (uint32_t)bf * kBN;
            bool ok = wait_bar(bar(B_SF + bf), (k >> 1) & 1, abort_flag, status);
            if (!__all_sync(0xffffffffu, ok)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            float s[kPart];
#if D3D_ATTN_WG == 2
            tmem_ld64(tS + (uint32_t)(w * kPart), s);
#else
            tmem_ld32(tS + (uint32_t)(w * kPart), s);
#endif
            bool pre;
            const int krow = tile_row(k, pre);
            if (pre) {
                const int valid = b.L - (pb + k) * kBN - w * kPart;
                if (valid < kPart) {
#pragma unroll
                    for (int e = 0; e < kPart; ++e)
                        if (e >= valid)
                            s[e] = -INFINITY;
                }
            } else {
                // this row's visible keys of the part as a mask: two half-open
                // intervals cut into 32-key words
                uint32_t wbits[kPart / 32];
#pragma unroll
                for (int q = 0; q < kPart / 32; ++q) {
                    const int base = krow - b.q0 + w * kPart + 32 * q;
                    wbits[q] = range_bits(vis.own_lo - base, vis.own_hi - base) |
                               range_bits(vis.par_lo - base, vis.par_hi - base);
                }
#pragma unroll
                for (int e = 0; e < kPart; ++e)
                    s[e] = ((wbits[e >> 5] >> (e & 31)) & 1u) ? s[e] : -INFINITY;
            }
            // max of this part with eight independent chains, then the row max
            // from all parts (published in shared memory, bounded wait)
            float m8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                m8[e] = s[e];
#pragma unroll
            for (int e0 = 8; e0 < kPart; e0 += 8)
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    m8[e] = fmaxf(m8[e], s[e0 + e]);
            const float mloc = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                     fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
            s_mx[(bf * kWG + w) * kBM + row] = mloc;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(B_MX + bf));
            ok = wait_bar(bar(B_MX + bf), (k >> 1) & 1, abort_flag, status);
            if (!__all_sync(0xffffffffu, ok)) {
                aborted = true;
                break;
            }
            // every part of the S buffer is in registers by now: P may overwrite it
            float mrow = mloc;
#pragma unroll
            for (int w2 = 0; w2 < kWG; ++w2)
                mrow = fmaxf(mrow, s_mx[(bf * kWG + w2) * kBM + row]);
            const float mx = mrow * p.scale_log2;
            float factor = 1.f;
            if (mx > m_ref + kRescaleLog2) {
                factor = ex2(m_ref - mx);  // 0 when m_ref = -inf
                m_ref = mx;
            }
            const float msub = (m_ref == -INFINITY) ? 0.f : m_ref;
            // exponent arguments and the row sum in packed pairs (two sum chains of
            // two lanes each)
            float r4[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t pk[kPart / 2];
#pragma unroll
            for (int e = 0; e < kPart / 2; ++e) {
                float x0, x1;
                ffma2(x0, x1, s[2 * e], s[2 * e + 1], p.scale_log2, p.scale_log2, -msub, -msub);
                const float e0 = ex2(x0), e1 = ex2(x1);
                float &ra = r4[2 * (e & 1)], &rb = r4[2 * (e & 1) + 1];
                fadd2(ra, rb, ra, rb, e0, e1);
                pk[e] = pack_bf16x2(e0, e1);
            }
            l = l * factor + (r4[0] + r4[1]) + (r4[2] + r4[3]);
            // rescale this thread's part of O once PV(k-1) has landed (rare: only
            // when the max grows by more than 2^8)
            if (k > 0 && __any_sync(0xffffffffu, factor != 1.f)) {
                ok = wait_bar(bar(B_OW), (k - 1) & 1, abort_flag, status);
                if (!__all_sync(0xffffffffu, ok)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int q = 0; q < D / kWG / 8; ++q) {
                    float o[8];
                    const uint32_t col = (uint32_t)(w * (D / kWG) + q * 8);
                    tmem_ld8(tO + col, o);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        o[e] *= factor;
                    tmem_st8(tO + col, o);
                }
            }
            // P of keys kPart*w.. over columns (kPart/2)*w..
#if D3D_ATTN_WG == 2
            tmem_st32u(tS + (uint32_t)(w * (kPart / 2)), pk);
#else
            tmem_st16(tS + (uint32_t)(w * (kPart / 2)), pk);
#endif
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (kDuo && crank != 0)
                    mbar_arrive_remote(dsmem_addr(bar(B_PR + bf), 0u));
                else
                    mbar_arrive(bar(B_PR + bf));
            }
            n_done = k + 1;
        }

        // ---- epilogue: every MMA done, then the warpgroups' parts combine
        wait_drain(bar(B_DONE), 0, status);
        // (max, column-half sum, tiles done) of this thread's row; a negative sum
        // marks a void row (failed descriptor check or an abandoned wait)
        // a single request whose device offsets disagree with the host's: every row is void
        const bool bad_req = p.one_request && !one_request_matches(p, braw);
        if (bad_req && tid == 0 && sp == 0)
            record_status(status, D3D_ERR_DEVICE_INPUT);
        s_ml[w * kBM + row] = make_float4(m_ref, (aborted || row_bad || bad_req) ? -1.f : l, (float)n_done, 0.f);
        tc_fence_before();
        asm volatile("bar.sync 2, %0;" ::"n"(kSoftmaxThreads) : "memory");
        tc_fence_after();
        bool void_row = false;
        float M = -INFINITY, L = 0.f, done = 1e30f;
#pragma unroll
        for (int w2 = 0; w2 < kWG; ++w2) {
            const float4 t = s_ml[w2 * kBM + row];
            void_row = void_row || t.y < 0.f;
            M = fmaxf(M, t.x);  // every part keeps the same running max
            L += fmaxf(t.y, 0.f);
            done = fminf(done, t.z);
        }
        const bool have = done > 0.f;  // uniform over each warp
        const float inv = (void_row || !(L > 0.f)) ? 0.f : 1.f / L;
        // this thread's part of the head dimension: columns [w*D/kWG, (w+1)*D/kWG),
        // staged in the V ring (free once every MMA is done) and stored below
        const uint32_t part = Xchg<D>::part(sK);
        // the thread's D/kWG columns of O in one TMEM load (one wait)
        constexpr int kCols = D / kWG;
        float xo[kCols];
        if (have) {
            const uint32_t t0 = tO + (uint32_t)(w * kCols);
            if constexpr (kCols == 64) {
                tmem_ld64(t0, xo);
            } else if constexpr (kCols == 32) {
                tmem_ld32(t0, xo);
            } else {
#pragma unroll
                for (int q = 0; q < kCols / 8; ++q)
                    tmem_ld8(t0 + (uint32_t)(q * 8), *reinterpret_cast<float(*)[8]>(xo + 8 * q));
            }
        } else {
#pragma unroll
            for (int e = 0; e < kCols; ++e)
                xo[e] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < kCols / 8; ++q) {
            const uint4 v = pack8(xo + 8 * q, inv);
            const int unit = w * (D / kWG / 8) + q;
            if (p.S == 1) {
                smem_st_v4(stage_addr(sV, row, unit), v);
            } else {
                // the CTA's partial for the cluster's combine (every MMA is done)
                smem_st_v4(part + ((uint32_t)unit * kBM + (uint32_t)row) * 16u, v);
            }
        }
        if (p.S > 1 && w == 0)
            smem_st_f2(Xchg<D>::ml(sK) + (uint32_t)row * 8u, make_float2(M, void_row ? -1.f : L));
        if (!aborted && row_valid && row_bad && w == 0)
            record_status(status, D3D_ERR_DEVICE_INPUT);
        if (p.S == 1) {
            // a tile whose rows all belong to the request leaves by tensor stores
            // of the staged column blocks (one thread), another by plain stores
            fence_async_smem();
            asm volatile("bar.sync 3, %0;" ::"n"(kSoftmaxThreads) : "memory");
            if ((mt + 1) * p.TQ <= b.n_q) {
                if (tid == 0) {
                    for (int cb = 0; cb < D / 64; ++cb)
                        tma_store_3d(tm_o, sV + (uint32_t)cb * kBlockBytes, cb * 64, hk * p.G, b.q0 + mt * p.TQ);
                    bulk_commit();
                    bulk_wait_read();
                }
            } else {
                store_staged(sV, 0u, kBM, 0, D / 8, tid, kSoftmaxThreads, out_row);
            }
        }
        mg_on = true;
    }

    // ---- every role is done (all waits are bounded, copies and MMAs drained)
    tc_fence_before();
    __syncthreads();
    if constexpr (kDuo) {
        // neither CTA of a pair leaves (or frees TMEM) while the other's
        // MMAs or copies may still use it
        cluster_arrive();
        cluster_wait();
    }
    if (!kDuo && p.S > 1) {
        // split combine across the cluster: every thread of every CTA passes
        // both cluster barriers exactly once
        cluster_arrive();
        cluster_wait();
        if (mg_on) {
            const int w = warp >> 2, row = tid & 127;
            const uint32_t part = Xchg<D>::part(sK), ml = Xchg<D>::ml(sK);
            switch (p.S) {
            case 2: cluster_merge<D, 2>(sp, w, part, ml, row, sV); break;
            case 3: cluster_merge<D, 3>(sp, w, part, ml, row, sV); break;
            case 4: cluster_merge<D, 4>(sp, w, part, ml, row, sV); break;
            case 5: cluster_merge<D, 5>(sp, w, part, ml, row, sV); break;
            case 6: cluster_merge<D, 6>(sp, w, part, ml, row, sV); break;
            case 7: cluster_merge<D, 7>(sp, w, part, ml, row, sV); break;
            default: cluster_merge<D, 8>(sp, w, part, ml, row, sV); break;
            }
            fence_async_smem();
            asm volatile("bar.sync 3, %0;" ::"n"(kSoftmaxThreads) : "memory");
            // the CTA's units leave by tensor stores when they are whole column
            // blocks of a tile whose rows all belong to the request
            const int u0 = split_unit_begin(sp, p.S, D / 8), u1 = split_unit_begin(sp + 1, p.S, D / 8);
            if (u0 % 8 == 0 && u1 % 8 == 0 && (mt + 1) * p.TQ <= b.n_q) {
                if (tid == 0) {
                    for (int cb = u0 / 8; cb < u1 / 8; ++cb)
                        tma_store_3d(tm_o, sV + (uint32_t)cb * kBlockBytes, cb * 64, hk * p.G, b.q0 + mt * p.TQ);
                    bulk_commit();
                    bulk_wait_read();
                }
            } else {
                store_staged(sV, 0u, kBM, u0, u1, tid, kSoftmaxThreads, out_row);
            }
        }
        // no CTA leaves while another may still read its shared memory
        cluster_arrive();
        cluster_wait();
    }
    // release TMEM
    if (warp == kMmaWarp) {
        tc_fence_after();
        if constexpr (kDuo)
            tmem_dealloc_pair(tmem, kTmemCols);
        else
            tmem_dealloc(tmem, kTmemCols);
    }
    pdl_wait();
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kp,
                   const __grid_constant__ CUtensorMap tm_vp, const __grid_constant__ CUtensorMap tm_kn,
                   const __grid_constant__ CUtensorMap tm_vn, const __grid_constant__ CUtensorMap tm_o,
                   const AttnParams p)
{
    attn_body<D, false>(blockIdx.x, &tm_q, &tm_kp, &tm_vp, &tm_kn, &tm_vn, &tm_o, p);
}

// CTA pairs: launched in clusters of two, one query tile per CTA, the MMAs of
// both tiles issued by the even CTA over both SMs (the K maps' boxes hold 64
// keys: each CTA loads half of every K tile and half of every V tile's
// head-dim columns).
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_duo_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kp,
                    const __grid_constant__ CUtensorMap tm_vp, const __grid_constant__ CUtensorMap tm_kn,
                    const __grid_constant__ CUtensorMap tm_vn, const __grid_constant__ CUtensorMap tm_o,
                    const AttnParams p)
{
    attn_body<D, true>(blockIdx.x, &tm_q, &tm_kp, &tm_vp, &tm_kn, &tm_vn, &tm_o, p);
}

// One launch for the asynchronous round ([D3D] "Background: asynchronous
// drafting and cache hits": the drafter's packed pass runs while the current
// block is verified): CTAs [0, n_attn) are the drafting attention's units,
// the others the verification's CTAs (512 threads, every one resident: the
// launch is cooperative).  Each CTA holds one SM, so the two parts share the
// GPU exactly as the split launches do, without a second launch.
template <int D, typename T>
__global__ void __launch_bounds__(kNTLimited, 1)
    round_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kp,
                 const __grid_constant__ CUtensorMap tm_vp, const __grid_constant__ CUtensorMap tm_kn,
                 const __grid_constant__ CUtensorMap tm_vn, const __grid_constant__ CUtensorMap tm_o,
                   const AttnParams p, const VArgs va, int n_attn)
{
    if (blockIdx.x < (unsigned)n_attn)
        attn_body<D, false>(blockIdx.x, &tm_q, &tm_kp, &tm_vp, &tm_kn, &tm_vn, &tm_o, p);
    else
        verify_body<T, kNTLimited>(blockIdx.x - (unsigned)n_attn, gridDim.x - (unsigned)n_attn, va);
}
static_assert(kThreads <= kNTLimited, "the fused round launch holds the attention's roles");

// ===========================================================================
// Two query tiles per CTA.
//
// Work unit (one CTA, which holds one SM): request r, KV head hk, the pair of
// 128-row query tiles 2mp and 2mp+1, and one key split.  Both tiles read
// every K/V tile of the unit's key list, so a CTA moves half the K/V bytes
// per flop of attn_body, whose one tile per CTA leaves the kernel bound by
// the rate at which an SM receives K/V tiles.  The key list is as in
// attn_body: the split's prefix tiles, then (last split only) the packed
// tiles that some row of either query tile can see.
//
// Roles (320 threads):
//   warps 4t..4t+3  softmax of query tile t (t = 0, 1): thread i owns TMEM
//              lane i = row i of the tile and all 128 key columns of a key
//              tile.  Per key tile: the row max from the whole S_t row (four
//              32-column TMEM loads in flight, the mask only on a tile that is
//              not a full prefix tile, three-input maxima), a rescale of the
//              thread's O_t row only when the max grows by more than 2^8,
//              then per 32-column chunk (loaded again while the previous one
//              is computed) the exponentials and the row sum (packed f32x2
//              arithmetic) and P_t as bf16 pairs over the first 64 columns of
//              S_t.  The output is staged in shared memory and leaves by
//              tensor stores (whole tiles) or coalesced stores.
//   warp 8     TMA producer: Q0, K0, Q1, K1, then V and K tiles into 2-deep
//              rings (3-D tensor maps, 128-byte swizzle) in the tensor core's
//              order.
//   warp 9     MMA issuer and TMEM owner (warp-uniform loop, one elected
//              lane issues).  Per key tile k and tile t = 0, 1: once P_t(k)
//              is written, O_t += P_t(k) V_k, then S_t(k+1) = Q_t K_{k+1}^T
//              into the columns P_t(k) came from (one thread's MMAs run in
//              issue order, so S_t(k+1) never overwrites P_t(k) before its
//              PV has read it).  The tensor core alternates between the two
//              tiles: it computes the PV and the next S of one tile while the
//              softmax of the other runs.
// TMEM: S_0 [0, 128), S_1 [128, 256), O_0 [256, 256 + D), O_1 [384, 384 + D).
// With S > 1 splits the S CTAs of a tile pair form a thread-block cluster and
// combine through distributed shared memory as in attn_body (the exchange
// area spans the K and V rings, free once every MMA is done).
// ===========================================================================
// 320 threads: an SM sub-partition holds three of the ten warps, so a thread
// may use at most 168 registers (16384 per sub-partition) -- enough for a
// softmax thread to hold a whole 128-column S row.  The host checks that the
// compiled kernel fits one CTA per SM before it plans with it.
constexpr int kPairThreads = 320;
constexpr int kPairTmaWarp = 8;
constexpr int kPairMmaWarp = 9;
constexpr int kPStages = 2;  // K and V ring depth

enum {
    P_Q = 0,                  // 2: query tile t landed
    P_KF = P_Q + 2,           // kPStages
    P_KE = P_KF + kPStages,   // kPStages: released after S_1 of the tile
    P_VF = P_KE + kPStages,   // kPStages
    P_VE = P_VF + kPStages,   // kPStages: released after PV_1 of the tile
    P_SF = P_VE + kPStages,   // 2: S_t(k) in TMEM
    P_PR = P_SF + 2,          // 2: P_t(k) written (one arrival per softmax warp of tile t)
    P_OW = P_PR + 2,          // 2: PV_t(k) complete (O_t written, P_t read)
    P_MASK = P_OW + 2,        // visibility mask complete (256 arrivals)
    P_DONE = P_MASK + 1,      // every MMA of the CTA complete
    P_COUNT = P_DONE + 1
};

template <int D> struct PairLayout {
    static constexpr uint32_t kQBytes = kBM * D * 2;  // one query tile
    static constexpr uint32_t kKBytes = kBN * D * 2;
    static constexpr uint32_t q = 0;  // Q0 then Q1
    static constexpr uint32_t k = q + 2 * kQBytes;
    static constexpr uint32_t v = k + kPStages * kKBytes;
    static constexpr uint32_t bars = v + kPStages * kKBytes;
    static constexpr uint32_t misc = bars + P_COUNT * 8;
    static constexpr uint32_t segs = misc + 64;
    static constexpr uint32_t total = segs + kStagedSegs * sizeof(d3d_segment_t);
    static constexpr uint32_t alloc = total + 1024;  // room to align the base to 1024 bytes
};
static_assert(PairLayout<128>::alloc <= 227 * 1024, "two-tile shared memory fits an SM");

// Split-combine exchange of the two-tile kernel (over the K and V rings):
// 16-byte unit u (head-dim columns 8u..8u+7) of pair row i (tile t's row j is
// i = 128t + j) at (u * 256 + i) * 16, then (max, sum) per pair row.
template <int D> struct PairXchg {
    static constexpr uint32_t kPartBytes = (D / 8) * 2 * kBM * 16;
    static __device__ uint32_t part(uint32_t sK) { return sK; }
    static __device__ uint32_t ml(uint32_t sK) { return sK + kPartBytes; }
};
static_assert(PairXchg<128>::kPartBytes + 2 * kBM * 8 <= 2 * kPStages * PairLayout<128>::kKBytes,
              "two-tile exchange fits the K and V rings");
static_assert(PairXchg<64>::kPartBytes + 2 * kBM * 8 <= 2 * kPStages * PairLayout<64>::kKBytes,
              "two-tile exchange fits the K and V rings");

// Split combine of one pair row over the S CTAs of the cluster: the thread
// combines the units of its row in the CTA's range and stages them (tile
// prow / 128 of the two staged tiles at `stage`).
template <int D, int S>
__device__ __forceinline__ void pair_merge(int sp, uint32_t part, uint32_t ml, int prow, uint32_t stage)
{
    constexpr int kUnits = D / 8;
    constexpr int kMine = (kUnits + S - 1) / S;
    const int u0 = split_unit_begin(sp, S, kUnits), u1 = split_unit_begin(sp + 1, S, kUnits);
    float ms[S], ls[S];
#pragma unroll
    for (int s2 = 0; s2 < S; ++s2) {
        const float2 v = dsmem_ld_f2(dsmem_addr(ml + (uint32_t)prow * 8u, (uint32_t)s2));
        ms[s2] = v.x;
        ls[s2] = v.y;
    }
    float M = -INFINITY;
    bool bad = false;
#pragma unroll
    for (int s2 = 0; s2 < S; ++s2) {
        M = fmaxf(M, ms[s2]);
        bad = bad || ls[s2] < 0.f;
    }
    float coef[S], Lsum = 0.f;
#pragma unroll
    for (int s2 = 0; s2 < S; ++s2) {
        const float wt = (M == -INFINITY) ? 0.f : ex2(ms[s2] - M);
        coef[s2] = wt * fmaxf(ls[s2], 0.f);  // every partial was divided by its own sum
        Lsum += coef[s2];
    }
    const float sc = (bad || !(Lsum > 0.f)) ? 0.f : 1.f / Lsum;
    // every partial unit is in flight before the first is used (each CTA
    // wrote all of its units, zeros for a void row)
    uint4 rem[kMine][S];
#pragma unroll
    for (int k = 0; k < kMine; ++k) {
        const int u = u0 + k;
#pragma unroll
        for (int s2 = 0; s2 < S; ++s2)
            rem[k][s2] = u < u1 ? dsmem_ld_v4(dsmem_addr(part + ((uint32_t)u * 2u * kBM + (uint32_t)prow) * 16u,
                                                         (uint32_t)s2))
                                : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < kMine; ++k) {
        const int u = u0 + k;
        if (u >= u1)
            break;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s2 = 0; s2 < S; ++s2) {
            if (coef[s2] == 0.f || sc == 0.f)
                continue;
            const uint32_t wd[4] = {rem[k][s2].x, rem[k][s2].y, rem[k][s2].z, rem[k][s2].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[2 * e] += coef[s2] * __uint_as_float(wd[e] << 16);
                acc[2 * e + 1] += coef[s2] * __uint_as_float(wd[e] & 0xffff0000u);
            }
        }
        smem_st_v4(stage_addr(stage + (uint32_t)(prow >> 7) * (kBM * D * 2), prow & 127, u), pack8(acc, sc));
    }
}

// The attention of two-tile work unit `unit`; p.MT counts tile pairs here.
template <int D>
__device__ __forceinline__ void attn_pair_body(unsigned unit, const CUtensorMap *tm_q, const CUtensorMap *tm_kp,
                                               const CUtensorMap *tm_vp, const CUtensorMap *tm_kn,
                                               const CUtensorMap *tm_vn, const CUtensorMap *tm_o,
                                          const AttnParams &p)
{
    using Lay = PairLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- unit: ((r * Hkv + hk) * pairs + mp) * S + sp
    unsigned u = unit;
    const int sp = (int)(u % (unsigned)p.S);
    u /= (unsigned)p.S;
    const int mp = (int)(u % (unsigned)p.MT);
    u /= (unsigned)p.MT;
    const int hk = (int)(u % (unsigned)p.Hkv);
    const int r = (int)(u / (unsigned)p.Hkv);
    int32_t *status = reinterpret_cast<int32_t *>(p.ws);
    if (tid == 0)
        pdl_trigger();
    // the request's offsets: loaded now, checked once the setup below is done
    // (the setup does not depend on them and hides their latency)
    // (after a kernel whose output this one may read, nothing is read before
    // it has finished: the offsets load after the setup then)
    ReqRaw braw{};
    if (!p.wait_first)
        braw = load_bounds(p.cu_prefix, p.cu_q, p.cu_seg, r);
    const int mt0 = 2 * mp;  // first query tile of the pair

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

    if (tid == 0) {
        mbar_init(bar(P_Q), 1);
        mbar_init(bar(P_Q + 1), 1);
        for (int i = 0; i < kPStages; ++i) {
            mbar_init(bar(P_KF + i), 1);
            mbar_init(bar(P_KE + i), 1);
            mbar_init(bar(P_VF + i), 1);
            mbar_init(bar(P_VE + i), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(P_SF + t), 1);
            mbar_init(bar(P_PR + t), 4);
            mbar_init(bar(P_OW + t), 1);
        }
        mbar_init(bar(P_MASK), 256);
        mbar_init(bar(P_DONE), 1);
        *abort_flag = 0u;
        mask[0] = mask[1] = 0u;
        fence_barrier_init();
    }
    if (warp == kPairTmaWarp && lane == 0) {
        prefetch_tmap(tm_q);
        prefetch_tmap(tm_kp);
        prefetch_tmap(tm_vp);
        prefetch_tmap(tm_kn);
        prefetch_tmap(tm_vn);
        prefetch_tmap(tm_o);
    }
    if (warp == kPairMmaWarp) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // the offsets are used only from here on (the empty asm keeps the compiler
    // from moving their first use, and so the wait for the loads, above the
    // barrier); early exits are uniform over the CTAs of a cluster (same r and
    // pair) and come before any copy or cluster barrier
    if (p.wait_first) {  // the kernel ahead has finished and its writes are visible after this
        pdl_wait();
        braw = load_bounds(p.cu_prefix, p.cu_q, p.cu_seg, r);
    }
    if (!p.one_request)  // a single request's bounds come from the host: nothing to wait for here
        asm volatile("" : "+r"(braw.q0), "+r"(braw.q1), "+r"(braw.p0), "+r"(braw.p1), "+r"(braw.s0), "+r"(braw.s1));
    ReqBounds b;
    const bool bounds_ok = kernel_bounds(p, braw, b);
    if (!bounds_ok || mt0 * p.TQ >= b.n_q) {
        if (!bounds_ok && tid == 0 && sp == 0)
            record_status(status, D3D_ERR_DEVICE_INPUT);
        if (warp == kPairMmaWarp)
            tmem_dealloc(tmem, kTmemCols);
        pdl_wait();
        return;
    }

    // ---- this split's key list: prefix tiles [pb, pe), then (last split only) packed tiles
    const int nP = (b.L + kBN - 1) / kBN;
    const int pb = split_prefix_begin(sp, p.S, nP, p.PK);
    const int pe = (sp == p.S - 1) ? nP : split_prefix_begin(sp + 1, p.S, nP, p.PK);
    const int n_pre = pe - pb;
    const bool last_split = sp == p.S - 1;

    // number of packed tiles of the pair; waits for the mask on first use
    // (called by whole warps: the vote keeps the answer warp-uniform)
    int npk_cache = -1;
    uint32_t mk0 = 0, mk1 = 0;
    auto npk = [&]() -> int {
        if (npk_cache < 0) {
            if (!__all_sync(0xffffffffu, wait_bar(bar(P_MASK), 0, abort_flag, status)))
                return -1;
            mk0 = *(volatile uint32_t *)&mask[0];
            mk1 = *(volatile uint32_t *)&mask[1];
            npk_cache = __popc(mk0) + __popc(mk1);
        }
        return npk_cache;
    };
    // does list tile k of this split exist (-1: gave up waiting)
    auto exists = [&](int k) -> int {
        if (k < n_pre)
            return 1;
        if (!last_split)
            return 0;
        const int c = npk();
        return c < 0 ? -1 : (k - n_pre < c ? 1 : 0);
    };
    // global K/V row of list tile k (call only when it exists)
    auto tile_row = [&](int k, bool &pre) -> int {
        pre = k < n_pre;
        return pre ? b.p0 + (pb + k) * kBN : b.q0 + nth_set_bit(mk0, mk1, k - n_pre) * kBN;
    };

    bool mg_on = false;  // a softmax thread that reached the epilogue
    int mg_prow = 0;
    // output row of staged pair row i (tile i / 128), or null beyond the request
    auto out_row = [&](int i) -> uint16_t * {
        const int tok = (mt0 + (i >> 7)) * p.TQ + (i & 127) / p.G;
        if (tok >= b.n_q || !dbg_ok(b.q0 + tok < p.total_q && hk * p.G + ((i & 127) % p.G) < p.Hq, status))
            return nullptr;
        return p.out + ((size_t)(b.q0 + tok) * p.Hq + hk * p.G + ((i & 127) % p.G)) * D;
    };


    if (warp == kPairTmaWarp) {
        // =================== TMA producer ===================
        // issue order = the tensor core's consumption order: Q0, K0, Q1, K1,
        // then V(k), K(k+2) for k = 0, 1, ...
        const bool leader = elect_one();
        int nk = 0, nv = 0;     // K / V tiles handled, in list order
        bool skipped0 = false;  // the injected fault left K tile 0 unissued
        auto load_q = [&](int t) {
            if (leader) {
                mbar_arrive_expect_tx(bar(P_Q + t), Lay::kQBytes);
                for (int cb = 0; cb < D / 64; ++cb)
                    tma_load_3d(sQ + (uint32_t)t * Lay::kQBytes + cb * kBlockBytes, tm_q, bar(P_Q + t), cb * 64,
                                hk * p.G, b.q0 + (mt0 + t) * p.TQ);
            }
            __syncwarp();
        };
        load_q(0);
        auto issue = [&](int k, bool is_k) -> bool {
            const int s = k % kPStages;
            const int empty = is_k ? P_KE : P_VE, full = is_k ? P_KF : P_VF;
            if (k >= kPStages &&
                !__all_sync(0xffffffffu, wait_bar(bar(empty + s), ((k - kPStages) / kPStages) & 1, abort_flag, status)))
                return false;
            ++(is_k ? nk : nv);
            if (p.fault == 1 && is_k && k == 0) {
                skipped0 = true;  // injected fault: this tile never arrives
                return true;
            }
            bool pre;
            int row = tile_row(k, pre);
            // debug build: the tile's first row lies in the request's prefix or
            // packed rows (else the copy reads row 0 and the status says so)
            if (!dbg_ok(pre ? (row >= b.p0 && row < b.p0 + b.L) : (row >= b.q0 && row < b.q0 + b.n_q), status))
                row = 0;
            const CUtensorMap *m = is_k ? (pre ? tm_kp : tm_kn) : (pre ? tm_vp : tm_vn);
            const uint32_t dst = (is_k ? sK : sV) + s * Lay::kKBytes;
            if (leader) {
                mbar_arrive_expect_tx(bar(full + s), Lay::kKBytes);
                for (int cb = 0; cb < D / 64; ++cb)
                    tma_load_3d(dst + cb * kBlockBytes, m, bar(full + s), cb * 64, hk, row);
            }
            __syncwarp();
            return true;
        };
        bool ok = true;
        for (int k = 0; k < 2; ++k) {
            if (ok) {
                const int e = exists(k);
                ok = e >= 0;
                if (e == 1)
                    ok = issue(k, true);
            }
            if (k == 0)
                load_q(1);  // always issued: the drain below waits for it
        }
        for (int k = 0; ok; ++k) {
            const int e = exists(k);
            if (e != 1)
                break;
            ok = issue(k, false);
            const int e2 = ok ? exists(k + 2) : -1;
            if (e2 < 0)
                break;
            if (e2 == 1)
                ok = issue(k + 2, true);
        }
        // every copy this warp started must land before the CTA exits
        auto issued = [](int n, int s, int ns) { return n > s ? (n - 1 - s) / ns + 1 : 0; };
        wait_drain(bar(P_Q), 0, status);
        wait_drain(bar(P_Q + 1), 0, status);
        for (int s = 0; s < kPStages; ++s) {
            const int ck = issued(nk, s, kPStages) - ((s == 0 && skipped0) ? 1 : 0);
            if (ck > 0)
                wait_drain(bar(P_KF + s), (ck - 1) & 1, status);
            const int cv = issued(nv, s, kPStages);
            if (cv > 0)
                wait_drain(bar(P_VF + s), (cv - 1) & 1, status);
        }
        __syncwarp();
    } else if (warp == kPairMmaWarp) {
        // =================== MMA issuer ===================
        const bool leader = elect_one();
        constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, 0, 0);
        constexpr uint32_t idO = idesc_bf16_f32(kBM, D, 0, 1);
        auto wait_all = [&](uint32_t bar_addr, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, wait_bar(bar_addr, parity, abort_flag, status));
        };
        // S_t(k) = Q_t K_k^T into columns [128t, 128t + 128); the K stage is
        // released after S_1(k)
        auto issue_s = [&](int t, int k) {
            const int ks = k % kPStages;
            const uint32_t tS = tmem + (uint32_t)t * kBN;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * kBlockBytes + (kk % 4) * 32;
                    const uint64_t a = sdesc_sw128(sQ + (uint32_t)t * Lay::kQBytes + off, 16, 1024);
                    const uint64_t bd = sdesc_sw128(sK + ks * Lay::kKBytes + off, 16, 1024);
                    mma_bf16_ss(tS, a, bd, idS, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(P_SF + t));
                if (t == 1)
                    mma_commit(bar(P_KE + ks));
            }
            __syncwarp();
        };
        // O_t += P_t(k) V_k with P_t read from the first half of its S columns;
        // the V stage is released after PV_1(k)
        auto issue_pv = [&](int t, int k) {
            const int vs = k % kPStages;
            const uint32_t tP = tmem + (uint32_t)t * kBN, tO = tmem + 2u * kBN + (uint32_t)t * kBN;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint64_t bd = sdesc_sw128(sV + vs * Lay::kKBytes + kk * 2048, kBlockBytes, 1024);
                    mma_bf16_ts(tO, tP + kk * 8, bd, idO, (k > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar(P_OW + t));
                if (t == 1)
                    mma_commit(bar(P_VE + vs));
            }
            __syncwarp();
        };
        bool ok = wait_all(bar(P_Q), 0);
        if (ok) {
            const int e = exists(0);
            ok = e >= 0;
            if (e == 1) {
                ok = wait_all(bar(P_KF), 0);
                if (ok) {
                    tc_fence_after();
                    issue_s(0, 0);
                    ok = wait_all(bar(P_Q + 1), 0);
                }
                if (ok) {
                    tc_fence_after();
                    issue_s(1, 0);
                }
            }
        }
        // per key tile k and query tile t: PV_t(k) once P_t(k) is written, then
        // S_t(k+1) into the columns PV_t(k) has just read
        for (int k = 0; ok; ++k) {
            const int e = exists(k);
            if (e != 1) {
                ok = e >= 0;
                break;
            }
            const int e1 = exists(k + 1);
            ok = e1 >= 0 && wait_all(bar(P_VF + k % kPStages), (k / kPStages) & 1);
            for (int t = 0; ok && t < 2; ++t) {
                ok = wait_all(bar(P_PR + t), k & 1);
                if (!ok)
                    break;
                tc_fence_after();
                issue_pv(t, k);
                if (e1 == 1) {
                    if (t == 0)
                        ok = wait_all(bar(P_KF + (k + 1) % kPStages), ((k + 1) / kPStages) & 1);
                    if (ok) {
                        tc_fence_after();
                        issue_s(t, k + 1);
                    }
                }
            }
        }
        // every MMA is complete when P_DONE fires; TMEM is released only after it
        if (leader)
            mma_commit(bar(P_DONE));
        __syncwarp();
        wait_drain(bar(P_DONE), 0, status);
        __syncwarp();
    } else if (warp < kPairTmaWarp) {
        // =================== softmax: warpgroup t, query tile t ===================
        const int t = warp >> 2;
        const int row = tid & 127;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + (uint32_t)t * kBN;
        const uint32_t tO = tmem + lane_off + 2u * kBN + (uint32_t)t * kBN;
        const int token = (mt0 + t) * p.TQ + row / p.G;
        const bool row_valid = token < b.n_q;
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
            for (int i = tid; i < n_seg * 5; i += 256)
                dst[i] = src[i];
            asm volatile("bar.sync 1, 256;" ::: "memory");
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
        mbar_arrive(bar(P_MASK));

        float m_ref = -INFINITY, l = 0.f;
        bool aborted = false;
        int n_done = 0;
        for (int k = 0;; ++k) {
            const int ex = exists(k);
            if (!__all_sync(0xffffffffu, ex >= 0)) {
                aborted = true;
                break;
            }
            if (ex == 0)
                break;
            bool ok = wait_bar(bar(P_SF + t), k & 1, abort_flag, status);
            if (!__all_sync(0xffffffffu, ok)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            bool pre;
            const int krow = tile_row(k, pre);
            // a prefix tile with all 128 keys in range is visible to every row
            // in full (uniform over the CTA): no mask
            const bool full = pre && b.L - (pb + k) * kBN >= kBN;
            // this row's visible keys of 32-key word q of the tile, for a tile that
            // is not full: the valid ones of the last prefix tile, the two
            // half-open intervals of a packed tile
            auto word_bits = [&](int q) -> uint32_t {
                const int c0 = 32 * q;  // first key column of the word
                if (pre)
                    return range_bits(0, b.L - (pb + k) * kBN - c0);
                const int base = krow - b.q0 + c0;
                return range_bits(vis.own_lo - base, vis.own_hi - base) |
                       range_bits(vis.par_lo - base, vis.par_hi - base);
            };
            // pass 1: the row max from the whole S row (four loads in flight, one
            // wait; eight chains of three-input maxima)
            float mrow;
            {
                float s[kBN];
                tmem_ld32x4(tS, s);
                if (!full) {
                    uint32_t wb[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        wb[q] = word_bits(q);
#pragma unroll
                    for (int e = 0; e < kBN; ++e)
                        s[e] = ((wb[e >> 5] >> (e & 31)) & 1u) ? s[e] : -INFINITY;
                }
                float m8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    m8[e] = fmax3(s[e], s[8 + e], s[16 + e]);
#pragma unroll
                for (int j = 24; j + 16 <= kBN; j += 16)
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        m8[e] = fmax3(m8[e], s[j + e], s[j + 8 + e]);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    m8[e] = fmaxf(m8[e], s[kBN - 8 + e]);
                mrow = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
            }
            const float mx = mrow * p.scale_log2;
            float factor = 1.f;
            if (mx > m_ref + kRescaleLog2) {
                factor = ex2(m_ref - mx);  // 0 when m_ref = -inf
                m_ref = mx;
            }
            const float msub = (m_ref == -INFINITY) ? 0.f : m_ref;
            // pass 2, per 32-key chunk c (loaded again while the previous chunk is
            // computed): the exponentials and the row sum (packed pairs, two sum
            // chains of two lanes each), P as bf16 pairs over columns
            // [16c, 16c + 16) of S_t -- S columns whose load has completed.
            float r4[4] = {0.f, 0.f, 0.f, 0.f};
            float sc[2][32];
            tmem_ld32_async(tS, sc[0]);
            tmem_wait_ld32(sc[0]);
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) {
                float (&v)[32] = sc[c & 1];
                if (c + 1 < kBN / 32)
                    tmem_ld32_async(tS + (uint32_t)(32 * (c + 1)), sc[(c + 1) & 1]);
                if (!full) {
                    const uint32_t wbits = word_bits(c);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        v[e] = ((wbits >> e) & 1u) ? v[e] : -INFINITY;
                }
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float x0, x1, e0, e1;
                    ffma2(x0, x1, v[2 * e], v[2 * e + 1], p.scale_log2, p.scale_log2, -msub, -msub);
                    e0 = ex2(x0);
                    e1 = ex2(x1);
                    float &ra = r4[2 * (e & 1)], &rb = r4[2 * (e & 1) + 1];
                    fadd2(ra, rb, ra, rb, e0, e1);
                    pk[e] = pack_bf16x2(e0, e1);
                }
                if (c + 1 < kBN / 32)
                    tmem_wait_ld32(sc[(c + 1) & 1]);
                tmem_st16(tS + (uint32_t)(16 * c), pk);
            }
            l = l * factor + (r4[0] + r4[1]) + (r4[2] + r4[3]);
            // rescale the thread's O_t row once PV_t(k-1) has landed (rare: only
            // when the max grows by more than 2^8)
            if (k > 0 && __any_sync(0xffffffffu, factor != 1.f)) {
                ok = wait_bar(bar(P_OW + t), (k - 1) & 1, abort_flag, status);
                if (!__all_sync(0xffffffffu, ok)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    float o[32];
                    tmem_ld32(tO + (uint32_t)(q * 32), o);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        o[e] *= factor;
                    tmem_st32(tO + (uint32_t)(q * 32), o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(P_PR + t));
            n_done = k + 1;
        }

        // ---- epilogue: every MMA done; the thread owns its whole row
        wait_drain(bar(P_DONE), 0, status);
        // a single request whose device offsets disagree with the host's: every row is void
        const bool bad_req = p.one_request && !one_request_matches(p, braw);
        if (bad_req && tid == 0 && sp == 0)
            record_status(status, D3D_ERR_DEVICE_INPUT);
        const bool void_row = aborted || row_bad || bad_req;
        const float inv = (void_row || !(l > 0.f)) ? 0.f : 1.f / l;
        const bool have = n_done > 0;
        const int prow = t * kBM + row;
        const uint32_t part = PairXchg<D>::part(sK);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
            float o[64];
            if (have) {
                tc_fence_after();
                tmem_ld64(tO + (uint32_t)(h * 64), o);
            } else {
#pragma unroll
                for (int e = 0; e < 64; ++e)
                    o[e] = 0.f;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint4 v = pack8(o + 8 * q, inv);
                if (p.S == 1) {
                    // staged over the tile's own Q (free once every MMA is done)
                    smem_st_v4(stage_addr(sQ + (uint32_t)t * Lay::kQBytes, row, h * 8 + q), v);
                } else {
                    // the CTA's partial for the cluster's combine (every MMA is done)
                    const uint32_t unit8 = (uint32_t)(h * 8 + q);
                    smem_st_v4(part + (unit8 * 2u * kBM + (uint32_t)prow) * 16u, v);
                }
            }
        }
        if (p.S > 1)
            smem_st_f2(PairXchg<D>::ml(sK) + (uint32_t)prow * 8u, make_float2(m_ref, void_row ? -1.f : l));
        if (!aborted && row_valid && row_bad)
            record_status(status, D3D_ERR_DEVICE_INPUT);
        if (p.S == 1) {
            // a tile whose rows all belong to the request leaves by tensor stores
            // of the staged column blocks (one thread), another by plain stores
            const uint32_t stage = sQ + (uint32_t)t * Lay::kQBytes;
            fence_async_smem();
            if (t == 0)
                asm volatile("bar.sync 2, 128;" ::: "memory");
            else
                asm volatile("bar.sync 3, 128;" ::: "memory");
            if ((mt0 + t + 1) * p.TQ <= b.n_q) {
                if (row == 0) {
                    for (int cb = 0; cb < D / 64; ++cb)
                        tma_store_3d(tm_o, stage + (uint32_t)cb * kBlockBytes, cb * 64, hk * p.G,
                                     b.q0 + (mt0 + t) * p.TQ);
                    bulk_commit();
                    bulk_wait_read();
                }
            } else {
                store_staged(stage, 0u, kBM, 0, D / 8, row, kBM, [&](int i) { return out_row(t * kBM + i); });
            }
        }
        mg_on = true;
        mg_prow = prow;
    }

    // ---- every role is done (all waits are bounded, copies and MMAs drained)
    tc_fence_before();
    __syncthreads();
    if (p.S > 1) {
        // split combine across the cluster: every thread of every CTA passes
        // both cluster barriers exactly once
        cluster_arrive();
        cluster_wait();
        if (mg_on) {
            const uint32_t part = PairXchg<D>::part(sK), ml = PairXchg<D>::ml(sK);
            switch (p.S) {
            case 2: pair_merge<D, 2>(sp, part, ml, mg_prow, sQ); break;
            case 3: pair_merge<D, 3>(sp, part, ml, mg_prow, sQ); break;
            case 4: pair_merge<D, 4>(sp, part, ml, mg_prow, sQ); break;
            case 5: pair_merge<D, 5>(sp, part, ml, mg_prow, sQ); break;
            case 6: pair_merge<D, 6>(sp, part, ml, mg_prow, sQ); break;
            case 7: pair_merge<D, 7>(sp, part, ml, mg_prow, sQ); break;
            default: pair_merge<D, 8>(sp, part, ml, mg_prow, sQ); break;
            }
            fence_async_smem();
            asm volatile("bar.sync 2, 256;" ::: "memory");
            // the CTA's units of a tile leave by tensor stores when they are whole
            // column blocks and the tile's rows all belong to the request
            const int u0 = split_unit_begin(sp, p.S, D / 8), u1 = split_unit_begin(sp + 1, p.S, D / 8);
            auto by_tma = [&](int t) { return u0 % 8 == 0 && u1 % 8 == 0 && (mt0 + t + 1) * p.TQ <= b.n_q; };
            if (mg_prow == 0) {
                bool any = false;
                for (int t = 0; t < 2; ++t) {
                    if (!by_tma(t))
                        continue;
                    for (int cb = u0 / 8; cb < u1 / 8; ++cb)
                        tma_store_3d(tm_o, sQ + (uint32_t)t * Lay::kQBytes + (uint32_t)cb * kBlockBytes, cb * 64,
                                     hk * p.G, b.q0 + (mt0 + t) * p.TQ);
                    any = true;
                }
                if (any) {
                    bulk_commit();
                    bulk_wait_read();
                }
            }
            store_staged(sQ, Lay::kQBytes, 2 * kBM, u0, u1, mg_prow, 2 * kBM,
                         [&](int i) { return by_tma(i >> 7) ? nullptr : out_row(i); });
        }
        // no CTA leaves while another may still read its shared memory
        cluster_arrive();
        cluster_wait();
    }
    // release TMEM
    if (warp == kPairMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    pdl_wait();
}

template <int D>
__global__ void __launch_bounds__(kPairThreads, 1)
    attn_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kp,
                     const __grid_constant__ CUtensorMap tm_vp, const __grid_constant__ CUtensorMap tm_kn,
                     const __grid_constant__ CUtensorMap tm_vn, const __grid_constant__ CUtensorMap tm_o,
                   const AttnParams p)
{
    attn_pair_body<D>(blockIdx.x, &tm_q, &tm_kp, &tm_vp, &tm_kn, &tm_vn, &tm_o, p);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// Kernel the plan is restricted to (d3d_debug_force_attn_kernel): 0 any,
// 1 one tile per CTA, 2 two tiles per CTA, 3 CTA pairs.
inline int &forced_attn_kernel()
{
    static int kind = 0;
    return kind;
}

struct AttnPlan {
    int G, TQ, MT, S, PK;
    bool pair;  // two query tiles per CTA (attn_pair_kernel); MT then counts tile pairs
    bool duo;   // one query tile per CTA, CTA pairs sharing MMAs (attn_duo_kernel); MT then even, S = 1
    long long units;
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

template <int D> cudaError_t set_smem_attr()
{
    return set_max_dyn_smem<attn_tc_kernel<D>>((int)Layout<D>::alloc);
}

// The CTA-pair kernel (head dim 128 only): its shared-memory attribute and the
// CTAs resident at once in clusters of two (one CTA per SM), cached per
// device; 0 when the query fails or the kernel does not apply.
template <int D> int duo_capacity()
{
    if constexpr (D != 128) {
        return 0;
    } else {
        constexpr int kDev = 64;
        static std::mutex mu;
        static int cache[kDev];
        static bool have[kDev];
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDev) {
            cudaGetLastError();
            return 0;
        }
        std::lock_guard<std::mutex> lock(mu);
        if (!have[dev]) {
            int n = 0;
            if (set_max_dyn_smem<attn_duo_kernel<D>>((int)Layout<D, true>::alloc) == cudaSuccess) {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(128u);
                cfg.blockDim = dim3(kThreads);
                cfg.dynamicSmemBytes = Layout<D, true>::alloc;
                cudaLaunchAttribute a[1];
                a[0].id = cudaLaunchAttributeClusterDimension;
                a[0].val.clusterDim.x = 2;
                a[0].val.clusterDim.y = 1;
                a[0].val.clusterDim.z = 1;
                cfg.attrs = a;
                cfg.numAttrs = 1;
                if (cudaOccupancyMaxActiveClusters(&n, attn_duo_kernel<D>, &cfg) != cudaSuccess) {
                    cudaGetLastError();
                    n = 0;
                }
            } else {
                cudaGetLastError();
            }
            cache[dev] = 2 * n;
            have[dev] = true;
        }
        return cache[dev];
    }
}

// CTAs of the attention kernel resident at once when launched in clusters of
// S (one CTA per SM; a cluster needs S free SMs of one GPC).  Cached per
// device and S; 0 when the query fails.
// The two-tile kernel's shared-memory attribute, and whether one CTA of it
// fits an SM (its registers per thread decide that); the plan uses it only
// then.  Cached per device.
template <int D> cudaError_t set_pair_smem_attr()
{
    const cudaError_t e = set_max_dyn_smem<attn_pair_kernel<D>>((int)PairLayout<D>::alloc);
    if (e != cudaSuccess)
        return e;
    static std::mutex mu;
    static int fits[64];  // 0 unknown, 1 fits, 2 does not
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return cudaErrorInvalidDevice;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (fits[dev] == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_pair_kernel<D>, kPairThreads,
                                                          PairLayout<D>::alloc) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        fits[dev] = n >= 1 ? 1 : 2;
    }
    return fits[dev] == 1 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

// CTAs of the one-tile (pair = false) or two-tile attention kernel resident
// at once when launched in clusters of S (one CTA per SM; a cluster needs S
// free SMs of one GPC).  Cached per device, kernel and S; 0 when the query
// fails.
template <int D> int cluster_capacity(int S, bool pair = false)
{
    constexpr int kDev = 64;
    static std::mutex mu;
    static int cache[kDev][2][kMaxSplits + 1];
    static bool have[kDev][2][kMaxSplits + 1];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDev) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev][pair][S]) {
        int n = 0;
        if ((pair ? set_pair_smem_attr<D>() : set_smem_attr<D>()) == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(S * 64));
            cfg.blockDim = dim3(pair ? kPairThreads : kThreads);
            cfg.dynamicSmemBytes = pair ? PairLayout<D>::alloc : Layout<D>::alloc;
            cudaLaunchAttribute a[1];
            a[0].id = cudaLaunchAttributeClusterDimension;
            a[0].val.clusterDim.x = (unsigned)S;
            a[0].val.clusterDim.y = 1;
            a[0].val.clusterDim.z = 1;
            cfg.attrs = a;
            cfg.numAttrs = 1;
            const cudaError_t e = pair ? cudaOccupancyMaxActiveClusters(&n, attn_pair_kernel<D>, &cfg)
                                       : cudaOccupancyMaxActiveClusters(&n, attn_tc_kernel<D>, &cfg);
            if (e != cudaSuccess) {
                cudaGetLastError();
                n = 0;
            }
        }
        cache[dev][pair][S] = n * S;
        have[dev][pair][S] = true;
    }
    return cache[dev][pair][S];
}

// Kernel and split count S (a cluster of S CTAs per query tile or tile
// pair): minimise (waves of resident CTAs) x (the CTA's time: its key tiles
// times the cost of one, plus a fixed per-CTA cost for the prologue,
// pipeline fill and epilogue, plus the cluster combine when splitting).
// Costs in units of one key tile of the one-tile kernel (about 1,900 cycles:
// bound by the rate at which an SM receives K/V tiles), measured on GB300:
// 1.75 per key tile of the two-tile kernel (two query tiles per K/V tile; its
// softmax of one tile plus that tile's MMAs make the step), 5 for the
// prologue (the first Q and K tiles' round trip) and epilogue, 3.5 for a
// cluster's combine (waiting for the slowest split, the exchange, the
// stores).  max_ctas > 0 caps the CTAs of one wave (the SMs left to a kernel
// running beside the attention).
template <int D>
AttnPlan make_plan(int R, int Hq, int Hkv, int max_q, int max_prefix, int max_ctas = 0, bool allow_duo = true)
{
    constexpr double kTileCost1 = 1.0, kTileCost2 = 1.75, kFixed = 5.0, kCombine = 3.5;
    AttnPlan pl{};
    pl.G = Hq / Hkv;
    pl.TQ = kBM / pl.G;
    const int MT = (max_q + pl.TQ - 1) / pl.TQ;
    pl.PK = (max_q + kBN - 1) / kBN < 2 ? (max_q + kBN - 1) / kBN : 2;
    const int tiles = (max_prefix + kBN - 1) / kBN + packed_tile_weight(pl.PK);  // in prefix-tile units
    int budget = num_sms();
    if (max_ctas > 0 && max_ctas < budget)
        budget = max_ctas;
    double best = 1e300;
    pl.MT = MT;
    pl.S = 1;
    pl.pair = false;
    pl.duo = false;
    // a forced kernel that does not apply here leaves the choice to the plan
    int force = forced_attn_kernel();
    if (force == 2 && (MT < 2 || set_pair_smem_attr<D>() != cudaSuccess))
        force = 0;
    if (force == 3 && (!allow_duo || duo_capacity<D>() < 2))
        force = 0;
    for (int pair = 0; pair < 2; ++pair) {
        if (pair && (MT < 2 || set_pair_smem_attr<D>() != cudaSuccess))
            continue;
        if ((force == 1 && pair) || (force == 2 && !pair) || force == 3)
            continue;
        const int units_m = pair ? (MT + 1) / 2 : MT;
        const long long base = (long long)R * Hkv * units_m;
        for (int S = 1; S <= kMaxSplits && S <= tiles; ++S) {
            int cap = S == 1 ? budget : cluster_capacity<D>(S, pair != 0);
            if (cap > budget)
                cap = budget / S * S;
            if (cap < S)
                continue;
            const double waves = (double)((base * S + cap - 1) / cap);
            const int per_split = (tiles + S - 1) / S;
            const double cost = waves * (per_split * (pair ? kTileCost2 : kTileCost1) + kFixed + (S > 1 ? kCombine : 0.0));
            if (cost < best - 1e-9) {
                best = cost;
                pl.S = S;
                pl.pair = pair != 0;
                pl.MT = units_m;
            }
        }
    }
    // CTA pairs: every query tile in its own CTA (tiles rounded up to pairs),
    // no key splits; each SM receives half of every K/V tile.  Measured on
    // GB300 slower than the one-tile kernel on every workload here (its MMAs
    // wait for the slower CTA's softmax of each tile, and it cannot split
    // keys), so the plan takes it only when d3d_debug_force_attn_kernel asks.
    constexpr double kTileCostDuo = 1.1;
    if (allow_duo && force == 3) {
        const int MT2 = (MT + 1) / 2 * 2;
        int cap = duo_capacity<D>();
        if (cap > budget)
            cap = budget / 2 * 2;
        if (cap >= 2) {
            const double waves = (double)(((long long)R * Hkv * MT2 + cap - 1) / cap);
            const double cost = waves * (tiles * kTileCostDuo + kFixed);
            if (cost < best - 1e-9 || force == 3) {
                best = cost;
                pl.S = 1;
                pl.pair = false;
                pl.duo = true;
                pl.MT = MT2;
            }
        }
    }
    pl.units = (long long)R * Hkv * pl.MT * pl.S;
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

template <int D>
int launch_attn(const CUtensorMap (&maps)[6], const AttnParams &prm, long long units, bool pair, bool duo, int flags,
                cudaStream_t stream)
{
    if (duo) {
        if (D != 128 || duo_capacity<D>() < 2 || units % 2 != 0)
            return D3D_ERR_INTERNAL;
    } else if ((pair ? set_pair_smem_attr<D>() : set_smem_attr<D>()) != cudaSuccess) {
        return D3D_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)units);
    cfg.blockDim = dim3(pair ? kPairThreads : kThreads);
    cfg.dynamicSmemBytes = pair ? PairLayout<D>::alloc : duo ? Layout<128, true>::alloc : Layout<D>::alloc;
    cfg.stream = stream;
    cudaLaunchAttribute a[2];
    unsigned na = 0;
    if (prm.S > 1 || duo) {  // the splits of one query tile, or a CTA pair, form a cluster (consecutive CTAs)
        a[na].id = cudaLaunchAttributeClusterDimension;
        a[na].val.clusterDim.x = duo ? 2u : (unsigned)prm.S;
        a[na].val.clusterDim.y = 1;
        a[na].val.clusterDim.z = 1;
        ++na;
    }
    if (flags & (D3D_ATTN_AFTER_INDEPENDENT | D3D_ATTN_AFTER_DEPENDENT)) {  // may start while the previous kernel runs
        a[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        a[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = na ? a : nullptr;
    cfg.numAttrs = na;
    if (pair)
        return cuda_status(
            cudaLaunchKernelEx(&cfg, attn_pair_kernel<D>, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], prm));
    if constexpr (D == 128) {
        if (duo)
            return cuda_status(
                cudaLaunchKernelEx(&cfg, attn_duo_kernel<D>, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], prm));
    }
    return cuda_status(cudaLaunchKernelEx(&cfg, attn_tc_kernel<D>, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], prm));
}

// Host-side checks of d3d_packed_draft_attn's arguments and the tensor maps,
// parameters and plan of its launch.  Returns D3D_OK, a status, or 1 when
// there is nothing to compute.
int attn_prepare(const void *q, const void *k_prefix, const void *v_prefix, const void *k_packed,
                 const void *v_packed, const d3d_segment_t *segs, const int32_t *cu_prefix, const int32_t *cu_q,
                 const int32_t *cu_seg, int R, int Hq, int Hkv, int d, int max_q, int max_prefix, int total_q,
                 int total_prefix, int total_segs, float scale, void *out, void *ws, size_t ws_bytes,
                 CUtensorMap (&maps)[6], AttnParams &prm, AttnPlan &pl, int max_ctas = 0, bool one_tile = false)
{
    if (R < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || max_q < 0 || max_prefix < 0 || total_q < 0 ||
        total_prefix < 0 || total_segs < 0 || !(scale > 0.f) || !isfinite(scale))
        return D3D_ERR_INVALID_ARG;
    if (d != 64 && d != 128)
        return D3D_ERR_UNSUPPORTED;
    if (kBM % (Hq / Hkv) != 0 || max_q > kMaxPackedTiles * kBN)
        return D3D_ERR_UNSUPPORTED;
    if (R == 0 || max_q == 0)
        return 1;
    if (!q || !k_packed || !v_packed || !segs || !cu_prefix || !cu_q || !cu_seg || !out ||
        (total_prefix > 0 && (!k_prefix || !v_prefix)) || total_q < 1)
        return D3D_ERR_INVALID_ARG;
    const void *aligned_ptrs[4] = {q, k_packed, v_packed, out};
    for (const void *ptr : aligned_ptrs)
        if (reinterpret_cast<uintptr_t>(ptr) % 16)
            return D3D_ERR_INVALID_ARG;
    if (total_prefix > 0 && (reinterpret_cast<uintptr_t>(k_prefix) % 16 || reinterpret_cast<uintptr_t>(v_prefix) % 16))
        return D3D_ERR_INVALID_ARG;
    if (!ws_ok(ws, ws_bytes, sizeof(WsHeader)))
        return D3D_ERR_WORKSPACE;
    if (max_ctas < 0)
        return D3D_ERR_INVALID_ARG;
    pl = d == 64 ? make_plan<64>(R, Hq, Hkv, max_q, max_prefix, max_ctas, !one_tile)
                 : make_plan<128>(R, Hq, Hkv, max_q, max_prefix, max_ctas, !one_tile);
    if (one_tile && pl.pair) {  // the fused round launch holds the one-tile kernel only
        pl.pair = false;
        pl.S = 1;
        pl.MT = (max_q + pl.TQ - 1) / pl.TQ;
        pl.units = (long long)R * Hkv * pl.MT;
    }
    if (pl.units > 0x7fffffffLL)
        return D3D_ERR_UNSUPPORTED;
    // the output map has the query map's shape: a query tile's output box is
    // stored from the shared-memory staging in the same swizzled layout
    // (a CTA pair loads half of every K tile's keys per CTA)
    const int k_box = pl.duo ? kBN / 2 : kBN;
    if (!make_map(&maps[0], q, d, Hq, total_q, pl.G, pl.TQ) || !make_map(&maps[3], k_packed, d, Hkv, total_q, 1, k_box) ||
        !make_map(&maps[4], v_packed, d, Hkv, total_q, 1, kBN) || !make_map(&maps[5], out, d, Hq, total_q, pl.G, pl.TQ))
        return D3D_ERR_CUDA;
    if (total_prefix > 0) {
        if (!make_map(&maps[1], k_prefix, d, Hkv, total_prefix, 1, k_box) ||
            !make_map(&maps[2], v_prefix, d, Hkv, total_prefix, 1, kBN))
            return D3D_ERR_CUDA;
    } else {  // no prefix rows anywhere: the prefix maps are never used
        maps[1] = maps[3];
        maps[2] = maps[4];
    }
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
    prm.PK = pl.PK;
    prm.max_q = max_q;
    prm.max_prefix = max_prefix;
    prm.total_q = total_q;
    prm.total_prefix = total_prefix;
    prm.total_segs = total_segs;
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.fault = fault_mode();
    prm.one_request = R == 1 && total_q <= max_q && total_prefix <= max_prefix;
    prm.wait_first = 0;
    return D3D_OK;
}

// The fused round launch: n_attn attention CTAs, then n_verify verification
// CTAs, one per SM, cooperative.
template <int D, typename T>
int launch_round(const CUtensorMap (&maps)[6], const AttnParams &prm, int n_attn, const VArgs &va_in,
                 cudaStream_t stream)
{
    VArgs va = va_in;
    if (ring_fits<T, kNTLimited>(va) && Ring<kNTLimited>::bytes(kRingSlots) <= Layout<D>::alloc)
        va.ring = kRingSlots;  // the attention's shared memory holds the verification's phase-A ring
    const VerifyLayout L = verify_layout(va.R, va.B, va.V, VCfg<kNTLimited>::kChunk);
    const long long nA = (long long)va.R * va.B * L.nch;
    size_t dyn = verify_dyn_smem(va.B, L.nch);
    if (dyn < Layout<D>::alloc)
        dyn = Layout<D>::alloc;
    // the attention's carve-up is the larger one (a verification CTA stages at
    // most 32 KB of records); the static shared memory of the verification
    // part comes on top of it
    if (dyn > Layout<D>::alloc)
        return D3D_ERR_UNSUPPORTED;
    dyn = Layout<D>::alloc;
    const cudaError_t attr_err = set_max_dyn_smem<round_kernel<D, T>>((int)Layout<D>::alloc);
    int dev = 0, nsm = 0, per_sm = 0;
    if (attr_err != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, round_kernel<D, T>, kNTLimited, dyn) != cudaSuccess ||
        per_sm < 1) {
        cudaGetLastError();
        return D3D_ERR_CUDA;
    }
    if (n_attn >= nsm * per_sm || nA > 0x7fffffffLL)
        return D3D_ERR_UNSUPPORTED;
    const long long room = (long long)nsm * per_sm - n_attn;
    const int n_verify = (int)(nA < room ? nA : room);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_attn + n_verify));
    cfg.blockDim = dim3(kNTLimited);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, round_kernel<D, T>, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], prm,
                                          va, n_attn));
}

}  // namespace
}  // namespace d3d

extern "C" {

size_t d3d_packed_draft_attn_workspace_size(int R, int Hq, int Hkv, int d, int max_q, int max_prefix)
{
    if (R < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || max_q < 0 || max_prefix < 0 || (d != 64 && d != 128) ||
        d3d::kBM % (Hq / Hkv) != 0)
        return 0;
    return sizeof(d3d::WsHeader);  // the status word: the split combine needs no global scratch
}

int d3d_packed_draft_attn_ctas(int R, int Hq, int Hkv, int d, int max_q, int max_prefix, int max_ctas)
{
    if (R < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || max_q < 0 || max_prefix < 0 || max_ctas < 0)
        return D3D_ERR_INVALID_ARG;
    if (d != 64 && d != 128)
        return D3D_ERR_UNSUPPORTED;
    if (d3d::kBM % (Hq / Hkv) != 0 || max_q > d3d::kMaxPackedTiles * d3d::kBN)
        return D3D_ERR_UNSUPPORTED;
    if (R == 0 || max_q == 0)
        return 0;
    const d3d::AttnPlan pl = d == 64 ? d3d::make_plan<64>(R, Hq, Hkv, max_q, max_prefix, max_ctas)
                                     : d3d::make_plan<128>(R, Hq, Hkv, max_q, max_prefix, max_ctas);
    return pl.units > 0x7fffffffLL ? D3D_ERR_UNSUPPORTED : (int)pl.units;
}

void d3d_debug_inject_fault(int mode) { d3d::fault_mode() = mode; }

void d3d_debug_force_attn_kernel(int kind)
{
    if (kind >= 0 && kind <= 3)
        d3d::forced_attn_kernel() = kind;
}

int d3d_packed_draft_attn(const void *q, const void *k_prefix, const void *v_prefix, const void *k_packed,
                          const void *v_packed, const d3d_segment_t *segs, const int32_t *cu_prefix,
                          const int32_t *cu_q, const int32_t *cu_seg, int R, int Hq, int Hkv, int d, int max_q,
                          int max_prefix, int total_q, int total_prefix, int total_segs, float scale, void *out,
                          void *ws, size_t ws_bytes, int max_ctas, int flags, cudaStream_t stream)
{
    if ((flags & ~(D3D_ATTN_AFTER_INDEPENDENT | D3D_ATTN_AFTER_DEPENDENT)) != 0 ||
        (flags & D3D_ATTN_AFTER_INDEPENDENT && flags & D3D_ATTN_AFTER_DEPENDENT))
        return D3D_ERR_INVALID_ARG;
    CUtensorMap maps[6];
    d3d::AttnParams prm;
    d3d::AttnPlan pl;
    const int rc = d3d::attn_prepare(q, k_prefix, v_prefix, k_packed, v_packed, segs, cu_prefix, cu_q, cu_seg, R, Hq,
                                     Hkv, d, max_q, max_prefix, total_q, total_prefix, total_segs, scale, out, ws,
                                     ws_bytes, maps, prm, pl, max_ctas);
    if (rc != D3D_OK)
        return rc == 1 ? D3D_OK : rc;
    prm.wait_first = (flags & D3D_ATTN_AFTER_DEPENDENT) != 0;
    if (d == 64)
        return d3d::launch_attn<64>(maps, prm, pl.units, pl.pair, pl.duo, flags, stream);
    return d3d::launch_attn<128>(maps, prm, pl.units, pl.pair, pl.duo, flags, stream);
}

int d3d_async_round(const d3d_attn_call_t *a, const d3d_verify_call_t *v, cudaStream_t stream)
{
    if (!a || !v)
        return D3D_ERR_INVALID_ARG;
    // the verification's checks first: they make no CUDA call
    d3d::VArgs va;
    const int rv = d3d::verify_prepare(v->target_logits, v->draft_logits, v->logits_dtype, v->draft_tokens,
                                       v->u_accept, v->u_sample, v->R, v->B, v->V, v->temperature, v->accept_len,
                                       v->out_tokens, v->num_tokens, v->alpha, v->p_draft, v->q_draft,
                                       v->awl_weight, v->heads, v->head_len, v->M, v->branch, va);
    if (rv < 0)
        return rv;
    if (v->temperature == 0.f)  // greedy verification has its own launch
        return D3D_ERR_UNSUPPORTED;
    CUtensorMap maps[6];
    d3d::AttnParams prm;
    d3d::AttnPlan pl;
    const int ra = d3d::attn_prepare(a->q, a->k_prefix, a->v_prefix, a->k_packed, a->v_packed, a->segs, a->cu_prefix,
                                     a->cu_q, a->cu_seg, a->R, a->Hq, a->Hkv, a->d, a->max_q, a->max_prefix,
                                     a->total_q, a->total_prefix, a->total_segs, a->scale, a->out, a->ws,
                                     a->ws_bytes, maps, prm, pl, 0, true);
    if (ra < 0)
        return ra;
    if (ra == 1 || rv == 1)  // a part with nothing to compute: nothing to fuse
        return D3D_ERR_UNSUPPORTED;
    if (!d3d::ws_ok(v->ws, v->ws_bytes, d3d::verify_layout(v->R, v->B, v->V, d3d::kVChunkMin).total))
        return D3D_ERR_WORKSPACE;
    va.ws = static_cast<unsigned char *>(v->ws);
    if (pl.S != 1)  // the fused launch takes whole query tiles only (no key-split clusters)
        return D3D_ERR_UNSUPPORTED;
    const int n_attn = (int)pl.units;
    if (a->d == 64)
        return v->logits_dtype == D3D_DTYPE_BF16 ? d3d::launch_round<64, uint16_t>(maps, prm, n_attn, va, stream)
                                                 : d3d::launch_round<64, float>(maps, prm, n_attn, va, stream);
    return v->logits_dtype == D3D_DTYPE_BF16 ? d3d::launch_round<128, uint16_t>(maps, prm, n_attn, va, stream)
                                             : d3d::launch_round<128, float>(maps, prm, n_attn, va, stream);
}

}  // extern "C"
