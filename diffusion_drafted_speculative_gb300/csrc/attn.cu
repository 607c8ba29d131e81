// Packed drafting attention (entry point and argument checks).
//
// [D3D] "Core method", "Method steps" steps 2 and 4; [DScout] "Background:
// block-diffusion drafter".  See attn_common.cuh for the visibility rule.
//
// This first kernel is a plain warp-per-row online-softmax loop on the CUDA
// cores: one warp per (packed token, query head), lanes split the head
// dimension, keys are visited in order (prefix, own interval, parent
// interval) so masked keys are never touched.
#include <math.h>

#include "attn_common.cuh"

namespace d3d {
namespace {

constexpr int kAThreads = 256;
constexpr int kAWarps = kAThreads / 32;

template <int D>
__global__ void __launch_bounds__(kAThreads)
    attn_rows_kernel(const uint16_t *__restrict__ q, const uint16_t *__restrict__ kp, const uint16_t *__restrict__ vp,
                     const uint16_t *__restrict__ kn, const uint16_t *__restrict__ vn,
                     const d3d_segment_t *__restrict__ segs, const int32_t *__restrict__ cu_prefix,
                     const int32_t *__restrict__ cu_q, const int32_t *__restrict__ cu_seg, int Hq, int Hkv, int max_q,
                     int max_prefix, int total_q, int total_prefix, int total_segs, float scale_log2,
                     uint16_t *__restrict__ out, int32_t *__restrict__ status)
{
    constexpr int E = D / 32;  // head-dim elements per lane
    const int r = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kAWarps + warp;
    ReqBounds b;
    if (!request_bounds(cu_prefix, cu_q, cu_seg, r, max_q, max_prefix, total_q, total_prefix, total_segs, b)) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            record_status(status, D3D_ERR_DEVICE_INPUT);
        return;
    }
    const int i = row / Hq, h = row % Hq;
    if (i >= b.n_q)
        return;
    uint16_t *orow = out + ((size_t)(b.q0 + i) * Hq + h) * D + lane * E;
    RowVis vis;
    if (!row_visibility(segs, b.s0, b.s1, b.n_q, i, vis)) {
        if (lane == 0)
            record_status(status, D3D_ERR_DEVICE_INPUT);
#pragma unroll
        for (int e = 0; e < E; ++e)
            orow[e] = 0;
        return;
    }
    const int hk = h / (Hq / Hkv);
    float qv[E], acc[E];
    const uint16_t *qrow = q + ((size_t)(b.q0 + i) * Hq + h) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        qv[e] = bf16_bits_to_float(qrow[e]) * scale_log2;
        acc[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    auto visit = [&](const uint16_t *krow, const uint16_t *vrow) {
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e)
            s += qv[e] * bf16_bits_to_float(krow[lane * E + e]);
#pragma unroll
        for (int o = 16; o; o >>= 1)
            s += __shfl_xor_sync(0xffffffffu, s, o);
        const float mn = fmaxf(m, s);
        const float corr = exp2f(m - mn), p = exp2f(s - mn);
        l = l * corr + p;
#pragma unroll
        for (int e = 0; e < E; ++e)
            acc[e] = acc[e] * corr + p * bf16_bits_to_float(vrow[lane * E + e]);
        m = mn;
    };
    for (int k = 0; k < b.L; ++k) {
        const size_t o = ((size_t)(b.p0 + k) * Hkv + hk) * D;
        visit(kp + o, vp + o);
    }
    for (int j = vis.own_lo; j < vis.own_hi; ++j) {
        const size_t o = ((size_t)(b.q0 + j) * Hkv + hk) * D;
        visit(kn + o, vn + o);
    }
    for (int j = vis.par_lo; j < vis.par_hi; ++j) {
        const size_t o = ((size_t)(b.q0 + j) * Hkv + hk) * D;
        visit(kn + o, vn + o);
    }
    const float inv = 1.f / l;
#pragma unroll
    for (int e = 0; e < E; ++e)
        orow[e] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[e] * inv));
}

}  // namespace
}  // namespace d3d

extern "C" {

size_t d3d_packed_draft_attn_workspace_size(int R, int Hq, int Hkv, int d, int max_q, int max_prefix)
{
    if (R < 0 || Hq < 1 || Hkv < 1 || max_q < 0 || max_prefix < 0)
        return 0;
    (void)d;
    return sizeof(d3d::WsHeader);
}

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
    if (128 % (Hq / Hkv) != 0)
        return D3D_ERR_UNSUPPORTED;
    if (R == 0 || max_q == 0)
        return D3D_OK;
    if (R > 65535)
        return D3D_ERR_UNSUPPORTED;
    if (!q || !k_packed || !v_packed || !segs || !cu_prefix || !cu_q || !cu_seg || !out ||
        (total_prefix > 0 && (!k_prefix || !v_prefix)))
        return D3D_ERR_INVALID_ARG;
    if (!d3d::ws_ok(ws, ws_bytes, d3d_packed_draft_attn_workspace_size(R, Hq, Hkv, d, max_q, max_prefix)))
        return D3D_ERR_WORKSPACE;
    const float scale_log2 = scale * 1.4426950408889634f;
    const size_t rows = (size_t)max_q * Hq;
    const dim3 grid((unsigned)((rows + d3d::kAWarps - 1) / d3d::kAWarps), (unsigned)R);
    auto *st = static_cast<int32_t *>(ws);
#define D3D_ATTN_ARGS                                                                                              \
    static_cast<const uint16_t *>(q), static_cast<const uint16_t *>(k_prefix),                                    \
        static_cast<const uint16_t *>(v_prefix), static_cast<const uint16_t *>(k_packed),                         \
        static_cast<const uint16_t *>(v_packed), segs, cu_prefix, cu_q, cu_seg, Hq, Hkv, max_q, max_prefix,       \
        total_q, total_prefix, total_segs, scale_log2, static_cast<uint16_t *>(out), st
    if (d == 64)
        d3d::attn_rows_kernel<64><<<grid, d3d::kAThreads, 0, stream>>>(D3D_ATTN_ARGS);
    else
        d3d::attn_rows_kernel<128><<<grid, d3d::kAThreads, 0, stream>>>(D3D_ATTN_ARGS);
#undef D3D_ATTN_ARGS
    return d3d::cuda_status(cudaGetLastError());
}

}  // extern "C"
