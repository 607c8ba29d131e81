// Host-side pieces of the C ABI shared by all entry points: status text,
// version, workspace initialisation and status read-back, and the host check
// of a packed segment table.
#include <string.h>

#include "d3d_common.cuh"

extern "C" {

const char *d3d_status_string(int status)
{
    switch (status) {
    case D3D_OK: return "ok";
    case D3D_ERR_INVALID_ARG: return "invalid argument";
    case D3D_ERR_UNSUPPORTED: return "unsupported configuration";
    case D3D_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case D3D_ERR_CUDA: return "CUDA runtime error at enqueue time";
    case D3D_ERR_DEVICE_TIMEOUT: return "device: bounded wait expired";
    case D3D_ERR_DEVICE_INPUT: return "device: input data out of range";
    case D3D_ERR_INTERNAL: return "device: internal index check failed (debug build)";
    default: return "unknown status";
    }
}

int d3d_version(void) { return 10000 * 0 + 100 * 1 + 0; }

int d3d_workspace_init(void *ws, size_t bytes, cudaStream_t stream)
{
    if (ws == nullptr || bytes < sizeof(d3d::WsHeader))
        return D3D_ERR_WORKSPACE;
    return d3d::cuda_status(cudaMemsetAsync(ws, 0, bytes, stream));
}

int d3d_workspace_status(const void *ws, int32_t *status_host, int clear, cudaStream_t stream)
{
    if (ws == nullptr || status_host == nullptr)
        return D3D_ERR_INVALID_ARG;
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess)
        return D3D_ERR_CUDA;
    *status_host = v;
    if (clear && v != D3D_OK) {
        e = cudaMemsetAsync(const_cast<void *>(ws), 0, sizeof(int32_t), stream);
        if (e != cudaSuccess)
            return D3D_ERR_CUDA;
    }
    return D3D_OK;
}

int d3d_validate_segments(const d3d_segment_t *segs, const int32_t *cu_q, const int32_t *cu_seg, int R)
{
    if (R < 0)
        return D3D_ERR_INVALID_ARG;
    if (R == 0)
        return D3D_OK;
    if (cu_q == nullptr || cu_seg == nullptr || cu_q[0] != 0 || cu_seg[0] != 0)
        return D3D_ERR_INVALID_ARG;
    for (int r = 0; r < R; ++r) {
        const int32_t n_q = cu_q[r + 1] - cu_q[r];
        const int32_t s0 = cu_seg[r], s1 = cu_seg[r + 1];
        if (n_q < 0 || s1 < s0 || (s1 > s0 && segs == nullptr))
            return D3D_ERR_INVALID_ARG;
        int64_t next = 0;
        for (int32_t s = s0; s < s1; ++s) {
            const d3d_segment_t &g = segs[s];
            if (g.q_start != next || g.len < 1)
                return D3D_ERR_INVALID_ARG;
            if (g.mode != D3D_SEG_CAUSAL && g.mode != D3D_SEG_BIDIR)
                return D3D_ERR_INVALID_ARG;
            if (g.parent == -1) {
                if (g.parent_len != 0)
                    return D3D_ERR_INVALID_ARG;
            } else {
                if (g.parent < 0 || g.parent >= s - s0)
                    return D3D_ERR_INVALID_ARG;
                const d3d_segment_t &p = segs[s0 + g.parent];
                if (p.mode != D3D_SEG_CAUSAL || p.parent != -1)
                    return D3D_ERR_INVALID_ARG;
                if (g.parent_len < 0 || g.parent_len > p.len)
                    return D3D_ERR_INVALID_ARG;
            }
            next += g.len;
        }
        if (next != n_q)
            return D3D_ERR_INVALID_ARG;
    }
    return D3D_OK;
}

}  // extern "C"
