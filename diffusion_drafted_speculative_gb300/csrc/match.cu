// Branch cache-hit match.
//
// [D3D] "Background: asynchronous drafting and cache hits": a hit is an exact
// match of the verified prefix with the beginning (head) of a pre-drafted
// branch; the branch's remaining drafts are then reused.
//
// One warp per request.  Lane k compares head k0 + k with the verified prefix
// (lengths first, then tokens); a warp ballot gives the lowest matching
// index, so the lowest-index rule holds for duplicate heads.  Groups of 32
// heads are tried in order until one hits.
#include "d3d_common.cuh"

namespace d3d {
namespace {

constexpr int kMThreads = 128;

__global__ void __launch_bounds__(kMThreads)
    branch_match_kernel(const int32_t *__restrict__ verified, const int32_t *__restrict__ verified_len,
                        const int32_t *__restrict__ heads, const int32_t *__restrict__ head_len, int R, int M,
                        int B, int32_t *__restrict__ branch)
{
    const int req = (int)((blockIdx.x * (size_t)kMThreads + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (req >= R)
        return;
    const int n = __ldg(verified_len + req);
    const int32_t *v = verified + (size_t)req * B;
    int hit = -1;
    if (n >= 0 && n <= B) {
        for (int k0 = 0; k0 < M && hit < 0; k0 += 32) {
            const int k = k0 + lane;
            bool same = false;
            if (k < M && __ldg(head_len + (size_t)req * M + k) == n) {
                const int32_t *h = heads + ((size_t)req * M + k) * B;
                same = true;
                for (int i = 0; i < n; ++i)
                    if (__ldg(h + i) != __ldg(v + i)) {
                        same = false;
                        break;
                    }
            }
            const unsigned ballot = __ballot_sync(0xffffffffu, same);
            if (ballot)
                hit = k0 + __ffs(ballot) - 1;
        }
    }
    if (lane == 0)
        branch[req] = hit;
}

}  // namespace
}  // namespace d3d

extern "C" int d3d_branch_match(const int32_t *verified, const int32_t *verified_len, const int32_t *heads,
                                const int32_t *head_len, int R, int M, int B, int32_t *branch, cudaStream_t stream)
{
    if (R < 0 || M < 0 || B < 1)
        return D3D_ERR_INVALID_ARG;
    if (R == 0)
        return D3D_OK;
    if (!verified || !verified_len || !branch || (M > 0 && (!heads || !head_len)))
        return D3D_ERR_INVALID_ARG;
    const size_t warps_per_block = d3d::kMThreads / 32;
    const size_t blocks = ((size_t)R + warps_per_block - 1) / warps_per_block;
    if (blocks > 0x7fffffffull)
        return D3D_ERR_UNSUPPORTED;
    d3d::branch_match_kernel<<<(unsigned)blocks, d3d::kMThreads, 0, stream>>>(verified, verified_len, heads,
                                                                             head_len, R, M, B, branch);
    return d3d::cuda_status(cudaGetLastError());
}
