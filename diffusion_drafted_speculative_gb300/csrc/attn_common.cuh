// Visibility of packed keys, derived on the device from the segment table.
//
// [D3D] "Core method", "Method steps" steps 2 and 4: a draft block sees the
// shared prefix, the hypothesised accepted tokens of its branch, and itself
// bidirectionally; the block under verification is encoded causally.  For a
// packed query token the visible packed keys are therefore at most two
// half-open intervals (request-local indices): its own segment (clipped at
// itself when causal) and the first parent_len tokens of its parent.  The
// prefix is visible to every query and is not part of this.
#pragma once

#include "d3d_common.cuh"

namespace d3d {

struct RowVis {
    int own_lo, own_hi;  // own segment keys [own_lo, own_hi)
    int par_lo, par_hi;  // parent keys [par_lo, par_hi), empty without a parent
};

__device__ inline bool vis_has(const RowVis &v, int j)
{
    return (j >= v.own_lo && j < v.own_hi) || (j >= v.par_lo && j < v.par_hi);
}

// Bounds of one request, read from the offset arrays and checked against the
// host-side totals and maxima.  Returns false if the offsets lie.
struct ReqBounds {
    int q0, n_q, p0, L, s0, s1;
};

__device__ inline bool request_bounds(const int32_t *cu_prefix, const int32_t *cu_q, const int32_t *cu_seg, int r,
                                      int max_q, int max_prefix, int total_q, int total_prefix, int total_segs,
                                      ReqBounds &b)
{
    const int q0 = cu_q[r], q1 = cu_q[r + 1];
    const int p0 = cu_prefix[r], p1 = cu_prefix[r + 1];
    const int s0 = cu_seg[r], s1 = cu_seg[r + 1];
    b.q0 = q0, b.n_q = q1 - q0, b.p0 = p0, b.L = p1 - p0, b.s0 = s0, b.s1 = s1;
    return 0 <= q0 && q0 <= q1 && q1 <= total_q && q1 - q0 <= max_q && 0 <= p0 && p0 <= p1 &&
           p1 <= total_prefix && p1 - p0 <= max_prefix && 0 <= s0 && s0 <= s1 && s1 <= total_segs;
}

// Visible packed-key intervals of local token i (0 <= i < n_q) of a request
// whose segments are segs[s0, s1).  Returns false when the table is
// malformed around i (every read stays inside segs[s0, s1)).
__device__ inline bool row_visibility(const d3d_segment_t *segs, int s0, int s1, int n_q, int i, RowVis &v)
{
    v.own_lo = v.own_hi = v.par_lo = v.par_hi = 0;
    int lo = s0, hi = s1 - 1, s = -1;
    while (lo <= hi) {  // last segment with q_start <= i
        const int mid = (lo + hi) >> 1;
        if (segs[mid].q_start <= i) {
            s = mid;
            lo = mid + 1;
        } else {
            hi = mid - 1;
        }
    }
    if (s < 0)
        return false;
    const d3d_segment_t g = segs[s];
    if (g.len < 1 || g.q_start < 0 || i >= g.q_start + g.len || g.q_start + g.len > n_q)
        return false;
    if (g.mode != D3D_SEG_CAUSAL && g.mode != D3D_SEG_BIDIR)
        return false;
    v.own_lo = g.q_start;
    v.own_hi = (g.mode == D3D_SEG_BIDIR) ? g.q_start + g.len : i + 1;
    if (g.parent == -1) {
        if (g.parent_len != 0)
            return false;
        return true;
    }
    if (g.parent < 0 || g.parent >= s - s0)
        return false;
    const d3d_segment_t p = segs[s0 + g.parent];
    if (p.mode != D3D_SEG_CAUSAL || p.parent != -1 || g.parent_len < 0 || g.parent_len > p.len || p.q_start < 0 ||
        p.q_start + p.len > g.q_start)
        return false;
    v.par_lo = p.q_start;
    v.par_hi = p.q_start + g.parent_len;
    return true;
}

}  // namespace d3d
