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

// The six offsets of request r as loaded (load_bounds issues the loads; a
// caller may do other work before check_bounds consumes them).
struct ReqRaw {
    int q0, q1, p0, p1, s0, s1;
};

__device__ inline ReqRaw load_bounds(const int32_t *cu_prefix, const int32_t *cu_q, const int32_t *cu_seg, int r)
{
    ReqRaw w;
    w.q0 = cu_q[r], w.q1 = cu_q[r + 1];
    w.p0 = cu_prefix[r], w.p1 = cu_prefix[r + 1];
    w.s0 = cu_seg[r], w.s1 = cu_seg[r + 1];
    return w;
}

__device__ inline bool check_bounds(const ReqRaw &w, int max_q, int max_prefix, int total_q, int total_prefix,
                                    int total_segs, ReqBounds &b)
{
    b.q0 = w.q0, b.n_q = w.q1 - w.q0, b.p0 = w.p0, b.L = w.p1 - w.p0, b.s0 = w.s0, b.s1 = w.s1;
    return 0 <= w.q0 && w.q0 <= w.q1 && w.q1 <= total_q && w.q1 - w.q0 <= max_q && 0 <= w.p0 && w.p0 <= w.p1 &&
           w.p1 <= total_prefix && w.p1 - w.p0 <= max_prefix && 0 <= w.s0 && w.s0 <= w.s1 && w.s1 <= total_segs;
}

__device__ inline bool request_bounds(const int32_t *cu_prefix, const int32_t *cu_q, const int32_t *cu_seg, int r,
                                      int max_q, int max_prefix, int total_q, int total_prefix, int total_segs,
                                      ReqBounds &b)
{
    return check_bounds(load_bounds(cu_prefix, cu_q, cu_seg, r), max_q, max_prefix, total_q, total_prefix,
                        total_segs, b);
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
