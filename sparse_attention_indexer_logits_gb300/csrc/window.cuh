// The producer's window over a CTA's range of KV blocks, shared by the
// paged-logits kernels: up to 32 consecutive sub-tiles (one or two blocks of
// one request each) described at once, one per lane, by a warp scan over the
// requests' lengths and a shuffle search, with each lane's block-table
// entries read in parallel.  `Args` supplies batch, seq_lens, block_table,
// bt_stride and max_context.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace pml {

// Producer window: up to 32 consecutive sub-tiles of the CTA's range, one per
// lane, built by the whole warp at once.  Within the range, request b's
// sub-tiles pair its blocks from j0(b) (sj for the first request, else 0):
// (j0, j0+1), (j0+2, j0+3), ..., the last one single if the request's part of
// the range has an odd number of blocks.  A window starts at a sub-tile
// boundary (cb, cj) and holds a whole number of stages unless it is the last.
struct Window {
    int b, j, cnt, len;    // this lane's sub-tile (lanes < n)
    bool first, last;      // first / last sub-tile of request b in the range
    bool ld0, ld1;         // which of its two blocks lie below max_context
    int phys0, phys1;      // their physical blocks (read from block_table)
    int n;                 // sub-tiles in the window
    int nb, nj;            // where the next window starts; nb < 0: nothing left
    unsigned first_mask;   // lanes holding a first sub-tile
};

// Number of lanes r whose inclusive prefix p_r is <= v (p non-decreasing over
// the lanes): the lane index whose range of sub-tiles contains sub-tile v.
__device__ __forceinline__ int warp_locate(int p, int v)
{
    int pos = 0;
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) {
        const int t = __shfl_sync(0xffffffffu, p, pos + k - 1);
        if (t <= v) pos += k;
    }
    return pos;
}

template <int KT, class Args>
__device__ __forceinline__ Window make_window(const Args& a, int cb, int cj, int sb, int sj,
                                              int eb, int ej, int lane)
{
    Window w;
    // lane r describes request cb + r: its blocks in the range from this
    // window's start, and the sub-tiles they make
    const int rq = cb + lane;
    const bool in_rng = rq < a.batch && rq <= eb;
    const int len_r = in_rng ? __ldg(a.seq_lens + rq) : 0;
    const int nb_r = blocks_of(len_r);
    const int lim_r = rq == eb ? ej : nb_r;               // end of the request's part of the range
    const int blk_r = in_rng ? max(0, lim_r - (lane == 0 ? cj : 0)) : 0;
    const int st_r = (blk_r + 1) >> 1;
    int p = st_r;                                         // inclusive prefix over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, p, o);
        if (lane >= o) p += t;
    }
    const int total = __shfl_sync(0xffffffffu, p, 31);
    // lane l takes sub-tile l
    const int r = warp_locate(p, lane);
    const int p_r = __shfl_sync(0xffffffffu, p, r);
    const int s_r = __shfl_sync(0xffffffffu, st_r, r);
    const int l_r = __shfl_sync(0xffffffffu, lim_r, r);
    const int n_r = __shfl_sync(0xffffffffu, len_r, r);
    w.b = cb + r;
    w.j = (r == 0 ? cj : 0) + 2 * (lane - (p_r - s_r));
    w.cnt = min(2, l_r - w.j);
    w.len = min(n_r, a.max_context);
    w.first = w.j == (w.b == sb ? sj : 0);
    w.last = w.j + w.cnt == l_r;
    // extent of the window and the start of the next one
    const bool beyond = cb + 32 <= eb && cb + 32 < a.batch;   // requests not yet looked at
    w.n = min(total, 32);
    if (total > 32) {
        const int r32 = warp_locate(p, 32);
        const int p32 = __shfl_sync(0xffffffffu, p, r32);
        const int s32 = __shfl_sync(0xffffffffu, st_r, r32);
        w.nb = cb + r32;
        w.nj = (r32 == 0 ? cj : 0) + 2 * (32 - (p32 - s32));
    } else if (beyond) {
        w.nb = cb + 32;
        w.nj = 0;
    } else {
        w.nb = -1;
        w.nj = 0;
    }
    if (KT == 2 && w.nb >= 0 && (w.n & 1)) {
        // keep whole stages: the odd sub-tile opens the next window
        --w.n;
        w.nb = __shfl_sync(0xffffffffu, w.b, w.n);
        w.nj = __shfl_sync(0xffffffffu, w.j, w.n);
    }
    const bool mine = lane < w.n;
    w.first_mask = __ballot_sync(0xffffffffu, mine && w.first);
    w.ld0 = mine && (long long)w.j * kBlockKeys < a.max_context;
    w.ld1 = mine && w.cnt == 2 && (long long)(w.j + 1) * kBlockKeys < a.max_context;
    const int32_t* row = a.block_table + (long long)w.b * a.bt_stride + w.j;
    w.phys0 = w.ld0 ? __ldg(row) : 0;
    w.phys1 = w.ld1 ? __ldg(row + 1) : 0;
    return w;
}

}  // namespace pml
