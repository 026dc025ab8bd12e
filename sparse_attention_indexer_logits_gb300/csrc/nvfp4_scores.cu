// Single-head NVFP4 indexer scores on sm_103a.
//
//   scores[r, k] = query[r] . key_k     for k < min(context_lengths[g], max_context)
//
// ("flashinfer.sdsa.indexer_scores": the NVFP4 forms of query [rows, 64] and
// key_cache [pages, 64, 64] -- E2M1 values two to a byte -- with E4M3
// query_scales [rows, 8] and key_scales [pages, 64, 8], one scale per 16
// values; key pages any multiple of 16 bytes apart, scale pages any multiple
// of 8; a score is the plain dot product of the dequantised query row and
// key.)
//
// A dequantising stage in front of the tensor cores.  A value is an E2M1 code
// (at most 2 significant bits) times an E4M3 scale (at most 4), so it has at
// most 6 significant bits and |v| <= 6 * 448 = 2688: exact in f16.  Each tile
// of two 64-key pages therefore becomes an f16 operand with no rounding, and
// tcgen05.mma kind::f16 accumulates the exact f16 products in fp32.  The key
// tile (A) is written to tensor memory, not shared memory: that halves the
// shared-memory traffic of a tile, which would otherwise bound the kernel.
//
//   (every role comes twice, one copy for each side: the even tiles and the
//   odd tiles)
//   warps 0,10 producers: per tile one bulk copy per page -- 4608 bytes of
//              codes and scales when the scales follow the codes, else the
//              4 KB of codes and 8-byte cp.async copies of the 512 scale bytes
//              (their pages need only 8-byte alignment) -- completing on the
//              staging slot's `full` barrier, plus a 8-byte record of the
//              tile's group.  Staging slots (9 KB) fill most of the shared
//              memory, so many copies are in flight.
//   warps 1,11 MMA issue: 8 tcgen05.mma (K = 16) per tile, A from tensor
//              memory, B the group's rows (padded to N = 16) in shared memory,
//              one commit, into one of eight TMEM accumulators (16 columns
//              each; a side uses the four of its parity).
//   warps 2-5, 16-19 epilogues: one key per thread, up to 8 scores per key.
//   warps 6-9, 12-15 dequantisation: a thread expands one key row --
//              cvt.rn.f16x2.e2m1x2 per byte and one f16x2 multiply by the
//              group's scale -- into its TMEM lane (tcgen05.st, 64 columns);
//              per group of query rows, the rows into one of the side's two
//              Q slots (shared memory, 128-byte-swizzled K-major).
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace pml {

namespace {

constexpr int kN = 16;                                   // MMA N: group rows padded
constexpr int kPackedRow = kHeadDim / 2;                 // 64 bytes of codes per row
constexpr int kScalesPerRow = kHeadDim / 16;             // 8
constexpr int kPackedPage = kBlockKeys * kPackedRow;     // 4096
constexpr int kScalePage = kBlockKeys * kScalesPerRow;   // 512
constexpr int kStagePage = kPackedPage + kScalePage;     // 4608: a staged page, codes then scales
constexpr int kQHalfBytes = kN * 128;                    // 2 KB
constexpr int kQSlotBytes = 2 * kQHalfBytes;             // 4 KB
// Every role comes twice, one copy for each side of the tile sequence (side
// p = tile index & 1): one role's per-tile chain (waits, lookups, copy
// issues, conversions, TMEM loads) is longer than a tile's share of HBM time.
// Each side has its own half of the staging slots, key tiles, accumulators
// and Q slots, so every barrier has one side's roles on it, in tile order.
constexpr int kProducerWarp = 0;      // and kProducerWarp2
constexpr int kMmaWarp = 1;           // and kMmaWarp2; warp 1 also allocates TMEM
constexpr int kFirstEpiWarp = 2;      // warps 2-5, and 16-19
constexpr int kFirstDeqWarp = 6;      // warps 6-9, and 12-15
constexpr int kProducerWarp2 = 10;
constexpr int kMmaWarp2 = 11;
constexpr int kFirstDeqWarp2 = 12;
constexpr int kFirstEpiWarp2 = 16;
constexpr int kThreads = 640;
constexpr int kRecFirst = 1;
// Tensor memory: eight accumulators of N = 16 columns (a side uses the four of
// its parity), then the f16 key tiles, 64 columns each (128 values of a key
// row, two per column), `tiles` of them.
constexpr int kAcc = 8;
constexpr uint32_t kAccCols = kAcc * kN;                 // 128
constexpr uint32_t kTileCols = kHeadDim / 2;             // 64
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxTiles = (int)((kTmemCols - kAccCols) / kTileCols);   // 6

// Shared memory: `stages` staging slots of one tile's two pages (codes then
// scales, as HBM delivers them; deep, so that many copies are in flight), half
// of them per side, and two Q slots per side.  The f16 key tiles live in
// tensor memory (half of `tiles` per side), freed by the MMA's commit.
struct Nvfp4Layout {
    uint32_t stage, q, rec, bar, misc, total;
};

__host__ __device__ inline Nvfp4Layout nvfp4_layout(int stages, int tiles)
{
    Nvfp4Layout L;
    L.stage = 0;                                               // slot s, page p: 2s + p
    L.q = L.stage + (uint32_t)stages * 2 * kStagePage;
    L.rec = L.q + 4 * kQSlotBytes;                             // per staging slot
    L.bar = L.rec + (uint32_t)stages * 8;
    L.misc = L.bar + (uint32_t)(2 * stages + 2 * tiles + 24) * 8;
    L.total = L.misc + 64;
    return L;
}

// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled
// K-major region whose rows are 128 bytes (8-row atoms of 1 KB).
__device__ __forceinline__ uint32_t sw128(int r, int c)
{
    return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// Dequantise the 16 values of group g (8 packed bytes w0, w1) with scale code
// sc into chunks 2(g%4), 2(g%4)+1 of row `row` of K-half g/4.
__device__ __forceinline__ void dequant_group(uint32_t w0, uint32_t w1, uint32_t sc, int g,
                                              uint32_t half0, uint32_t half1, int row)
{
    const uint32_t s2 = e4m3_to_f16x2_dup(sc);
    uint32_t lo[4], hi[4], h[8];
    e2m1x8_to_f16x2x4(w0, lo);
    e2m1x8_to_f16x2x4(w1, hi);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        h[b] = mul_f16x2(lo[b], s2);
        h[4 + b] = mul_f16x2(hi[b], s2);
    }
    const uint32_t base = (g < 4) ? half0 : half1;
    const int c = (g % 4) * 2;
    st_shared_v4(base + sw128(row, c), h[0], h[1], h[2], h[3]);
    st_shared_v4(base + sw128(row, c + 1), h[4], h[5], h[6], h[7]);
}

// Dequantise one 128-value row: 64 packed bytes at `packed` (four 16-byte
// chunks, two groups each) and 8 scale codes -> f16 in the swizzled layout.
// The chunks are read starting at chunk `rot`, so that the rows a warp reads
// together (64 bytes apart) fall in distinct banks when rot = (row / 2) % 4.
__device__ __forceinline__ void dequant_row(const uint4* packed, uint2 scales, uint32_t half0,
                                            uint32_t half1, int row, int rot)
{
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int c = (k + rot) & 3;
        const uint4 v = packed[c];
        const uint32_t sw = c < 2 ? scales.x : scales.y;
        dequant_group(v.x, v.y, (sw >> (16 * (c & 1))) & 0xFF, 2 * c, half0, half1, row);
        dequant_group(v.z, v.w, (sw >> (16 * (c & 1) + 8)) & 0xFF, 2 * c + 1, half0, half1, row);
    }
}

// Position in a ring of n slots and the parity of its current pass, advanced
// one step at a time (no division by the runtime ring size in the loops).
struct RingPos {
    int idx = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next(int n)
    {
        if (++idx == n) {
            idx = 0;
            phase ^= 1u;
        }
    }
};

// Dequantise one 16-byte chunk (32 codes: two groups of 16 with scale codes
// sa, sb) into 16 f16x2 words, byte i -> word i.
__device__ __forceinline__ void dequant_chunk(uint4 v, uint32_t sa, uint32_t sb,
                                              uint32_t (&out)[16])
{
    const uint32_t s_a = e4m3_to_f16x2_dup(sa);
    const uint32_t s_b = e4m3_to_f16x2_dup(sb);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t h[4];
        e2m1x8_to_f16x2x4(w[q], h);
        const uint32_t s2 = q < 2 ? s_a : s_b;
#pragma unroll
        for (int b = 0; b < 4; ++b) out[4 * q + b] = mul_f16x2(h[b], s2);
    }
}

__global__ void __launch_bounds__(kThreads, 1) nvfp4_scores_kernel(const Nvfp4Args a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = a.stages;     // staging slots
    const int T = a.tiles;      // f16 tiles
    const int G = a.group_size;
    const Nvfp4Layout L = nvfp4_layout(S, T);

    const uint32_t base = smem_addr(smem);
    const uint32_t stage_base = base + L.stage;
    // per staging slot, written by the producer before the slot's `full`
    // arrival: {group b, kRecFirst if the side's first tile of b}, or {-1, 0}
    // after the side's last tile
    const uint32_t rec_base = base + L.rec;
    const uint32_t q_base = base + L.q;
    const uint32_t bar = base + L.bar;
    auto full_bar = [&](int s) { return bar + 8u * s; };                  // staging landed
    auto sfree_bar = [&](int s) { return bar + 8u * (S + s); };           // staging read
    auto deq_bar = [&](int t) { return bar + 8u * (2 * S + t); };         // tile written
    auto tfree_bar = [&](int t) { return bar + 8u * (2 * S + T + t); };   // tile consumed
    const uint32_t tfull_bar0 = bar + 8u * (2 * S + 2 * T);              // + 8*acc
    const uint32_t tempty_bar0 = tfull_bar0 + 8u * 8;
    const uint32_t qfull_bar0 = tempty_bar0 + 8u * 8;                    // + 8*(2*side+slot)
    const uint32_t qempty_bar0 = qfull_bar0 + 8u * 4;
    const int S2 = S / 2, T2 = T / 2;   // per side
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);
    int* sched = reinterpret_cast<int*>(smem + L.misc + 16);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int prod = warp == kProducerWarp ? 0 : warp == kProducerWarp2 ? 1 : -1;
    const int mmaw = warp == kMmaWarp ? 0 : warp == kMmaWarp2 ? 1 : -1;
    const int dgrp = (warp >= kFirstDeqWarp && warp < kFirstDeqWarp + 4) ? 0
                     : (warp >= kFirstDeqWarp2 && warp < kFirstDeqWarp2 + 4) ? 1 : -1;
    const int egrp = (warp >= kFirstEpiWarp && warp < kFirstEpiWarp + 4) ? 0
                     : warp >= kFirstEpiWarp2 ? 1 : -1;

    if (warp == kProducerWarp) {
        const long long total = warp_total_blocks(a.context_lengths, a.groups);
        const long long s0 = range_start(total, gridDim.x, blockIdx.x);
        const long long s1 = range_start(total, gridDim.x, blockIdx.x + 1);
        int sb, sj, eb, ej;
        warp_locate2(a.context_lengths, a.groups, s0, s1, sb, sj, eb, ej);
        if (lane == 0) {
            sched[0] = sb; sched[1] = sj; sched[2] = eb; sched[3] = ej;
            *abort_flag = 0;
            for (int s = 0; s < S; ++s) {
                // expect_tx arrive (+ each lane's cp.async of scales, unless fused)
                mbar_init(full_bar(s), a.fused ? 1 : 1 + 32);
                mbar_init(sfree_bar(s), 4);
            }
            for (int t = 0; t < T; ++t) {
                mbar_init(deq_bar(t), 4);
                mbar_init(tfree_bar(t), 1);       // the MMA's commit
            }
            for (int i = 0; i < kAcc; ++i) {
                mbar_init(tfull_bar0 + 8u * i, 1);
                mbar_init(tempty_bar0 + 8u * i, 4);
            }
            for (int i = 0; i < 4; ++i) {
                mbar_init(qfull_bar0 + 8u * i, 4);
                mbar_init(qempty_bar0 + 8u * i, 4);
            }
            fence_mbar_init();
        }
    } else if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int sb = sched[0], sj = sched[1], eb = sched[2], ej = sched[3];

    if (prod >= 0) {
        // ------------------------------------------------------------ producers
        const uint64_t policy = policy_evict_first();
        Walk w;
        w.init(a.context_lengths, a.groups, sb, sj, eb, ej);
        int it = 0, k = 0, prev_g = -1;   // it: tile; k: this side's tiles so far
        RingPos sp;                        // this side's staging slot
        long long bt_row = 0;
        // block-table entries come 32 at a time, one per lane, the next 32
        // already in flight: lane i of `cur` holds block cur_j + i
        int nbl = 0, cur_j = 0, cur = 0, nxt = 0;
        auto fetch = [&](int j0) {
            return j0 + lane < nbl ? __ldg(a.block_table + bt_row + j0 + lane) : 0;
        };
        bool ok = true;
        while (!w.done()) {
            const int c = w.cnt();
            if ((it & 1) != prod) {               // the other side's tile
                w.advance(c);
                ++it;
                continue;
            }
            const bool first = w.b != prev_g;
            if (first) {
                int req = __ldg(a.requests + w.b);
                if (req < 0 || req >= a.num_requests) {
                    if (lane == 0) atomicOr(a.status, kStatusBadRequest);
                    req = 0;
                }
                bt_row = (long long)req * a.bt_stride;
                nbl = blocks_of(min(w.len, a.max_context));
                cur_j = w.j;
                cur = fetch(cur_j);
                nxt = fetch(cur_j + 32);
                prev_g = w.b;
            }
            // the entries of blocks w.j and w.j + 1: `cur` and `nxt` hold the
            // window [cur_j, cur_j + 64), which covers both
            while (w.j >= cur_j + 32) {
                cur_j += 32;
                cur = nxt;
                nxt = fetch(cur_j + 32);
            }
            const int i0 = w.j - cur_j;
            const int e0 = __shfl_sync(0xffffffffu, cur, i0);
            const int e1c = __shfl_sync(0xffffffffu, cur, (i0 + 1) & 31);
            const int e1n = __shfl_sync(0xffffffffu, nxt, 0);
            // pages of the tile below max_context
            const int nload = (long long)w.j * kBlockKeys >= a.max_context ? 0
                              : (c > 1 && (long long)(w.j + 1) * kBlockKeys < a.max_context) ? 2
                                                                                             : 1;
            long long page0 = e0, page1 = i0 < 31 ? e1c : e1n;
            if (nload >= 1 && (page0 < 0 || page0 >= a.num_pages)) {
                if (lane == 0) atomicOr(a.status, kStatusBadBlock);
                page0 = 0;
            }
            if (nload == 2 && (page1 < 0 || page1 >= a.num_pages)) {
                if (lane == 0) atomicOr(a.status, kStatusBadBlock);
                page1 = 0;
            }
            const int s = prod * S2 + sp.idx;
            if (lane == 0) ok = mbar_wait(sfree_bar(s), sp.phase ^ 1u, abort_flag, a.status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            const uint32_t dst = stage_base + (uint32_t)(2 * s) * kStagePage;
            if (lane == 0) st_shared_v2_s32(rec_base + 8u * s, w.b, first ? kRecFirst : 0);
            if (a.fused) {
                // a page's codes and scales are one run of 4608 bytes
                if (lane == 0) {
                    mbar_arrive_expect_tx(full_bar(s), (uint32_t)nload * kStagePage);
                    if (nload >= 1)
                        bulk_load_stream(dst, a.key_cache + page0 * a.page_stride, kStagePage,
                                         full_bar(s), policy);
                    if (nload == 2)
                        bulk_load_stream(dst + kStagePage, a.key_cache + page1 * a.page_stride,
                                         kStagePage, full_bar(s), policy);
                }
            } else {
                // codes by bulk copies; scales (pages only 8-byte aligned) by
                // 8-byte cp.async, two per lane per page
                if (lane == 0) {
                    mbar_arrive_expect_tx(full_bar(s), (uint32_t)nload * kPackedPage);
                    if (nload >= 1)
                        bulk_load_stream(dst, a.key_cache + page0 * a.page_stride, kPackedPage,
                                         full_bar(s), policy);
                    if (nload == 2)
                        bulk_load_stream(dst + kStagePage, a.key_cache + page1 * a.page_stride,
                                         kPackedPage, full_bar(s), policy);
                }
                for (int cc = 0; cc < nload; ++cc) {
                    const uint8_t* src = a.key_scales + (cc ? page1 : page0) * a.scale_stride;
                    const uint32_t sdst = dst + (uint32_t)cc * kStagePage + kPackedPage;
                    cp_async8(sdst + lane * 8, src + lane * 8);
                    cp_async8(sdst + (lane + 32) * 8, src + (lane + 32) * 8);
                }
                cp_async_arrive(full_bar(s));
            }
            w.advance(c);
            ++it;
            ++k;
            sp.next(S2);
        }
        if (ok) {
            // the end mark, in the next slot
            const int s = prod * S2 + sp.idx;
            if (lane == 0) ok = mbar_wait(sfree_bar(s), sp.phase ^ 1u, abort_flag, a.status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (ok) {
                if (lane == 0) {
                    st_shared_v2_s32(rec_base + 8u * s, -1, 0);
                    mbar_arrive_expect_tx(full_bar(s), 0u);
                }
                if (!a.fused) cp_async_arrive(full_bar(s));
            }
        }
        if (!ok && lane == 0) {
            for (int t = (k > S2 ? k - S2 : 0); t < k; ++t)
                mbar_wait_drain(full_bar(prod * S2 + t % S2), (t / S2) & 1);
        }
        cp_async_wait_all();
    } else if (mmaw >= 0) {
        // ------------------------------------------------------------ MMA issue
        const uint32_t idesc = make_idesc(0, 0, kTileKeys, kN);   // f16 x f16 -> f32
        Walk w;
        w.init(a.context_lengths, a.groups, sb, sj, eb, ej);
        // kg: tile within the request; qk: requests this side has tiles of
        int it = 0, kg = 0, prev_g = -1, qk = 0, slot = 0, last = -1;
        RingPos tp;                        // this side's f16 tile
        bool ok = true;
        while (!w.done()) {
            const int c = w.cnt();
            if (w.b != prev_g) {
                kg = 0;
                prev_g = w.b;
            }
            if ((it & 1) == mmaw) {
                if (kg < 2) {                     // this side's first tile of the request
                    slot = 2 * mmaw + (qk & 1);
                    ok = mbar_wait(qfull_bar0 + 8u * slot, (qk >> 1) & 1, abort_flag, a.status);
                    if (!ok) break;
                    ++qk;
                }
                const int tt = mmaw * T2 + tp.idx;
                ok = mbar_wait(deq_bar(tt), tp.phase, abort_flag, a.status);
                if (!ok) break;
                const int acc = it % kAcc;        // this side's accumulators: it's parity
                ok = mbar_wait(tempty_bar0 + 8u * acc, ((it / kAcc) & 1) ^ 1, abort_flag, a.status);
                if (!ok) break;
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t d = tmem_base + (uint32_t)(acc * kN);
                    const uint32_t at = tmem_base + kAccCols + (uint32_t)tt * kTileCols;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint64_t bd =
                            smem_desc_sw128(q_base + slot * kQSlotBytes + h * kQHalfBytes);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)   // K = 16: 8 columns of A
                            mma_f16_tmem_a(d, at + 8u * (4 * h + kk), bd + 2u * kk, idesc,
                                           (h | kk) ? 1u : 0u);
                    }
                    mma_commit(tfull_bar0 + 8u * acc);
                    mma_commit(tfree_bar(tt));    // the tile may be rewritten once these complete
                }
                __syncwarp();
                last = it;
                tp.next(T2);
            }
            w.advance(c);
            ++it;
            ++kg;
        }
        if (!ok && last >= 0) mbar_wait_drain(tfull_bar0 + 8u * (last % kAcc), (last / kAcc) & 1);
    } else if (egrp >= 0) {
        // ------------------------------------------------------------ epilogues
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int pg = row >> 6;
        const int key = row & 63;
        const uint32_t lane_addr = tmem_base + ((uint32_t)(quad * 32) << 16);
        Walk w;
        w.init(a.context_lengths, a.groups, sb, sj, eb, ej);
        int it = 0, prev_g = -1, len = 0, qk = 0;
        bool ok = true;
        while (!w.done()) {
            const int c = w.cnt();
            if ((it & 1) != egrp) {               // the other side's tile
                w.advance(c);
                ++it;
                continue;
            }
            if (w.b != prev_g) {
                prev_g = w.b;
                len = min(__ldg(a.context_lengths + w.b), a.max_context);
            }
            // the request's last two tiles are the last of each side: each
            // frees its side's q slot
            const bool last_of_side = w.blocks_after(c) <= 2;
            const int acc = it % kAcc;
            ok = mbar_wait(tfull_bar0 + 8u * acc, (it / kAcc) & 1, abort_flag, a.status);
            if (!ok) break;
            tc_fence_after();
            float v[8];
            tmem_ld8(lane_addr + (uint32_t)(acc * kN), v);
            const int pos = (w.j + pg) * kBlockKeys + key;
            if (pg < c && pos < len) {
                float* dst = a.scores + (long long)w.b * G * a.scores_stride + pos;
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    if (r < G) dst[(long long)r * a.scores_stride] = v[r];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(tempty_bar0 + 8u * acc);
                if (last_of_side) mbar_arrive(qempty_bar0 + 8u * (2 * egrp + (qk & 1)));
            }
            if (last_of_side) ++qk;
            w.advance(c);
            ++it;
        }
    } else if (dgrp >= 0) {
        // ------------------------------------------------------------ dequantisation
        const int t = threadIdx.x - 32 * (dgrp == 0 ? kFirstDeqWarp : kFirstDeqWarp2);
        // key tiles: a warp may reach only its own quarter of the TMEM lanes,
        // so the thread expands tile row (key) 32 * (warp % 4) + lane into that
        // lane: page row / 64, row row % 64 of it
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t row_off = (uint32_t)((row >> 6) * kStagePage + (row & 63) * kPackedRow);
        const uint32_t sc_row_off =
            (uint32_t)((row >> 6) * kStagePage + kPackedPage + (row & 63) * kScalesPerRow);
        const uint32_t lane_tmem = tmem_base + ((uint32_t)(quad * 32) << 16) + kAccCols;
        int qk = 0;
        RingPos sp, tp;                    // this side's staging slot and f16 tile
        bool ok = true;
        while (true) {
            const int s = dgrp * S2 + sp.idx, tt = dgrp * T2 + tp.idx;
            // both waits issued before either result is needed
            const bool got_full = mbar_try_wait(full_bar(s), sp.phase);
            const bool got_tile = mbar_try_wait(tfree_bar(tt), tp.phase ^ 1u);
            if (!got_full) {
                ok = mbar_wait(full_bar(s), sp.phase, abort_flag, a.status);
                if (!ok) break;
            }
            const int2 rec = ld_shared_v2_s32(rec_base + 8u * s);
            if (rec.x < 0) break;                 // the producer's end mark
            if (rec.y & kRecFirst) {
                // this side's first tile of group rec.x: its query rows into
                // this side's next Q slot (rows G..15 zero)
                const int slot = 2 * dgrp + (qk & 1);
                ok = mbar_wait(qempty_bar0 + 8u * slot, ((qk >> 1) & 1) ^ 1, abort_flag, a.status);
                if (!ok) break;
                const uint32_t qh0 = q_base + slot * kQSlotBytes;
                if (t < G) {
                    const long long qrow = (long long)rec.x * G + t;
                    const uint4* src = reinterpret_cast<const uint4*>(a.query + qrow * kPackedRow);
                    const uint4 pk[4] = {__ldg(src), __ldg(src + 1), __ldg(src + 2),
                                         __ldg(src + 3)};
                    const uint2 sc = __ldg(
                        reinterpret_cast<const uint2*>(a.query_scales + qrow * kScalesPerRow));
                    dequant_row(pk, sc, qh0, qh0 + kQHalfBytes, t, 0);
                } else if (t < kN) {
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        st_shared_v4(qh0 + sw128(t, c8), 0u, 0u, 0u, 0u);
                        st_shared_v4(qh0 + kQHalfBytes + sw128(t, c8), 0u, 0u, 0u, 0u);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(qfull_bar0 + 8u * slot);
                ++qk;
            }
            if (!got_tile) {
                ok = mbar_wait(tfree_bar(tt), tp.phase ^ 1u, abort_flag, a.status);
                if (!ok) break;
            }
            tc_fence_after();                     // the tile's last MMA read before our stores
            // every row: a page past the request's end or max_context holds
            // stale bytes, which only reach accumulator rows the epilogue does
            // not store
            const uint32_t slot = stage_base + (uint32_t)(2 * s) * kStagePage;
            uint4 v[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) v[c] = ld_shared_v4(slot + row_off + 16u * c);
            const uint2 sc = ld_shared_v2_u32(slot + sc_row_off);
            const uint32_t ta = lane_tmem + (uint32_t)tt * kTileCols;
#pragma unroll
            for (int c = 0; c < 4; ++c) {         // 16-byte chunk c: columns 16c..16c+15
                const uint32_t sw = c < 2 ? sc.x : sc.y;
                uint32_t w16[16];
                dequant_chunk(v[c], (sw >> (16 * (c & 1))) & 0xFF, (sw >> (16 * (c & 1) + 8)) & 0xFF,
                              w16);
                tmem_st16(ta + 16u * c, w16);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(sfree_bar(s));        // staging slot read: refill it
                mbar_arrive(deq_bar(tt));
            }
            sp.next(S2);
            tp.next(T2);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

size_t nvfp4_smem_bytes(int stages, int tiles)
{
    return (size_t)nvfp4_layout(stages, tiles).total + 1024;
}

cudaError_t launch_nvfp4_scores(const Nvfp4Args& a, int num_ctas, cudaStream_t stream)
{
    // both rings split between the two sides; the key tiles must fit the
    // tensor memory the kernel allocates
    if (a.stages < 2 || (a.stages & 1) || a.tiles < 2 || (a.tiles & 1) || a.tiles > kMaxTiles)
        return cudaErrorInvalidValue;
    const size_t smem = nvfp4_smem_bytes(a.stages, a.tiles);
    static int configured_device = -1;
    static size_t configured_smem = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev || configured_smem < smem) {
        e = cudaFuncSetAttribute(nvfp4_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        configured_device = dev;
        configured_smem = smem;
    }
    nvfp4_scores_kernel<<<num_ctas, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace pml
