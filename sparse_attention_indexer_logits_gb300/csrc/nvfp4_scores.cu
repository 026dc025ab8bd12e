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
// The tensor cores take the format as stored.  tcgen05.mma kind::mxf4nvf4
// with 16-element scale blocks multiplies E2M1 codes of A (128 keys, K-major)
// and B (the group's rows padded to N = 16), scales each block's partial sum
// by the two E4M3 scales it reads from tensor memory and accumulates in fp32:
// no dequantising pass, two MMAs (K = 64) per 128 keys.  The MMA reads a scale
// byte without its sign (and 0x7f / 0xff as NaN, like the format), so a
// negative scale is applied by flipping the sign bits of its block's sixteen
// codes in shared memory (bit 3 of each nibble) before the MMA reads them.
//
// Scale layout in tensor memory (one 32-bit column holds the four scales of a
// row's K = 64 half, byte b for elements 16b..16b+15):
//   A: row m is read from lane m, column sfa + m / 32;
//   B: row n, for the output rows of lane quadrant q, from lane 32 q + n,
//      column sfb + n / 32 -- every quadrant holds its own copy.
// Writing each lane's word to all four columns sfa..sfa+3 (and its second
// K-half's word to sfa+4..sfa+7) satisfies both with one tcgen05.st.
//
// A tile is four 64-key pages (two MMA halves of M = 128): the codes arrive by
// TMA with the 64-byte swizzle (a row of 64 bytes is one swizzle span), so the
// two pages of a half are the K-major operand as they land; the scales by
// cp.async into the stage's scale area.
//
//   warps 0,2,3 producers, tile i to warp i % 3: per tile the block-table
//               entries (a 64-entry window in two registers per lane), a TMA
//               per page for the codes and one or two cp.async per lane and
//               page for the scales, all completing on the stage's `full`
//               barrier, and a record of the tile's group; an end mark after
//               the last tile.  One warp's round per tile (~1.9k cycles,
//               mostly issue latency) is twice a tile's share of HBM time, so
//               three take turns.
//   warp 1      MMA issue: per tile 2 x 2 MMAs into one of four accumulators
//               (two 16-column halves each); commits free the accumulator's
//               readers, the stage and, after a group's last tile, its Q slot.
//   warps 4-7   scales: per tile each thread writes the scale words of keys
//               (row, 128 + row) to the stage's columns, fixing signs; on a
//               group's first tile, the query rows into a Q slot (shared
//               memory, sign-fixed, swizzled) and their scales into the slot's
//               columns.
//   warps 8-15  two epilogue warpgroups, even and odd tiles: two keys per
//               thread, up to 8 scores per key.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace pml {

namespace {

constexpr int kN = 16;                                     // MMA N: group rows padded
constexpr int kRowBytes = kHeadDim / 2;                    // 64 bytes of codes per row
constexpr int kRowScales = kHeadDim / 16;                  // 8
constexpr int kPageCodes = kBlockKeys * kRowBytes;         // 4096
constexpr int kPageScales = kBlockKeys * kRowScales;       // 512
constexpr int kTileBlocks = 4;                             // pages per tile
constexpr int kHalfCodes = 2 * kPageCodes;                 // one M = 128 operand
constexpr int kStageCodes = kTileBlocks * kPageCodes;      // 16 KB
constexpr int kStageBytes = kStageCodes + kTileBlocks * kPageScales;   // 18 KB
constexpr int kQSlotBytes = kN * kRowBytes;                // 1 KB
constexpr int kAcc = 4;
constexpr uint32_t kAccCols = 2 * kN;                      // both halves of a tile
constexpr uint32_t kSfaCol0 = kAcc * kAccCols;             // 16 columns per stage
constexpr uint32_t kSfbCol0 = kSfaCol0 + 16u * kMaxNvfp4Stages;   // 8 columns per Q slot
constexpr uint32_t kTmemCols = 512;
static_assert(kSfbCol0 + 16 <= kTmemCols, "scale columns beyond the allocation");
constexpr int kProducers = kNvfp4Producers;   // warps 0, 2, 3: tile i is producer i % 3's
constexpr int kMmaWarp = 1;
constexpr int kScaleWarp0 = 4;      // a whole warpgroup: warp w writes lane quadrant w % 4
constexpr int kEpiWarp0 = 8;        // warps 8-11 even tiles, 12-15 odd tiles
constexpr int kThreads = 512;
constexpr int kRecFirst = 1;
constexpr uint32_t kSignBits = 0x80808080u;   // the sign bits of four E4M3 scales
constexpr uint32_t kCodeSigns = 0x88888888u;  // the sign bits of eight E2M1 codes

// Shared memory: `stages` stages of one tile (four pages of codes, then their
// scales), two Q slots, an 8-byte record per stage, barriers.
struct Nvfp4Layout {
    uint32_t stage, q, rec, bar, misc, total;
};

__host__ __device__ inline Nvfp4Layout nvfp4_layout(int stages)
{
    Nvfp4Layout L;
    L.stage = 0;
    L.q = L.stage + (uint32_t)stages * kStageBytes;
    L.rec = L.q + 2 * kQSlotBytes;
    L.bar = L.rec + (uint32_t)stages * 8;
    L.misc = L.bar + (uint32_t)(3 * stages + 2 * kAcc + 4) * 8;
    L.total = L.misc + 64;
    return L;
}

// Shared-memory matrix descriptor for a K-major operand with the 64-byte
// swizzle: rows of 64 bytes, groups of 8 rows 512 bytes apart; the base is
// 512-byte aligned and K advances by adding bytes/16 to the start address.
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);       // start address
    d |= static_cast<uint64_t>(1u) << 16;                     // leading byte offset (unused)
    d |= static_cast<uint64_t>(512u >> 4) << 32;              // stride byte offset
    d |= static_cast<uint64_t>(1u) << 46;                     // descriptor version
    d |= static_cast<uint64_t>(4u) << 61;                     // 64-byte swizzle
    return d;
}

// Instruction descriptor of kind::mxf4nvf4: E2M1 A and B (format 1), K-major,
// E4M3 scales (scale format 0), scale-data ids 0, dense.
__host__ __device__ constexpr uint32_t nvfp4_idesc(uint32_t M, uint32_t N)
{
    return (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D (+)= (A * B^T) with 16-element scale blocks, K = 64.
__device__ __forceinline__ void mma_nvfp4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X "
        "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Columns c..c+3 of this thread's lane := lo, c+4..c+7 := hi (warp-uniform c).
__device__ __forceinline__ void tmem_st_scales(uint32_t taddr, uint32_t lo, uint32_t hi)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%1,%1,%1,%2,%2,%2,%2};" ::"r"(taddr),
        "r"(lo), "r"(hi)
        : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_shared_v2_u32(uint32_t addr, uint32_t x, uint32_t y)
{
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(x), "r"(y) : "memory");
}

// Byte offset of 16-byte chunk c (0..3) of row r in a region written with the
// 64-byte swizzle (512-byte aligned base).
__device__ __forceinline__ uint32_t sw64(int r, int c)
{
    return (uint32_t)(r * kRowBytes + ((c ^ ((r >> 1) & 3)) << 4));
}

// The scale of block j (0..7) of a row's scale words is negative.
__device__ __forceinline__ bool scale_negative(uint2 sc, int j)
{
    const uint32_t w = j < 4 ? sc.x : sc.y;
    return (w >> (8 * (j & 3) + 7)) & 1u;
}

// Flip the code signs of every block of key row `kk` of a landed page whose
// scale is negative (rare: only then does a thread touch the codes).
__device__ __forceinline__ void fix_key_signs(uint32_t page, int kk, uint2 sc)
{
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (!scale_negative(sc, j)) continue;
        const uint32_t addr = page + sw64(kk, j >> 1) + 8u * (j & 1);
        const uint2 v = ld_shared_v2_u32(addr);
        st_shared_v2_u32(addr, v.x ^ kCodeSigns, v.y ^ kCodeSigns);
    }
}

// Blocks in the walk's current tile: up to four, within one group and range.
__device__ __forceinline__ int tile_blocks(const Walk& w)
{
    const int lim = (w.b == w.eb) ? w.ej : w.nbb;
    return min(lim - w.j, kTileBlocks);
}

// Position in a ring of n slots and the parity of its current pass.
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

__global__ void __launch_bounds__(kThreads, 1)
    nvfp4_scores_kernel(const __grid_constant__ CUtensorMap kmap, const Nvfp4Args a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = a.stages;
    const int G = a.group_size;
    const Nvfp4Layout L = nvfp4_layout(S);

    const uint32_t base = smem_addr(smem);
    const uint32_t stage_base = base + L.stage;
    const uint32_t q_base = base + L.q;
    // per stage, written by the producer before the stage's `full` arrival:
    // {group, kRecFirst on the group's first tile in this CTA}, or {-1, 0}
    // after the last tile
    const uint32_t rec_base = base + L.rec;
    const uint32_t bar = base + L.bar;
    auto full_bar = [&](int s) { return bar + 8u * s; };                // codes and scales landed
    auto sfa_bar = [&](int s) { return bar + 8u * (S + s); };           // key scales written
    auto sfree_bar = [&](int s) { return bar + 8u * (2 * S + s); };     // stage consumed
    const uint32_t tfull_bar0 = bar + 8u * (3 * S);                    // + 8 * acc
    const uint32_t tempty_bar0 = tfull_bar0 + 8u * kAcc;
    const uint32_t qfull_bar0 = tempty_bar0 + 8u * kAcc;               // + 8 * slot
    const uint32_t qempty_bar0 = qfull_bar0 + 16u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);
    int* sched = reinterpret_cast<int*>(smem + L.misc + 16);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int prod = warp == 0 ? 0 : (warp == 2 || warp == 3) ? warp - 1 : -1;

    if (warp == 0) {
        const long long total = warp_total_blocks(a.context_lengths, a.groups);
        const long long s0 = range_start(total, gridDim.x, blockIdx.x);
        const long long s1 = range_start(total, gridDim.x, blockIdx.x + 1);
        int sb, sj, eb, ej;
        warp_locate2(a.context_lengths, a.groups, s0, s1, sb, sj, eb, ej);
        if (lane == 0) {
            sched[0] = sb; sched[1] = sj; sched[2] = eb; sched[3] = ej;
            *abort_flag = 0;
            for (int s = 0; s < S; ++s) {
                mbar_init(full_bar(s), 1 + 32);   // expect_tx arrival + each lane's cp.async
                mbar_init(sfa_bar(s), 4);
                mbar_init(sfree_bar(s), 1);       // the MMA's commit
            }
            for (int i = 0; i < kAcc; ++i) {
                mbar_init(tfull_bar0 + 8u * i, 1);
                mbar_init(tempty_bar0 + 8u * i, 4);
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(qfull_bar0 + 8u * i, 4);
                mbar_init(qempty_bar0 + 8u * i, 1);
            }
            fence_mbar_init();
            tma_prefetch_map(&kmap);
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
        // Tile i (counted over the CTA's range) belongs to producer i % kProducers
        // and uses stage i % S; every producer walks every tile.
        const uint64_t policy = policy_evict_first();
        Walk w;
        w.init(a.context_lengths, a.groups, sb, sj, eb, ej);
        int it = 0, owner = 0, prev_g = -1, win_g = -1;
        RingPos sp;
        long long bt_row = 0;
        // block-table entries 32 at a time, one per lane, the next 32 already
        // in flight: lane i of `cur` holds block cur_j + i, of `nxt` cur_j + 32 + i
        int nbl = 0, cur_j = 0, cur = 0, nxt = 0;
        auto fetch = [&](int j0) {
            return j0 + lane < nbl ? __ldg(a.block_table + bt_row + j0 + lane) : 0;
        };
        bool ok = true;
        while (!w.done()) {
            const int c = tile_blocks(w);
            const bool first = w.b != prev_g;
            prev_g = w.b;
            if (owner == prod) {
                if (w.b != win_g) {
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
                    win_g = w.b;
                }
                while (w.j >= cur_j + 32) {
                    cur_j += 32;
                    cur = nxt;
                    nxt = fetch(cur_j + 32);
                }
                // blocks w.j .. w.j + 3 lie in the window [cur_j, cur_j + 64);
                // the pages below max_context are a prefix of the tile
                int page[kTileBlocks];
                int nload = 0;
#pragma unroll
                for (int cc = 0; cc < kTileBlocks; ++cc) {
                    const int i = w.j - cur_j + cc;
                    long long pg = __shfl_sync(0xffffffffu, i < 32 ? cur : nxt, i & 31);
                    page[cc] = 0;
                    if (cc < c && (long long)(w.j + cc) * kBlockKeys < a.max_context) {
                        if (pg < 0 || pg >= a.num_pages) {
                            if (lane == 0) atomicOr(a.status, kStatusBadBlock);
                            pg = 0;
                        }
                        page[cc] = (int)pg;
                        nload = cc + 1;
                    }
                }
                const int s = sp.idx;
                if (lane == 0) ok = mbar_wait(sfree_bar(s), sp.phase ^ 1u, abort_flag, a.status);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                const uint32_t dst = stage_base + (uint32_t)s * kStageBytes;
                if (lane == 0) {
                    st_shared_v2_s32(rec_base + 8u * s, w.b, first ? kRecFirst : 0);
                    mbar_arrive_expect_tx(full_bar(s), (uint32_t)nload * kPageCodes);
#pragma unroll
                    for (int cc = 0; cc < kTileBlocks; ++cc)
                        if (cc < nload)
                            tma_load_3d_stream(dst + cc * kPageCodes, &kmap, full_bar(s), 0, 0,
                                               page[cc], policy);
                }
#pragma unroll
                for (int cc = 0; cc < kTileBlocks; ++cc) {
                    if (cc >= nload) break;
                    const uint8_t* src = a.key_scales + (long long)page[cc] * a.scale_stride;
                    const uint32_t sdst = dst + kStageCodes + cc * kPageScales;
                    if (a.scales16) {
                        cp_async16(sdst + 16u * lane, src + 16 * lane);
                    } else {
                        cp_async8(sdst + 8u * lane, src + 8 * lane);
                        cp_async8(sdst + 8u * (lane + 32), src + 8 * (lane + 32));
                    }
                }
                cp_async_arrive(full_bar(s));
            }
            w.advance(c);
            ++it;
            if (++owner == kProducers) owner = 0;
            sp.next(S);
        }
        if (ok && owner == prod) {
            // the end mark, in the stage after the last tile
            const int s = sp.idx;
            if (lane == 0) ok = mbar_wait(sfree_bar(s), sp.phase ^ 1u, abort_flag, a.status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (ok) {
                if (lane == 0) {
                    st_shared_v2_s32(rec_base + 8u * s, -1, 0);
                    mbar_arrive_expect_tx(full_bar(s), 0u);
                }
                cp_async_arrive(full_bar(s));
                ++it;
            }
        }
        // every copy this warp issued lands before the CTA may exit, whatever
        // the other roles did: of its stages only the last S tiles' can be in
        // flight (S a multiple of kProducers: see the launch)
        cp_async_wait_all();
        if (lane == 0) {
            for (int t = (it > S ? it - S : 0); t < it; ++t)
                if (t % kProducers == prod)
                    mbar_wait_drain(full_bar(t % S), (uint32_t)(t / S) & 1u);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t idesc = nvfp4_idesc(128, kN);
            Walk w;
            w.init(a.context_lengths, a.groups, sb, sj, eb, ej);
            int prev_g = -1, qk = 0, slot = 0, last_acc = -1;
            uint32_t last_phase = 0;
            RingPos sp, ap;
            bool ok = true;
            while (!w.done()) {
                const int c = tile_blocks(w);
                if (w.b != prev_g) {
                    slot = qk & 1;
                    ok = mbar_wait(qfull_bar0 + 8u * slot, (qk >> 1) & 1, abort_flag, a.status);
                    if (!ok) break;
                    ++qk;
                    prev_g = w.b;
                }
                const int s = sp.idx;
                ok = mbar_wait(full_bar(s), sp.phase, abort_flag, a.status);
                if (!ok) break;
                ok = mbar_wait(sfa_bar(s), sp.phase, abort_flag, a.status);
                if (!ok) break;
                ok = mbar_wait(tempty_bar0 + 8u * ap.idx, ap.phase ^ 1u, abort_flag, a.status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)ap.idx * kAccCols;
                const uint32_t codes = stage_base + (uint32_t)s * kStageBytes;
                const uint32_t qb = q_base + (uint32_t)slot * kQSlotBytes;
                const uint32_t sfa = tmem_base + kSfaCol0 + 16u * s;
                const uint32_t sfb = tmem_base + kSfbCol0 + 8u * slot;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (h == 1 && c <= 2) break;       // the second half holds no page
#pragma unroll
                    for (int kc = 0; kc < 2; ++kc)
                        mma_nvfp4(d + kN * h, smem_desc_sw64(codes + h * kHalfCodes + 32 * kc),
                                  smem_desc_sw64(qb + 32 * kc), idesc, sfa + 8 * h + 4 * kc,
                                  sfb + 4 * kc, kc);
                }
                mma_commit(tfull_bar0 + 8u * ap.idx);
                mma_commit(sfree_bar(s));
                if (w.last_of_request(c)) mma_commit(qempty_bar0 + 8u * slot);
                last_acc = ap.idx;
                last_phase = ap.phase;
                w.advance(c);
                sp.next(S);
                ap.next(kAcc);
            }
            // the MMAs complete in order: the last commit covers them all
            if (!ok && last_acc >= 0) mbar_wait_drain(tfull_bar0 + 8u * last_acc, last_phase);
        }
    } else if (warp >= kScaleWarp0 && warp < kScaleWarp0 + 4) {
        // ------------------------------------------------------------ scales
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int t = threadIdx.x - 32 * kScaleWarp0;
        const uint32_t lane_tmem = tmem_base + ((uint32_t)(quad * 32) << 16);
        int qk = 0;
        RingPos sp;
        while (true) {
            const int s = sp.idx;
            if (!mbar_wait(full_bar(s), sp.phase, abort_flag, a.status)) break;
            const int2 rec = ld_shared_v2_s32(rec_base + 8u * s);
            if (rec.x < 0) break;                 // the producer's end mark
            if (rec.y & kRecFirst) {
                // the group's rows (zero beyond G) into the next Q slot: codes
                // sign-fixed and swizzled in shared memory, scale words in
                // every quadrant's lanes 0..15 of the slot's columns
                const int slot = qk & 1;
                if (!mbar_wait(qempty_bar0 + 8u * slot, ((qk >> 1) & 1) ^ 1, abort_flag, a.status))
                    break;
                if (t < kN * 4) {
                    const int r = t >> 2, c = t & 3;
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (r < G) {
                        const long long qrow = (long long)rec.x * G + r;
                        v = __ldg(reinterpret_cast<const uint4*>(a.query + qrow * kRowBytes) + c);
                        const uint2 sc = __ldg(
                            reinterpret_cast<const uint2*>(a.query_scales + qrow * kRowScales));
                        const uint32_t m0 = scale_negative(sc, 2 * c) ? kCodeSigns : 0u;
                        const uint32_t m1 = scale_negative(sc, 2 * c + 1) ? kCodeSigns : 0u;
                        v.x ^= m0;
                        v.y ^= m0;
                        v.z ^= m1;
                        v.w ^= m1;
                    }
                    st_shared_v4(q_base + slot * kQSlotBytes + sw64(r, c), v);
                }
                fence_proxy_async_smem();
                uint2 qs = make_uint2(0u, 0u);
                if (lane < G)
                    qs = __ldg(reinterpret_cast<const uint2*>(
                        a.query_scales + ((long long)rec.x * G + lane) * kRowScales));
                tmem_st_scales(lane_tmem + kSfbCol0 + 8u * slot, qs.x, qs.y);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(qfull_bar0 + 8u * slot);
                ++qk;
            }
            // keys row and 128 + row of the tile: page p, row kk of it.  A page
            // that was not loaded holds stale bytes, which only reach scores
            // the epilogue does not store.
            const uint32_t stage = stage_base + (uint32_t)s * kStageBytes;
            bool fixed = false;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int k = 128 * h + row, p = k >> 6, kk = k & 63;
                const uint2 sc =
                    ld_shared_v2_u32(stage + kStageCodes + p * kPageScales + kk * kRowScales);
                if ((sc.x | sc.y) & kSignBits) {
                    fix_key_signs(stage + p * kPageCodes, kk, sc);
                    fixed = true;
                }
                tmem_st_scales(lane_tmem + kSfaCol0 + 16u * s + 8u * h, sc.x, sc.y);
            }
            if (fixed) fence_proxy_async_smem();
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sfa_bar(s));
            sp.next(S);
        }
    } else if (warp >= kEpiWarp0) {
        // ------------------------------------------------------------ epilogues
        const int side = (warp - kEpiWarp0) >> 2;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_addr = tmem_base + ((uint32_t)(quad * 32) << 16);
        Walk w;
        w.init(a.context_lengths, a.groups, sb, sj, eb, ej);
        int it = 0, prev_g = -1, len = 0;
        while (!w.done()) {
            const int c = tile_blocks(w);
            if ((it & 1) == side) {
                if (w.b != prev_g) {
                    prev_g = w.b;
                    len = min(__ldg(a.context_lengths + w.b), a.max_context);
                }
                const int acc = it % kAcc;
                if (!mbar_wait(tfull_bar0 + 8u * acc, (uint32_t)(it / kAcc) & 1u, abort_flag,
                               a.status))
                    break;
                tc_fence_after();
                uint32_t v[2][8];
                tmem_ld8_async(lane_addr + (uint32_t)acc * kAccCols, v[0]);
                tmem_ld8_async(lane_addr + (uint32_t)acc * kAccCols + kN, v[1]);
                tmem_wait_bind8(v[0]);
                tmem_wait_bind8(v[1]);
                float* dst = a.scores + (long long)w.b * G * a.scores_stride;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int pg = 2 * h + (row >> 6);
                    const int pos = (w.j + pg) * kBlockKeys + (row & 63);
                    if (pg < c && pos < len) {
#pragma unroll
                        for (int r = 0; r < 8; ++r)
                            if (r < G)
                                dst[(long long)r * a.scores_stride + pos] = __uint_as_float(v[h][r]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar0 + 8u * acc);
            }
            w.advance(c);
            ++it;
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

size_t nvfp4_smem_bytes(int stages) { return (size_t)nvfp4_layout(stages).total + 1024; }

cudaError_t launch_nvfp4_scores(const CUtensorMap& kmap, const Nvfp4Args& a, int num_ctas,
                                cudaStream_t stream)
{
    // each stage's scale columns must fit the tensor memory the kernel
    // allocates; a multiple of kProducers keeps stage T - S (T = tiles), whose
    // slot the end mark takes, with the producer that writes the mark, which
    // is the one that leaves it out of its drain
    if (a.stages < kProducers || a.stages > kMaxNvfp4Stages || a.stages % kProducers != 0)
        return cudaErrorInvalidValue;
    const size_t smem = nvfp4_smem_bytes(a.stages);
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
    nvfp4_scores_kernel<<<num_ctas, kThreads, smem, stream>>>(kmap, a);
    return cudaGetLastError();
}

}  // namespace pml
