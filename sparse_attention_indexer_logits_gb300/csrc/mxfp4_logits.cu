// MXFP4 paged MQA logits on sm_103a.
//
//   out[b*next_n + t, p] = sum_h w[b*next_n+t, h] * relu(q[b*next_n+t, h] . k_p)
//
// over MXFP4 queries and keys ("flashinfer.attn_scores", the paragraphs after
// the two bullets: the fp4 variant folds the MXFP4 block scales -- one per
// 32-element group, on both operands -- into the dequantised values; q packs
// two FP4 values per byte; 64 heads of 128; no per-position factor; the
// rectifier acts per head before the weighted sum, first bullet).
//
// Numerics.  A row (one key, or one head of one query slot) holds 128 E2M1
// codes and four E8M0 scales 2^(e_g - 127).  With E the row's largest scale
// exponent (its frame), element d of group g is  c_d * 2^(e_g - E) * 2^(E - 127).
// The tensor cores take the codes as stored and the scales relative to the
// frame -- E8M0 bytes e_g - E + 127, at most 1 -- through tcgen05.mma
// kind::mxf4 (32-element scale blocks, read from tensor memory):
//
//   S[p, h] = sum_g 2^(e_gp - E_p) 2^(e_gh - E_h) (codes_gp . codes_gh),
//   q_h . k_p = 2^(E_p + E_h - 254) * S[p, h]
//
// Each block's products are multiples of 2^-2 at most 36, so a block term is
// exact in fp32 while the two gaps E - e_g add up to at most 124; the tensor
// cores accumulate in fp32.  The frames never enter the MMA:
//
//   logit = 2^(E_p - 127) * 2^(R - 127) * sum_h [w_h * 2^(E_h - R)] * relu(S[p, h])
//
// with R the largest head frame of the slot, so the bracketed weights are at
// most |w_h| and the sum cannot overflow; the key's and slot's frames are
// applied last, as two exact power-of-two multiplies, so a logit outside the
// fp32 range becomes +-inf only at the end.  A key whose largest gap plus its
// request's largest query gap exceeds 124 sets PML_STATUS_FP4_INEXACT (block
// terms below 2^-124 of the frames may be rounded or dropped), as does a head
// whose frame is more than 100 binades below R (its weight is then subnormal
// or zero).  A gap beyond 127 has no E8M0 code: that block's codes are set to
// zero, its terms dropped (and flagged).  An E8M0 NaN scale (0xFF) reaches the
// MMA unchanged and turns its block into NaN; a NaN dot product rectifies to 0.
//
// Scale layout in tensor memory, one byte per 32-element block (measured): the
// scales of A row m (a key) for one K = 64 MMA are bytes 0, 1 of lane m,
// column sfa + m/32; those of B row n (a head), for the output rows of lane
// quadrant q, bytes 0, 1 of lane 32q + n%32, column sfb + n/32.
//
// A tile is 2H 64-key blocks (H = 2 halves of M = 128 at one query slot per
// pass, H = 1 at two): the codes land by TMA with the 64-byte swizzle (a
// 64-byte row is one swizzle span), two blocks of a half being the MMA's
// K-major operand as they land; the 256 scale bytes of a block by a bulk copy.
//
//   warps 0,2,3 producers, tile i to warp i % 3: block-table entries from a
//               64-entry window, per block a TMA of the codes and a bulk
//               copy of its scales onto the stage's barrier; for the
//               owner of a request's first tile also the request's query rows
//               (TMA, 64-byte swizzle), raw scales and weights (bulk copies)
//               into a Q slot.  One warp's round takes about twice a tile's
//               share of HBM time, so three take turns.
//   warp 1      MMA issue: per tile H x 2 MMAs (K = 64) into one of three
//               accumulators and one commit, which the tile's epilogue waits
//               for; that epilogue then frees the stage and the scale columns
//               (a tcgen05 instruction costs the issuing thread ~100 cycles).
//   warps 4-7   scales: per tile each thread takes H keys: frame, gap check,
//               relative scale bytes into the tile's columns, the frames into
//               the accumulator's frame columns; per request the query rows'
//               frames, relative scales (every quadrant's copy), framed
//               weights and slot frames.
//   warps 8-15  two epilogue warpgroups, even and odd tiles: H keys per
//               thread, 64 heads per slot rectified, weighted and summed.
//
// next_n = 3, 4 run as two passes over the cache (slots 0-1, then the rest),
// each with its own launch.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace pml {

namespace {

constexpr int kHeads = kMxfp4Heads;                         // 64
constexpr int kRowBytes = kHeadDim / 2;                     // 64 code bytes per row
constexpr int kRowScales = kHeadDim / 32;                   // 4
constexpr int kBlockCodeBytes = kBlockKeys * kRowBytes;     // 4096
constexpr int kBlockScaleBytes = kBlockKeys * kRowScales;   // 256
constexpr int kProducers = 3;                               // warps 0, 2, 3
constexpr int kMmaWarp = 1;
constexpr int kScaleWarp0 = 4;                              // a warpgroup: warp w -> quadrant w % 4
constexpr int kEpiWarp0 = 8;                                // warps 8-11 even tiles, 12-15 odd
constexpr int kThreads = 512;
constexpr int kAcc = 3;                                     // accumulators
constexpr int kSfaSlots = 4;                                // tiles' key-scale columns
constexpr uint32_t kTmemCols = 512;
constexpr int kExactGapSum = 124;                           // block terms stay normal fp32
constexpr int kWeightGapLimit = 100;

template <int NN>
struct Plan {
    static constexpr int N = kHeads * NN;                    // MMA N: query rows of the pass
    static constexpr int H = NN == 1 ? 2 : 1;                // M = 128 halves per tile
    static constexpr int TB = 2 * H;                         // blocks per tile
    // tensor memory: accumulators, key-scale columns per tile slot, query
    // scales per Q slot, the keys' frames per accumulator (one column a half)
    static constexpr uint32_t kAccCols = (uint32_t)(H * N);
    static constexpr uint32_t kSfaCols = 8u * H;
    static constexpr uint32_t kSfaCol0 = kAcc * kAccCols;
    static constexpr uint32_t kSfbCol0 = kSfaCol0 + kSfaSlots * kSfaCols;
    static constexpr uint32_t kFrameCol0 = kSfbCol0 + 16;
    static_assert(kFrameCol0 + 2 * kAcc <= kTmemCols, "tensor memory");
    static constexpr uint32_t kStageCodes = (uint32_t)TB * kBlockCodeBytes;
    static constexpr uint32_t kStageBytes = kStageCodes + (uint32_t)TB * kBlockScaleBytes;
    static_assert(kStageBytes % 512 == 0, "stages keep the 64-byte swizzle's alignment");
    // one Q slot: the codes (N rows, 64-byte swizzle), raw scales, raw
    // weights, framed weights, relative scale words, slot frames, the
    // conversion's partial results, the largest query gap
    static constexpr uint32_t kQCodes = 0;
    static constexpr uint32_t kQRawSf = (uint32_t)N * kRowBytes;
    static constexpr uint32_t kQRawW = kQRawSf + (uint32_t)N * 4;
    static constexpr uint32_t kQW = kQRawW + (uint32_t)N * 4;
    static constexpr uint32_t kQRel = kQW + (uint32_t)N * 4;
    static constexpr uint32_t kQFrame = kQRel + (uint32_t)N * 4;   // NN ints, padded to 16 B
    static constexpr uint32_t kQPart = kQFrame + 16;                // 4 warps x {max E, max gap}
    static constexpr uint32_t kQGap = kQPart + 32;
    static constexpr uint32_t kQSlotBytes = (kQGap + 16 + 1023) / 1024 * 1024;
    static constexpr uint32_t kQTx = (uint32_t)N * (kRowBytes + 4 + 4);
};

struct Layout {
    uint32_t q, stage, bar, misc, total;
};

// Shared memory: two Q slots, `stages` stages of one tile (codes, then
// scales), barriers.
template <int NN>
__host__ __device__ inline Layout layout_of(int stages)
{
    using P = Plan<NN>;
    Layout L;
    L.q = 0;
    L.stage = 2 * P::kQSlotBytes;
    L.bar = L.stage + (uint32_t)stages * P::kStageBytes;
    L.misc = L.bar + (uint32_t)(2 * stages + 2 * kSfaSlots + 2 * kAcc + 7) * 8;
    L.total = L.misc + 32;
    return L;
}

// 2^k as an fp32 for k in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2_small(int k)
{
    return k >= -126 ? __int_as_float((k + 127) << 23) : __int_as_float(0x00400000);
}

// 2^k for k <= 0, rounded to zero below the fp32 range.
__device__ __forceinline__ float pow2_down(int k)
{
    return k >= -126 ? __int_as_float((k + 127) << 23)
                     : (k >= -149 ? __int_as_float(1 << (k + 149)) : 0.0f);
}

// x * 2^F for F in [-254, 254], as two exact power-of-two multiplies (the
// second rounds once if the result leaves the normal range).
__device__ __forceinline__ float scale_pow2(float x, int F)
{
    const int f1 = F / 2;
    return (x * pow2_small(f1)) * pow2_small(F - f1);
}

// A row's four scale bytes (byte g for group g) relative to its frame: E the
// largest non-NaN exponent (0 if none), gap the largest distance below it,
// rel the bytes e - E + 127 (NaN kept), drop a mask of the groups whose gap
// has no E8M0 code (more than 127; their byte is then 0 and their codes must
// be zeroed).
struct RowScales {
    int E, gap;
    uint32_t rel, drop;
};

__device__ __forceinline__ RowScales row_scales(uint32_t sc)
{
    RowScales r;
    r.E = 0;
    int lo = 255;
    bool any = false;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int e = (int)((sc >> (8 * g)) & 0xFF);
        if (e != 0xFF) {
            r.E = max(r.E, e);
            lo = min(lo, e);
            any = true;
        }
    }
    r.gap = any ? r.E - lo : 0;
    r.rel = 0;
    r.drop = 0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int e = (int)((sc >> (8 * g)) & 0xFF);
        int v = e == 0xFF ? 0xFF : e - r.E + 127;
        if (v < 0) {
            v = 0;
            r.drop |= 1u << g;
        }
        r.rel |= (uint32_t)v << (8 * g);
    }
    return r;
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

// Instruction descriptor of kind::mxf4: E2M1 A and B (format 1), K-major,
// E8M0 scales (scale format 1), scale-data ids 0, dense.
__host__ __device__ constexpr uint32_t mxfp4_idesc(uint32_t M, uint32_t N)
{
    return (1u << 7) | (1u << 10) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24);
}

// D (+)= (A * B^T) with 32-element scale blocks, K = 64.
__device__ __forceinline__ void mma_mxfp4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X "
        "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Eight 32-bit columns of this thread's lane, from taddr on (warp-uniform).
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

__device__ __forceinline__ void tmem_st2(uint32_t taddr, uint32_t x, uint32_t y)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1,%2};" ::"r"(taddr), "r"(x),
                 "r"(y)
                 : "memory");
}

// Two columns of this thread's lane, waited for.
__device__ __forceinline__ void tmem_ld2(uint32_t taddr, uint32_t& x, uint32_t& y)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(x), "=r"(y)
                 : "r"(taddr)
                 : "memory");
}

__device__ __forceinline__ void st_shared_zero16(uint32_t addr)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

// Byte offset of 16-byte chunk c (0..3) of row r in a region written with the
// 64-byte swizzle (512-byte aligned base).
__device__ __forceinline__ uint32_t sw64(int r, int c)
{
    return (uint32_t)(r * kRowBytes + ((c ^ ((r >> 1) & 3)) << 4));
}

// Zero the codes of the groups in `drop` (group g = 16-byte chunk g) of row r.
__device__ __forceinline__ void zero_groups(uint32_t region, int r, uint32_t drop)
{
#pragma unroll
    for (int g = 0; g < 4; ++g)
        if ((drop >> g) & 1u) st_shared_zero16(region + sw64(r, g));
}

// Blocks in the walk's current tile: up to TB, within one request and range.
template <int TB>
__device__ __forceinline__ int tile_blocks(const Walk& w)
{
    const int lim = (w.b == w.eb) ? w.ej : w.nbb;
    return min(lim - w.j, TB);
}

// Position in a ring of n slots and the parity of its current pass.
struct Ring {
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

template <int NN>
__global__ void __launch_bounds__(kThreads, 1)
    mxfp4_logits_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap qmap, const Mxfp4Args a)
{
    using P = Plan<NN>;
    constexpr int N = P::N;
    constexpr int H = P::H;
    constexpr int TB = P::TB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = a.stages;
    const Layout L = layout_of<NN>(S);
    const uint32_t base = smem_addr(smem);
    const uint32_t q0 = base + L.q;
    const uint32_t stage0 = base + L.stage;
    const uint32_t bar = base + L.bar;
    auto full_bar = [&](int s) { return bar + 8u * s; };               // codes and scales landed
    auto sfree_bar = [&](int s) { return bar + 8u * (S + s); };        // stage read by the MMA
    const uint32_t sfa_full0 = bar + 8u * (2 * S);                    // key scales written
    const uint32_t sfa_free0 = sfa_full0 + 8u * kSfaSlots;             // ... read by the MMA
    const uint32_t tfull0 = sfa_free0 + 8u * kSfaSlots;
    const uint32_t tempty0 = tfull0 + 8u * kAcc;
    const uint32_t qfull0 = tempty0 + 8u * kAcc;                       // raw rows landed
    const uint32_t qready0 = qfull0 + 16u;                            // converted
    const uint32_t qempty0 = qready0 + 16u;                           // request done
    const uint32_t wgsync = qempty0 + 16u;                            // the scale warps meet
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);
    int* sched = reinterpret_cast<int*>(smem + L.misc + 16);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int prod = warp == 0 ? 0 : (warp == 2 || warp == 3) ? warp - 1 : -1;

    allow_dependent_launch();
    if (warp == 0) {
        grid_dependency_wait();
        int sb, sj, eb, ej;
        if (a.schedule_meta != nullptr) {
            sb = __ldg(a.schedule_meta + 2 * blockIdx.x);
            sj = __ldg(a.schedule_meta + 2 * blockIdx.x + 1);
            eb = __ldg(a.schedule_meta + 2 * blockIdx.x + 2);
            ej = __ldg(a.schedule_meta + 2 * blockIdx.x + 3);
        } else {
            const long long total = warp_total_blocks(a.seq_lens, a.batch);
            const long long s0 = range_start(total, gridDim.x, blockIdx.x);
            const long long s1 = range_start(total, gridDim.x, blockIdx.x + 1);
            warp_locate2(a.seq_lens, a.batch, s0, s1, sb, sj, eb, ej);
        }
        if (lane == 0) {
            sched[0] = sb; sched[1] = sj; sched[2] = eb; sched[3] = ej;
            *abort_flag = 0;
            for (int s = 0; s < S; ++s) {
                mbar_init(full_bar(s), 1);
                mbar_init(sfree_bar(s), 1);
            }
            for (int i = 0; i < kSfaSlots; ++i) {
                mbar_init(sfa_full0 + 8u * i, 4);
                mbar_init(sfa_free0 + 8u * i, 1);
            }
            for (int i = 0; i < kAcc; ++i) {
                mbar_init(tfull0 + 8u * i, 1);
                mbar_init(tempty0 + 8u * i, 4);
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(qfull0 + 8u * i, 1);
                mbar_init(qready0 + 8u * i, 4);
                mbar_init(qempty0 + 8u * i, 8);   // both epilogue warpgroups
            }
            mbar_init(wgsync, 4);
            fence_mbar_init();
            tma_prefetch_map(&kmap);
            tma_prefetch_map(&qmap);
        }
    } else if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    grid_dependency_wait();
    const int sb = sched[0], sj = sched[1], eb = sched[2], ej = sched[3];

    if (prod >= 0) {
        // ------------------------------------------------------------ producers
        // Tile i (counted over the CTA's range) belongs to producer i % 3 and
        // uses stage i % S; request r's Q slot is r & 1.  Every producer
        // walks every tile.
        const uint64_t policy = policy_evict_first();
        Walk w;
        w.init(a.seq_lens, a.batch, sb, sj, eb, ej);
        int it = 0, owner = 0, prev_b = -1, qidx = -1, win_b = -1;
        int own_q0 = -1, own_q1 = -1;     // this warp's latest query load per slot
        Ring sp;
        long long bt_row = 0;
        // block-table entries 32 at a time, one per lane, the next 32 already
        // in flight: lane i of `cur` holds block cur_j + i, of `nxt` cur_j + 32 + i
        int nbl = 0, cur_j = 0, cur = 0, nxt = 0;
        auto fetch = [&](int j0) {
            return j0 + lane < nbl ? __ldg(a.block_table + bt_row + j0 + lane) : 0;
        };
        bool ok = true;
        while (!w.done()) {
            const int c = tile_blocks<TB>(w);
            const bool first = w.b != prev_b;
            if (first) {
                prev_b = w.b;
                ++qidx;
            }
            if (owner == prod) {
                if (first) {
                    // the request's query rows of this pass into Q slot qidx & 1
                    const int slot = qidx & 1;
                    if (lane == 0)
                        ok = mbar_wait(qempty0 + 8u * slot, ((qidx >> 1) & 1) ^ 1, abort_flag, a.status);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    if (lane == 0) {
                        const uint32_t qs = q0 + slot * P::kQSlotBytes;
                        const uint32_t qf = qfull0 + 8u * slot;
                        const long long r0 = ((long long)w.b * a.next_n + a.slot0) * kHeads;
                        mbar_arrive_expect_tx(qf, P::kQTx);
#pragma unroll
                        for (int u = 0; u < NN; ++u)
                            tma_load_2d(qs + P::kQCodes + u * kHeads * kRowBytes, &qmap, qf, 0,
                                        (int)(r0 + u * kHeads));
                        bulk_load(qs + P::kQRawSf, a.q_sf + r0 * kRowScales, (uint32_t)N * 4, qf);
                        bulk_load(qs + P::kQRawW, a.weights + r0, (uint32_t)N * 4, qf);
                    }
                    if (slot) own_q1 = qidx;
                    else own_q0 = qidx;
                }
                if (w.b != win_b) {
                    bt_row = (long long)w.b * a.bt_stride;
                    nbl = blocks_of(min(w.len, a.max_context));
                    cur_j = w.j;
                    cur = fetch(cur_j);
                    nxt = fetch(cur_j + 32);
                    win_b = w.b;
                }
                while (w.j >= cur_j + 32) {
                    cur_j += 32;
                    cur = nxt;
                    nxt = fetch(cur_j + 32);
                }
                // blocks w.j .. w.j + TB - 1 lie in the window [cur_j, cur_j + 64);
                // those below max_context are a prefix of the tile
                int page[TB];
                int nload = 0;
#pragma unroll
                for (int cc = 0; cc < TB; ++cc) {
                    const int i = w.j - cur_j + cc;
                    long long pg = __shfl_sync(0xffffffffu, i < 32 ? cur : nxt, i & 31);
                    page[cc] = 0;
                    if (cc < c && (long long)(w.j + cc) * kBlockKeys < a.max_context) {
                        if (pg < 0 || pg >= a.num_blocks) {
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
                const uint32_t dst = stage0 + (uint32_t)s * P::kStageBytes;
                if (lane == 0) {
                    mbar_arrive_expect_tx(full_bar(s), (uint32_t)nload * (kBlockCodeBytes + kBlockScaleBytes));
#pragma unroll
                    for (int cc = 0; cc < TB; ++cc)
                        if (cc < nload) {
                            tma_load_3d_stream(dst + cc * kBlockCodeBytes, &kmap, full_bar(s), 0, 0,
                                               page[cc], policy);
                            bulk_load_stream(dst + P::kStageCodes + cc * kBlockScaleBytes,
                                             a.kv + (long long)page[cc] * kMxfp4BlockBytes + kBlockCodeBytes,
                                             kBlockScaleBytes, full_bar(s), policy);
                        }
                }
            }
            w.advance(c);
            ++it;
            if (++owner == kProducers) owner = 0;
            sp.next(S);
        }
        // every copy this warp issued lands before the CTA may exit: of its
        // stages only the last S tiles' can be in flight, of its query loads
        // only those of the last two requests
        if (lane == 0) {
            for (int t = (it > S ? it - S : 0); t < it; ++t)
                if (t % kProducers == prod) mbar_wait_drain(full_bar(t % S), (uint32_t)(t / S) & 1u);
            if (own_q0 >= 0 && own_q0 >= qidx - 1)
                mbar_wait_drain(qfull0, (uint32_t)(own_q0 >> 1) & 1u);
            if (own_q1 >= 0 && own_q1 >= qidx - 1)
                mbar_wait_drain(qfull0 + 8u, (uint32_t)(own_q1 >> 1) & 1u);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t idesc = mxfp4_idesc(128, N);
            Walk w;
            w.init(a.seq_lens, a.batch, sb, sj, eb, ej);
            int prev_b = -1, qidx = -1, slot = 0, last_acc = -1;
            uint32_t last_phase = 0;
            Ring sp, fp, ap;
            bool ok = true;
            while (!w.done()) {
                const int c = tile_blocks<TB>(w);
                if (w.b != prev_b) {
                    prev_b = w.b;
                    ++qidx;
                    slot = qidx & 1;
                    ok = mbar_wait(qready0 + 8u * slot, (uint32_t)(qidx >> 1) & 1u, abort_flag, a.status);
                    if (!ok) break;
                }
                // the key scales of the tile are written only after its stage landed
                const int s = sp.idx;
                ok = mbar_wait(sfa_full0 + 8u * fp.idx, fp.phase, abort_flag, a.status);
                if (!ok) break;
                ok = mbar_wait(tempty0 + 8u * ap.idx, ap.phase ^ 1u, abort_flag, a.status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)ap.idx * P::kAccCols;
                const uint32_t codes = stage0 + (uint32_t)s * P::kStageBytes;
                const uint32_t qb = q0 + (uint32_t)slot * P::kQSlotBytes + P::kQCodes;
                const uint32_t sfa = tmem_base + P::kSfaCol0 + (uint32_t)fp.idx * P::kSfaCols;
                const uint32_t sfb = tmem_base + P::kSfbCol0 + 8u * slot;
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    if (h == 1 && c <= 2) break;       // the second half holds no block
#pragma unroll
                    for (int kc = 0; kc < 2; ++kc)
                        mma_mxfp4(d + (uint32_t)(N * h),
                                  smem_desc_sw64(codes + h * 2 * kBlockCodeBytes + 32 * kc),
                                  smem_desc_sw64(qb + 32 * kc), idesc, sfa + 8 * h + 4 * kc,
                                  sfb + (uint32_t)(N / 32) * kc, kc);
                }
                // one commit: the epilogue that sees it also frees the stage and
                // the scale columns
                mma_commit(tfull0 + 8u * ap.idx);
                last_acc = ap.idx;
                last_phase = ap.phase;
                w.advance(c);
                sp.next(S);
                fp.next(kSfaSlots);
                ap.next(kAcc);
            }
            // the MMAs complete in order: the last commit covers them all
            if (!ok && last_acc >= 0) mbar_wait_drain(tfull0 + 8u * last_acc, last_phase);
        }
    } else if (warp >= kScaleWarp0 && warp < kScaleWarp0 + 4) {
        // ------------------------------------------------------------ scales
        const int quad = warp & 3;
        const int t = threadIdx.x - 32 * kScaleWarp0;          // 0..127
        const uint32_t lane_tmem = tmem_base + ((uint32_t)(quad * 32) << 16);
        uint32_t sync_ph = 0;
        // the four warps meet on an mbarrier (bounded like every other wait)
        auto wg_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(wgsync);
            const bool r = mbar_wait(wgsync, sync_ph, abort_flag, a.status);
            sync_ph ^= 1u;
            return r;
        };
        // The query rows of a request's pass in Q slot `slot`: frames,
        // relative scales (zeroing groups beyond reach), framed weights, slot
        // frames, the largest gap; then the relative scale words into every
        // quadrant's lanes of the slot's columns.  Row n = thread n.
        auto convert_q = [&](int slot, uint32_t par) -> bool {
            const uint32_t qs = q0 + slot * P::kQSlotBytes;
            if (!mbar_wait(qfull0 + 8u * slot, par, abort_flag, a.status)) return false;
            const bool mine = t < N;
            RowScales f{0, 0, 0u, 0u};
            if (mine) {
                f = row_scales(ld_shared_u32(qs + P::kQRawSf + 4u * t));
                st_shared_u32(qs + P::kQRel + 4u * t, f.rel);
                if (f.drop) zero_groups(qs + P::kQCodes, t, f.drop);
            }
            const int emax = (int)__reduce_max_sync(0xffffffffu, mine ? (uint32_t)f.E : 0u);
            const int gmax = (int)__reduce_max_sync(0xffffffffu, mine ? (uint32_t)f.gap : 0u);
            if (lane == 0) st_shared_v2_s32(qs + P::kQPart + 8u * quad, emax, gmax);
            if (!wg_sync()) return false;
            if (mine) {
                // rows 64u..64u+63 (slot u of the pass) are warps 2u, 2u+1
                const int u = t >> 6;
                const int R = max(ld_shared_v2_s32(qs + P::kQPart + 8u * (2 * u)).x,
                                  ld_shared_v2_s32(qs + P::kQPart + 8u * (2 * u + 1)).x);
                const float wt = __uint_as_float(ld_shared_u32(qs + P::kQRawW + 4u * t));
                st_shared_u32(qs + P::kQW + 4u * t, __float_as_uint(wt * pow2_down(f.E - R)));
                if (R - f.E > kWeightGapLimit) atomicOr(a.status, kStatusFp4Inexact);
                if ((t & 63) == 0) st_shared_u32(qs + P::kQFrame + 4u * u, (uint32_t)R);
            }
            if (t == 0) {
                int g = 0;
#pragma unroll
                for (int u = 0; u < 2 * NN; ++u) g = max(g, ld_shared_v2_s32(qs + P::kQPart + 8u * u).y);
                st_shared_u32(qs + P::kQGap, (uint32_t)g);
            }
            if (!wg_sync()) return false;
            // lane i of every quadrant: rows i + 32j, the words of chunk 0
            // (groups 0, 1) in columns j, of chunk 1 (groups 2, 3) in N/32 + j
            uint32_t v[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
            for (int j = 0; j < N / 32; ++j) {
                const uint32_t rel = ld_shared_u32(qs + P::kQRel + 4u * (lane + 32 * j));
                v[j] = rel & 0xFFFFu;
                v[N / 32 + j] = rel >> 16;
            }
            tmem_st8(lane_tmem + P::kSfbCol0 + 8u * slot, v);
            fence_proxy_async_smem();             // zeroed query codes, for the MMA
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(qready0 + 8u * slot);
            return true;
        };

        Walk w;
        w.init(a.seq_lens, a.batch, sb, sj, eb, ej);
        int prev_b = -1, qidx = -1, qgap = 0, len = 0;
        Ring sp, fp, ap;
        while (!w.done()) {
            const int c = tile_blocks<TB>(w);
            if (w.b != prev_b) {
                prev_b = w.b;
                ++qidx;
                len = min(w.len, a.max_context);
                if (!convert_q(qidx & 1, (uint32_t)(qidx >> 1) & 1u)) break;
                qgap = (int)ld_shared_u32(q0 + (qidx & 1) * P::kQSlotBytes + P::kQGap);
            }
            const int s = sp.idx;
            if (!mbar_wait(full_bar(s), sp.phase, abort_flag, a.status)) break;
            if (!mbar_wait(sfa_free0 + 8u * fp.idx, fp.phase ^ 1u, abort_flag, a.status)) break;
            // the accumulator's frame columns: free once its epilogue is done
            if (!mbar_wait(tempty0 + 8u * ap.idx, ap.phase ^ 1u, abort_flag, a.status)) break;
            tc_fence_after();
            const uint32_t stage = stage0 + (uint32_t)s * P::kStageBytes;
            uint32_t frame[2] = {0u, 0u};
            bool zeroed = false;
#pragma unroll
            for (int h = 0; h < H; ++h) {
                // key 128h + t: block p of the tile, row kk of it.  A block that
                // was not loaded holds stale bytes, which reach only logits the
                // epilogue does not store.
                const int k = 128 * h + t, p = k >> 6, kk = k & 63;
                const RowScales f = row_scales(
                    ld_shared_u32(stage + P::kStageCodes + p * kBlockScaleBytes + kk * kRowScales));
                if (f.drop) {
                    zero_groups(stage + p * kBlockCodeBytes, kk, f.drop);
                    zeroed = true;
                }
                const bool valid = p < c && (w.j + p) * kBlockKeys + kk < len;
                if (valid && f.gap + qgap > kExactGapSum) atomicOr(a.status, kStatusFp4Inexact);
                const uint32_t lo = f.rel & 0xFFFFu, hi = f.rel >> 16;
                const uint32_t v[8] = {lo, lo, lo, lo, hi, hi, hi, hi};
                tmem_st8(lane_tmem + P::kSfaCol0 + (uint32_t)fp.idx * P::kSfaCols + 8u * h, v);
                frame[h] = (uint32_t)f.E;
            }
            tmem_st2(lane_tmem + P::kFrameCol0 + 2u * ap.idx, frame[0], frame[1]);
            if (zeroed) fence_proxy_async_smem();
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sfa_full0 + 8u * fp.idx);
            w.advance(c);
            sp.next(S);
            fp.next(kSfaSlots);
            ap.next(kAcc);
        }
    } else if (warp >= kEpiWarp0) {
        // ------------------------------------------------------------ epilogues
        const int side = (warp - kEpiWarp0) >> 2;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_tmem = tmem_base + ((uint32_t)(quad * 32) << 16);
        constexpr int NC = N / 32;                      // 32-column chunks of a half
        Walk w;
        w.init(a.seq_lens, a.batch, sb, sj, eb, ej);
        int k = 0, prev_b = -1, qidx = -1, slot = 0, len = 0;
        bool need_q = false;
        Ring sp, fp;                                   // the tile's stage and scale columns
        while (!w.done()) {
            const int c = tile_blocks<TB>(w);
            if (w.b != prev_b) {
                prev_b = w.b;
                ++qidx;
                slot = qidx & 1;
                len = min(w.len, a.max_context);
                need_q = true;
            }
            const bool last = w.last_of_request(c);
            const int acc = k % kAcc;
            if ((k & 1) == side) {
                if (need_q) {
                    // the framed weights and frames of the request
                    if (!mbar_wait(qready0 + 8u * slot, (uint32_t)(qidx >> 1) & 1u, abort_flag, a.status))
                        break;
                    need_q = false;
                }
                if (!mbar_wait(tfull0 + 8u * acc, (uint32_t)(k / kAcc) & 1u, abort_flag, a.status)) break;
                tc_fence_after();
                if (quad == 0 && lane == 0) {
                    // the tile's MMAs are complete: its stage and scale columns are free
                    mbar_arrive(sfree_bar(sp.idx));
                    mbar_arrive(sfa_free0 + 8u * fp.idx);
                }
                const uint32_t qs = q0 + slot * P::kQSlotBytes;
                uint32_t E[2];
                tmem_ld2(lane_tmem + P::kFrameCol0 + 2u * acc, E[0], E[1]);
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const int key = 128 * h + row;
                    const int pg = key >> 6;
                    const int pos = (w.j + pg) * kBlockKeys + (key & 63);
                    const bool valid = pg < c && pos < len;
                    const uint32_t col = (uint32_t)(acc * P::kAccCols + N * h);
                    uint32_t buf[2][32];
                    uint64_t acc4[4];
                    tmem_ld32_async(lane_tmem + col, buf[0]);
                    tmem_wait_bind32(buf[0]);
#pragma unroll
                    for (int cc = 0; cc < NC; ++cc) {
                        if (cc + 1 < NC) tmem_ld32_async(lane_tmem + col + 32u * (cc + 1), buf[(cc + 1) & 1]);
                        if ((cc & 1) == 0) {
#pragma unroll
                            for (int u = 0; u < 4; ++u) acc4[u] = 0ull;
                        }
                        const uint32_t(&v)[32] = buf[cc & 1];
#pragma unroll
                        for (int hh = 0; hh < 32; hh += 4) {
                            const uint4 wv = ld_shared_v4(qs + P::kQW + 4u * (32 * cc + hh));
                            const uint64_t w01 = ((uint64_t)wv.y << 32) | wv.x;
                            const uint64_t w23 = ((uint64_t)wv.w << 32) | wv.z;
                            acc4[(hh / 2) % 4] =
                                fma2(w01, pack2(fmaxf(__uint_as_float(v[hh]), 0.f),
                                                fmaxf(__uint_as_float(v[hh + 1]), 0.f)),
                                     acc4[(hh / 2) % 4]);
                            acc4[(hh / 2 + 1) % 4] =
                                fma2(w23, pack2(fmaxf(__uint_as_float(v[hh + 2]), 0.f),
                                                fmaxf(__uint_as_float(v[hh + 3]), 0.f)),
                                     acc4[(hh / 2 + 1) % 4]);
                        }
                        if ((cc & 1) == 1 && valid) {
                            const int u = cc >> 1;            // query slot of the pass
                            const float r = (sum2(acc4[0]) + sum2(acc4[1])) + (sum2(acc4[2]) + sum2(acc4[3]));
                            const int R = (int)ld_shared_u32(qs + P::kQFrame + 4u * u);
                            const float logit = scale_pow2(r, (int)E[h] + R - 254);
                            const long long o = ((long long)w.b * a.next_n + a.slot0 + u) * a.out_stride + pos;
                            if (a.out_bf16)
                                reinterpret_cast<__nv_bfloat16*>(a.out)[o] = __float2bfloat16_rn(logit);
                            else
                                reinterpret_cast<float*>(a.out)[o] = logit;
                        }
                        if (cc + 1 < NC) tmem_wait_bind32(buf[(cc + 1) & 1]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty0 + 8u * acc);
            }
            if (last) {
                // this warpgroup is done with the request: its own tiles of it
                // came earlier in the walk
                __syncwarp();
                if (lane == 0) mbar_arrive(qempty0 + 8u * slot);
            }
            w.advance(c);
            ++k;
            sp.next(S);
            fp.next(kSfaSlots);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <int NN>
cudaError_t launch_pass(const CUtensorMap& kmap, const CUtensorMap& qmap, const Mxfp4Args& a,
                        int num_ctas, cudaStream_t stream)
{
    const size_t smem = mxfp4_smem_bytes(NN, a.stages);
    static int configured_device = -1;
    static size_t configured_smem = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev || configured_smem < smem) {
        e = cudaFuncSetAttribute(mxfp4_logits_kernel<NN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        configured_device = dev;
        configured_smem = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)num_ctas);
    cfg.blockDim = dim3((unsigned)kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, mxfp4_logits_kernel<NN>, kmap, qmap, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

size_t mxfp4_smem_bytes(int slots_per_pass, int stages)
{
    const uint32_t t = slots_per_pass == 1 ? layout_of<1>(stages).total : layout_of<2>(stages).total;
    return (size_t)t + 1024;
}

cudaError_t launch_mxfp4_logits(const CUtensorMap& kmap, const CUtensorMap& qmap,
                                const Mxfp4Args& args, int num_ctas, cudaStream_t stream)
{
    // passes of at most two slots each: N = 64 or 128
    for (int s0 = 0; s0 < args.next_n; s0 += 2) {
        Mxfp4Args a = args;
        a.slot0 = s0;
        const int nn = args.next_n - s0 >= 2 ? 2 : 1;
        a.stages = nn == 1 ? args.stages : args.stages2;
        const cudaError_t e = nn == 1 ? launch_pass<1>(kmap, qmap, a, num_ctas, stream)
                                      : launch_pass<2>(kmap, qmap, a, num_ctas, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace pml
