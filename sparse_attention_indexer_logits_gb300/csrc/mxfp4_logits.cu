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
// exponent, element d of group g is  c_d * 2^-(E - e_g) * 2^(E - 127):  a
// code shifted down by the group's gap G_g = E - e_g, times one power of two
// per row (the row's frame).  The shifted codes are exact in f16 while every
// gap is at most 23 and exact in bf16 up to 132 (codes have at most two
// significant bits), so a key tile and the query rows become 16-bit operands
// without rounding, and tcgen05.mma kind::f16 forms
//
//   S[p, h] = k'_p . q'_h,     q_h . k_p = 2^(E_p + E_h - 254) * S[p, h]
//
// with exact products accumulated in fp32.  A tile (128 keys) runs in f16 when
// all its keys' gaps and its request's query gaps are <= 23, else in bf16;
// the query rows are kept in both forms.  The frames never enter the MMA:
//
//   logit = 2^(E_p - 127) * 2^(R - 127) * sum_h [w_h * 2^(E_h - R)] * relu(S[p, h])
//
// with R the largest head frame of the slot, so the bracketed weights are at
// most |w_h| and the sum cannot overflow; the key's and slot's frames are
// applied last, as two exact power-of-two multiplies, so a logit outside the
// fp32 range becomes +-inf only at the end.  The products of the MMA are exact
// as long as, for every group, the key's and the head's gaps add up to at most
// 124 (the smallest product then stays a normal fp32); a tile where the two
// largest gaps add up to more sets PML_STATUS_FP4_INEXACT (products below
// 2^-124 of the frames may be dropped), as does a head whose frame is more than
// 100 binades below R (its weight is then subnormal or zero).  An E8M0 NaN
// scale (0xFF) turns its group into NaN; a NaN dot product rectifies to 0.
//
// Roles:
//   warp 0      producer: the CTA's range of 64-key blocks in windows of 32
//               sub-tiles (window.cuh); per 128-key sub-tile one bulk copy
//               of each block (4096 code bytes then 256 scale bytes, as the
//               cache holds them) into a staging slot and a 32-byte record;
//               per request the raw query codes, scales and weights of the
//               pass's slots into one of two Q slots.
//   warps 1, 3  MMA issue (warp 1 also allocates TMEM), the sub-tiles of the
//               even and the odd groups: per sub-tile eight tcgen05.mma
//               kind::f16 (K = 16) with A = the key tile in tensor memory,
//               B = the request's query rows in shared memory, into the
//               owning group's accumulator (64 * NN columns); commits free
//               the key tile and fill the accumulator.
//   warp 2      scout: per sub-tile, the largest scale gap among the keys
//               below the request's length, read from the staged scale bytes,
//               which fixes the tile's operand format.
//   warps 4..   NWG warpgroups (four for one slot per pass, two for two),
//               sub-tile k going to group k mod NWG.  A thread owns one key
//               row: it dequantises the row into its TMEM lane of the group's
//               key tile and, after the MMA, reads the row's head scores back
//               for the epilogue (the dequantisation of the group's next
//               sub-tile is done before the epilogue of its previous one,
//               which hides the MMA).  The group that takes a request's first
//               sub-tile also converts the request's query rows, frames and
//               weights; the epilogue of the request's last finished sub-tile
//               frees its Q slot.
//
// next_n = 3, 4 run as two passes over the cache (slots 0-1, then the rest),
// each with its own launch.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "window.cuh"

namespace pml {

namespace {

constexpr int kHeads = kMxfp4Heads;                       // 64
constexpr int kRowBytes = kHeadDim / 2;                   // 64 code bytes per row
constexpr int kRowScales = kHeadDim / 32;                 // 4
constexpr int kBlockCodeBytes = kBlockKeys * kRowBytes;   // 4096
constexpr int kStageBytes = 2 * kMxfp4BlockBytes;         // 8704: one 128-key sub-tile
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kScoutWarp = 2;
constexpr int kMmaWarp2 = 3;                              // second MMA issuer
constexpr int kFirstWgWarp = 4;
constexpr uint32_t kTileCols = kHeadDim / 2;              // 64: two 16-bit values per column
constexpr uint32_t kTmemCols = 512;
constexpr int kF16MaxGap = 23;                            // exact in f16 up to here
constexpr int kExactGapSum = 124;                         // products stay normal fp32
constexpr int kWeightGapLimit = 100;
constexpr int kFmtF16 = 0, kFmtBf16 = 1;                  // kind::f16 operand formats
constexpr int kDoneAll = 1 << 24;                         // Q-slot release count, see epilogue

// Record of a sub-tile (two 16-byte words): {request, first block, min(len,
// max_context), meta} and {request index in this CTA, sub-tile index within
// the request, 0, 0}; meta = block count | flags | Q slot.
constexpr int kMetaFirst = 1 << 8;
constexpr int kMetaLast = 1 << 9;
constexpr int kMetaSlotShift = 12;
constexpr int kStageEnd = 1 << 20;

template <int NN>
struct Plan {
    static constexpr int N = kHeads * NN;                  // MMA N: query rows of the pass
    static constexpr int NWG = NN == 1 ? 4 : 2;            // warpgroups
    static constexpr int KPW = NN == 1 ? 1 : 2;            // key tiles per warpgroup
    static constexpr int APW = 1;                          // accumulators per warpgroup
    static constexpr int kThreads = 32 * kFirstWgWarp + 128 * NWG;
    static constexpr uint32_t kAccCols = (uint32_t)(NWG * APW * N);
    static constexpr int kKeyTiles = NWG * KPW;
    static_assert(kAccCols + kKeyTiles * kTileCols <= kTmemCols, "tensor memory");
    // one Q slot: the 16-bit operand in both formats (two K halves of N rows
    // x 128 bytes each, 128-byte swizzled), then the raw rows as loaded, the
    // framed weights, the slot frames and the conversion's partial results
    static constexpr uint32_t kHalf = (uint32_t)N * 128;
    static constexpr uint32_t kFmtBytes = 2 * kHalf;
    static constexpr uint32_t kRawCodes = 2 * kFmtBytes;
    static constexpr uint32_t kRawSf = kRawCodes + (uint32_t)N * kRowBytes;
    static constexpr uint32_t kRawW = kRawSf + (uint32_t)N * kRowScales;
    static constexpr uint32_t kWq = kRawW + (uint32_t)N * 4;
    static constexpr uint32_t kFrame = kWq + (uint32_t)N * 4;      // NN ints, padded to 16 B
    static constexpr uint32_t kPart = kFrame + 16;                 // 4 warps x {max E, max gap}
    static constexpr uint32_t kMeta = kPart + 32;                  // {f16 ok, max gap}
    static constexpr uint32_t kSlotBytes = (kMeta + 16 + 1023) / 1024 * 1024;
    static constexpr uint32_t kRawBytes = (uint32_t)N * (kRowBytes + kRowScales + 4);
};

struct Layout {
    uint32_t stage, q, rec, gap, info, done, bar, misc, total;
};

// Shared memory: two Q slots, `stages` staging slots (one sub-tile's two raw
// blocks each), per stage its record and its tile gap, per key tile an
// information word for the MMA, the Q slots' release counters, barriers.
template <int NN>
__host__ __device__ inline Layout layout_of(int stages)
{
    using P = Plan<NN>;
    Layout L;
    L.q = 0;                                                   // 1024-aligned Q slots first
    L.stage = L.q + 2 * P::kSlotBytes;
    L.rec = L.stage + (uint32_t)stages * kStageBytes;
    L.gap = L.rec + (uint32_t)stages * 32;
    L.info = L.gap + ((uint32_t)stages * 4 + 15) / 16 * 16;
    L.done = L.info + (uint32_t)P::kKeyTiles * 16;
    L.bar = L.done + 16;
    L.misc = L.bar + (uint32_t)(3 * stages + 6 + 2 * P::kKeyTiles + (2 * P::APW + 1) * P::NWG) * 8;
    L.total = L.misc + 32;
    return L;
}

// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled
// K-major region whose rows are 128 bytes (8-row atoms of 1 KB).
__device__ __forceinline__ uint32_t sw128(int r, int c)
{
    return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
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

// The four scale exponents of a row (byte g of sc): the row frame E (largest
// non-NaN exponent, 0 if none), the largest gap, and a NaN mask per group.
struct RowFrame {
    int E, gap;
    uint32_t nan_mask;
};

__device__ __forceinline__ RowFrame row_frame(uint32_t sc)
{
    RowFrame f;
    f.E = 0;
    f.nan_mask = 0;
    int lo = 255;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int e = (int)((sc >> (8 * g)) & 0xFF);
        if (e == 0xFF) {
            f.nan_mask |= 1u << g;
        } else {
            f.E = max(f.E, e);
            lo = min(lo, e);
        }
    }
    f.gap = f.nan_mask == 0xF ? 0 : f.E - lo;
    return f;
}

// Multiplier of group g (gap G) for each format, in both halves of a word:
// f16 path: 2^-G as an f16 (G <= 23, subnormal from 15 on), times the f16
// value of the code; bf16 path: the code's f16 bits moved into bf16 position
// (its value times 2^-112, see to_bf16_bits) times 2^(112 - G).  NaN for a NaN
// scale.
__device__ __forceinline__ uint32_t factor_f16(int G, bool nan)
{
    uint32_t h = nan ? 0x7E00u : (G <= 14 ? (uint32_t)(15 - G) << 10 : (G <= 24 ? 1u << (24 - G) : 0u));
    return h | (h << 16);
}
__device__ __forceinline__ uint32_t factor_bf16(int G, bool nan)
{
    // 2^(112 - G) is a normal bf16 down to G = 238; the product rounds (to a
    // subnormal or zero) once it leaves bf16's range, from G = 133 on
    uint32_t h = nan ? 0x7FC0u : (G <= 238 ? (uint32_t)(239 - G) << 7 : 0u);
    return h | (h << 16);
}

// An f16x2 holding two E2M1 values (exact) -> the same values times 2^-112 as
// a bf16x2: the 5-bit exponent and the mantissa's top bit move down three
// places into bf16 position, the signs stay.
__device__ __forceinline__ uint32_t to_bf16_bits(uint32_t h)
{
    return ((h & 0x7FFF7FFFu) >> 3) | (h & 0x80008000u);
}

// One 16-byte chunk of a row (32 codes of group g, four code words) -> 16
// words of 16-bit operand pairs (byte i -> word i), in format fmt.
__device__ __forceinline__ void dequant_chunk(uint4 v, uint32_t fac, int fmt, uint32_t (&out)[16])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t h[4];
        e2m1x8_to_f16x2x4(w[q], h);
        if (fmt == kFmtF16) {
#pragma unroll
            for (int b = 0; b < 4; ++b) out[4 * q + b] = mul_f16x2(h[b], fac);
        } else {
#pragma unroll
            for (int b = 0; b < 4; ++b) out[4 * q + b] = mul_bf16x2(to_bf16_bits(h[b]), fac);
        }
    }
}

// v[i] holds chunk (i + rot) & 3 of a row; afterwards v[c] holds chunk c.
// Two conditional rotations (by one chunk, then by two), as selects.
__device__ __forceinline__ void rotate_back(uint4 (&v)[4], int rot)
{
    if (rot & 1) {
        const uint4 t = v[3];
        v[3] = v[2];
        v[2] = v[1];
        v[1] = v[0];
        v[0] = t;
    }
    if (rot & 2) {
        uint4 t = v[0];
        v[0] = v[2];
        v[2] = t;
        t = v[1];
        v[1] = v[3];
        v[3] = t;
    }
}

// Ring position and the parity of its current pass.
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
__global__ void __launch_bounds__(Plan<NN>::kThreads, 1) mxfp4_logits_kernel(const Mxfp4Args a)
{
    using P = Plan<NN>;
    constexpr int N = P::N;
    constexpr int NWG = P::NWG;
    constexpr int KPW = P::KPW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = a.stages;
    const Layout L = layout_of<NN>(S);
    const uint32_t base = smem_addr(smem);
    const uint32_t stage0 = base + L.stage;
    const uint32_t q0 = base + L.q;
    const uint32_t bar = base + L.bar;
    auto full_bar = [&](int s) { return bar + 8u * s; };             // staging landed
    auto empty_bar = [&](int s) { return bar + 8u * (S + s); };      // staging read
    auto scout_bar = [&](int s) { return bar + 8u * (2 * S + s); };  // tile gap known
    const uint32_t qfull0 = bar + 8u * (3 * S);           // raw rows landed, per Q slot
    const uint32_t qready0 = qfull0 + 16;                 // converted
    const uint32_t qempty0 = qready0 + 16;                // every sub-tile of the request done
    const uint32_t ktfull0 = qempty0 + 16;                // key tile written
    const uint32_t ktfree0 = ktfull0 + 8u * P::kKeyTiles; // key tile read by the MMA
    const uint32_t accfull0 = ktfree0 + 8u * P::kKeyTiles;
    const uint32_t accempty0 = accfull0 + 8u * NWG * P::APW;
    const uint32_t wgsync0 = accempty0 + 8u * NWG * P::APW;   // a group's four warps meet
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);
    int* done_cnt = reinterpret_cast<int*>(smem + L.done);   // per Q slot

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    allow_dependent_launch();
    int sb = 0, sj = 0, eb = 0, ej = 0;
    Window win;
    if (warp == kProducerWarp) {
        grid_dependency_wait();
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
        win = make_window<1>(a, sb, sj, sb, sj, eb, ej, lane);
    } else if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    } else if (warp == kScoutWarp && lane == 0) {
        *abort_flag = 0;
        done_cnt[0] = 0;
        done_cnt[1] = 0;
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 4);        // the owning group's four warps
            mbar_init(scout_bar(s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(qfull0 + 8u * i, 1);
            mbar_init(qready0 + 8u * i, 4);
            mbar_init(qempty0 + 8u * i, 1);
        }
        for (int i = 0; i < P::kKeyTiles; ++i) {
            mbar_init(ktfull0 + 8u * i, 4);
            mbar_init(ktfree0 + 8u * i, 1);
        }
        for (int i = 0; i < NWG * P::APW; ++i) {
            mbar_init(accfull0 + 8u * i, 1);
            mbar_init(accempty0 + 8u * i, 4);
        }
        for (int i = 0; i < NWG; ++i) mbar_init(wgsync0 + 8u * i, 4);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    grid_dependency_wait();

    if (warp == kProducerWarp) {
        // ---------------------------------------------------------------- producer
        const uint64_t policy = policy_evict_first();
        Ring st;
        int qbase = 0, issued = 0, q_issued = 0;
        bool ok = true;
        while (true) {
            Window nxt;
            bool have_nxt = false;
            const int qidx = qbase + __popc(win.first_mask & ((2u << lane) - 1u)) - 1;
            // sub-tile index within the request's part of this CTA's range
            const int j0 = win.b == sb ? sj : 0;
            const int sub_idx = (win.j - j0) >> 1;
            for (int k = 0; k < win.n; ++k) {
                if ((win.first_mask >> k) & 1u) {
                    if (lane == k) {
                        // this request's raw query rows, scales and weights
                        const int slot = qidx & 1;
                        ok = mbar_wait(qempty0 + 8u * slot, ((qidx >> 1) & 1) ^ 1, abort_flag, a.status);
                        if (ok) {
                            const uint32_t qs = q0 + slot * P::kSlotBytes;
                            const uint32_t qf = qfull0 + 8u * slot;
                            const long long r0 = ((long long)win.b * a.next_n + a.slot0) * kHeads;
                            mbar_arrive_expect_tx(qf, P::kRawBytes);
                            bulk_load(qs + P::kRawCodes, a.q + r0 * kRowBytes, (uint32_t)N * kRowBytes, qf);
                            bulk_load(qs + P::kRawSf, a.q_sf + r0 * kRowScales, (uint32_t)N * kRowScales, qf);
                            bulk_load(qs + P::kRawW, a.weights + r0, (uint32_t)N * 4, qf);
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, k);
                    if (!ok) break;
                    ++q_issued;
                }
                if (lane == 0) ok = mbar_wait(empty_bar(st.idx), st.phase ^ 1, abort_flag, a.status);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (lane == k) {
                    const int meta = win.cnt | (win.first ? kMetaFirst : 0) | (win.last ? kMetaLast : 0) |
                                     ((qidx & 1) << kMetaSlotShift);
                    const uint32_t rec = base + L.rec + 32u * st.idx;
                    st_shared_v4(rec, (uint32_t)win.b, (uint32_t)win.j, (uint32_t)win.len, (uint32_t)meta);
                    st_shared_v4(rec + 16, (uint32_t)qidx, (uint32_t)sub_idx, 0u, 0u);
                    const uint32_t fb = full_bar(st.idx);
                    mbar_arrive_expect_tx(fb, (uint32_t)((win.ld0 ? 1 : 0) + (win.ld1 ? 1 : 0)) *
                                                  kMxfp4BlockBytes);
                    const uint32_t dst = stage0 + (uint32_t)st.idx * kStageBytes;
                    int p0 = win.phys0, p1 = win.phys1;
                    if (win.ld0 && (p0 < 0 || (long long)p0 >= a.num_blocks)) {
                        atomicOr(a.status, kStatusBadBlock);
                        p0 = 0;
                    }
                    if (win.ld1 && (p1 < 0 || (long long)p1 >= a.num_blocks)) {
                        atomicOr(a.status, kStatusBadBlock);
                        p1 = 0;
                    }
                    if (win.ld0)
                        bulk_load_stream(dst, a.kv + (long long)p0 * kMxfp4BlockBytes, kMxfp4BlockBytes,
                                         fb, policy);
                    if (win.ld1)
                        bulk_load_stream(dst + kMxfp4BlockBytes, a.kv + (long long)p1 * kMxfp4BlockBytes,
                                         kMxfp4BlockBytes, fb, policy);
                }
                __syncwarp();
                ++issued;
                st.next(S);
                if (k == 0 && win.nb >= 0) {
                    nxt = make_window<1>(a, win.nb, win.nj, sb, sj, eb, ej, lane);
                    have_nxt = true;
                }
            }
            if (!ok || win.nb < 0) break;
            qbase += __popc(win.first_mask);
            if (!have_nxt) nxt = make_window<1>(a, win.nb, win.nj, sb, sj, eb, ej, lane);
            win = nxt;
        }
        // one end mark per group, in the stages after the last sub-tile
        for (int e = 0; ok && e < NWG; ++e) {
            if (lane == 0) {
                ok = mbar_wait(empty_bar(st.idx), st.phase ^ 1, abort_flag, a.status);
                if (ok) {
                    st_shared_v4(base + L.rec + 32u * st.idx, 0u, 0u, 0u, (uint32_t)kStageEnd);
                    mbar_arrive(full_bar(st.idx));
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            st.next(S);
        }
        if (!ok && lane == 0) {
            // drain: every copy this warp issued lands before the CTA exits
            Ring d = st;
            for (int t = 0; t < issued && t < S; ++t) {
                if (d.idx == 0) {
                    d.idx = S;
                    d.phase ^= 1u;
                }
                --d.idx;
                mbar_wait_drain(full_bar(d.idx), d.phase);
            }
            for (int qc = (q_issued > 2 ? q_issued - 2 : 0); qc < q_issued; ++qc)
                mbar_wait_drain(qfull0 + 8u * (qc & 1), (qc >> 1) & 1);
        }
    } else if (warp == kScoutWarp) {
        // ---------------------------------------------------------------- scout
        // Per sub-tile: the largest gap between a key's frame and its other
        // groups, over the keys below the request's length (a staged row past
        // it may hold anything, a block past max_context stale bytes).  Lane l
        // looks at rows l, l+32, l+64, l+96.
        Ring st;
        int ends = 0;
        while (ends < NWG) {
            if (!mbar_wait(full_bar(st.idx), st.phase, abort_flag, a.status)) break;
            const uint4 rec = ld_shared_v4(base + L.rec + 32u * st.idx);
            int gap = 0;
            if (rec.w & kStageEnd) {
                ++ends;
            } else {
                const int cnt = (int)(rec.w & 0xffu), j = (int)rec.y, len = (int)rec.z;
                const uint32_t stg = stage0 + (uint32_t)st.idx * kStageBytes;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = lane + 32 * i;
                    const int page = r >> 6, key = r & 63;
                    if (page < cnt && (j + page) * kBlockKeys + key < len) {
                        const uint32_t sc = ld_shared_u32(stg + (uint32_t)(page * kMxfp4BlockBytes +
                                                                           kBlockCodeBytes + key * kRowScales));
                        gap = max(gap, row_frame(sc).gap);
                    }
                }
                gap = (int)__reduce_max_sync(0xffffffffu, (uint32_t)gap);
            }
            if (lane == 0) {
                st_shared_u32(base + L.gap + 4u * st.idx, (uint32_t)gap);
                mbar_arrive(scout_bar(st.idx));
            }
            __syncwarp();
            st.next(S);
        }
    } else if (warp == kMmaWarp || warp == kMmaWarp2) {
        // ---------------------------------------------------------------- MMA issue
        // Issuing a tcgen05.mma takes a thread longer than the tensor pipe
        // needs to run it at N = 64, so two warps issue: warp 1 the sub-tiles
        // of the even groups, warp 3 those of the odd ones (k even / odd).
        const int m = warp == kMmaWarp ? 0 : 1;
        int last_q = -1, last_acc = -1;
        uint32_t last_ph = 0;
        bool ok = true;
        for (int k = m;; k += 2) {
            const int wg = k % NWG;
            const int i = k / NWG;                        // the group's own sub-tile count
            const int kt = wg * KPW + i % KPW;
            ok = mbar_wait(ktfull0 + 8u * kt, (uint32_t)(i / KPW) & 1u, abort_flag, a.status);
            if (!ok) break;
            const uint4 info = ld_shared_v4(base + L.info + 16u * kt);
            if (info.x & kStageEnd) break;
            const int slot = (int)info.y;
            if ((int)info.w != last_q) {
                // this warp's first sub-tile of the request: its query rows
                last_q = (int)info.w;
                ok = mbar_wait(qready0 + 8u * slot, (uint32_t)(last_q >> 1) & 1u, abort_flag, a.status);
                if (!ok) break;
            }
            const int acc = wg * P::APW + i % P::APW;
            const uint32_t aph = (uint32_t)(i / P::APW) & 1u;
            ok = mbar_wait(accempty0 + 8u * acc, aph ^ 1u, abort_flag, a.status);
            if (!ok) break;
            tc_fence_after();
            if (lane == 0) {
                const int fmt = (int)info.z;
                const uint32_t idesc = fmt == kFmtBf16 ? make_idesc(1, 1, kTileKeys, N)
                                                       : make_idesc(0, 0, kTileKeys, N);
                const uint32_t qb = q0 + slot * P::kSlotBytes + (uint32_t)fmt * P::kFmtBytes;
                const uint32_t d = tmem_base + (uint32_t)(acc * N);
                const uint32_t at = tmem_base + P::kAccCols + (uint32_t)kt * kTileCols;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint64_t bd = smem_desc_sw128(qb + h * P::kHalf);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)      // K = 16: 8 columns of A
                        mma_f16_tmem_a(d, at + 8u * (4 * h + kk), bd + 2u * kk, idesc,
                                       (h | kk) ? 1u : 0u);
                }
                mma_commit(accfull0 + 8u * acc);
                mma_commit(ktfree0 + 8u * kt);
            }
            __syncwarp();
            last_acc = acc;
            last_ph = aph;
        }
        if (last_acc >= 0) mbar_wait_drain(accfull0 + 8u * last_acc, last_ph);
    } else if (warp >= kFirstWgWarp) {
        // ---------------------------------------------------------------- dequantise + epilogue
        const int wg = (warp - kFirstWgWarp) >> 2;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;                 // key row of a sub-tile; query row n
        const int page = row >> 6, key = row & 63;
        const uint32_t lane_tmem = tmem_base + ((uint32_t)(quad * 32) << 16);
        const uint32_t stage_row = (uint32_t)(page * kMxfp4BlockBytes + key * kRowBytes);
        const uint32_t stage_sc = (uint32_t)(page * kMxfp4BlockBytes + kBlockCodeBytes + key * kRowScales);
        const int rot = (row >> 1) & 3;                  // chunk order: distinct banks per warp
        // the group's four warps meet on an mbarrier of their own (one
        // arrival per warp), so that the meeting is bounded like every other
        // wait: a warp that gave up elsewhere cannot hold the others forever
        const uint32_t wsync = wgsync0 + 8u * wg;
        uint32_t wsync_ph = 0;
        auto wg_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(wsync);
            const bool r = mbar_wait(wsync, wsync_ph, abort_flag, a.status);
            wsync_ph ^= 1u;
            return r;
        };
        // the group's sub-tile whose epilogue is still to run
        struct Pending {
            bool has;
            int acc;
            uint32_t aph;
            int slot, qidx, b, j, len, cnt, E, sub_idx;
            bool last;
        } pend;
        pend.has = false;

        // Epilogue of sub-tile p: the row's head scores from TMEM (32-column
        // chunks, the next one in flight while the current one is summed),
        // rectified, weighted by the framed weights, summed, times the key's
        // and slot's frames, stored.  Then the accumulator is handed back and
        // the sub-tile counted as done for its Q slot: the count reaches
        // kDoneAll exactly when every sub-tile of the request in this CTA is
        // done, and the warp whose count completes it frees the slot.
        auto epilogue = [&](const Pending& p) -> bool {
            if (!mbar_wait(accfull0 + 8u * p.acc, p.aph, abort_flag, a.status)) return false;
            tc_fence_after();
            const uint32_t qs = q0 + p.slot * P::kSlotBytes;
            const int pos = (p.j + page) * kBlockKeys + key;
            const bool valid = page < p.cnt && pos < p.len;
            constexpr int NC = NN * 2;                    // 32-column chunks
            uint32_t buf[2][32];
            uint64_t acc4[4];
            const uint32_t acc_col = (uint32_t)(p.acc * N);
            tmem_ld32_async(lane_tmem + acc_col, buf[0]);
            tmem_wait_bind32(buf[0]);
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                if (c + 1 < NC) tmem_ld32_async(lane_tmem + acc_col + 32u * (c + 1), buf[(c + 1) & 1]);
                if ((c & 1) == 0) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) acc4[u] = 0ull;
                }
                const uint32_t(&v)[32] = buf[c & 1];
#pragma unroll
                for (int h = 0; h < 32; h += 4) {
                    const uint4 wv = ld_shared_v4(qs + P::kWq + 4u * (32 * c + h));
                    const uint64_t w01 = ((uint64_t)wv.y << 32) | wv.x;
                    const uint64_t w23 = ((uint64_t)wv.w << 32) | wv.z;
                    acc4[(h / 2) % 4] =
                        fma2(w01, pack2(fmaxf(__uint_as_float(v[h]), 0.f), fmaxf(__uint_as_float(v[h + 1]), 0.f)),
                             acc4[(h / 2) % 4]);
                    acc4[(h / 2 + 1) % 4] =
                        fma2(w23, pack2(fmaxf(__uint_as_float(v[h + 2]), 0.f), fmaxf(__uint_as_float(v[h + 3]), 0.f)),
                             acc4[(h / 2 + 1) % 4]);
                }
                if ((c & 1) == 1 && valid) {
                    const int t = c >> 1;
                    const float r = (sum2(acc4[0]) + sum2(acc4[1])) + (sum2(acc4[2]) + sum2(acc4[3]));
                    const int R = (int)ld_shared_u32(qs + P::kFrame + 4u * t);
                    const float logit = scale_pow2(r, p.E + R - 254);
                    const long long o = ((long long)p.b * a.next_n + a.slot0 + t) * a.out_stride + pos;
                    if (a.out_bf16)
                        reinterpret_cast<__nv_bfloat16*>(a.out)[o] = __float2bfloat16_rn(logit);
                    else
                        reinterpret_cast<float*>(a.out)[o] = logit;
                }
                if (c + 1 < NC) tmem_wait_bind32(buf[(c + 1) & 1]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(accempty0 + 8u * p.acc);
                // Count this warp's part of the sub-tile towards the Q slot's
                // release.  A sub-tile counts 1 per warp, except the request's
                // last one (index T-1 of T), whose warps add kDoneAll/4 -
                // (T-1) each: the total reaches kDoneAll exactly when every
                // warp of every sub-tile of the request is done, in any order.
                const int inc = p.last ? kDoneAll / 4 - p.sub_idx : 1;
                __threadfence_block();
                const int old = atomicAdd(&done_cnt[p.slot], inc);
                if (old + inc == kDoneAll) {
                    __threadfence_block();
                    done_cnt[p.slot] = 0;
                    mbar_arrive(qempty0 + 8u * p.slot);
                }
            }
            return true;
        };

        auto flush = [&]() -> bool {
            if (!pend.has) return true;
            pend.has = false;
            return epilogue(pend);
        };

        // The query rows of a request's pass into Q slot `slot`: frames, both
        // operand formats, framed weights.  All 128 threads; row n = row.
        auto convert_q = [&](int slot, uint32_t qpar) -> bool {
            const uint32_t qs = q0 + slot * P::kSlotBytes;
            if (!mbar_wait(qfull0 + 8u * slot, qpar, abort_flag, a.status)) return false;
            const bool mine = row < N;
            RowFrame f{0, 0, 0};
            if (mine) {
                const uint32_t sc = ld_shared_u32(qs + P::kRawSf + 4u * row);
                f = row_frame(sc);
                const uint32_t src = qs + P::kRawCodes + (uint32_t)row * kRowBytes;
#pragma unroll
                for (int c = 0; c < 4; ++c) {                  // group c = 16-byte chunk c
                    const int e = (int)((sc >> (8 * c)) & 0xFF);
                    const bool nan = (f.nan_mask >> c) & 1u;
                    const uint4 v = ld_shared_v4(src + 16u * c);
                    uint32_t w16[16], wb[16];
                    dequant_chunk(v, factor_f16(f.E - e, nan), kFmtF16, w16);
                    dequant_chunk(v, factor_bf16(f.E - e, nan), kFmtBf16, wb);
                    // elements 32c..32c+31: half c/2, 16-byte chunks 4(c%2)..4(c%2)+3
                    const uint32_t hoff = (uint32_t)(c >> 1) * P::kHalf;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t off = hoff + sw128(row, 4 * (c & 1) + u);
                        st_shared_v4(qs + off, w16[4 * u], w16[4 * u + 1], w16[4 * u + 2], w16[4 * u + 3]);
                        st_shared_v4(qs + P::kFmtBytes + off, wb[4 * u], wb[4 * u + 1], wb[4 * u + 2],
                                     wb[4 * u + 3]);
                    }
                }
            }
            // per warp: largest head frame and largest gap, then across the group
            const int emax = __reduce_max_sync(0xffffffffu, mine ? f.E : 0);
            const int gmax = __reduce_max_sync(0xffffffffu, mine ? f.gap : 0);
            if (lane == 0) st_shared_v2_s32(qs + P::kPart + 8u * quad, emax, gmax);
            if (!wg_sync()) return false;
            if (mine) {
                // rows 64t..64t+63 (slot t) are warps 2t, 2t+1
                const int t = row >> 6;
                const int2 pa = ld_shared_v2_s32(qs + P::kPart + 8u * (2 * t));
                const int2 pb = ld_shared_v2_s32(qs + P::kPart + 8u * (2 * t + 1));
                const int R = max(pa.x, pb.x);
                const float w = __uint_as_float(ld_shared_u32(qs + P::kRawW + 4u * row));
                st_shared_u32(qs + P::kWq + 4u * row, __float_as_uint(w * pow2_down(f.E - R)));
                if (R - f.E > kWeightGapLimit) atomicOr(a.status, kStatusFp4Inexact);
                if ((row & 63) == 0) st_shared_u32(qs + P::kFrame + 4u * t, (uint32_t)R);
            }
            if (row == 0) {
                int g = 0;
#pragma unroll
                for (int w = 0; w < 2 * NN; ++w) g = max(g, ld_shared_v2_s32(qs + P::kPart + 8u * w).y);
                st_shared_v2_s32(qs + P::kMeta, g <= kF16MaxGap ? 1 : 0, g);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(qready0 + 8u * slot);
            return true;
        };

        // this group's sub-tiles: k = wg, wg + NWG, ...
        Ring st;
        for (int u = 0; u < wg; ++u) st.next(S);
        bool ok = true;
        for (int i = 0;; ++i) {
            // a pending epilogue is not held while waiting for the next
            // sub-tile: other groups (and the producer, through the Q slots)
            // may be waiting for it
            if (pend.has && !mbar_try_wait(scout_bar(st.idx), st.phase) && !flush()) {
                ok = false;
                break;
            }
            ok = mbar_wait(scout_bar(st.idx), st.phase, abort_flag, a.status);
            if (!ok) break;
            const uint32_t rec = base + L.rec + 32u * st.idx;
            const uint4 r0 = ld_shared_v4(rec);
            const int meta = (int)r0.w;
            const int kt = wg * KPW + i % KPW;
            const uint32_t ktph = (uint32_t)(i / KPW) & 1u;
            if (meta & kStageEnd) {
                // tell the MMA warp, through the key tile it would take next
                ok = flush() && mbar_wait(ktfree0 + 8u * kt, ktph ^ 1u, abort_flag, a.status);
                if (ok) {
                    if (row == 0) st_shared_v4(base + L.info + 16u * kt, (uint32_t)kStageEnd, 0u, 0u, 0u);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ktfull0 + 8u * kt);
                }
                break;
            }
            const uint4 r1 = ld_shared_v4(rec + 16);
            const int slot = (meta >> kMetaSlotShift) & 1;
            const int qidx = (int)r1.x;
            const uint32_t qpar = (uint32_t)(qidx >> 1) & 1u;
            // a pending sub-tile of an earlier request is finished before this
            // one waits on its own request's Q slot: that slot's reload may be
            // waiting for the earlier request's release
            if (pend.has && pend.qidx != qidx && !flush()) {
                ok = false;
                break;
            }
            if ((meta & kMetaFirst) && !convert_q(slot, qpar)) {
                ok = false;
                break;
            }
            ok = mbar_wait(ktfree0 + 8u * kt, ktph ^ 1u, abort_flag, a.status);
            if (ok) ok = mbar_wait(qready0 + 8u * slot, qpar, abort_flag, a.status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t stg = stage0 + (uint32_t)st.idx * kStageBytes;
            const uint32_t sc = ld_shared_u32(stg + stage_sc);
            const RowFrame f = row_frame(sc);
            const int tile_gap = (int)ld_shared_u32(base + L.gap + 4u * st.idx);
            const int2 qm = ld_shared_v2_s32(q0 + slot * P::kSlotBytes + P::kMeta);
            const int fmt = (tile_gap <= kF16MaxGap && qm.x) ? kFmtF16 : kFmtBf16;
            if (row == 0) {
                if (tile_gap + qm.y > kExactGapSum) atomicOr(a.status, kStatusFp4Inexact);
                st_shared_v4(base + L.info + 16u * kt, (uint32_t)meta, (uint32_t)slot, (uint32_t)fmt,
                             (uint32_t)qidx);
            }
            const uint32_t ta = lane_tmem + P::kAccCols + (uint32_t)kt * kTileCols;
            // the row's four 16-byte chunks (group c = chunk c), read in a
            // rotated order so that the rows a warp reads together fall in
            // distinct banks, then rotated back in registers: the TMEM stores
            // need the same column on every lane
            uint4 v[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) v[c] = ld_shared_v4(stg + stage_row + 16u * ((c + rot) & 3));
            rotate_back(v, rot);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int e = (int)((sc >> (8 * c)) & 0xFF);
                const bool nan = (f.nan_mask >> c) & 1u;
                uint32_t w16[16];
                if (fmt == kFmtF16) dequant_chunk(v[c], factor_f16(f.E - e, nan), kFmtF16, w16);
                else dequant_chunk(v[c], factor_bf16(f.E - e, nan), kFmtBf16, w16);
                tmem_st16(ta + 16u * c, w16);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(empty_bar(st.idx));   // staging slot read
                mbar_arrive(ktfull0 + 8u * kt);
            }
            if (!flush()) {
                ok = false;
                break;
            }
            pend.has = true;
            pend.acc = wg * P::APW + i % P::APW;
            pend.aph = (uint32_t)(i / P::APW) & 1u;
            pend.slot = slot;
            pend.qidx = qidx;
            pend.b = (int)r0.x;
            pend.j = (int)r0.y;
            pend.len = (int)r0.z;
            pend.cnt = meta & 0xff;
            pend.E = f.E;
            pend.sub_idx = (int)r1.y;
            pend.last = (meta & kMetaLast) != 0;
            for (int u = 0; u < NWG; ++u) st.next(S);
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
cudaError_t launch_pass(const Mxfp4Args& a, int num_ctas, cudaStream_t stream)
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
    cfg.blockDim = dim3((unsigned)Plan<NN>::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, mxfp4_logits_kernel<NN>, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

size_t mxfp4_smem_bytes(int slots_per_pass, int stages)
{
    const uint32_t t = slots_per_pass == 1 ? layout_of<1>(stages).total : layout_of<2>(stages).total;
    return (size_t)t + 1024;
}

cudaError_t launch_mxfp4_logits(const Mxfp4Args& args, int num_ctas, cudaStream_t stream)
{
    // passes of at most two slots each: N = 64 or 128
    for (int s0 = 0; s0 < args.next_n; s0 += 2) {
        Mxfp4Args a = args;
        a.slot0 = s0;
        const int nn = args.next_n - s0 >= 2 ? 2 : 1;
        a.stages = nn == 1 ? args.stages : args.stages2;
        const cudaError_t e = nn == 1 ? launch_pass<1>(a, num_ctas, stream)
                                      : launch_pass<2>(a, num_ctas, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace pml
