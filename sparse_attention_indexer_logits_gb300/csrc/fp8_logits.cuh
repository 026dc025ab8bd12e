// fp8 paged MQA logits on sm_103a: the kernel template.
//
//   out[b*next_n + t, p] = s_p * sum_h w[b*next_n+t, h] * relu(q[b*next_n+t, h] . k_p)
//
// ("flashinfer.attn_scores": math block; first bullet -- the rectifier acts
// per head, before the weighted sum; second bullet -- the fp8 variant is
// multiplied by the per-token fp32 scale s_p from the trailing scale region
// of each kv_fused block; note -- row b*next_n+t, empty requests untouched.)
//
// One persistent CTA per SM walks a contiguous range of 64-key blocks
// (common.cuh).  The unit of the MMA is a sub-tile of up to two blocks of one
// request (128 keys = the MMA's M); a pipeline stage holds KT sub-tiles
// (KT = 2 when next_n*H <= 128, so that four stages' accumulators still fit
// TMEM; else 1), so every barrier, descriptor and commit is paid once per 256
// keys where possible.
//
//   warps 0,3 MMA issue (warp 0 also allocates TMEM): warp m takes sub-tile
//             m of every stage; four tcgen05.mma kind::f8f6f4 (K = 32 each)
//             compute S = K (128 x 128) * Q^T into the stage's accumulator
//             (TMEM lanes = keys, columns = next_n*H), then tcgen05.commit.
//   warps 1-2 producers, stage i to warp 1 + i % 2: both walk the CTA's
//             range in windows of up to 32 sub-tiles, one per lane (request,
//             blocks and block-table entries read by the lanes in parallel);
//             per own stage the warp waits for the slot, publishes a stage
//             descriptor (per sub-tile: request, block, count, length,
//             flags) in shared memory, and the owning lanes issue the TMA
//             copy of each block's keys (8 KB, 3-D tensor map, 128-byte
//             swizzle) and the bulk copy of its 64 scales (256 B).  Per
//             request starting in an own stage, the q rows (next_n*H x 128
//             e4m3) and weights.  After the last stage an end marker.  One
//             warp issuing every copy (eight per 256 keys) is slower than the
//             stage's share of HBM time, hence two.
//   warps 4-11 epilogue, two warpgroups: with KT = 2 group g takes sub-tile g
//             of every stage (all slots), with KT = 1 both take the one
//             sub-tile and split the slots (t = g, g+2).  Each thread owns one
//             key (one TMEM lane), reads its head scores with tcgen05.ld in
//             chunks of 32 columns (the next chunk in flight while the current
//             one is computed), rectifies, weights and sums them with packed
//             f32x2 FMAs, multiplies by s_p and stores, for positions below
//             min(seq_len, max_context).
//
// The MMA and epilogue warps read the stage descriptors instead of walking
// the schedule, and every loop keeps its stage / accumulator index and phase
// bit as counters.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "window.cuh"

namespace pml {
namespace fp8 {

constexpr int kSubKeyBytes = kTileKeys * kHeadDim;     // 16 KB: one sub-tile of keys
constexpr int kSubScaleBytes = kTileKeys * 4;          // 512 B
constexpr int kMmaWarp = 0;                            // also allocates TMEM
constexpr int kProducers = 2;                          // warps 1, 2: stage i is warp 1 + i % 2's
constexpr int kMmaWarp2 = 3;                           // issues sub-tile 1 of each stage
constexpr int kFirstEpiWarp = 4;
// Two epilogue warpgroups: one per sub-tile when a stage holds two, else
// both on the one sub-tile with the slots split between them.
__host__ __device__ constexpr int epi_groups_of(int) { return 2; }
__host__ __device__ constexpr int threads_of(int next_n)
{
    return 32 * kFirstEpiWarp + 128 * epi_groups_of(next_n);
}

__host__ __device__ constexpr int n_pad_of(int next_n, int heads)
{
    return (next_n * heads + 15) / 16 * 16;
}
__host__ __device__ constexpr int subtiles_of(int n_pad) { return n_pad <= 128 ? 2 : 1; }
__host__ __device__ constexpr int acc_cols_of(int n_pad) { return subtiles_of(n_pad) * n_pad; }
__host__ __device__ constexpr int accumulators_of(int n_pad)
{
    return acc_cols_of(n_pad) <= 128 ? 4 : 2;
}
__host__ __device__ constexpr int tmem_cols_of(int n_pad)
{
    return accumulators_of(n_pad) * acc_cols_of(n_pad) <= 32    ? 32
           : accumulators_of(n_pad) * acc_cols_of(n_pad) <= 64  ? 64
           : accumulators_of(n_pad) * acc_cols_of(n_pad) <= 128 ? 128
           : accumulators_of(n_pad) * acc_cols_of(n_pad) <= 256 ? 256
                                                                : 512;
}

// One sub-tile of a stage, 16 bytes, so that a consumer reads it with one
// vector load: b = request, j = first block within it, len =
// min(seq_lens[b], max_context), meta = block count (1 or 2; 0 = no sub-tile
// here) | kTileFirst/kTileLast << 8 | q slot << 12, or kStageEnd in the first
// sub-tile of the stage after the CTA's last.
struct __align__(16) SubDesc {
    int b, j, len, meta;
};
struct StageDesc {
    SubDesc sub[2];
};
constexpr int kMetaFirst = kTileFirst << 8;
constexpr int kMetaLast = kTileLast << 8;
constexpr int kMetaSlotShift = 12;
constexpr int kStageEnd = 1 << 20;
__device__ __forceinline__ int4 load_sub(const StageDesc* d, int i)
{
    return *reinterpret_cast<const int4*>(&d->sub[i]);
}
__device__ __forceinline__ int meta_slot(int meta) { return (meta >> kMetaSlotShift) & 1; }

struct Layout {
    uint32_t k, q, s, w, desc, bar, misc, total;
    uint32_t q_bytes, w_bytes;
};

__host__ __device__ inline Layout layout(int n_pad, int next_n, int heads, int stages)
{
    const int kt = subtiles_of(n_pad);
    Layout L;
    L.q_bytes = (uint32_t)n_pad * kHeadDim;
    L.w_bytes = (uint32_t)((next_n * heads * 4 + 15) / 16 * 16);
    L.k = 0;
    L.q = L.k + (uint32_t)(stages * kt) * kSubKeyBytes;
    L.s = L.q + 2 * L.q_bytes;
    L.w = L.s + (uint32_t)(stages * kt) * kSubScaleBytes;
    L.desc = L.w + 2 * L.w_bytes;
    L.bar = L.desc + (uint32_t)stages * (uint32_t)sizeof(StageDesc);
    L.misc = L.bar + (uint32_t)(2 * stages + 12) * 8;
    L.total = L.misc + 64;
    return L;
}

template <int W>
__device__ __forceinline__ void tmem_ld_async(uint32_t taddr, uint32_t (&r)[W])
{
    if constexpr (W == 32) tmem_ld32_async(taddr, r);
    else if constexpr (W == 16) tmem_ld16_async(taddr, r);
    else tmem_ld8_async(taddr, r);
}

template <int W>
__device__ __forceinline__ void tmem_wait_bind(uint32_t (&r)[W])
{
    if constexpr (W == 32) tmem_wait_bind32(r);
    else if constexpr (W == 16) tmem_wait_bind16(r);
    else tmem_wait_bind8(r);
}

// The logits of this thread's key for every (sub-tile, slot) pass of a stage:
// NS sub-tiles x SL slots t = first_slot + k*GS.  The head scores are read
// from TMEM in chunks of up to CWMAX columns as one pipelined sequence, the
// load of the next chunk issued before the current one is computed (across
// pass boundaries too, so only the stage's first load is waited for in
// full), then rectified, weighted (packed f32x2 FMAs, four accumulators) and
// summed.  taddr[n] is the column of slot 0 of sub-tile n in this thread's
// lane and oidx[n] the output element of its slot 0.  wp holds packed weight pairs of the SL slots (slot k at
// wp[k*H/2 + i]) of request cur_b; a sub-tile of another request reloads them
// from its shared-memory weights wsrc[n] before its first chunk.  A sub-tile
// with no blocks (d.w == 0) is computed on stale columns and not stored.
// Logit v of output element idx: fp32, or bf16 rounded to nearest even.
__device__ __forceinline__ void store_logit(void* out, bool bf16, long long idx, float v)
{
    if (bf16) reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
    else reinterpret_cast<float*>(out)[idx] = v;
}

template <int H, int NN, int NS, int SL, int GS, int CWMAX, int WN>
__device__ __forceinline__ void stage_logits(const uint32_t (&taddr)[NS], const int4 (&d)[NS],
                                             const float (&sp)[NS], const bool (&valid)[NS],
                                             const long long (&oidx)[NS],
                                             const float4* const (&wsrc)[NS], uint64_t (&wp)[WN],
                                             int& cur_b, int first_slot, void* out, bool out_bf16,
                                             long long out_stride)
{
    static_assert(SL * H / 2 <= WN, "weights of every slot are held");
    constexpr int CW = H >= CWMAX ? CWMAX : H;   // chunk width (columns)
    constexpr int CPS = H / CW;                  // chunks per slot
    constexpr int CPP = SL * CPS;                // chunks per sub-tile
    constexpr int NC = NS * CPP;
    auto column = [&](int c) {
        return taddr[c / CPP] + (uint32_t)((first_slot + ((c % CPP) / CPS) * GS) * H + (c % CPS) * CW);
    };
    uint32_t buf[2][CW];
    uint64_t acc[4];
    tmem_ld_async<CW>(column(0), buf[0]);
    tmem_wait_bind<CW>(buf[0]);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const int n = c / CPP;
        const int k = (c % CPP) / CPS;
        const int t = first_slot + k * GS;
        if (c % CPP == 0 && (d[n].w & 0xff) != 0 && d[n].x != cur_b) {
            // first sub-tile of a new request for this warp
#pragma unroll
            for (int kk = 0; kk < SL; ++kk) {
                const int tt = first_slot + kk * GS;
#pragma unroll
                for (int h = 0; h < H; h += 4) {
                    const float4 v = tt < NN ? wsrc[n][tt * (H / 4) + h / 4]
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                    wp[(kk * H + h) / 2] = pack2(v.x, v.y);
                    wp[(kk * H + h) / 2 + 1] = pack2(v.z, v.w);
                }
            }
            cur_b = d[n].x;
        }
        if (c % CPS == 0) {
#pragma unroll
            for (int a = 0; a < 4; ++a) acc[a] = 0ull;
        }
        if (c + 1 < NC) tmem_ld_async<CW>(column(c + 1), buf[(c + 1) & 1]);
        const uint32_t(&v)[CW] = buf[c & 1];
        const int w0 = (k * H + (c % CPS) * CW) / 2;
#pragma unroll
        for (int i = 0; i < CW; i += 2) {
            const uint64_t x = pack2(fmaxf(__uint_as_float(v[i]), 0.f),
                                     fmaxf(__uint_as_float(v[i + 1]), 0.f));
            acc[(i / 2) % 4] = fma2(wp[w0 + i / 2], x, acc[(i / 2) % 4]);
        }
        if (c % CPS == CPS - 1) {
            const float r = (sum2(acc[0]) + sum2(acc[1])) + (sum2(acc[2]) + sum2(acc[3]));
            if (valid[n] && t < NN)
                store_logit(out, out_bf16, oidx[n] + t * out_stride, sp[n] * r);
        }
        if (c + 1 < NC) tmem_wait_bind<CW>(buf[(c + 1) & 1]);
    }
}

// How the two epilogue warpgroups share a stage.  Sub-tile split: group g
// takes sub-tile g (all slots); slot split: group g takes slots t = g, g+2 of
// every sub-tile.  A warp keeps the weights of its slots (SL x H) in
// registers, loaded when its request changes rather than read from shared
// memory for every key: the split is the one that keeps them to 64 where it
// can.  Only with next_n*H > 128 at one sub-tile per stage (H = 64,
// next_n >= 3) are there 128; then the CTA's registers are re-split, the
// MMA/producer warpgroup dropping to kLowRegs so that the two epilogue
// warpgroups can hold kHighRegs each (128 x 88 + 256 x 208 = 64512, the
// 384 x 168 registers of the block).  ptxas allocates each warpgroup's
// branch within its budget only if no call (a non-inlined function) sits in
// it, which is why the waits are fully inlined.
template <int H, int NN>
struct EpiPlan {
    static constexpr int KT = subtiles_of(n_pad_of(NN, H));
    static constexpr bool kSubSplit = KT == 2 && (NN * H <= 64 || (NN + 1) / 2 * H > 64);
    static constexpr int GS = kSubSplit ? 1 : 2;            // slot stride
    static constexpr int SL = (NN + GS - 1) / GS;           // slots of group 0
    static constexpr int kWeightPairs = SL * H / 2;
    static constexpr bool kSplitRegs = SL * H > 64;
    static constexpr int kLowRegs = 88;
    static constexpr int kHighRegs = 208;
    // TMEM columns per tcgen05.ld (two chunks in flight): narrower when the
    // registers also hold 128 weights
    static constexpr int kChunk = kSplitRegs ? 16 : 32;
};

template <int H, int NN>
__global__ void __launch_bounds__(threads_of(NN), 1)
    logits_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                  const Fp8Args a)
{
    constexpr int N = n_pad_of(NN, H);
    constexpr int KT = subtiles_of(N);
    constexpr int COLS = acc_cols_of(N);
    constexpr int NACC = accumulators_of(N);
    constexpr int NH = NN * H;
    constexpr uint32_t kStageKeyBytes = KT * kSubKeyBytes;
    constexpr uint32_t kStageScaleBytes = KT * kSubScaleBytes;
    constexpr int EG = epi_groups_of(NN);
    constexpr uint32_t kEpiWarps = 4 * EG;
    constexpr bool kCallWait = !EpiPlan<H, NN>::kSplitRegs;   // no calls with split registers

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = a.stages;
    const Layout L = layout(N, NN, H, S);

    const uint32_t base = smem_addr(smem);
    const uint32_t k_base = base + L.k;
    const uint32_t q_base = base + L.q;
    const uint32_t s_base = base + L.s;
    const float* scales_smem = reinterpret_cast<const float*>(smem + L.s);
    StageDesc* descs = reinterpret_cast<StageDesc*>(smem + L.desc);
    const uint32_t bar = base + L.bar;
    const uint32_t full_bar0 = bar;                        // + 8*stage
    const uint32_t empty_bar0 = bar + 8u * S;
    const uint32_t tfull_bar0 = bar + 8u * (2 * S);        // + 8*acc
    const uint32_t tempty_bar0 = bar + 8u * (2 * S + 4);
    const uint32_t qfull_bar0 = bar + 8u * (2 * S + 8);    // + 8*slot
    const uint32_t qempty_bar0 = bar + 8u * (2 * S + 10);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---------------------------------------------------------------- setup
    // The next call may be placed on SMs as this grid leaves them; nothing
    // here touches global memory before grid_dependency_wait.
    allow_dependent_launch();
    const int prod = (warp == 1 || warp == 2) ? warp - 1 : -1;
    const bool producer = prod >= 0;
    // The producers compute their range and first window (block-table reads
    // included) before the CTA-wide barrier, so that these global round trips
    // overlap the TMEM allocation and the barrier set-up.
    int sb = 0, sj = 0, eb = 0, ej = 0;
    Window win;
    if (producer) {
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
        win = make_window<KT>(a, sb, sj, sb, sj, eb, ej, lane);
    } else if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), tmem_cols_of(N));
        tmem_relinquish();
    } else if (warp == kMmaWarp2 && lane == 0) {
        *abort_flag = 0;
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar0 + 8u * s, 1);
            mbar_init(empty_bar0 + 8u * s, kEpiWarps);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(tfull_bar0 + 8u * i, KT);   // one commit per sub-tile
            mbar_init(tempty_bar0 + 8u * i, kEpiWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(qfull_bar0 + 8u * i, 1);
            mbar_init(qempty_bar0 + 8u * i, kEpiWarps);
        }
        fence_mbar_init();
        tma_prefetch_map(&kmap);
        tma_prefetch_map(&qmap);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    grid_dependency_wait();

    if (warp < kFirstEpiWarp) {
        // warpgroup 0: MMA issue and producers
        if constexpr (EpiPlan<H, NN>::kSplitRegs) regs_dec<EpiPlan<H, NN>::kLowRegs>();
        if (producer) {
            // ------------------------------------------------------------ producer
            const uint64_t policy = policy_evict_first();
            // Both producers walk every stage of the CTA's range (windows
            // included); producer p publishes stage i (counted from 0) when
            // i % 2 == p, with the q tiles of the requests starting in it.
            // One warp issuing every copy of a stage (eight per 256 keys)
            // takes longer than the stage's share of HBM time.
            uint32_t s = 0, ph = 0;
            int qbase = 0;                  // requests started in earlier windows
            int issued = 0, q_issued = 0;   // stages walked, q tiles of the range
            int own_q0 = -1, own_q1 = -1;   // this warp's latest q tile per slot
            bool ok = true;
            // TMA of one block's keys (8 KB, 128-byte swizzle) and bulk copy of
            // its 64 scales into stage s
            auto load_block = [&](uint32_t kdst, uint32_t sdst, int pb) {
                if (pb < 0 || (long long)pb >= a.num_blocks) {
                    atomicOr(a.status, kStatusBadBlock);
                    pb = 0;
                }
                tma_load_3d_stream(kdst, &kmap, full_bar0 + 8u * s, 0, 0, pb, policy);
                bulk_load_stream(sdst, a.kv_fused + (long long)pb * kFp8BlockBytes + kFp8BlockKeyBytes,
                                 kBlockKeys * 4, full_bar0 + 8u * s, policy);
            };
            while (true) {
                Window nxt;
                bool have_nxt = false;
                const int stages_here = (win.n + KT - 1) / KT;
                // q index of this lane's request: requests started before it
                const int qidx = qbase + __popc(win.first_mask & ((2u << lane) - 1u)) - 1;
                for (int st = 0; st < stages_here; ++st) {
                    const int o0 = st * KT;
                    const int i = lane - o0;                 // sub-tile slot this lane fills
                    const bool mine = issued % kProducers == prod;
                    const bool own = mine && i >= 0 && i < KT && lane < win.n;
                    // q / weights of each request starting in this stage, in order
#pragma unroll
                    for (int k = 0; k < KT; ++k) {
                        const int ol = o0 + k;
                        if (ol < win.n && ((win.first_mask >> ol) & 1u)) {
                            if (mine && lane == ol) {
                                const int slot = qidx & 1;
                                ok = mbar_wait<kCallWait>(qempty_bar0 + 8u * slot,
                                                          ((qidx >> 1) & 1) ^ 1, abort_flag, a.status, a.wait_limit_ns);
                                if (ok) {
                                    const uint32_t qfb = qfull_bar0 + 8u * slot;
                                    mbar_arrive_expect_tx(qfb,
                                                          (uint32_t)a.q_box_rows * kHeadDim + NH * 4u);
                                    tma_load_2d(q_base + slot * L.q_bytes, &qmap, qfb, 0, win.b * NH);
                                    bulk_load(base + L.w + slot * L.w_bytes,
                                              a.weights + (long long)win.b * NH, NH * 4u, qfb);
                                }
                            }
                            ok = __shfl_sync(0xffffffffu, ok, ol);
                            if (!ok) break;
                            if (mine) {
                                if (q_issued & 1) own_q1 = q_issued;
                                else own_q0 = q_issued;
                            }
                            ++q_issued;
                        }
                    }
                    if (!ok) break;
                    if (mine && lane == 0) ok = mbar_wait<kCallWait>(empty_bar0 + 8u * s, ph ^ 1, abort_flag, a.status, a.wait_limit_ns);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    // publish the stage: each owner lane its sub-tile, lane 0 the rest
                    // (not at all for the stage a test asks to leave out: the roles
                    // waiting on it then run out of time and the CTA aborts)
                    const bool publish = mine && issued != a.drop_stage;
                    StageDesc& sd = descs[s];
                    if (own && publish) {
                        const int meta = win.cnt | (win.first ? kMetaFirst : 0) |
                                         (win.last ? kMetaLast : 0) | ((qidx & 1) << kMetaSlotShift);
                        *reinterpret_cast<int4*>(&sd.sub[i]) = make_int4(win.b, win.j, win.len, meta);
                    }
                    if (lane == 0 && publish) {
                        for (int k = win.n - o0; k < KT; ++k)
                            *reinterpret_cast<int4*>(&sd.sub[k]) = make_int4(0, 0, 0, 0);
                    }
                    const unsigned m0 = __ballot_sync(0xffffffffu, own && win.ld0);
                    const unsigned m1 = __ballot_sync(0xffffffffu, own && win.ld1);
                    __syncwarp();
                    if (lane == 0 && publish)
                        mbar_arrive_expect_tx(full_bar0 + 8u * s,
                                              (uint32_t)(__popc(m0) + __popc(m1)) * kFp8BlockBytes);
                    __syncwarp();
                    if (own && publish) {
                        const uint32_t kdst = k_base + s * kStageKeyBytes + (uint32_t)i * kSubKeyBytes;
                        const uint32_t sdst = s_base + s * kStageScaleBytes + (uint32_t)i * kSubScaleBytes;
                        if (win.ld0) load_block(kdst, sdst, win.phys0);
                        if (win.ld1) load_block(kdst + kFp8BlockKeyBytes, sdst + kBlockKeys * 4, win.phys1);
                    }
                    ++issued;
                    if (++s == (uint32_t)S) { s = 0; ph ^= 1; }
                    if (st == 0 && win.nb >= 0) {
                        // the next window's block-table reads overlap this window's stages
                        nxt = make_window<KT>(a, win.nb, win.nj, sb, sj, eb, ej, lane);
                        have_nxt = true;
                    }
                }
                if (!ok || win.nb < 0) break;
                qbase += __popc(win.first_mask);
                if (!have_nxt) nxt = make_window<KT>(a, win.nb, win.nj, sb, sj, eb, ej, lane);
                win = nxt;
            }
            bool end_written = false;
            if (ok && lane == 0 && issued % kProducers == prod) {
                // end marker for the MMA and epilogue warps, in the stage after the
                // last one, from the producer whose turn it is
                ok = mbar_wait<kCallWait>(empty_bar0 + 8u * s, ph ^ 1, abort_flag, a.status, a.wait_limit_ns);
                if (ok) {
                    *reinterpret_cast<int4*>(&descs[s].sub[0]) = make_int4(0, 0, 0, kStageEnd);
                    mbar_arrive(full_bar0 + 8u * s);
                    end_written = true;
                }
            }
            if (lane == 0) {
                // drain: every copy this warp issued lands before the CTA exits,
                // also when the consumers stopped early (on the normal path these
                // phases have completed already).  The end marker's stage is left
                // out: its barrier has moved on, and the copies of its earlier use
                // were consumed before the marker could take the stage.
                // With S even, stage T - S (T = stages walked), whose slot the
                // marker takes, belongs to the marker's producer, which leaves it
                // out; the other producer owns none of the two.
                const int depth = end_written ? S - 1 : S;
                for (int t = (issued > depth ? issued - depth : 0); t < issued; ++t)
                    if (t % kProducers == prod && t != a.drop_stage)   // that one holds no copies
                        mbar_wait_drain<kCallWait>(full_bar0 + 8u * (uint32_t)(t % S),
                                                   (uint32_t)(t / S) & 1u, a.wait_limit_ns);
                // of its q tiles only those of the range's last two requests
                if (own_q0 >= q_issued - 2 && own_q0 >= 0)
                    mbar_wait_drain<kCallWait>(qfull_bar0, (uint32_t)(own_q0 >> 1) & 1u, a.wait_limit_ns);
                if (own_q1 >= q_issued - 2 && own_q1 >= 0)
                    mbar_wait_drain<kCallWait>(qfull_bar0 + 8u, (uint32_t)(own_q1 >> 1) & 1u, a.wait_limit_ns);
            }
        } else if (warp == kMmaWarp || warp == kMmaWarp2) {
            // ------------------------------------------------------------ MMA issuers
            // MMA warp m issues sub-tile m of every stage (one tcgen05.mma takes a
            // thread more cycles to issue than the tensor pipe needs to run it at
            // these N, so two issuers run in parallel when a stage has two).  The
            // whole warp runs the loop and lane 0 issues: a warp kept converged
            // is scheduled promptly, where one whose other lanes wait at the
            // CTA barrier is not.
            const int mw = warp == kMmaWarp ? 0 : 1;
            if (mw < KT) {
                constexpr uint32_t idesc = make_idesc(0, 0, kTileKeys, N);
                uint32_t s = 0, ph = 0, acc = 0, aph = 0, last_acc = 0, last_ph = 0;
                int qcount = 0, done = 0;
                bool ok = true;
                while (true) {
                    ok = mbar_wait<kCallWait>(full_bar0 + 8u * s, ph, abort_flag, a.status, a.wait_limit_ns);
                    if (!ok) break;
                    const int4 x0 = load_sub(descs + s, 0);
                    const int4 x1 = KT == 2 ? load_sub(descs + s, 1) : make_int4(0, 0, 0, 0);
                    if (x0.w & kStageEnd) break;
                    ok = mbar_wait<kCallWait>(tempty_bar0 + 8u * acc, aph ^ 1, abort_flag, a.status, a.wait_limit_ns);
                    if (!ok) break;
                    // q / weights of every request that starts in this stage, in order
#pragma unroll
                    for (int i = 0; i < KT; ++i) {
                        const int meta = i == 0 ? x0.w : x1.w;
                        if (ok && (meta & kMetaFirst)) {
                            ok = mbar_wait<kCallWait>(qfull_bar0 + 8u * meta_slot(meta),
                                                      (qcount >> 1) & 1, abort_flag, a.status, a.wait_limit_ns);
                            ++qcount;
                        }
                    }
                    if (!ok) break;
                    tc_fence_after();
                    const int mmeta = mw == 0 ? x0.w : x1.w;
                    if ((mmeta & 0xff) != 0) {
                        if (lane == 0) {
                            const int slot = meta_slot(mmeta);
                            const uint64_t ad =
                                smem_desc_sw128(k_base + s * kStageKeyBytes + mw * kSubKeyBytes);
                            const uint64_t bd = smem_desc_sw128(q_base + slot * L.q_bytes);
                            const uint32_t dt = tmem_base + acc * COLS + mw * N;
#pragma unroll
                            for (int kk = 0; kk < kHeadDim / 32; ++kk)
                                mma_f8(dt, ad + 2u * kk, bd + 2u * kk, idesc, kk > 0 ? 1u : 0u);
                            mma_commit(tfull_bar0 + 8u * acc);
                        }
                        last_acc = acc;
                        last_ph = aph;
                        ++done;
                    } else if (lane == 0) {
                        mbar_arrive(tfull_bar0 + 8u * acc);   // nothing issued for this sub-tile
                    }
                    __syncwarp();
                    if (++s == (uint32_t)S) { s = 0; ph ^= 1; }
                    if (++acc == NACC) { acc = 0; aph ^= 1; }
                }
                if (done > 0) {
                    // every MMA this warp issued has completed before TMEM is
                    // released: the phase of its last commit completes only then
                    mbar_wait_drain<kCallWait>(tfull_bar0 + 8u * last_acc, last_ph, a.wait_limit_ns);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        if constexpr (EpiPlan<H, NN>::kSplitRegs) regs_inc<EpiPlan<H, NN>::kHighRegs>();
        const int grp = (warp - kFirstEpiWarp) >> 2;
        const int quad = warp & 3;             // TMEM lane quadrant this warp may access
        const int row = quad * 32 + lane;      // key row within the sub-tile
        const int page = row >> 6;
        const int key = row & 63;
        using E = EpiPlan<H, NN>;
        // sub-tiles of each stage this group processes, and its slots
        constexpr int NSUB = E::kSubSplit ? 1 : KT;
        const int first_slot = E::kSubSplit ? 0 : grp;
        uint64_t wp[E::kWeightPairs];
        int cur_b = -1;                        // request whose weights wp holds
        const uint32_t lane_addr = tmem_base + ((uint32_t)(quad * 32) << 16);
        uint32_t s = 0, ph = 0, acc = 0, aph = 0;
        int qcount = 0;
        bool ok = true;
        while (true) {
            ok = mbar_wait<kCallWait>(full_bar0 + 8u * s, ph, abort_flag, a.status, a.wait_limit_ns);
            if (!ok) break;
            const int4 x0 = load_sub(descs + s, 0);
            const int4 x1 = KT == 2 ? load_sub(descs + s, 1) : make_int4(0, 0, 0, 0);
            if (x0.w & kStageEnd) break;
            // every warp waits for each request's q/weights in order, so that
            // its release of the slot below can never run a phase ahead
#pragma unroll
            for (int i = 0; i < KT; ++i) {
                const int meta = i == 0 ? x0.w : x1.w;
                if (ok && (meta & kMetaFirst)) {
                    ok = mbar_wait<kCallWait>(qfull_bar0 + 8u * meta_slot(meta), (qcount >> 1) & 1,
                                              abort_flag, a.status, a.wait_limit_ns);
                    ++qcount;
                }
            }
            if (!ok) break;
            ok = mbar_wait<kCallWait>(tfull_bar0 + 8u * acc, aph, abort_flag, a.status, a.wait_limit_ns);
            if (!ok) break;
            tc_fence_after();
            // The MMAs of this stage are complete, so its key buffers are no
            // longer read: take the descriptor fields and this key's scales
            // into registers and hand the stage back to the producers before
            // the arithmetic, which then overlaps with the next copies.
            int4 d[NSUB];   // (request, block, length, meta) of each sub-tile taken
            float sp[NSUB];
#pragma unroll
            for (int ii = 0; ii < NSUB; ++ii) {
                const int i = E::kSubSplit ? grp : ii;
                d[ii] = E::kSubSplit ? (grp == 0 ? x0 : x1) : (ii == 0 ? x0 : x1);
                sp[ii] = scales_smem[s * (kStageScaleBytes / 4) + i * kTileKeys + row];
            }
            const int rel0 = (x0.w & kMetaLast) ? meta_slot(x0.w) : -1;
            const int rel1 = (KT == 2 && (x1.w & kMetaLast)) ? meta_slot(x1.w) : -1;
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar0 + 8u * s);
            uint32_t taddr[NSUB];
            bool valid[NSUB];
            long long oidx[NSUB];
            const float4* wsrc[NSUB];
#pragma unroll
            for (int ii = 0; ii < NSUB; ++ii) {
                const int i = E::kSubSplit ? grp : ii;
                const int pos = (d[ii].y + page) * kBlockKeys + key;
                taddr[ii] = lane_addr + acc * COLS + i * N;
                valid[ii] = page < (d[ii].w & 0xff) && pos < d[ii].z;
                oidx[ii] = (long long)d[ii].x * NN * a.out_stride + pos;
                wsrc[ii] = reinterpret_cast<const float4*>(smem + L.w + meta_slot(d[ii].w) * L.w_bytes);
            }
            if constexpr (NSUB == 1) {
                stage_logits<H, NN, 1, E::SL, E::GS, E::kChunk>(taddr, d, sp, valid, oidx, wsrc, wp,
                                                                 cur_b, first_slot, a.out,
                                                                 a.out_bf16 != 0, a.out_stride);
            } else {
                // two sub-tiles: one pipelined pass each (measured faster than
                // one sequence over both at these register counts)
#pragma unroll
                for (int ii = 0; ii < NSUB; ++ii) {
                    if ((d[ii].w & 0xff) == 0) continue;
                    const uint32_t ta1[1] = {taddr[ii]};
                    const int4 d1[1] = {d[ii]};
                    const float sp1[1] = {sp[ii]};
                    const bool v1[1] = {valid[ii]};
                    const long long o1[1] = {oidx[ii]};
                    const float4* const w1[1] = {wsrc[ii]};
                    stage_logits<H, NN, 1, E::SL, E::GS, E::kChunk>(ta1, d1, sp1, v1, o1, w1, wp,
                                                                     cur_b, first_slot, a.out,
                                                                     a.out_bf16 != 0, a.out_stride);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(tempty_bar0 + 8u * acc);
                if (rel0 >= 0) mbar_arrive(qempty_bar0 + 8u * rel0);
                if (rel1 >= 0) mbar_arrive(qempty_bar0 + 8u * rel1);
            }
            if (++s == (uint32_t)S) { s = 0; ph ^= 1; }
            if (++acc == NACC) { acc = 0; aph ^= 1; }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem_base, tmem_cols_of(N));
    }
}

template <int H, int NN>
cudaError_t launch(const CUtensorMap& kmap, const CUtensorMap& qmap, const Fp8Args& a,
                   int num_ctas, cudaStream_t stream)
{
    constexpr int N = n_pad_of(NN, H);
    // the two producers take the stages in turn; the end marker's stage rule
    // in their drain needs an even count
    if (a.stages < 2 || (a.stages & 1)) return cudaErrorInvalidValue;
    const size_t smem = (size_t)layout(N, NN, H, a.stages).total + 1024;
    static int configured_device = -1;
    static size_t configured_smem = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev || configured_smem < smem) {
        e = cudaFuncSetAttribute(logits_kernel<H, NN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        if constexpr (EpiPlan<H, NN>::kSplitRegs) {
            // the warpgroups' register budgets must fit the block's allocation,
            // else the epilogue's setmaxnreg.inc would wait forever
            cudaFuncAttributes fa;
            e = cudaFuncGetAttributes(&fa, logits_kernel<H, NN>);
            if (e != cudaSuccess) return e;
            const long long pool = (long long)fa.numRegs * threads_of(NN);
            const long long need = 128LL * EpiPlan<H, NN>::kLowRegs +
                                   128LL * epi_groups_of(NN) * EpiPlan<H, NN>::kHighRegs;
            if (fa.numRegs > EpiPlan<H, NN>::kHighRegs || pool < need)
                return cudaErrorInvalidConfiguration;
        }
        configured_device = dev;
        configured_smem = smem;
    }
    // programmatic stream serialization: this launch may begin while the
    // previous kernel in the stream finishes (see grid_dependency_wait)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)num_ctas);
    cfg.blockDim = dim3((unsigned)threads_of(NN));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, logits_kernel<H, NN>, kmap, qmap, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int H>
cudaError_t launch_heads(const CUtensorMap& kmap, const CUtensorMap& qmap, const Fp8Args& a,
                         int num_ctas, cudaStream_t stream)
{
    switch (a.next_n) {
    case 1: return launch<H, 1>(kmap, qmap, a, num_ctas, stream);
    case 2: return launch<H, 2>(kmap, qmap, a, num_ctas, stream);
    case 3: return launch<H, 3>(kmap, qmap, a, num_ctas, stream);
    case 4: return launch<H, 4>(kmap, qmap, a, num_ctas, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace fp8
}  // namespace pml
