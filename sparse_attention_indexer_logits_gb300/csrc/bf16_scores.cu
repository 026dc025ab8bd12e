// Single-head bf16 indexer scores on sm_103a.
//
//   scores[r, k] = query[r] . key_k     for k < min(context_lengths[g], max_context)
//
// ("flashinfer.sdsa.indexer_scores": the paged MQA-logits computation with one
// head, so no weight and no rectifier; query rows come in groups of 1..8
// consecutive rows sharing one length and one request; only pages below a
// group's length are read and later entries are not written.)
//
// Same engine as the fp8 kernel with the group as the unit of work: the
// persistent schedule runs over context_lengths, a tile is two 64-key pages
// of one group (M = 128 keys), the B operand is the group's rows padded to
// N = 16, and the MMA is tcgen05.mma kind::f16 with bf16 operands.  A key row
// is 256 bytes, wider than the 128-byte swizzle span, so every page arrives
// as two K-halves of 64 elements (two TMA boxes) and the tile is consumed by
// 2 x 4 MMAs of K = 16.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace pml {

namespace {

constexpr int kN = 16;                                  // MMA N: group rows padded
constexpr int kHalfBytes = kTileKeys * 128;             // 16 KB: one K-half of a tile
constexpr int kStageBytes = 2 * kHalfBytes;             // 32 KB
constexpr int kQHalfBytes = kN * 128;                   // 2 KB
constexpr int kQSlotBytes = 2 * kQHalfBytes;            // 4 KB
constexpr int kPageHalfBytes = kBlockKeys * 128;        // 8 KB: one K-half of a page

struct Bf16Layout {
    uint32_t k, q, bar, misc, total;
};

__host__ __device__ inline Bf16Layout bf16_layout(int stages)
{
    Bf16Layout L;
    L.k = 0;
    L.q = L.k + (uint32_t)stages * kStageBytes;
    L.bar = L.q + 2 * kQSlotBytes;
    L.misc = L.bar + (uint32_t)(2 * stages + 8) * 8;
    L.total = L.misc + 64;
    return L;
}

__global__ void __launch_bounds__(192, 1)
    bf16_scores_kernel(const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap qmap, const Bf16Args a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = a.stages;
    const int G = a.group_size;
    const Bf16Layout L = bf16_layout(S);

    const uint32_t base = smem_addr(smem);
    const uint32_t k_base = base + L.k;
    const uint32_t q_base = base + L.q;
    const uint32_t bar = base + L.bar;
    auto full_bar = [&](int s) { return bar + 8u * s; };
    auto empty_bar = [&](int s) { return bar + 8u * (S + s); };
    const uint32_t tfull_bar0 = bar + 8u * (2 * S);
    const uint32_t tempty_bar0 = bar + 8u * (2 * S + 2);
    const uint32_t qfull_bar0 = bar + 8u * (2 * S + 4);
    const uint32_t qempty_bar0 = bar + 8u * (2 * S + 6);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);
    int* sched = reinterpret_cast<int*>(smem + L.misc + 16);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr uint32_t kTmemCols = 32;    // two accumulators of N = 16 columns

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
                mbar_init(full_bar(s), 1);
                mbar_init(empty_bar(s), 4);
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(tfull_bar0 + 8u * i, 1);
                mbar_init(tempty_bar0 + 8u * i, 4);
                mbar_init(qfull_bar0 + 8u * i, 1);
                mbar_init(qempty_bar0 + 8u * i, 4);
            }
            fence_mbar_init();
            tma_prefetch_map(&kmap);
            tma_prefetch_map(&qmap);
        }
    } else if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int sb = sched[0], sj = sched[1], eb = sched[2], ej = sched[3];

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t policy = policy_evict_first();
            Walk w;
            w.init(a.context_lengths, a.groups, sb, sj, eb, ej);
            int it = 0, qcount = 0, prev_g = -1;
            long long bt_row = 0;
            bool ok = true;
            while (!w.done()) {
                const int c = w.cnt();
                if (w.b != prev_g) {
                    const int slot = qcount & 1;
                    ok = mbar_wait(qempty_bar0 + 8u * slot, ((qcount >> 1) & 1) ^ 1, abort_flag,
                                   a.status);
                    if (!ok) break;
                    const uint32_t qb = q_base + slot * kQSlotBytes;
                    const uint32_t qfb = qfull_bar0 + 8u * slot;
                    mbar_arrive_expect_tx(qfb, 2u * a.q_box_rows * 128u);
                    tma_load_2d(qb, &qmap, qfb, 0, w.b * G);
                    tma_load_2d(qb + kQHalfBytes, &qmap, qfb, 64, w.b * G);
                    int req = __ldg(a.requests + w.b);
                    if (req < 0 || req >= a.num_requests) {
                        atomicOr(a.status, kStatusBadRequest);
                        req = 0;
                    }
                    bt_row = (long long)req * a.bt_stride;
                    ++qcount;
                    prev_g = w.b;
                }
                const int s = it % S;
                ok = mbar_wait(empty_bar(s), ((it / S) & 1) ^ 1, abort_flag, a.status);
                if (!ok) break;
                int page[2] = {0, 0};
                int nload = 0;
                for (int cc = 0; cc < c; ++cc) {
                    if ((long long)(w.j + cc) * kBlockKeys < a.max_context) {
                        long long pg = __ldg(a.block_table + bt_row + w.j + cc);
                        if (pg < 0 || pg >= a.num_pages) {
                            atomicOr(a.status, kStatusBadBlock);
                            pg = 0;
                        }
                        page[cc] = (int)pg;
                        nload = cc + 1;
                    }
                }
                mbar_arrive_expect_tx(full_bar(s), (uint32_t)nload * 2u * kPageHalfBytes);
                for (int cc = 0; cc < nload; ++cc) {
                    const uint32_t dst = k_base + s * kStageBytes + cc * kPageHalfBytes;
                    tma_load_3d_stream(dst, &kmap, full_bar(s), 0, 0, page[cc], policy);
                    tma_load_3d_stream(dst + kHalfBytes, &kmap, full_bar(s), 64, 0, page[cc], policy);
                }
                w.advance(c);
                ++it;
            }
            if (!ok) {
                for (int t = (it > S ? it - S : 0); t < it; ++t)
                    mbar_wait_drain(full_bar(t % S), (t / S) & 1);
                for (int qc = (qcount > 2 ? qcount - 2 : 0); qc < qcount; ++qc)
                    mbar_wait_drain(qfull_bar0 + 8u * (qc & 1), (qc >> 1) & 1);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = make_idesc(1, 1, kTileKeys, kN);
            Walk w;
            w.init(a.context_lengths, a.groups, sb, sj, eb, ej);
            int it = 0, qcount = 0, prev_g = -1, slot = 0;
            bool ok = true;
            while (!w.done()) {
                const int c = w.cnt();
                if (w.b != prev_g) {
                    slot = qcount & 1;
                    ok = mbar_wait(qfull_bar0 + 8u * slot, (qcount >> 1) & 1, abort_flag, a.status);
                    if (!ok) break;
                    ++qcount;
                    prev_g = w.b;
                }
                const int s = it % S;
                ok = mbar_wait(full_bar(s), (it / S) & 1, abort_flag, a.status);
                if (!ok) break;
                const int acc = it & 1;
                ok = mbar_wait(tempty_bar0 + 8u * acc, ((it >> 1) & 1) ^ 1, abort_flag, a.status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * kN);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint64_t ad = smem_desc_sw128(k_base + s * kStageBytes + h * kHalfBytes);
                    const uint64_t bd = smem_desc_sw128(q_base + slot * kQSlotBytes + h * kQHalfBytes);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_f16(d, ad + 2u * k, bd + 2u * k, idesc, (h | k) ? 1u : 0u);
                }
                mma_commit(tfull_bar0 + 8u * acc);
                w.advance(c);
                ++it;
            }
            if (!ok && it > 0) mbar_wait_drain(tfull_bar0 + 8u * ((it - 1) & 1), ((it - 1) >> 1) & 1);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int pg = row >> 6;
        const int key = row & 63;
        const uint32_t lane_addr = tmem_base + ((uint32_t)(quad * 32) << 16);
        Walk w;
        w.init(a.context_lengths, a.groups, sb, sj, eb, ej);
        int it = 0, qcount = 0, prev_g = -1, slot = 0, len = 0;
        bool ok = true;
        while (!w.done()) {
            const int c = w.cnt();
            if (w.b != prev_g) {
                slot = qcount & 1;
                ++qcount;
                prev_g = w.b;
                len = min(__ldg(a.context_lengths + w.b), a.max_context);
            }
            const bool last = w.last_of_request(c);
            const int s = it % S;
            const int acc = it & 1;
            ok = mbar_wait(tfull_bar0 + 8u * acc, (it >> 1) & 1, abort_flag, a.status);
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
                mbar_arrive(empty_bar(s));
                if (last) mbar_arrive(qempty_bar0 + 8u * slot);
            }
            w.advance(c);
            ++it;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

size_t bf16_smem_bytes(int stages) { return (size_t)bf16_layout(stages).total + 1024; }

cudaError_t launch_bf16_scores(const CUtensorMap& kmap, const CUtensorMap& qmap,
                               const Bf16Args& a, int num_ctas, cudaStream_t stream)
{
    const size_t smem = bf16_smem_bytes(a.stages);
    static int configured_device = -1;
    static size_t configured_smem = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev || configured_smem < smem) {
        e = cudaFuncSetAttribute(bf16_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        configured_device = dev;
        configured_smem = smem;
    }
    bf16_scores_kernel<<<num_ctas, 192, smem, stream>>>(kmap, qmap, a);
    return cudaGetLastError();
}

}  // namespace pml
