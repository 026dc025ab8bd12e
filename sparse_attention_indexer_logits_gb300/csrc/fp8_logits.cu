// fp8 paged MQA logits on sm_103a.
//
//   out[b*next_n + t, p] = s_p * sum_h w[b*next_n+t, h] * relu(q[b*next_n+t, h] . k_p)
//
// ("flashinfer.attn_scores": math block; first bullet -- the rectifier acts
// per head, before the weighted sum; second bullet -- the fp8 variant is
// multiplied by the per-token fp32 scale s_p from the trailing scale region
// of each kv_fused block; note -- row b*next_n+t, empty requests untouched.)
//
// One persistent CTA per SM walks a contiguous range of 64-key blocks
// (common.cuh) in tiles of two blocks = 128 keys:
//   warp 0      TMA producer: per tile, the keys of each block (8 KB, 3-D
//               tensor map, 128-byte swizzle) and its 64 scales (256 B bulk
//               copy) into a ring of shared-memory stages; per request, the
//               q rows (next_n*H x 128 e4m3, 2-D tensor map) and weights.
//   warp 1      TMEM allocation and MMA issue: four tcgen05.mma kind::f8f6f4
//               (K = 32 each) compute S = K_tile (128 x 128) * Q^T into one
//               of two TMEM accumulators (128 lanes = keys, N = next_n*H
//               columns), then tcgen05.commit.
//   warps 2..   epilogue (1 or 2 warpgroups; group g takes slots t = g, g+2):
//               each thread owns one key (one TMEM lane), loads its head
//               scores with tcgen05.ld, applies relu, weights and sums the
//               heads in registers, multiplies by s_p and stores to out, for
//               positions below min(seq_len, max_context).
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace pml {

namespace {

constexpr int kStageKeyBytes = kTileKeys * kHeadDim;   // 16 KB: two blocks of keys
constexpr int kStageScaleBytes = kTileKeys * 4;        // 512 B

struct Fp8Layout {
    uint32_t k, q, s, w, bar, misc, total;
    uint32_t q_bytes, w_bytes;
};

__host__ __device__ inline Fp8Layout fp8_layout(int n_pad, int next_n, int num_heads, int stages)
{
    Fp8Layout L;
    L.q_bytes = (uint32_t)n_pad * kHeadDim;
    L.w_bytes = (uint32_t)((next_n * num_heads * 4 + 15) / 16 * 16);
    L.k = 0;
    L.q = L.k + (uint32_t)stages * kStageKeyBytes;
    L.s = L.q + 2 * L.q_bytes;
    L.w = L.s + (uint32_t)stages * kStageScaleBytes;
    L.bar = L.w + 2 * L.w_bytes;
    L.misc = L.bar + (uint32_t)(2 * stages + 8) * 8;
    L.total = L.misc + 64;
    return L;
}

template <int H>
__device__ __forceinline__ float weighted_relu_sum(uint32_t taddr, const float* __restrict__ w)
{
    float acc = 0.f;
    if constexpr (H == 8) {
        float v[8];
        tmem_ld8(taddr, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc = fmaf(w[i], fmaxf(v[i], 0.f), acc);
    } else if constexpr (H == 16) {
        float v[16];
        tmem_ld16(taddr, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) acc = fmaf(w[i], fmaxf(v[i], 0.f), acc);
    } else {
#pragma unroll
        for (int c = 0; c < H; c += 32) {
            float v[32];
            tmem_ld32(taddr + c, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) acc = fmaf(w[c + i], fmaxf(v[i], 0.f), acc);
        }
    }
    return acc;
}

template <int H>
__global__ void __launch_bounds__(320, 1)
    fp8_logits_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap qmap, const Fp8Args a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = a.stages;
    const int n = a.next_n;
    const int N = a.n_pad;
    const Fp8Layout L = fp8_layout(N, n, H, S);

    const uint32_t base = smem_addr(smem);
    const uint32_t k_base = base + L.k;
    const uint32_t q_base = base + L.q;
    const uint32_t s_base = base + L.s;
    const float* scales_smem = reinterpret_cast<const float*>(smem + L.s);
    const float* w_smem = reinterpret_cast<const float*>(smem + L.w);
    const uint32_t bar = base + L.bar;
    auto full_bar = [&](int s) { return bar + 8u * s; };
    auto empty_bar = [&](int s) { return bar + 8u * (S + s); };
    const uint32_t tfull_bar0 = bar + 8u * (2 * S);       // +8*acc
    const uint32_t tempty_bar0 = bar + 8u * (2 * S + 2);
    const uint32_t qfull_bar0 = bar + 8u * (2 * S + 4);   // +8*slot
    const uint32_t qempty_bar0 = bar + 8u * (2 * S + 6);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);
    int* sched = reinterpret_cast<int*>(smem + L.misc + 16);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = a.epi_groups;
    const uint32_t epi_threads_warps = 4u * E;

    // ---------------------------------------------------------------- setup
    if (warp == 0) {
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
                mbar_init(empty_bar(s), epi_threads_warps);
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(tfull_bar0 + 8u * i, 1);
                mbar_init(tempty_bar0 + 8u * i, epi_threads_warps);
                mbar_init(qfull_bar0 + 8u * i, 1);
                mbar_init(qempty_bar0 + 8u * i, epi_threads_warps);
            }
            fence_mbar_init();
            tma_prefetch_map(&kmap);
            tma_prefetch_map(&qmap);
        }
    } else if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), a.tmem_cols);
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
            w.init(a.seq_lens, a.batch, sb, sj, eb, ej);
            int it = 0, qcount = 0, prev_b = -1;
            bool ok = true;
            while (ok && !w.done()) {
                const int c = w.cnt();
                if (w.b != prev_b) {
                    const int slot = qcount & 1;
                    ok = mbar_wait(qempty_bar0 + 8u * slot, ((qcount >> 1) & 1) ^ 1, abort_flag,
                                   a.status);
                    if (!ok) break;
                    const uint32_t qb = q_base + slot * L.q_bytes;
                    const int nH = n * H;
                    mbar_arrive_expect_tx(qfull_bar0 + 8u * slot,
                                          (uint32_t)a.q_box_rows * kHeadDim + (uint32_t)nH * 4);
                    tma_load_2d(qb, &qmap, qfull_bar0 + 8u * slot, 0, w.b * nH);
                    bulk_load(base + L.w + slot * L.w_bytes, a.weights + (long long)w.b * nH,
                              (uint32_t)nH * 4, qfull_bar0 + 8u * slot);
                    ++qcount;
                    prev_b = w.b;
                }
                const int s = it % S;
                ok = mbar_wait(empty_bar(s), ((it / S) & 1) ^ 1, abort_flag, a.status);
                if (!ok) break;
                int phys[2] = {0, 0};
                uint32_t bytes = 0;
                int nload = 0;
                for (int cc = 0; cc < c; ++cc) {
                    if ((long long)(w.j + cc) * kBlockKeys < a.max_context) {
                        long long pb = __ldg(a.block_table + (long long)w.b * a.bt_stride + w.j + cc);
                        if (pb < 0 || pb >= a.num_blocks) {
                            atomicOr(a.status, kStatusBadBlock);
                            pb = 0;
                        }
                        phys[cc] = (int)pb;
                        nload = cc + 1;
                        bytes += kFp8BlockBytes;
                    }
                }
                mbar_arrive_expect_tx(full_bar(s), bytes);
                for (int cc = 0; cc < nload; ++cc) {
                    tma_load_3d_stream(k_base + s * kStageKeyBytes + cc * kFp8BlockKeyBytes, &kmap,
                                       full_bar(s), 0, 0, phys[cc], policy);
                    bulk_load_stream(s_base + s * kStageScaleBytes + cc * (kBlockKeys * 4),
                                     a.kv_fused + (long long)phys[cc] * kFp8BlockBytes +
                                         kFp8BlockKeyBytes,
                                     kBlockKeys * 4, full_bar(s), policy);
                }
                w.advance(c);
                ++it;
            }
            if (!ok) {
                // drain: let every copy already issued land before the CTA exits
                for (int t = (it > S ? it - S : 0); t < it; ++t)
                    mbar_wait_drain(full_bar(t % S), (t / S) & 1);
                for (int qc = (qcount > 2 ? qcount - 2 : 0); qc < qcount; ++qc)
                    mbar_wait_drain(qfull_bar0 + 8u * (qc & 1), (qc >> 1) & 1);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = make_idesc(0, 0, kTileKeys, (uint32_t)N);
            Walk w;
            w.init(a.seq_lens, a.batch, sb, sj, eb, ej);
            int it = 0, qcount = 0, prev_b = -1, slot = 0;
            bool ok = true;
            while (!w.done()) {
                const int c = w.cnt();
                if (w.b != prev_b) {
                    slot = qcount & 1;
                    ok = mbar_wait(qfull_bar0 + 8u * slot, (qcount >> 1) & 1, abort_flag, a.status);
                    if (!ok) break;
                    ++qcount;
                    prev_b = w.b;
                }
                const int s = it % S;
                ok = mbar_wait(full_bar(s), (it / S) & 1, abort_flag, a.status);
                if (!ok) break;
                const int acc = it & 1;
                ok = mbar_wait(tempty_bar0 + 8u * acc, ((it >> 1) & 1) ^ 1, abort_flag, a.status);
                if (!ok) break;
                tc_fence_after();
                const uint64_t ad = smem_desc_sw128(k_base + s * kStageKeyBytes);
                const uint64_t bd = smem_desc_sw128(q_base + slot * L.q_bytes);
                const uint32_t d = tmem_base + (uint32_t)(acc * N);
#pragma unroll
                for (int k = 0; k < kHeadDim / 32; ++k)
                    mma_f8(d, ad + 2u * k, bd + 2u * k, idesc, k > 0 ? 1u : 0u);
                mma_commit(tfull_bar0 + 8u * acc);
                w.advance(c);
                ++it;
            }
            if (!ok && it > 0) mbar_wait_drain(tfull_bar0 + 8u * ((it - 1) & 1), ((it - 1) >> 1) & 1);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 2;
        const int grp = ew >> 2;
        const int quad = warp & 3;             // TMEM lane quadrant this warp may access
        const int row = quad * 32 + lane;      // key row within the tile
        const int page = row >> 6;
        const int key = row & 63;
        const uint32_t lane_addr = tmem_base + ((uint32_t)(quad * 32) << 16);
        Walk w;
        w.init(a.seq_lens, a.batch, sb, sj, eb, ej);
        int it = 0, qcount = 0, prev_b = -1, slot = 0, len = 0;
        bool ok = true;
        while (!w.done()) {
            const int c = w.cnt();
            if (w.b != prev_b) {
                slot = qcount & 1;
                ok = mbar_wait(qfull_bar0 + 8u * slot, (qcount >> 1) & 1, abort_flag, a.status);
                if (!ok) break;
                ++qcount;
                prev_b = w.b;
                len = min(__ldg(a.seq_lens + w.b), a.max_context);
            }
            const bool last = w.last_of_request(c);
            const int s = it % S;
            ok = mbar_wait(full_bar(s), (it / S) & 1, abort_flag, a.status);
            if (!ok) break;
            const int acc = it & 1;
            ok = mbar_wait(tfull_bar0 + 8u * acc, (it >> 1) & 1, abort_flag, a.status);
            if (!ok) break;
            tc_fence_after();
            const int pos = (w.j + page) * kBlockKeys + key;
            const bool valid = page < c && pos < len;
            const float sp = scales_smem[s * kTileKeys + row];
            const float* wq = w_smem + slot * (L.w_bytes / 4);
            for (int t = grp; t < n; t += E) {
                const float r = weighted_relu_sum<H>(lane_addr + (uint32_t)(acc * N + t * H), wq + t * H);
                if (valid)
                    a.out[((long long)w.b * n + t) * a.out_stride + pos] = sp * r;
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

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, a.tmem_cols);
    }
}

template <int H>
cudaError_t launch_h(const CUtensorMap& kmap, const CUtensorMap& qmap, const Fp8Args& a,
                     int num_ctas, cudaStream_t stream)
{
    const size_t smem = fp8_smem_bytes(a.n_pad, a.next_n, H, a.stages);
    static int configured_device = -1;
    static size_t configured_smem = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev || configured_smem < smem) {
        e = cudaFuncSetAttribute(fp8_logits_kernel<H>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        configured_device = dev;
        configured_smem = smem;
    }
    const int threads = 64 + 128 * a.epi_groups;
    fp8_logits_kernel<H><<<num_ctas, threads, smem, stream>>>(kmap, qmap, a);
    return cudaGetLastError();
}

}  // namespace

size_t fp8_smem_bytes(int n_pad, int next_n, int num_heads, int stages)
{
    return (size_t)fp8_layout(n_pad, next_n, num_heads, stages).total + 1024;
}

cudaError_t launch_fp8_logits(int num_heads, const CUtensorMap& kmap, const CUtensorMap& qmap,
                              const Fp8Args& a, int num_ctas, cudaStream_t stream)
{
    switch (num_heads) {
    case 8: return launch_h<8>(kmap, qmap, a, num_ctas, stream);
    case 16: return launch_h<16>(kmap, qmap, a, num_ctas, stream);
    case 32: return launch_h<32>(kmap, qmap, a, num_ctas, stream);
    case 64: return launch_h<64>(kmap, qmap, a, num_ctas, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pml
