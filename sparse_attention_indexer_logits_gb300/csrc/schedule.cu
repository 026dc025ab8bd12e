// The persistent work schedule as a standalone kernel
// ("flashinfer.attn_scores", "Scheduling and Setup": a per-call CTA work
// assignment computed on the GPU, which a caller may build once and pass back
// while seq_lens is unchanged).
//
// meta[2i], meta[2i+1] = (request, block) where CTA i's range starts, for
// i = 0 .. num_ctas; entry num_ctas is the end, (batch, 0).  One warp per
// entry, the same device code the logits kernel runs in its prologue when no
// schedule is passed, so the two agree bit for bit.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace pml {

namespace {

__global__ void __launch_bounds__(128) schedule_kernel(const int32_t* __restrict__ seq_lens,
                                                       int batch, int num_ctas,
                                                       int32_t* __restrict__ meta)
{
    const int warps = (blockDim.x >> 5) * gridDim.x;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw > num_ctas) return;   // whole warps exit together
    const long long total = warp_total_blocks(seq_lens, batch);
    // entries gw, gw + warps, ... (pairs located two at a time)
    for (int i = gw; i <= num_ctas; i += 2 * warps) {
        const int i2 = (i + warps <= num_ctas) ? i + warps : i;
        int b0, j0, b1, j1;
        warp_locate2(seq_lens, batch, range_start(total, num_ctas, i),
                     range_start(total, num_ctas, i2), b0, j0, b1, j1);
        if (lane == 0) {
            meta[2 * i] = b0;
            meta[2 * i + 1] = j0;
            meta[2 * i2] = b1;
            meta[2 * i2 + 1] = j1;
        }
    }
}

}  // namespace

cudaError_t launch_schedule(const int32_t* seq_lens, int batch, int num_ctas, int32_t* meta,
                            cudaStream_t stream)
{
    const int entries = num_ctas + 1;
    int blocks = (entries + 3) / 4;
    if (blocks > 64) blocks = 64;
    schedule_kernel<<<blocks, 128, 0, stream>>>(seq_lens, batch, num_ctas, meta);
    return cudaGetLastError();
}

}  // namespace pml
