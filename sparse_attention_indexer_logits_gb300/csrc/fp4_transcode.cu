// MXFP4 paged MQA logits, front half: re-encoding of the MXFP4 operands for
// the fp8 logits engine.
//
// ("flashinfer.attn_scores", the paragraphs after the math block: the fp4
// variant folds MXFP4 block scales -- one per 32-element group, on both
// operands -- into the dequantised values; q packs two FP4 values per byte;
// 64 heads of 128; no per-position factor.)
//
// A row (one key, or one head of one query slot) holds 128 E2M1 codes and
// four E8M0 group scales 2^(e_g - 127).  With e_max the largest of the four,
// every value is  code * 2^(e_g - e_max) * 2^(e_max - 127):  the first factor
// is an E2M1 value scaled down by 2^(e_max - e_g), which E4M3 holds exactly
// while e_max - e_g <= 8 (E4M3 reaches down to 2^-9; E2M1 values have at most
// two significant bits); the second factor is one power of two per row.  So
//
//   * a key becomes 128 E4M3 bytes and the fp32 per-token scale
//     s_p = 2^(e_max - 127) of the fp8 engine's kv_fused block;
//   * a query row (t, h) becomes 128 E4M3 bytes, and its 2^(e_max - 127)
//     joins the head weight: w' = w * 2^(e_max - 127), since
//     w * relu(c * x) = (w * c) * relu(x) for c > 0.
//
// The fp8 engine then computes s_p * sum_h w' * relu(q' . k'), which is the
// MXFP4 logit.  A value that E4M3 cannot hold exactly (a row whose group
// scales lie more than 8 binades apart and whose smaller groups hold small
// codes) is rounded and flagged with kStatusFp4Inexact.
//
// One thread per row.  Keys: only the blocks a request uses below
// max_context, read through the block table (a block two requests share is
// written twice with the same bytes).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "fp4_transcode.h"
#include "kernels.h"
#include "ptx.cuh"

namespace pml {

namespace {

constexpr int kMxRowBytes = kHeadDim / 2;                      // 64
constexpr int kMxBlockCodeBytes = kBlockKeys * kMxRowBytes;      // 4096

// Sign bits of four E2M1 codes (the low 16 bits of x, one per nibble) moved
// to the top bit of four bytes.
__device__ __forceinline__ uint32_t nibble_signs_to_bytes(uint32_t x)
{
    return ((x & 0x0008u) << 4) | ((x & 0x0080u) << 8) | ((x & 0x0800u) << 12) |
           ((x & 0x8000u) << 16);
}

// One row: 64 code bytes (four 16-byte chunks, chunk g = group g) and the
// four E8M0 scale bytes in `sc` (byte g = group g) -> 128 E4M3 bytes in
// `out` (byte d = element d) and the row's power of two.  Per group, the
// E4M3 bytes of the eight E2M1 magnitudes times 2^(e_g - e_max) form a table
// that one byte permute per four codes reads, the code's low three bits as
// the index; the sign bit is moved across.  Returns false if a code the row
// uses was not exact in E4M3.
__device__ __forceinline__ bool mx_row_to_e4m3(const uint4 (&codes)[4], uint32_t sc,
                                               uint32_t (&out)[32], float& row_scale)
{
    int e_max = 0;
    bool nan = false;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int e = (int)((sc >> (8 * g)) & 0xFF);
        nan |= e == 0xFF;
        e_max = max(e_max, e);
    }
    row_scale = nan ? __int_as_float(0x7FC00000) : ldexpf(1.0f, e_max - 127);
    uint32_t inexact = 0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int e = (int)((sc >> (8 * g)) & 0xFF);
        const float down = ldexpf(1.0f, e - e_max);       // 2^-(e_max - e_g), exact or 0
        uint32_t lut[2] = {0u, 0u}, bad[2] = {0u, 0u};
#pragma unroll
        for (int pr = 0; pr < 4; ++pr) {                   // magnitudes 2pr (low), 2pr+1
            const uint32_t h2 = e2m1x2_to_f16x2((uint32_t)(((2 * pr + 1) << 4) | (2 * pr)));
            const __half2 hv = *reinterpret_cast<const __half2*>(&h2);
            const float v0 = __low2float(hv) * down, v1 = __high2float(hv) * down;
            const __nv_fp8_storage_t b0 = __nv_cvt_float_to_fp8(v0, __NV_SATFINITE, __NV_E4M3);
            const __nv_fp8_storage_t b1 = __nv_cvt_float_to_fp8(v1, __NV_SATFINITE, __NV_E4M3);
            const bool x0 = __half2float(__half(__nv_cvt_fp8_to_halfraw(b0, __NV_E4M3))) == v0;
            const bool x1 = __half2float(__half(__nv_cvt_fp8_to_halfraw(b1, __NV_E4M3))) == v1;
            const int sh = 16 * (pr & 1);
            lut[pr >> 1] |= ((uint32_t)b0 | ((uint32_t)b1 << 8)) << sh;
            bad[pr >> 1] |= ((x0 ? 0u : 1u) | ((x1 ? 0u : 1u) << 8)) << sh;
        }
        const uint32_t w[4] = {codes[g].x, codes[g].y, codes[g].z, codes[g].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {                      // 8 codes -> 8 E4M3 bytes
            const uint32_t lo = w[q] & 0xFFFFu, hi = w[q] >> 16;
            const uint32_t sel_lo = lo & 0x7777u, sel_hi = hi & 0x7777u;
            out[g * 8 + 2 * q] = __byte_perm(lut[0], lut[1], sel_lo) | nibble_signs_to_bytes(lo);
            out[g * 8 + 2 * q + 1] = __byte_perm(lut[0], lut[1], sel_hi) | nibble_signs_to_bytes(hi);
            inexact |= __byte_perm(bad[0], bad[1], sel_lo) | __byte_perm(bad[0], bad[1], sel_hi);
        }
    }
    return inexact == 0;
}

__device__ __forceinline__ void store_row(uint8_t* dst, const uint32_t (&out)[32])
{
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int c = 0; c < 8; ++c)
        d[c] = make_uint4(out[4 * c], out[4 * c + 1], out[4 * c + 2], out[4 * c + 3]);
}

// grid (x, batch), 128 threads: two blocks of 64 keys per CTA and step.
__global__ void __launch_bounds__(128) fp4_transcode_kv_kernel(const Fp4TranscodeArgs a)
{
    const int b = blockIdx.y;
    const int L = min(__ldg(a.seq_lens + b), a.max_context);
    if (L <= 0) return;
    const int nb = blocks_of(L);
    const int r = threadIdx.x & 63;
    bool exact = true;
    for (int j = 2 * blockIdx.x + (threadIdx.x >> 6); j < nb; j += 2 * gridDim.x) {
        const long long P = __ldg(a.block_table + (long long)b * a.bt_stride + j);
        if (P < 0 || P >= a.num_blocks) continue;          // the logits kernel flags it
        const uint8_t* src = a.kv + P * kMxfp4BlockBytes;
        const uint4* cp = reinterpret_cast<const uint4*>(src + r * kMxRowBytes);
        const uint4 codes[4] = {__ldg(cp), __ldg(cp + 1), __ldg(cp + 2), __ldg(cp + 3)};
        const uint32_t sc =
            __ldg(reinterpret_cast<const uint32_t*>(src + kMxBlockCodeBytes + r * 4));
        uint32_t out[32];
        float s;
        exact &= mx_row_to_e4m3(codes, sc, out, s);
        uint8_t* dst = a.kv8 + P * kFp8BlockBytes;
        store_row(dst + r * kHeadDim, out);
        reinterpret_cast<float*>(dst + kBlockKeys * kHeadDim)[r] = s;
    }
    if (!exact) atomicOr(a.status, kStatusFp4Inexact);
}

// One thread per (slot row, head): rows * 64 threads.
__global__ void __launch_bounds__(256) fp4_transcode_q_kernel(const Fp4TranscodeArgs a)
{
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= a.q_rows) return;
    const uint4* cp = reinterpret_cast<const uint4*>(a.q + i * kMxRowBytes);
    const uint4 codes[4] = {__ldg(cp), __ldg(cp + 1), __ldg(cp + 2), __ldg(cp + 3)};
    const uint32_t sc = __ldg(reinterpret_cast<const uint32_t*>(a.q_sf + i * 4));
    uint32_t out[32];
    float s;
    const bool exact = mx_row_to_e4m3(codes, sc, out, s);
    store_row(a.q8 + i * kHeadDim, out);
    a.w8[i] = __ldg(a.weights + i) * s;
    if (!exact) atomicOr(a.status, kStatusFp4Inexact);
}

}  // namespace

cudaError_t launch_fp4_transcode(const Fp4TranscodeArgs& a, int batch, cudaStream_t stream)
{
    if (batch > 65535) return cudaErrorInvalidValue;
    if (batch > 0) {
        // one CTA per pair of blocks of the longest possible request (the
        // loop in the kernel covers the rest past 65535 pairs)
        const long long pairs = ((long long)blocks_of(a.max_context) + 1) / 2;
        const unsigned gx = (unsigned)(pairs < 1 ? 1 : pairs > 65535 ? 65535 : pairs);
        fp4_transcode_kv_kernel<<<dim3(gx, batch), 128, 0, stream>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (a.q_rows > 0) {
        const long long blocks = (a.q_rows + 255) / 256;
        if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
        fp4_transcode_q_kernel<<<(unsigned)blocks, 256, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace pml
