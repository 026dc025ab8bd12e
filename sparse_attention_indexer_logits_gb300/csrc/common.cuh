// Constants, device status bits and the persistent work schedule shared by
// the kernels of the paged MQA-logits library.
//
// Work model ("flashinfer.attn_scores", "Scheduling and Setup"): request b
// owns nb_b = ceil(len_b / 64) KV blocks of 64 keys; the blocks of all
// requests, in request order, are numbered 0 .. T-1 and cut into num_ctas
// contiguous ranges whose sizes differ by at most one (the first T mod
// num_ctas ranges are one block longer).  A range start is stored as the
// (request, block-within-request) it falls on; a start at T is (batch, 0).
// A persistent CTA walks its range in tiles of up to two consecutive blocks
// of one request (128 keys, the MMA's M).
#pragma once

#include <stdint.h>

namespace pml {

constexpr int kHeadDim = 128;                 // q / key length (elements)
constexpr int kBlockKeys = 64;                // keys per paged block
constexpr int kFp8BlockKeyBytes = kBlockKeys * kHeadDim;          // 8192
constexpr int kFp8BlockBytes = kFp8BlockKeyBytes + kBlockKeys * 4; // 8448: keys, then scales
constexpr int kTileKeys = 128;                // MMA M: two blocks
constexpr unsigned long long kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s per wait
constexpr unsigned int kWaitSuspendNs = 1000;   // longest hardware suspension per try_wait

// Bits of the device status word (sticky until cleared by the host).
constexpr unsigned int kStatusWaitTimeout = 1u;   // an mbarrier wait ran out; the CTA aborted
constexpr unsigned int kStatusBadBlock = 2u;      // a block/page index outside the cache
constexpr unsigned int kStatusBadRequest = 4u;    // a group's request outside the block table
// MXFP4 logits: a product of query and key values, or a head weight, may have
// fallen below the range of its row frames and been dropped (see mxfp4_logits.cu)
constexpr unsigned int kStatusFp4Inexact = 8u;

// MXFP4 paged cache: a block is 64 keys x 64 code bytes (E2M1, two per
// byte), then 64 x 4 E8M0 scale bytes (one per 32 values).
constexpr int kMxfp4Heads = 64;
constexpr int kMxfp4BlockBytes = kBlockKeys * (kHeadDim / 2 + kHeadDim / 32);   // 4352

__host__ __device__ __forceinline__ int blocks_of(int32_t len)
{
    return len > 0 ? (len + kBlockKeys - 1) / kBlockKeys : 0;
}

// Start of range `cta` in the flattened block order: cta*floor(T/G) + min(cta, T mod G).
__host__ __device__ __forceinline__ long long range_start(long long total, int num_ctas, int cta)
{
    const long long base = total / num_ctas, extra = total % num_ctas;
    return (long long)cta * base + (cta < extra ? cta : extra);
}

// Executed by one full warp: total block count of all requests.
__device__ __forceinline__ long long warp_total_blocks(const int32_t* lens, int batch)
{
    const int lane = threadIdx.x & 31;
    long long t = 0;
    for (int i = lane; i < batch; i += 32) t += blocks_of(__ldg(lens + i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}

// Executed by one full warp: (request, block) positions of two flattened
// block indices s0 <= s1 (a position at or past the end is (batch, 0)).
// Results are returned to every lane.
__device__ __forceinline__ void warp_locate2(const int32_t* lens, int batch, long long s0,
                                             long long s1, int& b0, int& j0, int& b1, int& j1)
{
    const int lane = threadIdx.x & 31;
    int fb0 = batch, fj0 = 0, fb1 = batch, fj1 = 0;
    long long prefix = 0;
    for (int c = 0; c < batch; c += 32) {
        const int i = c + lane;
        const long long v = (i < batch) ? blocks_of(__ldg(lens + i)) : 0;
        long long incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        const long long start = prefix + incl - v;
        if (v > 0 && start <= s0 && s0 < start + v) { fb0 = i; fj0 = (int)(s0 - start); }
        if (v > 0 && start <= s1 && s1 < start + v) { fb1 = i; fj1 = (int)(s1 - start); }
        prefix += __shfl_sync(0xffffffffu, incl, 31);
    }
    // exactly one lane (or none) found each position: take the minimum request
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const int ob0 = __shfl_xor_sync(0xffffffffu, fb0, o);
        const int oj0 = __shfl_xor_sync(0xffffffffu, fj0, o);
        const int ob1 = __shfl_xor_sync(0xffffffffu, fb1, o);
        const int oj1 = __shfl_xor_sync(0xffffffffu, fj1, o);
        if (ob0 < fb0) { fb0 = ob0; fj0 = oj0; }
        if (ob1 < fb1) { fb1 = ob1; fj1 = oj1; }
    }
    b0 = fb0; j0 = fj0; b1 = fb1; j1 = fj1;
}

// Walks one CTA's range in tiles of up to two blocks of one request.
struct Walk {
    const int32_t* lens;
    int batch;
    int b, j;      // current position (b < batch means j < blocks_of(lens[b]))
    int eb, ej;    // end of the range (exclusive)
    int nbb;       // blocks of request b
    int len;       // length of request b

    __device__ __forceinline__ void init(const int32_t* l, int B, int sb, int sj, int e_b, int e_j)
    {
        lens = l; batch = B; b = sb; j = sj; eb = e_b; ej = e_j;
        len = (b < batch) ? __ldg(lens + b) : 0;
        nbb = blocks_of(len);
    }
    __device__ __forceinline__ bool done() const { return b >= batch || (b == eb && j == ej); }
    // blocks in the current tile: 1 or 2
    __device__ __forceinline__ int cnt() const
    {
        const int lim = (b == eb) ? ej : nbb;
        return (lim - j) >= 2 ? 2 : 1;
    }
    // whether the current tile is the last one of request b in this range
    __device__ __forceinline__ bool last_of_request(int c) const
    {
        return (j + c == nbb) || (b == eb && j + c == ej);
    }
    // blocks of request b in this range after the current tile
    __device__ __forceinline__ int blocks_after(int c) const
    {
        return ((b == eb) ? ej : nbb) - j - c;
    }
    __device__ __forceinline__ void advance(int c)
    {
        j += c;
        if (j >= nbb) {
            j = 0;
            ++b;
            nbb = 0;
            while (b < batch && (nbb = blocks_of(len = __ldg(lens + b))) == 0) ++b;
        }
    }
};

// Flags of the per-tile records a producer publishes to the other roles.
constexpr int kTileFirst = 1;   // first tile of a request in this CTA: q / weights were loaded
constexpr int kTileLast = 2;    // last tile of a request in this CTA: release the q slot after it

}  // namespace pml
