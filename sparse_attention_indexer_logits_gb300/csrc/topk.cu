// Per-row top-k over paged MQA logits: the indexer's selection of KV
// positions ("flashinfer.attn_scores", intro: the logits are what a
// sparse-attention indexer uses to choose which KV tokens to keep; note: row
// b*next_n+t is meaningful for positions 0 .. seq_lens[b]-next_n+t).
//
// For row r = b*next_n+t the candidates are positions p < lim, lim =
// min(seq_lens[b]-next_n+t+1, max_context) (none for empty requests).  The
// order is the float32 bit order made unsigned (negative values inverted,
// others with the sign bit set: -NaN < -inf < ... < -0 < +0 < ... < +inf <
// +NaN), equal values by ascending position.
//
// One CTA per row: a radix select, 8 bits per pass over the row, finds the
// exact key T of the K-th largest candidate (K = min(k, lim)); one more pass
// collects every key above T, and the first (in position order) of the keys
// equal to T through a block-wide scan; a bitonic sort of (key, ~position)
// pairs in shared memory gives the output order.  A row whose candidates fit
// in the rest of shared memory is read from global memory once and the five
// passes run on that copy.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace pml {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

// Keys and values stay integer bit patterns throughout: a float register can
// be canonicalised on its way (a NaN payload or sign lost), and the order
// is defined on the bits.
__device__ __forceinline__ uint32_t order_key(uint32_t b)
{
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ uint32_t key_bits(uint32_t k)
{
    return (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
}

// (key, position) packed so that a larger value means earlier in the output.
__device__ __forceinline__ unsigned long long pack_cand(uint32_t key, int p)
{
    return ((unsigned long long)key << 32) | (0xFFFFFFFFu - (uint32_t)p);
}

// The candidates' bit patterns: from the shared-memory copy of the row when
// it fits (`cached`), else from global memory.
struct RowSource {
    const uint32_t* gx;
    const uint32_t* sx;
    bool cached;
    __device__ __forceinline__ uint32_t operator()(int p) const
    {
        return cached ? sx[p] : __ldg(gx + p);
    }
};

__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkArgs a, int cache_elems)
{
    __shared__ unsigned int hist[256];
    __shared__ unsigned long long cand[kTopkMax];
    __shared__ int warp_sums[kWarps];
    __shared__ int sel[2];
    extern __shared__ uint32_t row_cache[];

    const int row = blockIdx.x;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int b = row / a.next_n, t = row % a.next_n;
    const int len = __ldg(a.seq_lens + b);
    int lim = len > 0 ? min(len - a.next_n + t + 1, a.max_context) : 0;
    if (lim < 0) lim = 0;
    const int K = min(a.k, lim);
    const uint32_t* gx =
        reinterpret_cast<const uint32_t*>(a.logits) + (long long)row * a.logits_stride;
    // one read of the row from global memory when it fits in shared memory
    const bool cached = lim <= cache_elems;
    if (cached) {
        for (int p = tid; p < lim; p += kThreads) row_cache[p] = __ldg(gx + p);
        __syncthreads();
    }
    const RowSource x{gx, row_cache, cached};

    // radix select of the K-th largest key
    uint32_t prefix = 0, mask = 0;
    int need = K;
    for (int shift = 24; shift >= 0 && K > 0; shift -= 8) {
        for (int i = tid; i < 256; i += kThreads) hist[i] = 0;
        __syncthreads();
        for (int p = tid; p < lim; p += kThreads) {
            const uint32_t key = order_key(x(p));
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (warp == 0) {
            // lane l holds bins 255-8l .. 248-8l (descending); the first lane whose
            // inclusive count reaches `need` holds the bin of the K-th largest
            unsigned c[8], s = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = hist[255 - (lane * 8 + j)];
                s += c[j];
            }
            unsigned incl = s;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, incl >= (unsigned)need);
            if (lane == __ffs(hit) - 1) {
                unsigned cum = incl - s;
                int bin = 255 - lane * 8;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (cum + c[j] >= (unsigned)need) {
                        bin = 255 - (lane * 8 + j);
                        break;
                    }
                    cum += c[j];
                }
                sel[0] = bin;
                sel[1] = (int)cum;       // candidates above this bin
            }
        }
        __syncthreads();
        need -= sel[1];
        prefix |= (uint32_t)sel[0] << shift;
        mask |= 255u << shift;
        __syncthreads();
    }

    // collect: every key above T, then the first `need` keys equal to T
    const int n_above = K - need;
    if (K > 0) {
        if (tid == 0) sel[0] = 0;
        __syncthreads();
        for (int p = tid; p < lim; p += kThreads) {
            const uint32_t key = order_key(x(p));
            if (key > prefix) cand[atomicAdd(&sel[0], 1)] = pack_cand(key, p);
        }
        int taken = 0;
        for (int base = 0; base < lim && taken < need; base += kThreads) {
            const int p = base + tid;
            const bool eq = p < lim && order_key(x(p)) == prefix;
            const unsigned bal = __ballot_sync(0xffffffffu, eq);
            if (lane == 0) warp_sums[warp] = __popc(bal);
            __syncthreads();
            int before = 0, total = 0;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const int v = warp_sums[w];
                before += w < warp ? v : 0;
                total += v;
            }
            const int rank = taken + before + __popc(bal & ((1u << lane) - 1u));
            if (eq && rank < need) cand[n_above + rank] = pack_cand(prefix, p);
            taken += total;
            __syncthreads();
        }
    }

    // bitonic sort of K entries (padded with 0, which sorts last) into
    // descending order
    int P = 1;
    while (P < K) P <<= 1;
    for (int i = K + tid; i < P; i += kThreads) cand[i] = 0ull;
    __syncthreads();
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < P / 2; i += kThreads) {
                const int lo = 2 * i - (i & (stride - 1));
                const int hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const unsigned long long u = cand[lo], v = cand[hi];
                if ((u < v) == desc) {
                    cand[lo] = v;
                    cand[hi] = u;
                }
            }
            __syncthreads();
        }
    }

    int32_t* oi = a.indices + (long long)row * a.indices_stride;
    uint32_t* ov = a.values ? reinterpret_cast<uint32_t*>(a.values) + (long long)row * a.values_stride
                            : nullptr;
    for (int i = tid; i < a.k; i += kThreads) {
        if (i < K) {
            const unsigned long long c = cand[i];
            oi[i] = (int32_t)(0xFFFFFFFFu - (uint32_t)c);
            if (ov) ov[i] = key_bits((uint32_t)(c >> 32));
        } else {
            oi[i] = -1;
            if (ov) ov[i] = 0xFF800000u;     // -inf
        }
    }
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, int rows, int smem_optin, cudaStream_t stream)
{
    // static shared memory of the kernel, plus the largest row copy that fits
    constexpr int kStatic = 256 * 4 + kTopkMax * 8 + kWarps * 4 + 8;
    const int cache_bytes = (smem_optin - kStatic - 1024) & ~15;
    const int cache_elems = cache_bytes > 0 ? cache_bytes / 4 : 0;
    static int configured_device = -1;
    static int configured_bytes = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev || configured_bytes != cache_bytes) {
        e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 cache_bytes > 0 ? cache_bytes : 0);
        if (e != cudaSuccess) return e;
        configured_device = dev;
        configured_bytes = cache_bytes;
    }
    topk_kernel<<<rows, kThreads, cache_bytes > 0 ? cache_bytes : 0, stream>>>(a, cache_elems);
    return cudaGetLastError();
}

}  // namespace pml
