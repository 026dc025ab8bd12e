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
// A row is one cluster of kSlices CTAs; CTA s of the cluster holds the
// slice [s*chunk, min(lim, (s+1)*chunk)) of the row, chunk = ceil(lim /
// kSlices), in shared memory when it fits.
//   1. Radix select of the exact key T of the K-th largest candidate (K =
//      min(k, lim)), 8 bits per pass: each CTA histograms its slice, and
//      every CTA sums the kSlices histograms through distributed shared
//      memory (two histogram buffers, alternating, so one cluster barrier
//      per pass suffices).
//   2. Each CTA counts its keys above T and equal to T; after an exchange of
//      the counts it knows where its candidates go: all its keys above T,
//      and the first ones equal to T in position order that the slices
//      before it left over (K - #above in all).
//   3. Each CTA sorts its candidates, (key, ~position) descending, in its own
//      shared memory; after a cluster barrier it copies every other CTA's
//      sorted list next to its own and places each of its candidates at its
//      rank: its index in its own list plus, for every other list, the
//      number of entries there that come before it (binary search).
//      Candidates are distinct, so the ranks are a permutation of 0..K-1.
// Every CTA of a cluster takes the same path (K is the row's), so they all
// meet at every cluster barrier; the last one keeps each CTA's shared memory
// alive until the others are done reading it.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace pml {

namespace {

constexpr int kSlices = 8;          // CTAs per row (a portable cluster size)
constexpr int kThreads = 256;
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

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster arrives; shared-memory writes
// before it are visible to the cluster after it.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t remote_addr(const void* local, uint32_t rank)
{
    uint32_t la = static_cast<uint32_t>(__cvta_generic_to_shared(local)), ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
    return ra;
}

// Loads from another CTA's shared memory.  They carry no memory clobber, so
// that several can be in flight at once; being volatile they stay after the
// cluster barrier that precedes them, and a later write of this CTA's own
// shared memory does not alias anything they read.
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint4 ld_cluster_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ unsigned long long ld_cluster_u64(uint32_t addr)
{
    unsigned long long v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr));
    return v;
}

// The slice's candidates: from the shared-memory copy when it fits
// (`cached`), else from global memory.
struct SliceSource {
    const uint32_t* gx;    // the row, position 0
    const uint32_t* sx;    // the copy, slice position 0
    int s0;
    bool cached;
    __device__ __forceinline__ uint32_t operator()(int p) const
    {
        return cached ? sx[p - s0] : __ldg(gx + p);
    }
};

// Block-wide exclusive scan of one int per thread (kThreads threads); also
// returns the total.  Uses `buf` (kWarps ints).
__device__ __forceinline__ int block_exclusive_scan(int v, int* buf, int& total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) buf[warp] = incl;
    __syncthreads();
    int before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const int s = buf[w];
        before += w < warp ? s : 0;
        total += s;
    }
    __syncthreads();
    return before + incl - v;
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkArgs a, int cache_elems, int sort_cap)
{
    __shared__ __align__(16) unsigned int hist[2][256];
    __shared__ __align__(16) unsigned int merged[256];            // the slices' histograms summed
    __shared__ int slice_counts[4][kSlices];                      // counts[] of every slice
    __shared__ int counts[4];        // {above T, equal to T, list offset, list length} of this CTA
    __shared__ int sel[2];
    __shared__ int scan_buf[kWarps];
    extern __shared__ __align__(16) uint8_t dyn[];
    // dynamic: the sorted list (sort_cap entries), every CTA's lists
    // (k entries), the slice copy (cache_elems)
    unsigned long long* own = reinterpret_cast<unsigned long long*>(dyn);
    unsigned long long* all = own + sort_cap;
    uint32_t* slice_copy = reinterpret_cast<uint32_t*>(all + a.k);

    const int row = blockIdx.x / kSlices;
    const uint32_t rank = cluster_rank();
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int b = row / a.next_n, t = row % a.next_n;
    const int len = __ldg(a.seq_lens + b);
    int lim = len > 0 ? min(len - a.next_n + t + 1, a.max_context) : 0;
    if (lim < 0) lim = 0;
    const int K = min(a.k, lim);
    const int chunk = (lim + kSlices - 1) / kSlices;
    const int s0 = min(lim, (int)rank * chunk), s1 = min(lim, s0 + chunk);
    const uint32_t* gx =
        reinterpret_cast<const uint32_t*>(a.logits) + (long long)row * a.logits_stride;
    const bool cached = chunk <= cache_elems;
    if (cached) {
        for (int p = s0 + tid; p < s1; p += kThreads) slice_copy[p - s0] = __ldg(gx + p);
    }
    const SliceSource x{gx, slice_copy, s0, cached};

    // ---------------------------------------------------------------- 1. radix select
    uint32_t prefix = 0, mask = 0;
    int need = K;
    int buf = 0;
    for (int shift = 24; shift >= 0 && K > 0; shift -= 8, buf ^= 1) {
        hist[buf][tid] = 0u;                       // kThreads == 256 bins
        merged[tid] = 0u;
        __syncthreads();
        // four positions per thread per step, loaded before any is counted
        for (int p0 = s0; p0 < s1; p0 += 4 * kThreads) {
            int bins[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int p = p0 + u * kThreads + tid;
                const uint32_t key = p < s1 ? order_key(x(p)) : 0u;
                bins[u] = (p < s1 && (key & mask) == prefix) ? (int)((key >> shift) & 255u) : -1;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (bins[u] >= 0) atomicAdd(&hist[buf][bins[u]], 1u);
        }
        __syncthreads();
        cluster_sync();
        {
            // the slices' histograms summed in this CTA: thread t adds bins
            // 8(t%32) .. 8(t%32)+7 of slice t/32 (two 16-byte remote loads per
            // thread rather than many per thread, as remote loads of one
            // thread complete one after another)
            const int r = tid >> 5, b8 = (tid & 31) * 8;
            const uint32_t src = remote_addr(&hist[buf][b8], (uint32_t)r);
            const uint4 lo = ld_cluster_v4(src), hi = ld_cluster_v4(src + 16);
            atomicAdd(&merged[b8 + 0], lo.x); atomicAdd(&merged[b8 + 1], lo.y);
            atomicAdd(&merged[b8 + 2], lo.z); atomicAdd(&merged[b8 + 3], lo.w);
            atomicAdd(&merged[b8 + 4], hi.x); atomicAdd(&merged[b8 + 5], hi.y);
            atomicAdd(&merged[b8 + 6], hi.z); atomicAdd(&merged[b8 + 7], hi.w);
        }
        __syncthreads();
        if (warp == 0) {
            // lane l sums bins 255-8l .. 248-8l over the slices (descending);
            // the first lane whose inclusive count reaches `need` holds the
            // bin of the K-th largest
            unsigned c[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) c[j] = merged[255 - (lane * 8 + j)];
            unsigned s = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) s += c[j];
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
    }
    // T = prefix; the K-th largest key; `need` keys equal to T are taken

    // ---------------------------------------------------------------- 2. this CTA's candidates
    int n_above = 0, n_equal = 0;
    if (K > 0) {
        for (int p = s0 + tid; p < s1; p += kThreads) {
            const uint32_t key = order_key(x(p));
            n_above += key > prefix;
            n_equal += key == prefix;
        }
    }
    int tot_above, tot_equal;
    (void)block_exclusive_scan(n_above, scan_buf, tot_above);
    (void)block_exclusive_scan(n_equal, scan_buf, tot_equal);
    if (tid == 0) {
        counts[0] = tot_above;
        counts[1] = tot_equal;
    }
    __syncthreads();
    cluster_sync();
    // the slices before this one: their keys above T and equal to T
    if (tid < 2 * kSlices)
        slice_counts[tid / kSlices][tid % kSlices] =
            (int)ld_cluster_u32(remote_addr(&counts[tid / kSlices], (uint32_t)(tid % kSlices)));
    __syncthreads();
    int above_before = 0, equal_before = 0;
#pragma unroll
    for (int r = 0; r < kSlices; ++r) {
        if (r < (int)rank) {
            above_before += slice_counts[0][r];
            equal_before += slice_counts[1][r];
        }
    }
    // keys equal to T taken by this slice: the first take_e of its own
    const int take_e = K > 0 ? max(0, min(tot_equal, need - equal_before)) : 0;
    const int m = K > 0 ? tot_above + take_e : 0;          // this CTA's candidates
    // its list starts after the lists of the slices before it
    const int taken_before = above_before + min(equal_before, need);
    if (K > 0 && take_e == tot_equal) {
        // every key of the slice at or above T is a candidate: any order
        // (the list is sorted next), slots handed out per warp
        if (tid == 0) sel[0] = 0;
        __syncthreads();
        for (int p0 = s0; p0 < s1; p0 += kThreads) {
            const int p = p0 + tid;
            const uint32_t key = p < s1 ? order_key(x(p)) : 0u;
            const bool c = p < s1 && key >= prefix;
            const unsigned bal = __ballot_sync(0xffffffffu, c);
            int base = 0;
            if (lane == 0 && bal) base = atomicAdd(&sel[0], __popc(bal));
            base = __shfl_sync(0xffffffffu, base, 0);
            if (c) own[base + __popc(bal & ((1u << lane) - 1u))] = pack_cand(key, p);
        }
    } else if (K > 0) {
        // only the first take_e keys equal to T, in position order: thread
        // tid takes the contiguous positions [q0, q1) and finds where its
        // keys go from two block-wide scans
        const int per = (s1 - s0 + kThreads - 1) / kThreads;
        const int q0 = min(s1, s0 + tid * per), q1 = min(s1, q0 + per);
        int na = 0, ne = 0;
        for (int p = q0; p < q1; ++p) {
            const uint32_t key = order_key(x(p));
            na += key > prefix;
            ne += key == prefix;
        }
        int ta, te;
        int ia = block_exclusive_scan(na, scan_buf, ta);
        int ie = block_exclusive_scan(ne, scan_buf, te);
        for (int p = q0; p < q1; ++p) {
            const uint32_t key = order_key(x(p));
            if (key > prefix) own[ia++] = pack_cand(key, p);
            else if (key == prefix) {
                if (ie < take_e) own[tot_above + ie] = pack_cand(key, p);
                ++ie;
            }
        }
    }
    // pad to a power of two with 0 (sorts last)
    int P = 1;
    while (P < m) P <<= 1;
    for (int i = m + tid; i < P; i += kThreads) own[i] = 0ull;
    __syncthreads();

    // ---------------------------------------------------------------- 3. sort, rank, place
    if (P <= kThreads) {
        // one entry per thread (threads past P hold 0): the same network, the
        // partner within the warp reached by a shuffle, beyond it through
        // shared memory
        unsigned long long v = tid < P ? own[tid] : 0ull;
        for (int size = 2; size <= kThreads; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                unsigned long long o;
                if (stride >= 32) {
                    __syncthreads();
                    own[tid] = v;
                    __syncthreads();
                    o = own[tid ^ stride];
                } else {
                    o = __shfl_xor_sync(0xffffffffu, v, stride);
                }
                // the lower index of a pair keeps the larger value in a
                // descending block, the smaller in an ascending one
                const bool desc = (tid & size) == 0;
                const bool lower = (tid & stride) == 0;
                v = (lower == desc) ? (v > o ? v : o) : (v < o ? v : o);
            }
        }
        __syncthreads();
        if (tid < P) own[tid] = v;
        __syncthreads();
    } else {
        for (int size = 2; size <= P; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int i = tid; i < P / 2; i += kThreads) {
                    const int lo = 2 * i - (i & (stride - 1));
                    const int hi = lo + stride;
                    const bool desc = (lo & size) == 0;
                    const unsigned long long u = own[lo], w = own[hi];
                    if ((u < w) == desc) {
                        own[lo] = w;
                        own[hi] = u;
                    }
                }
                __syncthreads();
            }
        }
    }
    if (tid == 0) {
        counts[2] = taken_before;
        counts[3] = m;
    }
    __syncthreads();
    cluster_sync();
    // every list into `all`, each at its offset (this CTA's own too)
    if (tid < 2 * kSlices)
        slice_counts[2 + tid / kSlices][tid % kSlices] =
            (int)ld_cluster_u32(remote_addr(&counts[2 + tid / kSlices], (uint32_t)(tid % kSlices)));
    __syncthreads();
    int offs[kSlices], lens[kSlices];
#pragma unroll
    for (int r = 0; r < kSlices; ++r) {
        offs[r] = slice_counts[2][r];
        lens[r] = slice_counts[3][r];
    }
    // entry j of the concatenated lists (list r holds [offs[r], offs[r] +
    // lens[r])), eight loads in flight per thread
    for (int j0 = 0; j0 < K; j0 += 8 * kThreads) {
        unsigned long long v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int j = j0 + u * kThreads + tid;
            v[u] = 0ull;
            if (j < K) {
                int r = 0;
#pragma unroll
                for (int q = 1; q < kSlices; ++q) r += j >= offs[q] ? 1 : 0;
                v[u] = ld_cluster_u64(remote_addr(own + (j - offs[r]), (uint32_t)r));
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int j = j0 + u * kThreads + tid;
            if (j < K) all[j] = v[u];
        }
    }
    __syncthreads();
    int32_t* oi = a.indices + (long long)row * a.indices_stride;
    uint32_t* ov = a.values ? reinterpret_cast<uint32_t*>(a.values) + (long long)row * a.values_stride
                            : nullptr;
    for (int i = tid; i < m; i += kThreads) {
        const unsigned long long c = own[i];
        int rk = i;
        for (int r = 0; r < kSlices; ++r) {
            if (r == (int)rank) continue;
            // entries of list r greater than c (the list is descending)
            int lo = 0, hi = lens[r];
            const unsigned long long* L = all + offs[r];
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (L[mid] > c) lo = mid + 1;
                else hi = mid;
            }
            rk += lo;
        }
        oi[rk] = (int32_t)(0xFFFFFFFFu - (uint32_t)c);
        if (ov) ov[rk] = key_bits((uint32_t)(c >> 32));
    }
    if (rank == 0) {
        for (int i = K + tid; i < a.k; i += kThreads) {
            oi[i] = -1;
            if (ov) ov[i] = 0xFF800000u;     // -inf
        }
    }
    // no CTA leaves while another may still read its shared memory
    cluster_sync();
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, int rows, int smem_optin, cudaStream_t stream)
{
    // dynamic shared memory: the sort buffer (k rounded up to a power of
    // two, at least kThreads), the lists of all slices (k), and the largest slice copy that fits
    // under a budget that keeps four CTAs on an SM (larger slices are read
    // from global memory on every pass)
    // (at least one entry per thread: the in-register sort goes through it)
    int sort_cap = kThreads;
    while (sort_cap < a.k) sort_cap <<= 1;
    const size_t lists = (size_t)(sort_cap + a.k) * 8;
    const size_t budget = 54 * 1024;
    const long long chunk = ((long long)a.max_context + kSlices - 1) / kSlices;
    long long cache_elems = budget > lists ? (long long)(budget - lists) / 4 : 0;
    if (cache_elems > chunk) cache_elems = chunk;
    const size_t smem = lists + (size_t)cache_elems * 4;
    if (smem + 4 * 1024 > (size_t)smem_optin) return cudaErrorInvalidConfiguration;
    static int configured_device = -1;
    static size_t configured_bytes = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev || configured_bytes < smem) {
        e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured_device = dev;
        configured_bytes = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows * kSlices);
    cfg.blockDim = dim3((unsigned)kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSlices;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, topk_kernel, a, (int)cache_elems, sort_cap);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace pml
