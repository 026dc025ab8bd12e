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
// kSlices), as order keys: in registers, kPer a thread, when the slice has
// at most kRegKeys of them; else in shared memory when it fits, or read from
// global memory on every pass.  Every exchange
// between the CTAs is a push: a CTA stores into the others' shared memory
// (distributed shared memory) and one cluster barrier later they read it
// locally.
//   1. Radix select, 8 bits per pass from the top: each CTA histograms its
//      slice and pushes the histogram to every CTA, each CTA sums the eight
//      and finds the bin that holds the K-th largest key (K = min(k, lim)).
//      The passes stop as soon as the keys at or above that bin's lower
//      edge lo number at most K + kCapExtra -- after two passes on
//      Gaussian-like rows -- and these keys, sorted, give the answer in
//      their first K places.  Otherwise (many keys equal to the K-th one)
//      the four passes give it exactly, T; the keys above T are sorted
//      and the first keys equal to T in position order fill the rest.
//   2. The keys to sort are cut into at most 256 bins, ascending in key:
//      each top-8-bit digit that holds some of them (counted by the first
//      pass) gets a share of the bins in proportion to its count, bins of
//      equal power-of-two width over its range (from lo, or the digit's
//      start, to the digit's end or the row's largest key).  The CTAs push
//      and sum the bins' histograms, which gives each bin's place in the
//      output; the bins are dealt out in descending order to the CTAs in
//      runs of about an eighth of the keys each.  Each CTA stores every one
//      of its keys, packed with its position, into the shared memory of
//      the bin's owner at the bin's place.
//   3. After a last cluster barrier each CTA ranks the entries it received:
//      an entry's place is the number of keys in higher bins plus the
//      number of entries of its own bin that come before it (a bin holds a
//      few dozen entries on such rows).
// All CTAs of a cluster take the same path (their histograms are the
// row's), so they meet at every cluster barrier; none touches another's
// shared memory after the last, so none waits for the others to leave.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace pml {

namespace {

constexpr int kSlices = 8;          // CTAs per row (a portable cluster size)
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 256;          // radix digits; bins of the keys to sort
constexpr int kCapExtra = 256;      // keys past K a row may take into the sort
constexpr int kPer = 16;            // keys a thread holds in registers
constexpr int kRegKeys = kPer * kThreads;   // the largest slice held in registers

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

// Bin of a key to sort (key >= lo): its digit D = key >> 24 has bins from
// first[D] = info[D] & 0xFFFF on, each 2^(info[D] >> 16) keys wide from
// base[D].
__device__ __forceinline__ int key_bin(uint32_t key, const uint32_t* base, const int* info)
{
    const int d = (int)(key >> 24), i = info[d];
    return (i & 0xFFFF) + (int)((unsigned long long)(key - base[d]) >> (i >> 16));
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster arrives; shared-memory writes
// before it (local or into another CTA) are visible to the cluster after it.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Address of the shared-memory location `local` (a shared-window address of
// this CTA) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t remote_addr(uint32_t local, uint32_t rank)
{
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local), "r"(rank));
    return ra;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint4 v)
{
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void st_cluster_u64(uint32_t addr, unsigned long long v)
{
    asm volatile("st.shared::cluster.u64 [%0], %1;" :: "r"(addr), "l"(v) : "memory");
}

// The slice's order keys: from the shared-memory copy when it fits
// (`cached`), else converted from global memory.
struct SliceKeys {
    const uint32_t* gx;    // the row, position 0
    const uint32_t* sk;    // the copy, slice position 0
    int s0;
    bool cached;
    __device__ __forceinline__ uint32_t operator()(int p) const
    {
        return cached ? sk[p - s0] : order_key(__ldg(gx + p));
    }
};

// Calls f(key, p) for every key of the slice [s0, s1): from the registers
// (key u of thread t at position s0 + u*kThreads + t) when the slice fits
// them, else from `x`, kPer keys per thread loaded before any is visited.
template <bool kRegs, typename F>
__device__ __forceinline__ void visit_keys(const uint32_t (&reg)[kPer], const SliceKeys& x, int s0,
                                           int s1, F&& f)
{
    const int tid = threadIdx.x;
    if constexpr (kRegs) {
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int p = s0 + u * kThreads + tid;
            if (p < s1) f(reg[u], p);
        }
    } else {
        for (int p0 = s0; p0 < s1; p0 += kRegKeys) {
            uint32_t v[kPer];
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int p = p0 + u * kThreads + tid;
                v[u] = p < s1 ? x(p) : 0u;
            }
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int p = p0 + u * kThreads + tid;
                if (p < s1) f(v[u], p);
            }
        }
    }
}

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

// This CTA's 256-bin histogram into row `rank` of inbox `box` (a shared-window
// address) of every CTA of the cluster: thread t stores 16 bytes into two
// CTAs.
__device__ __forceinline__ void push_hist(const uint32_t* hist, uint32_t box, uint32_t rank)
{
    const int tid = threadIdx.x, part = tid & 63, c0 = 2 * (tid >> 6);
    const uint4 v = reinterpret_cast<const uint4*>(hist)[part];
    const uint32_t local = box + (rank * kBins + 4 * part) * 4;
    st_cluster_v4(remote_addr(local, (uint32_t)c0), v);
    st_cluster_v4(remote_addr(local, (uint32_t)c0 + 1), v);
}

// kRegs: the slice (at most kRegKeys keys) is held in registers; else in
// shared memory when it fits (cache_elems), or read from global memory.
template <bool kRegs>
__global__ void __launch_bounds__(kThreads, 4) topk_kernel(const TopkArgs a, int cache_elems, int cap)
{
    __shared__ __align__(16) uint32_t inbox[2][kSlices][kBins];   // the slices' histograms
    __shared__ __align__(16) uint32_t hist[kBins];   // this CTA's histogram, then the bins' slot counters
    __shared__ int abv[kBins];        // summed histogram (radix passes); keys in higher bins (sort)
    __shared__ int dest[kBins];       // a bin's owner << 24 | where this CTA's keys of it go there
    int* const h1 = dest;             // before it: the row's first-pass histogram
    __shared__ uint32_t dbase[kBins];  // per digit: lowest key of its bins
    __shared__ int dinfo[kBins];       // per digit: first bin | bin width bits << 16
    __shared__ uint32_t eq_in[kSlices];   // the slices' counts of keys equal to T
    __shared__ uint32_t max_in[kSlices];  // the slices' largest keys
    __shared__ uint32_t wmax[kWarps];
    __shared__ int sel[3];
    __shared__ int span[2];
    __shared__ int scan_buf[kWarps];
    extern __shared__ __align__(16) uint8_t dyn[];
    // dynamic: the received entries (cap), the slice's keys (cache_elems)
    unsigned long long* recv = reinterpret_cast<unsigned long long*>(dyn);
    uint32_t* sk = reinterpret_cast<uint32_t*>(recv + cap);

    const int row = blockIdx.x / kSlices;
    const uint32_t rank = cluster_rank();
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int b = row / a.next_n, t = row % a.next_n;
    const int len = __ldg(a.seq_lens + b);
    int lim = len > 0 ? min(len - a.next_n + t + 1, a.max_context) : 0;
    if (lim < 0) lim = 0;
    const int K = min(a.k, lim);
    int32_t* oi = a.indices + (long long)row * a.indices_stride;
    uint32_t* ov = a.values ? reinterpret_cast<uint32_t*>(a.values) + (long long)row * a.values_stride
                            : nullptr;
    if (rank == 0) {
        for (int i = K + tid; i < a.k; i += kThreads) {
            oi[i] = -1;
            if (ov) ov[i] = 0xFF800000u;     // -inf
        }
    }
    if (K == 0) return;                      // the whole cluster: no barrier follows

    const int chunk = (lim + kSlices - 1) / kSlices;
    const int s0 = min(lim, (int)rank * chunk), s1 = min(lim, s0 + chunk);
    const uint32_t* gx =
        reinterpret_cast<const uint32_t*>(a.logits) + (long long)row * a.logits_stride;
    const bool cached = !kRegs && chunk <= cache_elems;
    const uint32_t box0 = smem_addr(&inbox[0][0][0]);

    // ------------------------------------------------ the slice's keys and the first histogram
    hist[tid] = 0u;
    __syncthreads();
    uint32_t kmax = 0u;
    uint32_t reg[kPer];
    if constexpr (kRegs) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int u = h * 8; u < h * 8 + 8; ++u) {
                const int p = s0 + u * kThreads + tid;
                reg[u] = p < s1 ? order_key(__ldg(gx + p)) : 0u;
            }
#pragma unroll
            for (int u = h * 8; u < h * 8 + 8; ++u) {
                if (s0 + u * kThreads + tid < s1) {
                    kmax = max(kmax, reg[u]);
                    atomicAdd(&hist[reg[u] >> 24], 1u);
                }
            }
        }
    } else {
        for (int p0 = s0; p0 < s1; p0 += 8 * kThreads) {
            uint32_t v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int p = p0 + u * kThreads + tid;
                v[u] = p < s1 ? __ldg(gx + p) : 0u;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int p = p0 + u * kThreads + tid;
                if (p < s1) {
                    const uint32_t key = order_key(v[u]);
                    if (cached) sk[p - s0] = key;
                    kmax = max(kmax, key);
                    atomicAdd(&hist[key >> 24], 1u);
                }
            }
        }
    }
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    if (lane == 0) wmax[warp] = kmax;
    const SliceKeys x{gx, sk, s0, cached};

    // ------------------------------------------------ 1. radix select
    uint32_t prefix = 0, mask = 0;
    int need = K;           // keys still to take from the current bin
    int box = 0;
    int shift = 24;
    bool sort_all = false;  // the keys at or above the bin's lower edge are few enough
    int bin_count = 0;
    for (;;) {
        if (shift != 24) {
            visit_keys<kRegs>(reg, x, s0, s1, [&](uint32_t key, int) {
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
            });
        }
        __syncthreads();
        push_hist(hist, box0 + box * kSlices * kBins * 4, rank);
        if (shift == 24 && tid < kSlices) {
            uint32_t m = 0u;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) m = max(m, wmax[w]);
            st_cluster_u32(remote_addr(smem_addr(&max_in[rank]), (uint32_t)tid), m);
        }
        cluster_sync();
        {
            uint32_t m = 0;
#pragma unroll
            for (int r = 0; r < kSlices; ++r) m += inbox[box][r][tid];
            abv[tid] = (int)m;
            if (shift == 24) h1[tid] = (int)m;
            hist[tid] = 0u;
        }
        __syncthreads();
        if (warp == 0) {
            // lane l sums bins 255-8l .. 248-8l (descending); the first lane
            // whose inclusive count reaches `need` holds the bin of the K-th
            // largest
            unsigned c[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) c[j] = (unsigned)abv[255 - (lane * 8 + j)];
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
                int bin = 255 - lane * 8, cnt = (int)c[0];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (cum + c[j] >= (unsigned)need) {
                        bin = 255 - (lane * 8 + j);
                        cnt = (int)c[j];
                        break;
                    }
                    cum += c[j];
                }
                sel[0] = bin;
                sel[1] = (int)cum;       // keys above this bin
                sel[2] = cnt;            // keys in it
            }
        }
        __syncthreads();
        need -= sel[1];
        prefix |= (uint32_t)sel[0] << shift;
        mask |= 255u << shift;
        box ^= 1;
        bin_count = sel[2];
        if (K - need + bin_count <= cap) {
            sort_all = true;
            break;
        }
        if (shift == 0) break;           // T = prefix exactly
        shift -= 8;
    }
    // The keys to sort: key >= lo.  With sort_all lo is the bin's lower
    // edge (its low bits are zero); else the keys above T = prefix, and the
    // first `need` keys equal to T are placed by position.
    const uint32_t T = prefix;
    const bool any = sort_all || T != 0xFFFFFFFFu;
    const uint32_t lo = sort_all ? T : T + 1u;

    // ------------------------------------------------ 2. bins, exchange, scatter
    {
        // thread tid takes digit tid: its keys to sort, c (digits above lo's
        // from the first pass, lo's digit the rest), its share of the bins
        const int cand = sort_all ? K - need + bin_count : K - need;
        const int dlo = any ? (int)(lo >> 24) : kBins;
        int c = tid > dlo ? h1[tid] : 0, above_dlo;
        (void)block_exclusive_scan(c, scan_buf, above_dlo);
        if (tid == dlo) c = cand - above_dlo;
        const int nz = __syncthreads_count(c > 0);
        int used = 0, width = 0;
        uint32_t base = 0u;
        if (c > 0) {
            uint32_t top = 0u;
#pragma unroll
            for (int r = 0; r < kSlices; ++r) top = max(top, max_in[r]);
            top = min(top, ((uint32_t)tid << 24) | 0xFFFFFFu);
            base = max(lo, (uint32_t)tid << 24);
            // at most `share` bins of width 2^width: the least width with
            // (span - 1) >> width < share
            const long long share = max(1LL, (long long)c * (kBins - nz) / cand);
            const unsigned long long last = (unsigned long long)(top - base);   // span - 1
            if ((long long)last >= share) {
                width = (64 - __clzll((long long)last)) - (64 - __clzll(share));
                width += (long long)(last >> width) >= share ? 1 : 0;
            }
            used = (int)(last >> width) + 1;
        }
        int nbins;
        const int first = block_exclusive_scan(used, scan_buf, nbins);
        dbase[tid] = base;
        dinfo[tid] = first | (width << 16);
        __syncthreads();
    }
    int n_eq = 0;
    visit_keys<kRegs>(reg, x, s0, s1, [&](uint32_t key, int) {
        if (any && key >= lo) atomicAdd(&hist[key_bin(key, dbase, dinfo)], 1u);
        n_eq += key == T ? 1 : 0;
    });
    int eq_me = 0;
    if (!sort_all) (void)block_exclusive_scan(n_eq, scan_buf, eq_me);
    __syncthreads();
    push_hist(hist, box0 + box * kSlices * kBins * 4, rank);
    if (!sort_all && tid < kSlices)
        st_cluster_u32(remote_addr(smem_addr(&eq_in[rank]), (uint32_t)tid), (uint32_t)eq_me);
    cluster_sync();

    // thread tid takes bin kBins-1-tid, so that a block scan runs over the
    // bins in descending order
    int total, target;
    {
        const int bn = kBins - 1 - tid;
        int m = 0, before_me = 0;
#pragma unroll
        for (int r = 0; r < kSlices; ++r) {
            const int c = (int)inbox[box][r][bn];
            m += c;
            before_me += r < (int)rank ? c : 0;
        }
        const int above = block_exclusive_scan(m, scan_buf, total);
        target = (total + kSlices - 1) / kSlices;
        const int owner = target ? min(kSlices - 1, above / target) : 0;
        abv[bn] = above;
        dest[bn] = (owner << 24) | (above - owner * target + before_me);
        hist[bn] = 0u;
        if (tid == 0) {
            span[0] = cap;               // no entries: an empty range
            span[1] = 0;
        }
        __syncthreads();
        if (m > 0 && owner == (int)rank) {
            atomicMin(&span[0], above - owner * target);
            atomicMax(&span[1], above - owner * target + m);
        }
    }
    const uint32_t recv0 = smem_addr(recv);
    if (any) {
        visit_keys<kRegs>(reg, x, s0, s1, [&](uint32_t key, int p) {
            if (key >= lo) {
                const int bn = key_bin(key, dbase, dinfo);
                const int slot = (int)atomicAdd(&hist[bn], 1u);
                const int d = dest[bn];
                st_cluster_u64(remote_addr(recv0 + 8u * (uint32_t)((d & 0xFFFFFF) + slot), (uint32_t)(d >> 24)),
                               pack_cand(key, p));
            }
        });
    }
    if (!sort_all) {
        // the first `need` keys equal to T, in position order over the
        // slices, take places K-need .. K-1: thread tid walks the contiguous
        // positions [q0, q1) (read through `x`: from global memory when the
        // slice is in registers) and finds its keys' places from a block scan
        int eq_before = 0;
#pragma unroll
        for (int r = 0; r < kSlices; ++r) eq_before += r < (int)rank ? (int)eq_in[r] : 0;
        const int take = max(0, min(eq_me, need - eq_before));
        if (take > 0) {
            const int per = (s1 - s0 + kThreads - 1) / kThreads;
            const int q0 = min(s1, s0 + tid * per), q1 = min(s1, q0 + per);
            int ne = 0;
            for (int p = q0; p < q1; ++p) ne += x(p) == T ? 1 : 0;
            int te;
            int ie = block_exclusive_scan(ne, scan_buf, te);
            for (int p = q0; p < q1 && ie < take; ++p) {
                if (x(p) == T) {
                    const int rk = K - need + eq_before + ie;
                    oi[rk] = p;
                    if (ov) ov[rk] = key_bits(T);
                    ++ie;
                }
            }
        }
    }
    cluster_sync();

    // ------------------------------------------------ 3. rank the received entries
    for (int i = span[0] + tid; i < span[1]; i += kThreads) {
        const unsigned long long e = recv[i];
        const uint32_t key = (uint32_t)(e >> 32);
        const int bn = key_bin(key, dbase, dinfo);
        const int first = abv[bn] - (int)rank * target;
        const int n = (bn == 0 ? total : abv[bn - 1]) - abv[bn];
        int before = 0;
        for (int j = first; j < first + n; ++j) before += recv[j] > e ? 1 : 0;
        const int rk = abv[bn] + before;
        if (rk < K) {
            oi[rk] = (int32_t)(0xFFFFFFFFu - (uint32_t)e);
            if (ov) ov[rk] = key_bits(key);
        }
    }
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, int rows, int smem_optin, cudaStream_t stream)
{
    // dynamic shared memory: the received entries (k + kCapExtra) and the
    // largest slice copy that fits under a budget that keeps four CTAs on an
    // SM (k <= 2048; beyond, enough for a 32768-position row's slice) --
    // larger slices are read from global memory on every pass
    const int cap = a.k + kCapExtra;
    const size_t entries = (size_t)cap * 8;
    const long long chunk = ((long long)a.max_context + kSlices - 1) / kSlices;
    const bool regs = chunk <= kRegKeys;
    long long cache_elems = 0;
    if (!regs) {
        const size_t budget = entries <= 20 * 1024 ? 36 * 1024 : entries + 16 * 1024;
        cache_elems = (long long)(budget - entries) / 4;
        if (cache_elems > chunk) cache_elems = chunk;
    }
    const size_t smem = entries + (size_t)cache_elems * 4;
    if (smem + 24 * 1024 > (size_t)smem_optin) return cudaErrorInvalidConfiguration;
    void (*kernel)(const TopkArgs, int, int) = regs ? topk_kernel<true> : topk_kernel<false>;
    static int configured_device[2] = {-1, -1};
    static size_t configured_bytes[2] = {0, 0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device[regs] != dev || configured_bytes[regs] < smem) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured_device[regs] = dev;
        configured_bytes[regs] = smem;
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
    e = cudaLaunchKernelEx(&cfg, kernel, a, (int)cache_elems, cap);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace pml
