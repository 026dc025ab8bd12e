// C ABI of libpml.so (declared in include/pml.h): argument checks, TMA tensor
// map encoding, grid / pipeline sizing and kernel launches.  No allocation,
// no synchronisation except in pml_device_status.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "pml.h"

namespace {

using namespace pml;

constexpr int kMaxDevices = 64;
constexpr int kMaxFp8Stages = 12;
constexpr int kMaxBf16Stages = 8;
constexpr int kMaxMxfp4Stages = 24;

thread_local int g_last_cuda_error = 0;

// Sticky per-device status word written by the kernels (PML_STATUS_* bits).
__device__ unsigned int g_device_status;

std::mutex g_mutex;
int g_sm_count[kMaxDevices];
int g_smem_optin[kMaxDevices];
unsigned int* g_status_ptr[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int cuda_fail(cudaError_t e)
{
    g_last_cuda_error = static_cast<int>(e);
    return PML_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct DeviceInfo {
    int device, sm_count, smem_optin;
    unsigned int* status;
};

// Device properties and the status word's device address, looked up once per
// device with that device current.
cudaError_t device_info(DeviceInfo& d)
{
    cudaError_t e = cudaGetDevice(&d.device);
    if (e != cudaSuccess) return e;
    if (d.device < 0 || d.device >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_status_ptr[d.device] == nullptr) {
        int sms = 0, optin = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d.device);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d.device);
        if (e != cudaSuccess) return e;
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_device_status);
        if (e != cudaSuccess) return e;
        g_sm_count[d.device] = sms;
        g_smem_optin[d.device] = optin;
        g_status_ptr[d.device] = static_cast<unsigned int*>(ptr);
    }
    d.sm_count = g_sm_count[d.device];
    d.smem_optin = g_smem_optin[d.device];
    d.status = g_status_ptr[d.device];
    return cudaSuccess;
}

cudaError_t encoder(PFN_cuTensorMapEncodeTiled_v12000& fn)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_encode == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e =
            cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || p == nullptr) return cudaErrorSymbolNotFound;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    fn = g_encode;
    return cudaSuccess;
}

// Tiled map: dims/strides innermost first, strides in bytes for dimensions 1.. .
cudaError_t encode_tiled(CUtensorMap& map, CUtensorMapDataType dtype, int rank, const void* base,
                         const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                         CUtensorMapSwizzle swizzle)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn;
    cudaError_t e = encoder(fn);
    if (e != cudaSuccess) return e;
    const uint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(&map, dtype, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The same with the 128-byte swizzle.
cudaError_t encode_sw128(CUtensorMap& map, CUtensorMapDataType dtype, int rank, const void* base,
                         const uint64_t* dims, const uint64_t* strides, const uint32_t* box)
{
    return encode_tiled(map, dtype, rank, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

extern "C" {

int pml_version(void) { return 101; }

const char* pml_error_string(int code)
{
    switch (code) {
    case PML_OK: return "ok";
    case PML_ERR_INVALID_ARG: return "invalid argument";
    case PML_ERR_UNSUPPORTED: return "unsupported shape";
    case PML_ERR_ALIGNMENT: return "misaligned pointer or stride";
    case PML_ERR_CUDA: return "CUDA error";
    default: return "unknown error code";
    }
}

int pml_last_cuda_error(void) { return g_last_cuda_error; }

int pml_default_num_ctas(int device)
{
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
    return sms;
}

int pml_schedule_meta_elems(int num_ctas) { return num_ctas < 0 ? 0 : (num_ctas + 1) * 2; }

int pml_min_block_table_width(int max_seq_len)
{
    return max_seq_len <= 0 ? 0 : (max_seq_len + kBlockKeys - 1) / kBlockKeys;
}

int pml_padded_seq_len(int max_seq_len)
{
    return pml_min_block_table_width(max_seq_len) * kBlockKeys;
}

int pml_schedule(const int32_t* seq_lens, int batch, int next_n, int num_ctas,
                 int32_t* schedule_meta, void* stream)
{
    if (batch < 0 || num_ctas <= 0 || schedule_meta == nullptr) return PML_ERR_INVALID_ARG;
    if (batch > 0 && seq_lens == nullptr) return PML_ERR_INVALID_ARG;
    if (next_n < 1 || next_n > 4) return PML_ERR_UNSUPPORTED;
    if (!aligned(seq_lens, 4) || !aligned(schedule_meta, 4)) return PML_ERR_ALIGNMENT;
    cudaError_t e = launch_schedule(seq_lens, batch, num_ctas, schedule_meta,
                                    static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PML_OK : cuda_fail(e);
}

int pml_fp8_paged_mqa_logits(const uint8_t* q, const uint8_t* kv_fused, int64_t num_blocks,
                             const float* weights, const int32_t* seq_lens,
                             const int32_t* block_table, int64_t bt_stride,
                             const int32_t* schedule_meta, int num_ctas, float* out,
                             int64_t out_stride, int max_context, int batch, int next_n,
                             int num_heads, void* stream)
{
    return pml_fp8_paged_mqa_logits_ex(q, kv_fused, num_blocks, weights, seq_lens, block_table,
                                       bt_stride, schedule_meta, num_ctas, out, out_stride,
                                       PML_DTYPE_FLOAT32, max_context, batch, next_n, num_heads,
                                       stream);
}

}  // extern "C"

namespace {

// The fp8 logits call with the longest wait of any role and, for tests, a
// stage the producer leaves unpublished (-1: none).
int fp8_logits_call(const uint8_t* q, const uint8_t* kv_fused, int64_t num_blocks,
                    const float* weights, const int32_t* seq_lens, const int32_t* block_table,
                    int64_t bt_stride, const int32_t* schedule_meta, int num_ctas, void* out,
                    int64_t out_stride, int output_dtype, int max_context, int batch, int next_n,
                    int num_heads, void* stream, unsigned long long wait_limit_ns, int drop_stage)
{
    if (batch < 0 || num_ctas < 0) return PML_ERR_INVALID_ARG;
    if (output_dtype != PML_DTYPE_FLOAT32 && output_dtype != PML_DTYPE_BFLOAT16)
        return PML_ERR_UNSUPPORTED;
    const int out_bytes = output_dtype == PML_DTYPE_BFLOAT16 ? 2 : 4;
    if (next_n < 1 || next_n > 4) return PML_ERR_UNSUPPORTED;
    if (num_heads != 8 && num_heads != 16 && num_heads != 32 && num_heads != 64)
        return PML_ERR_UNSUPPORTED;
    if (batch == 0) return PML_OK;
    if (!q || !kv_fused || !weights || !seq_lens || !block_table || !out) return PML_ERR_INVALID_ARG;
    if (num_blocks < 1 || num_blocks > 0x7fffffffLL) return PML_ERR_INVALID_ARG;
    if (max_context < 1 || out_stride < max_context) return PML_ERR_INVALID_ARG;
    if (bt_stride < pml_min_block_table_width(max_context)) return PML_ERR_INVALID_ARG;
    const long long rows_total = (long long)batch * next_n * num_heads;
    if (rows_total > 0x7fffffffLL) return PML_ERR_INVALID_ARG;
    if (schedule_meta != nullptr && num_ctas == 0) return PML_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(kv_fused, 16) || !aligned(weights, 16) || !aligned(out, out_bytes) ||
        !aligned(seq_lens, 4) || !aligned(block_table, 4) || !aligned(schedule_meta, 4))
        return PML_ERR_ALIGNMENT;

    DeviceInfo dev;
    cudaError_t e = device_info(dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (num_ctas == 0) num_ctas = dev.sm_count;

    Fp8Args a;
    a.seq_lens = seq_lens;
    a.block_table = block_table;
    a.schedule_meta = schedule_meta;
    a.weights = weights;
    a.kv_fused = kv_fused;
    a.out = out;
    a.out_bf16 = output_dtype == PML_DTYPE_BFLOAT16 ? 1 : 0;
    a.status = dev.status;
    a.bt_stride = bt_stride;
    a.out_stride = out_stride;
    a.num_blocks = num_blocks;
    a.batch = batch;
    a.next_n = next_n;
    a.max_context = max_context;
    a.wait_limit_ns = wait_limit_ns;
    a.drop_stage = drop_stage;
    const int n_pad = (next_n * num_heads + 15) / 16 * 16;
    a.q_box_rows = (int)(rows_total < n_pad ? rows_total : n_pad);
    const size_t fixed = fp8_smem_bytes(next_n, num_heads, 0);
    const size_t per_stage = fp8_smem_bytes(next_n, num_heads, 1) - fixed;
    int stages = (int)(((size_t)dev.smem_optin - fixed) / per_stage);
    if (stages > kMaxFp8Stages) stages = kMaxFp8Stages;
    // an even count: the kernel's two producers take the stages in turn
    stages &= ~1;
    if (stages < 2) return PML_ERR_UNSUPPORTED;
    a.stages = stages;

    CUtensorMap kmap, qmap;
    {
        const uint64_t dims[3] = {(uint64_t)kHeadDim, (uint64_t)kBlockKeys, (uint64_t)num_blocks};
        const uint64_t strides[2] = {(uint64_t)kHeadDim, (uint64_t)kFp8BlockBytes};
        const uint32_t box[3] = {(uint32_t)kHeadDim, (uint32_t)kBlockKeys, 1};
        e = encode_sw128(kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, kv_fused, dims, strides, box);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    {
        const uint64_t dims[2] = {(uint64_t)kHeadDim, (uint64_t)rows_total};
        const uint64_t strides[1] = {(uint64_t)kHeadDim};
        const uint32_t box[2] = {(uint32_t)kHeadDim, (uint32_t)a.q_box_rows};
        e = encode_sw128(qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, q, dims, strides, box);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    e = launch_fp8_logits(num_heads, kmap, qmap, a, num_ctas, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PML_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

int pml_fp8_paged_mqa_logits_ex(const uint8_t* q, const uint8_t* kv_fused, int64_t num_blocks,
                                const float* weights, const int32_t* seq_lens,
                                const int32_t* block_table, int64_t bt_stride,
                                const int32_t* schedule_meta, int num_ctas, void* out,
                                int64_t out_stride, int output_dtype, int max_context, int batch,
                                int next_n, int num_heads, void* stream)
{
    return fp8_logits_call(q, kv_fused, num_blocks, weights, seq_lens, block_table, bt_stride,
                           schedule_meta, num_ctas, out, out_stride, output_dtype, max_context,
                           batch, next_n, num_heads, stream, kWaitLimitNs, -1);
}

int pml_fp8_paged_mqa_logits_wait_test(const uint8_t* q, const uint8_t* kv_fused,
                                       int64_t num_blocks, const float* weights,
                                       const int32_t* seq_lens, const int32_t* block_table,
                                       int64_t bt_stride, float* out, int64_t out_stride,
                                       int max_context, int batch, int next_n, int num_heads,
                                       int drop_stage, int64_t wait_limit_us, void* stream)
{
    if (drop_stage < 0 || wait_limit_us < 1 || wait_limit_us > 1000000) return PML_ERR_INVALID_ARG;
    return fp8_logits_call(q, kv_fused, num_blocks, weights, seq_lens, block_table, bt_stride,
                           nullptr, 0, out, out_stride, PML_DTYPE_FLOAT32, max_context, batch,
                           next_n, num_heads, stream,
                           (unsigned long long)wait_limit_us * 1000ull, drop_stage);
}

int pml_fp4_paged_mqa_logits(const uint8_t* q, const uint8_t* q_sf, const uint8_t* kv_cache,
                             int64_t num_blocks, const float* weights, const int32_t* seq_lens,
                             const int32_t* block_table, int64_t bt_stride,
                             const int32_t* schedule_meta, int num_ctas, void* out,
                             int64_t out_stride, int output_dtype, int max_context, int batch,
                             int next_n, void* stream)
{
    if (batch < 0 || num_ctas < 0) return PML_ERR_INVALID_ARG;
    if (output_dtype != PML_DTYPE_FLOAT32 && output_dtype != PML_DTYPE_BFLOAT16)
        return PML_ERR_UNSUPPORTED;
    if (next_n < 1 || next_n > 4) return PML_ERR_UNSUPPORTED;
    if (batch == 0) return PML_OK;
    if (batch > 65535) return PML_ERR_UNSUPPORTED;
    if (!q || !q_sf || !kv_cache || !weights || !seq_lens || !block_table || !out)
        return PML_ERR_INVALID_ARG;
    if (num_blocks < 1 || num_blocks > 0x7fffffffLL) return PML_ERR_INVALID_ARG;
    if (max_context < 1 || out_stride < max_context) return PML_ERR_INVALID_ARG;
    if (bt_stride < pml_min_block_table_width(max_context)) return PML_ERR_INVALID_ARG;
    if (schedule_meta != nullptr && num_ctas == 0) return PML_ERR_INVALID_ARG;
    const int out_bytes = output_dtype == PML_DTYPE_BFLOAT16 ? 2 : 4;
    if (!aligned(q, 16) || !aligned(q_sf, 16) || !aligned(kv_cache, 16) || !aligned(weights, 16) ||
        !aligned(seq_lens, 4) || !aligned(block_table, 4) || !aligned(out, out_bytes) ||
        !aligned(schedule_meta, 4))
        return PML_ERR_ALIGNMENT;
    DeviceInfo dev;
    cudaError_t e = device_info(dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (num_ctas == 0) num_ctas = dev.sm_count;

    Mxfp4Args a;
    a.q = q;
    a.q_sf = q_sf;
    a.weights = weights;
    a.kv = kv_cache;
    a.seq_lens = seq_lens;
    a.block_table = block_table;
    a.schedule_meta = schedule_meta;
    a.out = out;
    a.status = dev.status;
    a.bt_stride = bt_stride;
    a.out_stride = out_stride;
    a.num_blocks = num_blocks;
    a.batch = batch;
    a.next_n = next_n;
    a.slot0 = 0;
    a.max_context = max_context;
    a.out_bf16 = output_dtype == PML_DTYPE_BFLOAT16 ? 1 : 0;
    // as many staging slots as fit, for a one-slot and a two-slot pass
    for (int nn = 1; nn <= 2; ++nn) {
        const size_t fixed = mxfp4_smem_bytes(nn, 0);
        const size_t per_stage = mxfp4_smem_bytes(nn, 1) - fixed;
        if ((size_t)dev.smem_optin < fixed + 2 * per_stage) return PML_ERR_UNSUPPORTED;
        int stages = (int)(((size_t)dev.smem_optin - fixed) / per_stage);
        if (stages > kMaxMxfp4Stages) stages = kMaxMxfp4Stages;
        (nn == 1 ? a.stages : a.stages2) = stages;
    }
    // the codes of block P: 64 rows of 64 bytes at P * 4352; the query rows:
    // 64 bytes each, 64 (one slot's heads) per copy; both land with the
    // 64-byte swizzle the MMA reads
    CUtensorMap kmap, qmap;
    {
        const uint64_t dims[3] = {(uint64_t)kHeadDim / 2, (uint64_t)kBlockKeys, (uint64_t)num_blocks};
        const uint64_t strides[2] = {(uint64_t)kHeadDim / 2, (uint64_t)kMxfp4BlockBytes};
        const uint32_t box[3] = {(uint32_t)kHeadDim / 2, (uint32_t)kBlockKeys, 1};
        e = encode_tiled(kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, kv_cache, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_64B);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    {
        const uint64_t dims[2] = {(uint64_t)kHeadDim / 2, (uint64_t)batch * next_n * kMxfp4Heads};
        const uint64_t strides[1] = {(uint64_t)kHeadDim / 2};
        const uint32_t box[2] = {(uint32_t)kHeadDim / 2, (uint32_t)kMxfp4Heads};
        e = encode_tiled(qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, q, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_64B);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    e = launch_mxfp4_logits(kmap, qmap, a, num_ctas, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PML_OK : cuda_fail(e);
}

int pml_topk_logits(const float* logits, int64_t logits_stride, const int32_t* seq_lens, int batch,
                    int next_n, int max_context, int k, int32_t* indices, int64_t indices_stride,
                    float* values, int64_t values_stride, void* stream)
{
    if (batch < 0 || next_n < 1 || max_context < 1) return PML_ERR_INVALID_ARG;
    if (k < 1 || k > kTopkMax) return PML_ERR_UNSUPPORTED;
    if (batch == 0) return PML_OK;
    if (!logits || !seq_lens || !indices) return PML_ERR_INVALID_ARG;
    const long long rows = (long long)batch * next_n;
    if (rows > 0x7fffffffLL) return PML_ERR_INVALID_ARG;
    if (logits_stride < max_context || indices_stride < k) return PML_ERR_INVALID_ARG;
    if (values && values_stride < k) return PML_ERR_INVALID_ARG;
    if (!aligned(logits, 4) || !aligned(seq_lens, 4) || !aligned(indices, 4) ||
        !aligned(values, 4))
        return PML_ERR_ALIGNMENT;
    TopkArgs a;
    a.logits = logits;
    a.seq_lens = seq_lens;
    a.indices = indices;
    a.values = values;
    a.logits_stride = logits_stride;
    a.indices_stride = indices_stride;
    a.values_stride = values_stride;
    a.next_n = next_n;
    a.max_context = max_context;
    a.k = k;
    DeviceInfo dev;
    cudaError_t e = device_info(dev);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_topk(a, (int)rows, dev.smem_optin, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PML_OK : cuda_fail(e);
}

int pml_indexer_scores_nvfp4(const uint8_t* query, const uint8_t* query_scales, int rows,
                             const uint8_t* key_cache, int64_t page_stride_bytes,
                             const uint8_t* key_scales, int64_t scale_page_stride_bytes,
                             int64_t num_pages, const int32_t* block_table, int64_t bt_stride,
                             int num_requests, const int32_t* context_lengths,
                             const int32_t* requests, int groups, float* scores,
                             int64_t scores_stride, int max_context, void* stream)
{
    if (rows < 0 || groups < 0) return PML_ERR_INVALID_ARG;
    if (groups == 0) return rows == 0 ? PML_OK : PML_ERR_INVALID_ARG;
    if (rows % groups != 0) return PML_ERR_INVALID_ARG;
    const int G = rows / groups;
    if (G < 1 || G > 8) return PML_ERR_UNSUPPORTED;
    if (!query || !query_scales || !key_cache || !key_scales || !block_table ||
        !context_lengths || !requests || !scores)
        return PML_ERR_INVALID_ARG;
    if (num_pages < 1 || num_pages > 0x7fffffffLL || num_requests < 1) return PML_ERR_INVALID_ARG;
    if (page_stride_bytes < (int64_t)kBlockKeys * kHeadDim / 2) return PML_ERR_INVALID_ARG;
    if (scale_page_stride_bytes < (int64_t)kBlockKeys * kHeadDim / 16) return PML_ERR_INVALID_ARG;
    if (page_stride_bytes % 16 != 0 || scale_page_stride_bytes % 8 != 0) return PML_ERR_ALIGNMENT;
    if (max_context < 1 || scores_stride < max_context) return PML_ERR_INVALID_ARG;
    if (bt_stride < pml_min_block_table_width(max_context)) return PML_ERR_INVALID_ARG;
    if (!aligned(query, 16) || !aligned(query_scales, 8) || !aligned(key_cache, 16) ||
        !aligned(key_scales, 8) || !aligned(scores, 4) || !aligned(block_table, 4) ||
        !aligned(context_lengths, 4) || !aligned(requests, 4))
        return PML_ERR_ALIGNMENT;

    DeviceInfo dev;
    cudaError_t e = device_info(dev);
    if (e != cudaSuccess) return cuda_fail(e);

    Nvfp4Args a;
    a.query = query;
    a.query_scales = query_scales;
    a.key_cache = key_cache;
    a.key_scales = key_scales;
    a.context_lengths = context_lengths;
    a.requests = requests;
    a.block_table = block_table;
    a.scores = scores;
    a.status = dev.status;
    a.page_stride = page_stride_bytes;
    a.scale_stride = scale_page_stride_bytes;
    a.bt_stride = bt_stride;
    a.scores_stride = scores_stride;
    a.num_pages = num_pages;
    a.num_requests = num_requests;
    a.groups = groups;
    a.group_size = G;
    a.max_context = max_context;
    a.scales16 = (aligned(key_scales, 16) && scale_page_stride_bytes % 16 == 0) ? 1 : 0;
    // as many four-page stages (18 KB) as fit
    const size_t fixed = nvfp4_smem_bytes(0);
    const size_t per_stage = nvfp4_smem_bytes(1) - fixed;
    if ((size_t)dev.smem_optin < fixed + 2 * per_stage) return PML_ERR_UNSUPPORTED;
    int stages = (int)(((size_t)dev.smem_optin - fixed) / per_stage);
    if (stages > kMaxNvfp4Stages) stages = kMaxNvfp4Stages;
    a.stages = stages - stages % kNvfp4Producers;   // the kernel's producers share the ring
    // the codes of page P: 64 rows of 64 bytes at P * page_stride, landing
    // with the 64-byte swizzle the MMA reads
    CUtensorMap kmap;
    {
        const uint64_t dims[3] = {(uint64_t)kHeadDim / 2, (uint64_t)kBlockKeys, (uint64_t)num_pages};
        const uint64_t strides[2] = {(uint64_t)kHeadDim / 2, (uint64_t)page_stride_bytes};
        const uint32_t box[3] = {(uint32_t)kHeadDim / 2, (uint32_t)kBlockKeys, 1};
        e = encode_tiled(kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, key_cache, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_64B);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    e = launch_nvfp4_scores(kmap, a, dev.sm_count, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PML_OK : cuda_fail(e);
}

int pml_indexer_scores_bf16(const uint16_t* query, int rows, const uint16_t* key_cache,
                            int64_t page_stride_bytes, int64_t num_pages,
                            const int32_t* block_table, int64_t bt_stride, int num_requests,
                            const int32_t* context_lengths, const int32_t* requests, int groups,
                            float* scores, int64_t scores_stride, int max_context, void* stream)
{
    if (rows < 0 || groups < 0) return PML_ERR_INVALID_ARG;
    if (groups == 0) return rows == 0 ? PML_OK : PML_ERR_INVALID_ARG;
    if (rows % groups != 0) return PML_ERR_INVALID_ARG;
    const int G = rows / groups;
    if (G < 1 || G > 8) return PML_ERR_UNSUPPORTED;
    if (!query || !key_cache || !block_table || !context_lengths || !requests || !scores)
        return PML_ERR_INVALID_ARG;
    if (num_pages < 1 || num_pages > 0x7fffffffLL || num_requests < 1) return PML_ERR_INVALID_ARG;
    if (page_stride_bytes < (int64_t)kBlockKeys * kHeadDim * 2) return PML_ERR_INVALID_ARG;
    if (page_stride_bytes % 16 != 0) return PML_ERR_ALIGNMENT;
    if (max_context < 1 || scores_stride < max_context) return PML_ERR_INVALID_ARG;
    if (bt_stride < pml_min_block_table_width(max_context)) return PML_ERR_INVALID_ARG;
    if (!aligned(query, 16) || !aligned(key_cache, 16) || !aligned(scores, 4) ||
        !aligned(block_table, 4) || !aligned(context_lengths, 4) || !aligned(requests, 4))
        return PML_ERR_ALIGNMENT;

    DeviceInfo dev;
    cudaError_t e = device_info(dev);
    if (e != cudaSuccess) return cuda_fail(e);

    Bf16Args a;
    a.context_lengths = context_lengths;
    a.requests = requests;
    a.block_table = block_table;
    a.scores = scores;
    a.status = dev.status;
    a.bt_stride = bt_stride;
    a.scores_stride = scores_stride;
    a.num_pages = num_pages;
    a.num_requests = num_requests;
    a.groups = groups;
    a.group_size = G;
    a.max_context = max_context;
    a.q_box_rows = rows < 16 ? rows : 16;
    const size_t fixed = bf16_smem_bytes(0);
    const size_t per_stage = bf16_smem_bytes(1) - fixed;
    int stages = (int)(((size_t)dev.smem_optin - fixed) / per_stage);
    if (stages > kMaxBf16Stages) stages = kMaxBf16Stages;
    if (stages < 2) return PML_ERR_UNSUPPORTED;
    a.stages = stages;

    CUtensorMap kmap, qmap;
    {
        const uint64_t dims[3] = {(uint64_t)kHeadDim, (uint64_t)kBlockKeys, (uint64_t)num_pages};
        const uint64_t strides[2] = {(uint64_t)kHeadDim * 2, (uint64_t)page_stride_bytes};
        const uint32_t box[3] = {64, (uint32_t)kBlockKeys, 1};
        e = encode_sw128(kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, key_cache, dims, strides, box);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    {
        const uint64_t dims[2] = {(uint64_t)kHeadDim, (uint64_t)rows};
        const uint64_t strides[1] = {(uint64_t)kHeadDim * 2};
        const uint32_t box[2] = {64, (uint32_t)a.q_box_rows};
        e = encode_sw128(qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, query, dims, strides, box);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    e = launch_bf16_scores(kmap, qmap, a, dev.sm_count, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PML_OK : cuda_fail(e);
}

int pml_device_status(unsigned int* status, int clear)
{
    if (status == nullptr) return PML_ERR_INVALID_ARG;
    DeviceInfo dev;
    cudaError_t e = device_info(dev);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaMemcpyFromSymbol(status, g_device_status, sizeof(unsigned int));
    if (e != cudaSuccess) return cuda_fail(e);
    if (clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(unsigned int));
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return PML_OK;
}

}  // extern "C"
