// Allocation-free variant of the two-step fp8 logits call.
//
// The regular two-step path asks the caller for a device buffer that carries
// the per-CTA schedule from pml_schedule to pml_fp8_paged_mqa_logits.  Here
// that buffer is a fixed array in the library's own device memory, so the
// caller passes only the inputs and the output.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "pml.h"

namespace {

constexpr int kNoAllocMaxCtas = 1024;
constexpr int kNoAllocEntries = (kNoAllocMaxCtas + 1) * 2;
constexpr int kMaxDevices = 64;

// Schedule scratch: (request, block) start of every CTA's range plus the end
// entry.  Every device that loads the library holds these 8200 bytes until the
// process exits.  The name is only a host-side handle; kernels get the device
// address looked up below.
static __device__ __align__(256) int32_t g_noalloc_schedule[kNoAllocEntries];

std::mutex g_noalloc_mutex;
int32_t* g_noalloc_ptr[kMaxDevices];

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
cudaError_t noalloc_scratch(int32_t** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_schedule);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" {

int pml_noalloc_max_ctas(void) { return kNoAllocMaxCtas; }

int pml_fp8_paged_mqa_logits_noalloc(const uint8_t* q, const uint8_t* kv_fused, int64_t num_blocks,
                                     const float* weights, const int32_t* seq_lens,
                                     const int32_t* block_table, int64_t bt_stride, int num_ctas,
                                     float* out, int64_t out_stride, int max_context, int batch,
                                     int next_n, int num_heads, void* stream)
{
    if (batch < 0 || num_ctas < 0) return PML_ERR_INVALID_ARG;
    if (num_ctas > kNoAllocMaxCtas) return PML_ERR_INVALID_ARG;
    if (batch == 0) return PML_OK;
    if (num_ctas == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return PML_ERR_CUDA;
        num_ctas = pml_default_num_ctas(dev);
        if (num_ctas <= 0) return PML_ERR_CUDA;
        if (num_ctas > kNoAllocMaxCtas) num_ctas = kNoAllocMaxCtas;
    }
    int32_t* scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess) return PML_ERR_CUDA;
    int rc = pml_schedule(seq_lens, batch, next_n, num_ctas, scratch, stream);
    if (rc != PML_OK) return rc;
    return pml_fp8_paged_mqa_logits(q, kv_fused, num_blocks, weights, seq_lens, block_table,
                                    bt_stride, scratch, num_ctas, out, out_stride, max_context,
                                    batch, next_n, num_heads, stream);
}

}  // extern "C"
