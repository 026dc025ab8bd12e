// Host-side launch records for the kernels of the paged MQA-logits library.
// Internal to the library: the public C ABI is include/pml.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pml {

struct Fp8Args {
    const int32_t* seq_lens;
    const int32_t* block_table;
    const int32_t* schedule_meta;  // nullptr: computed by each CTA
    const float* weights;
    const uint8_t* kv_fused;
    void* out;        // fp32, or bf16 when out_bf16
    unsigned int* status;
    long long bt_stride;
    long long out_stride;   // elements
    long long num_blocks;
    int batch;
    int next_n;
    int max_context;
    int stages;       // depth of the K-page ring
    int q_box_rows;   // rows one Q load brings (<= MMA N)
    int out_bf16;     // 1: logits stored as bf16 (round to nearest even)
    unsigned long long wait_limit_ns;   // longest wait of any role (kWaitLimitNs normally)
    int drop_stage;   // test support: the stage (count within each CTA) the producer
                      // leaves unpublished, so the roles waiting on it run out of time; -1: none
};

struct Bf16Args {
    const int32_t* context_lengths;
    const int32_t* requests;
    const int32_t* block_table;
    float* scores;
    unsigned int* status;
    long long bt_stride;
    long long scores_stride;
    long long num_pages;
    int num_requests;
    int groups;
    int group_size;
    int max_context;
    int stages;
    int q_box_rows;
};

// Stages of the NVFP4 kernel: each has 16 tensor-memory columns of key scales;
// their count is a multiple of the kernel's producer warps.
constexpr int kMaxNvfp4Stages = 20;
constexpr int kNvfp4Producers = 3;

struct Nvfp4Args {
    const uint8_t* query;          // [rows][64] packed E2M1
    const uint8_t* query_scales;   // [rows][8] E4M3
    const uint8_t* key_cache;      // page P at P * page_stride: [64][64] packed E2M1
    const uint8_t* key_scales;     // page P at P * scale_stride: [64][8] E4M3
    const int32_t* context_lengths;
    const int32_t* requests;
    const int32_t* block_table;
    float* scores;
    unsigned int* status;
    long long page_stride;
    long long scale_stride;
    long long bt_stride;
    long long scores_stride;
    long long num_pages;
    int num_requests;
    int groups;
    int group_size;
    int max_context;
    int stages;      // stages of one four-page tile (codes, then scales), <= kMaxNvfp4Stages
    int scales16;    // 1: key_scales and its page stride are 16-byte aligned (one
                     // 16-byte cp.async per lane and page), else two of 8 bytes
};

struct Mxfp4Args {
    const uint8_t* q;              // [batch*next_n][64 heads][64] packed E2M1
    const uint8_t* q_sf;           // [batch*next_n][64][4] E8M0
    const float* weights;          // [batch*next_n][64]
    const uint8_t* kv;             // [num_blocks][4352]
    const int32_t* seq_lens;
    const int32_t* block_table;
    const int32_t* schedule_meta;  // nullptr: computed by each CTA
    void* out;                     // fp32, or bf16 when out_bf16
    unsigned int* status;
    long long bt_stride;
    long long out_stride;          // elements
    long long num_blocks;
    int batch;
    int next_n;
    int slot0;                     // first query slot of this pass (set per launch)
    int max_context;
    int stages;                    // staging slots of a one-slot pass
    int stages2;                   // ... of a two-slot pass
    int out_bf16;
};

constexpr int kTopkMax = 4096;     // largest k of the top-k selection

struct TopkArgs {
    const float* logits;
    const int32_t* seq_lens;
    int32_t* indices;
    float* values;                // may be null
    long long logits_stride;
    long long indices_stride;
    long long values_stride;
    int next_n;
    int max_context;
    int k;
};

// Bytes of dynamic shared memory the fp8 kernel needs for `stages`.
size_t fp8_smem_bytes(int next_n, int num_heads, int stages);
size_t bf16_smem_bytes(int stages);
size_t nvfp4_smem_bytes(int stages);
size_t mxfp4_smem_bytes(int slots_per_pass, int stages);

cudaError_t launch_fp8_logits(int num_heads, const CUtensorMap& kmap, const CUtensorMap& qmap,
                              const Fp8Args& a, int num_ctas, cudaStream_t stream);
cudaError_t launch_bf16_scores(const CUtensorMap& kmap, const CUtensorMap& qmap,
                               const Bf16Args& a, int num_ctas, cudaStream_t stream);
cudaError_t launch_nvfp4_scores(const CUtensorMap& kmap, const Nvfp4Args& a, int num_ctas,
                                cudaStream_t stream);
// The MXFP4 logits: one launch per pass of at most two query slots.
cudaError_t launch_mxfp4_logits(const CUtensorMap& kmap, const CUtensorMap& qmap,
                                const Mxfp4Args& a, int num_ctas, cudaStream_t stream);
cudaError_t launch_topk(const TopkArgs& a, int rows, int smem_optin, cudaStream_t stream);
cudaError_t launch_schedule(const int32_t* seq_lens, int batch, int num_ctas, int32_t* meta,
                            cudaStream_t stream);

}  // namespace pml
