// The MXFP4 variant's re-encoding into the fp8 logits engine's formats
// (fp4_transcode.cu; the logits call in api.cu).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "common.cuh"

namespace pml {

// One MXFP4 KV block: 64 keys x 64 code bytes, then 64 x 4 E8M0 scale bytes.
constexpr int kMxfp4BlockBytes = kBlockKeys * (kHeadDim / 2 + kHeadDim / 32);   // 4352
// Status bit: an MXFP4 value that E4M3 could not hold exactly was rounded.
constexpr unsigned int kStatusFp4Inexact = 8u;

struct Fp4TranscodeArgs {
    const uint8_t* q;              // [q_rows][64] packed E2M1, q_rows = batch*next_n*64
    const uint8_t* q_sf;           // [q_rows][4] E8M0
    const float* weights;          // [q_rows]
    const uint8_t* kv;             // [num_blocks][4352]
    const int32_t* seq_lens;
    const int32_t* block_table;
    uint8_t* q8;                   // out: [q_rows][128] E4M3
    float* w8;                     // out: [q_rows] weights times the rows' powers of two
    uint8_t* kv8;                  // out: [num_blocks][8448] kv_fused blocks (used ones only)
    unsigned int* status;
    long long q_rows;
    long long bt_stride;
    long long num_blocks;
    int max_context;
};

cudaError_t launch_fp4_transcode(const Fp4TranscodeArgs& a, int batch, cudaStream_t stream);

}  // namespace pml
