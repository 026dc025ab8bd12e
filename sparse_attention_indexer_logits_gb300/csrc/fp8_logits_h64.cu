// Instantiation of the fp8 paged MQA-logits kernel for 64 heads
// (next_n = 1..4); one translation unit per head count so they build in
// parallel.
#include "fp8_logits.cuh"

namespace pml {

cudaError_t launch_fp8_h64(const CUtensorMap& kmap, const CUtensorMap& qmap, const Fp8Args& a,
                           int num_ctas, cudaStream_t stream)
{
    return fp8::launch_heads<64>(kmap, qmap, a, num_ctas, stream);
}

}  // namespace pml
