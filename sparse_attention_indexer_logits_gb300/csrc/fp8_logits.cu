// Dispatch of the fp8 paged MQA-logits kernel (fp8_logits.cuh) by head
// count, and its shared-memory footprint for the host's pipeline sizing.
#include "fp8_logits.cuh"

namespace pml {

cudaError_t launch_fp8_h8(const CUtensorMap&, const CUtensorMap&, const Fp8Args&, int, cudaStream_t);
cudaError_t launch_fp8_h16(const CUtensorMap&, const CUtensorMap&, const Fp8Args&, int, cudaStream_t);
cudaError_t launch_fp8_h32(const CUtensorMap&, const CUtensorMap&, const Fp8Args&, int, cudaStream_t);
cudaError_t launch_fp8_h64(const CUtensorMap&, const CUtensorMap&, const Fp8Args&, int, cudaStream_t);

size_t fp8_smem_bytes(int next_n, int num_heads, int stages)
{
    return (size_t)fp8::layout(fp8::n_pad_of(next_n, num_heads), next_n, num_heads, stages).total +
           1024;
}

cudaError_t launch_fp8_logits(int num_heads, const CUtensorMap& kmap, const CUtensorMap& qmap,
                              const Fp8Args& a, int num_ctas, cudaStream_t stream)
{
    switch (num_heads) {
    case 8: return launch_fp8_h8(kmap, qmap, a, num_ctas, stream);
    case 16: return launch_fp8_h16(kmap, qmap, a, num_ctas, stream);
    case 32: return launch_fp8_h32(kmap, qmap, a, num_ctas, stream);
    case 64: return launch_fp8_h64(kmap, qmap, a, num_ctas, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pml
