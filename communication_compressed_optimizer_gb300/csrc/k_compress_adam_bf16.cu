// Fused compression kernels for the 1-bit Adam variant with bfloat16 error
// buffers, every chunk size and gradient kind (templates in k_compress.cuh).
#include "k_compress.cuh"

namespace lamb1b {

template <>
cudaError_t launch_fused<true, true>(const Problem& P, const Dev& D, const Grads& G, cudaStream_t st)
{
    return launch_fused_all_chunks<true, true>(P, D, G, st);
}

}  // namespace lamb1b
