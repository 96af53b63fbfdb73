// Fused compression kernels for the 1-bit Adam variant with binary32 error
// buffers, every chunk size and gradient kind (templates in k_compress.cuh).
#include "k_compress.cuh"

namespace lamb1b {

template <>
cudaError_t launch_fused<true, false>(const Problem& P, const Dev& D, const Grads& G, cudaStream_t st)
{
    return launch_fused_all_chunks<true, false>(P, D, G, st);
}

}  // namespace lamb1b
