// Compression stage of 1-bit LAMB (arXiv 2104.06069): dispatch of the fused
// worker + server pass (k_compress.cuh, one translation unit per variant and
// error storage), the per-tensor factor kernel and the update.
#include "k_compress.cuh"

namespace lamb1b {

// Per tensor: soft-thresholded factor from the max ratio, coefficient, and
// reset of the max for the next step.
__global__ void k_factor(const Problem P, const Dev D)
{
    const int l = blockIdx.x * blockDim.x + threadIdx.x;
    if (l >= P.L) return;
    const float R = __uint_as_float(D.Rmax[l]);
    D.Rmax[l] = 0u;
    const float rp = D.r_prev[l];
    const float r = clip(clip(R, P.fmin, P.fmax), fmul(P.fthr_lo, rp), fmul(P.fthr_hi, rp));
    const float c = fmul(D.c_bar[l], r);
    D.R_last[l] = R;
    D.r_prev[l] = r;
    D.c_cur[l] = c;
    D.gc[l] = fmul(P.lr, c);
}

int64_t padded_length(int64_t N, int C)
{
    const int64_t tile = C > 4096 ? C : 4096;
    return (N + tile - 1) / tile * tile;
}

cudaError_t launch_compress(const Problem& P, const Dev& D, const Grads& G, float* x,
                            cudaStream_t st, const cudaEvent_t* ev)
{
    cudaError_t e;
    if ((e = trace(ev, 0, st)) != cudaSuccess) return e;
    // 4096-element tiles (256 threads x 4 float4 groups) holding 4096/C chunks;
    // 8192-element chunks use 512-thread tiles of one chunk.
    if (P.adam)
        e = P.ebf16 ? launch_fused<true, true>(P, D, G, st) : launch_fused<true, false>(P, D, G, st);
    else
        e = P.ebf16 ? launch_fused<false, true>(P, D, G, st) : launch_fused<false, false>(P, D, G, st);
    if (e != cudaSuccess) return e;
    if ((e = trace(ev, 1, st)) != cudaSuccess) return e;
    if (!P.adam) {   // 1-bit Adam: c = 1, gc = lr from the initialisation
        k_factor<<<(P.L + 255) / 256, 256, 0, st>>>(P, D);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if ((e = trace(ev, 2, st)) != cudaSuccess) return e;
    // the update reads this step's server sign words and chunk scales (m is
    // exactly server sign x server scale) instead of the dense m
    if ((e = launch_update(P, D, x, 1, st)) != cudaSuccess) return e;
    return trace(ev, 3, st);
}

}  // namespace lamb1b
