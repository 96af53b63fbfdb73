// On-device generation of the seeded synthetic workload (include/lamb1b_gen.h).
#include <cuda_runtime.h>

#include "lamb1b_gen.h"
#include "lamb1b.h"
#include "philox.cuh"
#include "device_ptr.h"

namespace lamb1b {

// One thread per aligned group of 4 elements q that meets the tensor
// [lo, hi); grid.y = worker.
template <bool BF16>
__global__ void k_gen_grads(void* out, int64_t ld, uint64_t seed, uint32_t t, int64_t lo,
                            int64_t hi, float std, int heavy, float heavy_scale)
{
    const int64_t q = lo / 4 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (q * 4 >= hi) return;
    const uint32_t w = blockIdx.y;
    float g[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (!heavy) {
        float z[4];
        gen::grads_normal4(seed, (uint64_t)q, t, w, z);
#pragma unroll
        for (int c = 0; c < 4; ++c) g[c] = __fmul_rn(std, z[c]);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int64_t i = q * 4 + c;
        if (i < lo || i >= hi) continue;
        if (heavy) g[c] = __fmul_rn(heavy_scale, gen::student_t3(seed, i, t, w));
        if (BF16)
            static_cast<uint16_t*>(out)[(int64_t)w * ld + i] = gen::bf16_rne(g[c]);
        else
            static_cast<float*>(out)[(int64_t)w * ld + i] = g[c];
    }
}

__global__ void k_gen_params(float* out, int64_t lo, int64_t hi, float std, uint64_t seed)
{
    const int64_t q = lo / 4 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (q * 4 >= hi) return;
    float z[4];
    gen::normal4(seed, gen::u4{(uint32_t)q, (uint32_t)((uint64_t)q >> 32), 0u, 0x7FFFFFFFu}, z);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int64_t i = q * 4 + c;
        if (i >= lo && i < hi) out[i - lo] = __fmul_rn(std, z[c]);
    }
}

// ---- self-check of the transform's fast division and square root -----------
// counts[0]: log-series quotients (all 2^23 f) where div_logq differs from
// __fdiv_rn; counts[1]: non-negative floats where div3 differs from
// __fdiv_rn(x, 3); counts[2]: floats in [2^-102, +max] where sqrt_big differs
// from __fsqrt_rn; counts[3]: draws of 2^22 counters where normal4 differs
// from normal4_reference (any of the four values); counts[4]: the same for
// student_t3 on 2^22 elements.
__global__ void k_check_logq(unsigned long long* counts)
{
    const uint32_t m = blockIdx.x * blockDim.x + threadIdx.x;
    if (m >= (1u << 23)) return;
    float f = __uint_as_float(m | 0x3F800000u);
    if (f > 0x1.6a09e6p+0f) f = __fmul_rn(f, 0.5f);
    const float a = __fsub_rn(f, 1.0f), b = __fadd_rn(f, 1.0f);
    if (__float_as_uint(gen::div_logq(a, b)) != __float_as_uint(__fdiv_rn(a, b))) atomicAdd(&counts[0], 1ull);
}

__global__ void k_check_floats(unsigned long long* counts, uint32_t first)
{
    const uint32_t bits = first + blockIdx.x * blockDim.x + threadIdx.x;   // +0 .. +max, in order
    if (bits >= 0x7F800000u) return;
    const float x = __uint_as_float(bits);
    if (__float_as_uint(gen::div3(x)) != __float_as_uint(__fdiv_rn(x, 3.0f))) atomicAdd(&counts[1], 1ull);
    if (x >= 0x1p-102f && __float_as_uint(gen::sqrt_big(x)) != __float_as_uint(__fsqrt_rn(x)))
        atomicAdd(&counts[2], 1ull);
}

__global__ void k_check_draws(unsigned long long* counts, uint64_t seed)
{
    const uint32_t q = blockIdx.x * blockDim.x + threadIdx.x;
    if (q >= (1u << 22)) return;
    float a[4], b[4];
    gen::normal4(seed, gen::u4{q, 0u, 5u, 3u}, a);
    gen::normal4_reference(seed, gen::u4{q, 0u, 5u, 3u}, b);
    bool bad = false;
#pragma unroll
    for (int c = 0; c < 4; ++c) bad = bad || __float_as_uint(a[c]) != __float_as_uint(b[c]);
    if (bad) atomicAdd(&counts[3], 1ull);
    if (__float_as_uint(gen::student_t3(seed, q, 5u, 3u)) !=
        __float_as_uint(gen::student_t3_reference(seed, q, 5u, 3u)))
        atomicAdd(&counts[4], 1ull);
}

}  // namespace lamb1b

extern "C" int lamb1b_gen_selfcheck(unsigned long long* counts_dev, uint64_t seed, void* stream)
{
    if (!counts_dev) return LAMB1B_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(counts_dev) & 7u) return LAMB1B_ERR_ALIGN;
    if (!lamb1b::is_current_device_ptr(counts_dev)) return LAMB1B_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(counts_dev, 0, 5 * sizeof(unsigned long long), st) != cudaSuccess) {
        cudaGetLastError();
        return LAMB1B_ERR_CUDA;
    }
    lamb1b::k_check_logq<<<(1u << 23) / 256, 256, 0, st>>>(counts_dev);
    for (uint32_t first = 0; first < 0x7F800000u; first += (1u << 28))
        lamb1b::k_check_floats<<<(1u << 28) / 256, 256, 0, st>>>(counts_dev, first);
    lamb1b::k_check_draws<<<(1u << 22) / 256, 256, 0, st>>>(counts_dev, seed);
    return cudaGetLastError() == cudaSuccess ? LAMB1B_OK : LAMB1B_ERR_CUDA;
}

extern "C" int lamb1b_gen_grads(void* out_dev, int64_t ld, int32_t W, int32_t bf16,
                                uint64_t seed, int64_t t, const int64_t* layer_off,
                                const int64_t* layer_numel, int32_t L, const float* layer_std,
                                const uint8_t* layer_heavy, float heavy_scale, void* stream)
{
    if (!out_dev || !layer_off || !layer_numel || !layer_std || L <= 0 || W <= 0 || W > 65535 ||
        t < 0 || t > 0xFFFFFFFFll)
        return LAMB1B_ERR_ARG;
    int64_t N = 0;
    for (int32_t l = 0; l < L; ++l) {
        if (layer_off[l] != N || layer_numel[l] <= 0) return LAMB1B_ERR_ARG;
        N += layer_numel[l];
    }
    if (ld < N) return LAMB1B_ERR_ARG;
    if (!lamb1b::is_current_device_ptr(out_dev)) return LAMB1B_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int32_t l = 0; l < L; ++l) {
        const int64_t lo = layer_off[l], hi = lo + layer_numel[l];
        const int64_t nq = (hi - 1) / 4 - lo / 4 + 1;
        const dim3 grid((unsigned)((nq + 255) / 256), (unsigned)W);
        const int heavy = layer_heavy ? (layer_heavy[l] != 0) : 0;
        if (bf16)
            lamb1b::k_gen_grads<true><<<grid, 256, 0, st>>>(out_dev, ld, seed, (uint32_t)t, lo, hi,
                                                            layer_std[l], heavy, heavy_scale);
        else
            lamb1b::k_gen_grads<false><<<grid, 256, 0, st>>>(out_dev, ld, seed, (uint32_t)t, lo, hi,
                                                             layer_std[l], heavy, heavy_scale);
        if (cudaGetLastError() != cudaSuccess) return LAMB1B_ERR_CUDA;
    }
    return LAMB1B_OK;
}

extern "C" int lamb1b_gen_params(float* out_dev, int64_t lo, int64_t hi, float std, uint64_t seed,
                                 void* stream)
{
    if (!out_dev || lo < 0 || hi < lo) return LAMB1B_ERR_ARG;
    if (hi == lo) return LAMB1B_OK;
    if (!lamb1b::is_current_device_ptr(out_dev)) return LAMB1B_ERR_ARG;
    const int64_t nq = (hi - 1) / 4 - lo / 4 + 1;
    lamb1b::k_gen_params<<<(unsigned)((nq + 255) / 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        out_dev, lo, hi, std, seed);
    return cudaGetLastError() == cudaSuccess ? LAMB1B_OK : LAMB1B_ERR_CUDA;
}
