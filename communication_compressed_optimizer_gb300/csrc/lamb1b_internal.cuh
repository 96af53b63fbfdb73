// Internal structures shared by the lamb1b translation units: the problem
// description, the workspace layout, the gradient source, and the device
// helpers every kernel uses (explicitly rounded binary32 arithmetic, the
// warp-level pairwise tree, sign-word packing, layer lookup).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "f32x2.cuh"
#include "philox.cuh"

namespace lamb1b {

constexpr int kGranule = 256;        // level-0 block of the canonical pairwise tree
// The level-1 tree of a tensor (over its granule sums, zero-padded to a power
// of two) is evaluated as subtrees over aligned blocks of kLevel1Block granule
// sums, then a tree over the block sums.  All partial sums are >= +0, so a
// subtree over a block that reaches past the padded length adds only +0.
constexpr int64_t kLevel1Block = 4096;
__host__ __device__ constexpr int64_t level1_blocks(int64_t granules)
{
    return (granules + kLevel1Block - 1) / kLevel1Block;
}
constexpr int kMaxChunkLayers = 64;  // per-chunk layer slots kept in shared memory

// Default bound of a shared-memory copy wait, in mbarrier.try_wait calls
// (each suspends for a hardware-defined time): seconds, far beyond any copy.
constexpr uint32_t kDefaultWaitTries = 1u << 24;

struct Problem {
    int64_t N;        // parameters
    int64_t Np;       // padded vector length: a multiple of max(C, 4096) >= K * C
    int64_t K;        // chunks
    int64_t words_ld; // Np / 32
    int32_t L, W, C;
    int64_t NB;       // level-1 blocks of all tensors (warmup norms)
    float lr, beta1, beta2, eps, wd;
    float omega1, omega2;             // fl(1 - beta1), fl(1 - beta2)
    float cmin, cmax, cema, one_m_cema;
    float fmin, fmax, fthr_lo, fthr_hi; // fl(1 - thr), fl(1 + thr)
    int32_t check_finite;
    int32_t adam;       // 1-bit Adam variant: no layerwise coefficient, no fresh variance
    int32_t ebf16;      // e_w and e_s stored as bfloat16
    int32_t log2c;      // C = 2^log2c
    int32_t w_pow2;     // W is a power of two
    float inv_w;        // 1 / W (exact when w_pow2)
    int32_t m_packed;    // compression stage after its first step: m is held as the
                         // server's sign words and chunk scales (signs_s, scale_s)
    uint32_t wait_tries; // bound of every shared-memory copy wait (try_wait calls)
    int32_t skip_copy;   // fault injection: copy position left out by CTA 0, or -1
};

// Device pointers into the caller's workspace.
struct Dev {
    float* m;         // [Np]
    float* v;         // [Np]  second moment; frozen after the stage switch
    float* v_fresh;   // [Np]
    float* d_frz;     // [Np]  fl(sqrt(v) + eps) of the frozen v (compression stage)
    float* e_s;       // [Np]     binary32, or bfloat16 bits when P.ebf16
    float* e_w;       // [W][Np]  binary32, or bfloat16 bits when P.ebf16
    uint32_t* signs_w;// [W][words_ld]
    uint32_t* signs_s;// [words_ld]
    float* scale_w;   // [W][K]
    float* scale_s;   // [K]
    float* c_bar;     // [L]
    float* r_prev;    // [L]
    float* c_cur;     // [L]
    float* gc;        // [L] fl(lr * c_cur)
    float* R_last;    // [L]
    float* Sx;        // [L]
    float* Su;        // [L]
    uint32_t* Rmax;   // [L] bit patterns of positive floats, max-reduced
    int64_t* layer_off;  // [L]
    int64_t* layer_end;  // [L] off + numel
    int64_t* hbase;      // [L+1] first half-granule partial of each layer
    int32_t* chunk_l0;   // [K] layer of the chunk's first element
    int32_t* chunk_l1;   // [K] layer of the chunk's last element
    float* part_x;       // [hbase[L]] warmup half-granule sums of x^2
    float* part_u;       // [hbase[L]] warmup half-granule sums of u^2
    int64_t* bbase;      // [L+1] first level-1 block of each layer
    float* blk_x;        // [NB] level-1 block sums of x^2 (kLevel1Block granule sums each)
    float* blk_u;        // [NB] the same for u^2
    uint32_t* flags;     // [4] bit 0: non-finite gradient seen
};

struct Grads {
    int32_t kind;     // 0 f32, 1 bf16, 2 philox
    const void* ptr;
    int64_t ld;
    uint64_t seed;
    const float* layer_std;
    const uint8_t* layer_heavy;
    float heavy_scale;
    uint32_t t;       // global step index (Philox counter word 2)
};

enum { kGradF32 = 0, kGradBF16 = 1, kGradPhilox = 2 };

// ---- explicitly rounded binary32 arithmetic --------------------------------
__device__ __forceinline__ float fadd(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float fsub(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ float fmul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float fdiv(float a, float b) { return __fdiv_rn(a, b); }
__device__ __forceinline__ float fsqrt(float a) { return __fsqrt_rn(a); }
// clip(x, a, b) = min{max{x, a}, b} by comparisons (a NaN x passes through)
__device__ __forceinline__ float clip(float x, float a, float b)
{
    const float r = (x < a) ? a : x;
    return (r > b) ? b : r;
}

// Pairwise tree of the 128 leaves held by a warp, 4 consecutive leaves per
// lane (lane l holds leaves 4l..4l+3): ((f0+f1)+(f2+f3)) then butterfly
// partners 1, 2, 4, 8, 16.  Every lane returns the total.
__device__ __forceinline__ float warp_tree128(float f0, float f1, float f2, float f3)
{
    float v = fadd(fadd(f0, f1), fadd(f2, f3));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) v = fadd(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// fl(a / W).  For W = 2^k the quotient a 2^-k is the exact product with the
// exact reciprocal, so one rounded multiplication gives the same bits as the
// rounded division for every a (zeros, subnormals, infinities, NaN).
__device__ __forceinline__ float div_w(float a, const Problem& P)
{
    return P.w_pow2 ? fmul(a, P.inv_w) : fdiv(a, (float)P.W);
}

// Pairwise trees of S independent 128-leaf blocks at once (S a power of two,
// S <= 32).  Lane l holds leaf-group sums v[s] = ((f0+f1)+(f2+f3)) of leaves
// 4l..4l+3 of block s.  The butterfly over partners 1, 2, 4, 8, 16 is the same
// tree as warp_tree128 for every block, but while a lane still holds n > 1
// blocks it passes half of them to its partner and keeps the other half, so S
// blocks cost about as many exchanges as two.  Lane l returns the total of
// block tree_block<S>(l).
template <int S>
__device__ __forceinline__ int tree_block(int lane)
{
    int b = 0, o = 1;
#pragma unroll
    for (int n = S; n > 1; n >>= 1, o <<= 1)
        if (lane & o) b += n / 2;
    return b;
}

template <int S>
__device__ __forceinline__ float warp_trees128(float (&v)[S], int lane)
{
    static_assert(S >= 1 && S <= 32 && (S & (S - 1)) == 0, "S a power of two");
    int o = 1;
#pragma unroll
    for (int n = S; n > 1; n >>= 1, o <<= 1) {
        const bool hi = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < n / 2; ++j) {
            const float send = hi ? v[j] : v[j + n / 2];
            const float keep = hi ? v[j + n / 2] : v[j];
            v[j] = fadd(keep, __shfl_xor_sync(0xFFFFFFFFu, send, o));
        }
    }
    float t = v[0];
#pragma unroll
    for (; o < 32; o <<= 1) t = fadd(t, __shfl_xor_sync(0xFFFFFFFFu, t, o));
    return t;
}

// Two binary32 values -> packed bfloat16 bits (lo in bits 0-15), each
// rounded to nearest even by one hardware conversion (cvt.rn.bf16x2.f32);
// a NaN is stored as 0x7FC0.
__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    uint32_t u = (uint32_t)__bfloat16_as_ushort(v.x) | ((uint32_t)__bfloat16_as_ushort(v.y) << 16);
    if (lo != lo) u = (u & 0xFFFF0000u) | 0x7FC0u;
    if (hi != hi) u = (u & 0x0000FFFFu) | 0x7FC00000u;
    return u;
}

// ---- launchers (one translation unit each) ---------------------------------
// `ev` is NULL or 4 events recorded before the first kernel and after each
// of the three kernels of a step.
cudaError_t launch_warmup(const Problem& P, const Dev& D, const Grads& G, float* x,
                          cudaStream_t st, int first_warmup, const cudaEvent_t* ev);
cudaError_t launch_freeze(const Problem& P, const Dev& D, cudaStream_t st);
cudaError_t launch_unpack_momentum(const Problem& P, const Dev& D, cudaStream_t st);
cudaError_t launch_frozen_denominator(const Problem& P, const Dev& D, cudaStream_t st);
cudaError_t launch_compress(const Problem& P, const Dev& D, const Grads& G, float* x,
                            cudaStream_t st, const cudaEvent_t* ev);

inline cudaError_t trace(const cudaEvent_t* ev, int i, cudaStream_t st)
{
    return ev ? cudaEventRecord(ev[i], st) : cudaSuccess;
}
cudaError_t launch_init_layers(const Problem& P, const Dev& D, cudaStream_t st);
// padded vector length for N elements and chunk C (whole compression tiles)
int64_t padded_length(int64_t N, int C);

}  // namespace lamb1b
