// Allocation-free entry point: per-tensor sums of squares of a device vector,
// reduced in the same canonical pairwise-tree order as the warmup step's
// trust-ratio norms, with all scratch in a fixed device array owned by this
// file.  See lamb1b_tensor_sumsq_noalloc in include/lamb1b.h.
#include <cstdint>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "lamb1b.h"
#include "lamb1b_internal.cuh"
#include "device_ptr.h"

namespace lamb1b {
namespace noalloc {

constexpr int32_t kMaxLayers = 4096;
constexpr int64_t kMaxHalves = int64_t(1) << 22;   // half-granule partial sums (16 MiB)
constexpr int kMaxDevices = 64;

// Everything the two kernels need besides their input and output.  Device
// memory for it is set aside when the library's module is loaded on a GPU and
// stays until the process exits; every call reuses it.
struct Scratch {
    int64_t off[kMaxLayers];
    int64_t end[kMaxLayers];
    int64_t hbase[kMaxLayers + 1];
    float part[kMaxHalves];
};

static __device__ __align__(256) Scratch g_scratch;

// Host side: the device address of g_scratch, looked up once per device.
static std::mutex g_mu;
static Scratch* g_addr[kMaxDevices] = {};

static int scratch_on_current_device(Scratch** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LAMB1B_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return LAMB1B_ERR_CUDA;
        }
        g_addr[dev] = static_cast<Scratch*>(p);
    }
    *out = g_addr[dev];
    return LAMB1B_OK;
}

constexpr int kNT = 256;
constexpr int kSlots = 4;
constexpr int kBlock = kNT * 4 * kSlots;

// Layer holding flat index i (binary search over the tensor ends).
__device__ __forceinline__ int layer_of(const Scratch* S, int32_t L, int64_t i)
{
    int lo = 0, hi = L - 1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (S->end[mid] <= i) lo = mid + 1; else hi = mid;
    }
    return lo;
}

// Level 0: for every aligned 128-element block and every tensor meeting it,
// the pairwise tree of the block's squares with leaves outside the tensor at
// +0, stored at the tensor's half-granule slot.
__global__ void __launch_bounds__(kNT) k_half_sums(const float* __restrict__ x, int64_t N, int32_t L,
                                                   Scratch* S)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t b0 = (int64_t)blockIdx.x * kBlock;
    int l = layer_of(S, L, b0);
    int64_t lend = S->end[l];
#pragma unroll 1
    for (int s = 0; s < kSlots; ++s) {
        const int64_t idx = b0 + s * kNT * 4 + tid * 4;
        const int64_t r = N - idx;
        const int nv = r >= 4 ? 4 : (r > 0 ? (int)r : 0);
        float f[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        int lay[4] = {-1, -1, -1, -1};
        if (nv == 4) {
            const float4 v = *reinterpret_cast<const float4*>(x + idx);
            f[0] = fmul(v.x, v.x); f[1] = fmul(v.y, v.y); f[2] = fmul(v.z, v.z); f[3] = fmul(v.w, v.w);
        } else {
            for (int c = 0; c < nv; ++c) f[c] = fmul(x[idx + c], x[idx + c]);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (c < nv) {
                while (idx + c >= lend) { ++l; lend = S->end[l]; }
                lay[c] = l;
            }
        }
        int lo = 0x7FFFFFFF, hi = -1;
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (lay[c] >= 0) { lo = min(lo, lay[c]); hi = max(hi, lay[c]); }
        lo = __reduce_min_sync(0xFFFFFFFFu, lo);
        hi = __reduce_max_sync(0xFFFFFFFFu, hi);
        const int64_t blk = b0 + s * kNT * 4 + warp * 128;
        for (int lj = lo; lj <= hi; ++lj) {
            const float t = warp_tree128(lay[0] == lj ? f[0] : 0.0f, lay[1] == lj ? f[1] : 0.0f,
                                         lay[2] == lj ? f[2] : 0.0f, lay[3] == lj ? f[3] : 0.0f);
            if (lane == 0)
                S->part[S->hbase[lj] + blk / 128 - 2 * (S->off[lj] / kGranule)] = t;
        }
    }
}

// Level 1 per tensor: pairwise tree over its granule sums (half + half),
// split into 256 aligned blocks, one per thread; then across the block.
__device__ float seq_tree_halves(const float* part, int64_t j0, int64_t B, int64_t cnt)
{
    float stk[40];
    int lvl[40];
    int sp = 0;
    for (int64_t j = j0; j < j0 + B; ++j) {
        float v = (j < cnt) ? fadd(part[2 * j], part[2 * j + 1]) : 0.0f;
        int lv = 0;
        while (sp > 0 && lvl[sp - 1] == lv) { v = fadd(stk[sp - 1], v); ++lv; --sp; }
        stk[sp] = v; lvl[sp] = lv; ++sp;
    }
    return stk[0];
}

__global__ void __launch_bounds__(kNT) k_tensor_totals(const Scratch* S, float* __restrict__ out)
{
    __shared__ float sh[kNT / 32];
    const int l = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t hb = S->hbase[l];
    const int64_t cnt = (S->hbase[l + 1] - hb) / 2;
    int64_t p2 = 1;
    while (p2 < cnt) p2 <<= 1;
    const int64_t B = p2 > kNT ? p2 / kNT : 1;
    float v = seq_tree_halves(S->part + hb, (int64_t)threadIdx.x * B, B, cnt);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) v = fadd(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float r = (lane < kNT / 32) ? sh[lane] : 0.0f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) r = fadd(r, __shfl_xor_sync(0xFFFFFFFFu, r, o));
        if (lane == 0) out[l] = r;
    }
}

}  // namespace noalloc
}  // namespace lamb1b

extern "C" int lamb1b_tensor_sumsq_noalloc(const float* x_dev, const lamb1b_layer* layers, int32_t L,
                                           float* out_dev, void* stream)
{
    using namespace lamb1b::noalloc;
    if (!x_dev || !out_dev || !layers || L < 1) return LAMB1B_ERR_ARG;
    if (L > kMaxLayers) return LAMB1B_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(x_dev) & 15u) return LAMB1B_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the tables are staged from host memory local to this call, which a
    // captured graph could not replay: refuse a capturing stream
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) {
        cudaGetLastError();
        return LAMB1B_ERR_CUDA;
    }
    if (cap != cudaStreamCaptureStatusNone) return LAMB1B_ERR_ARG;
    if (!lamb1b::is_current_device_ptr(x_dev) || !lamb1b::is_current_device_ptr(out_dev))
        return LAMB1B_ERR_ARG;
    std::vector<int64_t> tab(3 * (size_t)L + 1);
    int64_t* off = tab.data();
    int64_t* end = off + L;
    int64_t* hbase = end + L;
    int64_t N = 0;
    hbase[0] = 0;
    for (int32_t l = 0; l < L; ++l) {
        if (layers[l].offset != N || layers[l].numel < 1) return LAMB1B_ERR_ARG;
        if (layers[l].numel > (int64_t(1) << 40) - N) return LAMB1B_ERR_ARG;
        off[l] = N;
        N += layers[l].numel;
        end[l] = N;
        const int64_t g0 = off[l] / lamb1b::kGranule, g1 = (end[l] - 1) / lamb1b::kGranule;
        hbase[l + 1] = hbase[l] + 2 * (g1 - g0 + 1);
        if (hbase[l + 1] > kMaxHalves) return LAMB1B_ERR_ARG;   // vector too long for the scratch
    }
    Scratch* S = nullptr;
    int rc = scratch_on_current_device(&S);
    if (rc) return rc;
    // tables, then zeros in every half-granule slot a tensor could read
    if (cudaMemcpyAsync(S->off, off, sizeof(int64_t) * L, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(S->end, end, sizeof(int64_t) * L, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(S->hbase, hbase, sizeof(int64_t) * (L + 1), cudaMemcpyHostToDevice, st) !=
            cudaSuccess ||
        cudaMemsetAsync(S->part, 0, sizeof(float) * hbase[L], st) != cudaSuccess) {
        cudaGetLastError();
        return LAMB1B_ERR_CUDA;
    }
    const unsigned grid = (unsigned)((N + kBlock - 1) / kBlock);
    k_half_sums<<<grid, kNT, 0, st>>>(x_dev, N, L, S);
    if (cudaGetLastError() != cudaSuccess) return LAMB1B_ERR_CUDA;
    k_tensor_totals<<<(unsigned)L, kNT, 0, st>>>(S, out_dev);
    if (cudaGetLastError() != cudaSuccess) return LAMB1B_ERR_CUDA;
    return LAMB1B_OK;
}
