// Warmup stage of 1-bit LAMB (LAMB, arXiv 2104.06069 background on LAMB),
// the parameter update shared by both stages, the stage switch and the
// context's layer-state initialisation.
//
// Block map of the streaming kernels here: 256 threads, 4 aligned float4
// groups per thread, group s of thread tid at block offset s*1024 + tid*4, so
// each warp-group covers one aligned 128-element leaf block of the canonical
// pairwise tree.
#include "lamb1b_internal.cuh"

namespace lamb1b {

constexpr int kNT = 256;
constexpr int kSlots = 4;
constexpr int kBlock = kNT * 4 * kSlots;   // 4096 elements per CTA

__device__ __forceinline__ int first_layer_of_block(const Problem& P, const Dev& D, int64_t b0)
{
    return D.chunk_l0[b0 >> P.log2c];   // the chunk holding b0 starts at or before it
}

// Momentum of 4 elements at idx (a multiple of 4): the dense copy, or (msig)
// the server's sign bits of this step times its chunk scale.
__device__ __forceinline__ void update_momentum4(const Problem& P, const Dev& D, int msig, int64_t idx,
                                                 float mm[4])
{
    if (msig) {
        const uint32_t word = D.signs_s[idx >> 5];
        const float sc = D.scale_s[idx >> P.log2c];
#pragma unroll
        for (int c = 0; c < 4; ++c) mm[c] = ((word >> ((idx & 31) + c)) & 1u) ? sc : -sc;
    } else {
        const float4 m4 = *reinterpret_cast<const float4*>(D.m + idx);
        mm[0] = m4.x; mm[1] = m4.y; mm[2] = m4.z; mm[3] = m4.w;
    }
}

// The preconditioner fl(sqrt(v) + eps) of 4 elements at idx: precomputed from
// the frozen v in the compression stage (msig), else formed from v.
__device__ __forceinline__ void update_denominator4(const Problem& P, const Dev& D, int msig, int64_t idx,
                                                    float d[4])
{
    if (msig) {
        const float4 d4 = *reinterpret_cast<const float4*>(D.d_frz + idx);
        d[0] = d4.x; d[1] = d4.y; d[2] = d4.z; d[3] = d4.w;
    } else {
        const float4 v4 = *reinterpret_cast<const float4*>(D.v + idx);
        d[0] = fadd(fsqrt(v4.x), P.eps); d[1] = fadd(fsqrt(v4.y), P.eps);
        d[2] = fadd(fsqrt(v4.z), P.eps); d[3] = fadd(fsqrt(v4.w), P.eps);
    }
}

// ---- update: x = x - (lr c_l) (m / (sqrt(v) + eps) + wd x) ----------------
// Warmup: m, v are this step's moments.  Compression stage: m is the
// decompressed server momentum and v the frozen second moment, whose
// sqrt(v) + eps is precomputed (d_frz).
// msig: m is the decompressed server momentum of this step, read from its sign
// words and chunk scales (1/32 of the bytes) instead of the dense copy.
__global__ void __launch_bounds__(kNT) k_update(const Problem P, const Dev D, float* __restrict__ x,
                                                int msig)
{
    const int tid = threadIdx.x;
    const int64_t b0 = (int64_t)blockIdx.x * kBlock;
    int l = first_layer_of_block(P, D, b0);
    int64_t lend = D.layer_end[l];
    float gcl = D.gc[l];
    if (b0 + kBlock <= P.N && lend >= b0 + kBlock) {
        // the whole block lies in tensor l: every load is issued before any
        // arithmetic or store
        float mm[kSlots][4], dd[kSlots][4], xv[kSlots][4];
#pragma unroll
        for (int s = 0; s < kSlots; ++s) {
            const int64_t idx = b0 + s * kNT * 4 + tid * 4;
            update_momentum4(P, D, msig, idx, mm[s]);
            update_denominator4(P, D, msig, idx, dd[s]);
            const float4 x4 = *reinterpret_cast<const float4*>(x + idx);
            xv[s][0] = x4.x; xv[s][1] = x4.y; xv[s][2] = x4.z; xv[s][3] = x4.w;
        }
#pragma unroll
        for (int s = 0; s < kSlots; ++s) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float u = fadd(fdiv(mm[s][c], dd[s][c]), fmul(P.wd, xv[s][c]));
                xv[s][c] = fsub(xv[s][c], fmul(gcl, u));
            }
            *reinterpret_cast<float4*>(x + b0 + s * kNT * 4 + tid * 4) =
                make_float4(xv[s][0], xv[s][1], xv[s][2], xv[s][3]);
        }
        return;
    }
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        const int64_t idx = b0 + s * kNT * 4 + tid * 4;
        if (idx >= P.N) break;
        float mm[4];
        update_momentum4(P, D, msig, idx, mm);
        float dd[4];
        update_denominator4(P, D, msig, idx, dd);
        const bool full = idx + 4 <= P.N;
        float xv[4];
        if (full) {
            const float4 x4 = *reinterpret_cast<const float4*>(x + idx);
            xv[0] = x4.x; xv[1] = x4.y; xv[2] = x4.z; xv[3] = x4.w;
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) xv[c] = (idx + c < P.N) ? x[idx + c] : 0.0f;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int64_t i = idx + c;
            if (i < P.N) {
                while (i >= lend) { ++l; lend = D.layer_end[l]; gcl = D.gc[l]; }
                const float u = fadd(fdiv(mm[c], dd[c]), fmul(P.wd, xv[c]));
                xv[c] = fsub(xv[c], fmul(gcl, u));
            }
        }
        if (full) {
            *reinterpret_cast<float4*>(x + idx) = make_float4(xv[0], xv[1], xv[2], xv[3]);
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) if (idx + c < P.N) x[idx + c] = xv[c];
        }
    }
}

// ---- dense momentum from the server's sign words and chunk scales ---------
// m[i] = sign_i x scale_k for i < N (elements >= N stay 0): the values a
// compression step leaves in m, written out for inspection and checkpoints.
__global__ void __launch_bounds__(kNT) k_unpack_momentum(const Problem P, const Dev D)
{
    const int64_t b0 = (int64_t)blockIdx.x * kBlock;
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        const int64_t idx = b0 + s * kNT * 4 + threadIdx.x * 4;
        if (idx >= P.N) break;
        float mm[4];
        update_momentum4(P, D, 1, idx, mm);
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (idx + c >= P.N) mm[c] = 0.0f;
        *reinterpret_cast<float4*>(D.m + idx) = make_float4(mm[0], mm[1], mm[2], mm[3]);
    }
}

cudaError_t launch_unpack_momentum(const Problem& P, const Dev& D, cudaStream_t st)
{
    const unsigned grid = (unsigned)((P.N + kBlock - 1) / kBlock);
    k_unpack_momentum<<<grid, kNT, 0, st>>>(P, D);
    return cudaGetLastError();
}

// ---- the frozen preconditioner: d = fl(fl(sqrt(v)) + eps) over [0, Np) -----
// v does not change in the compression stage, so both compression-stage
// kernels read d instead of recomputing it (same bits, one square root and
// one addition less per element and step).
__global__ void __launch_bounds__(kNT) k_frozen_denominator(const Problem P, const Dev D)
{
    const int64_t idx = ((int64_t)blockIdx.x * kNT + threadIdx.x) * 4;
    if (idx >= P.Np) return;
    const float4 v4 = *reinterpret_cast<const float4*>(D.v + idx);
    *reinterpret_cast<float4*>(D.d_frz + idx) =
        make_float4(fadd(fsqrt(v4.x), P.eps), fadd(fsqrt(v4.y), P.eps),
                    fadd(fsqrt(v4.z), P.eps), fadd(fsqrt(v4.w), P.eps));
}

cudaError_t launch_frozen_denominator(const Problem& P, const Dev& D, cudaStream_t st)
{
    const unsigned grid = (unsigned)((P.Np / 4 + kNT - 1) / kNT);
    k_frozen_denominator<<<grid, kNT, 0, st>>>(P, D);
    return cudaGetLastError();
}

cudaError_t launch_update(const Problem& P, const Dev& D, float* x, int msig, cudaStream_t st)
{
    const unsigned grid = (unsigned)((P.N + kBlock - 1) / kBlock);
    k_update<<<grid, kNT, 0, st>>>(P, D, x, msig);
    return cudaGetLastError();
}

// ---- warmup moments and half-granule sums of x^2, u^2 ------------------------
template <int GK>
__device__ __forceinline__ void warm_grad4(const Grads& G, int w, int64_t idx, int nv,
                                           const float stdv[4], uint32_t heavy, float g[4])
{
    g[0] = g[1] = g[2] = g[3] = 0.0f;
    if (nv <= 0) return;
    if constexpr (GK == kGradF32) {
        const float4 v = *reinterpret_cast<const float4*>(
            static_cast<const float*>(G.ptr) + (int64_t)w * G.ld + idx);
        g[0] = v.x; g[1] = v.y; g[2] = v.z; g[3] = v.w;
    } else if constexpr (GK == kGradBF16) {
        const uint2 v = *reinterpret_cast<const uint2*>(
            static_cast<const uint16_t*>(G.ptr) + (int64_t)w * G.ld + idx);
        g[0] = __uint_as_float(v.x << 16);
        g[1] = __uint_as_float(v.x & 0xFFFF0000u);
        g[2] = __uint_as_float(v.y << 16);
        g[3] = __uint_as_float(v.y & 0xFFFF0000u);
    } else {
        if (heavy != 0xFu) {
            float z[4];
            gen::grads_normal4(G.seed, (uint64_t)idx >> 2, G.t, (uint32_t)w, z);
#pragma unroll
            for (int c = 0; c < 4; ++c) g[c] = fmul(stdv[c], z[c]);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if ((heavy >> c) & 1u)
                g[c] = fmul(G.heavy_scale, gen::student_t3(G.seed, idx + c, G.t, (uint32_t)w));
    }
#pragma unroll
    for (int c = 0; c < 4; ++c)
        if (c >= nv) g[c] = 0.0f;
}

template <int GK>
__global__ void __launch_bounds__(kNT) k_warmup_moments(const Problem P, const Dev D, const Grads G,
                                                        const float* __restrict__ x)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t b0 = (int64_t)blockIdx.x * kBlock;
    int l = first_layer_of_block(P, D, b0);
    int64_t lend = D.layer_end[l];
    bool bad = false;
#pragma unroll 1
    for (int s = 0; s < kSlots; ++s) {
        const int64_t idx = b0 + s * kNT * 4 + tid * 4;
        const int64_t r = P.N - idx;
        const int nv = r >= 4 ? 4 : (r > 0 ? (int)r : 0);
        // layers of the lane's elements (ascending)
        int lay[4] = {-1, -1, -1, -1};
        float stdv[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        uint32_t heavy = 0u;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (c < nv) {
                while (idx + c >= lend) { ++l; lend = D.layer_end[l]; }
                lay[c] = l;
                if constexpr (GK == kGradPhilox) {
                    stdv[c] = G.layer_std[l];
                    if (G.layer_heavy && G.layer_heavy[l]) heavy |= 1u << c;
                }
            }
        }
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int w = 0; w < P.W; ++w) {
            float g[4];
            warm_grad4<GK>(G, w, idx, nv, stdv, heavy, g);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (P.check_finite && c < nv && !isfinite(g[c])) bad = true;
                acc[c] = fadd(acc[c], g[c]);
            }
        }
        float fx[4] = {0.0f, 0.0f, 0.0f, 0.0f}, fu[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (nv > 0) {
            const float4 m4 = *reinterpret_cast<const float4*>(D.m + idx);
            const float4 v4 = *reinterpret_cast<const float4*>(D.v + idx);
            float mm[4] = {m4.x, m4.y, m4.z, m4.w};
            float vv[4] = {v4.x, v4.y, v4.z, v4.w};
            float xv[4];
            if (nv == 4) {
                const float4 x4 = *reinterpret_cast<const float4*>(x + idx);
                xv[0] = x4.x; xv[1] = x4.y; xv[2] = x4.z; xv[3] = x4.w;
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) xv[c] = (c < nv) ? x[idx + c] : 0.0f;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (c < nv) {
                    const float gb = div_w(acc[c], P);
                    mm[c] = fadd(fmul(P.beta1, mm[c]), fmul(P.omega1, gb));
                    vv[c] = fadd(fmul(P.beta2, vv[c]), fmul(P.omega2, fmul(gb, gb)));
                    const float d = fadd(fsqrt(vv[c]), P.eps);
                    const float u = fadd(fdiv(mm[c], d), fmul(P.wd, xv[c]));
                    fx[c] = fmul(xv[c], xv[c]);
                    fu[c] = fmul(u, u);
                }
            }
            *reinterpret_cast<float4*>(D.m + idx) = make_float4(mm[0], mm[1], mm[2], mm[3]);
            *reinterpret_cast<float4*>(D.v + idx) = make_float4(vv[0], vv[1], vv[2], vv[3]);
        }
        if (P.adam) continue;   // Adam: no per-tensor norms
        // half-granule partial sums, one per layer meeting this 128-block
        int lo = 0x7FFFFFFF, hi = -1;
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (lay[c] >= 0) { lo = min(lo, lay[c]); hi = max(hi, lay[c]); }
        lo = __reduce_min_sync(0xFFFFFFFFu, lo);
        hi = __reduce_max_sync(0xFFFFFFFFu, hi);
        const int64_t blk = b0 + s * kNT * 4 + warp * 128;   // first element of the block
        for (int lj = lo; lj <= hi; ++lj) {
            const float tx = warp_tree128(lay[0] == lj ? fx[0] : 0.0f, lay[1] == lj ? fx[1] : 0.0f,
                                          lay[2] == lj ? fx[2] : 0.0f, lay[3] == lj ? fx[3] : 0.0f);
            const float tu = warp_tree128(lay[0] == lj ? fu[0] : 0.0f, lay[1] == lj ? fu[1] : 0.0f,
                                          lay[2] == lj ? fu[2] : 0.0f, lay[3] == lj ? fu[3] : 0.0f);
            if (lane == 0) {
                const int64_t h = blk / 128 - 2 * (D.layer_off[lj] / kGranule);
                D.part_x[D.hbase[lj] + h] = tx;
                D.part_u[D.hbase[lj] + h] = tu;
            }
        }
    }
    if (bad) atomicOr(D.flags, 1u);
}

// ---- per tensor: level-1 tree over granule sums, trust ratio, coefficient -----
// Leaf j of tensor l is granule sum j = half 2j + half 2j+1.  The tensor's
// level-1 tree (zero-padded to a power of two) is evaluated in two passes:
// k_layer_blocks forms the subtrees over aligned blocks of kLevel1Block
// leaves, many CTAs per large tensor; k_layer_finish forms the tree over a
// tensor's block sums.  Both split their leaves into 256 aligned runs, one
// per thread, so every partial sum is a subtree of the canonical tree.
__device__ float block_tree256(float v, float* sh)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) v = fadd(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    __syncthreads();
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    float r = 0.0f;
    if (warp == 0) {
        r = (lane < kNT / 32) ? sh[lane] : 0.0f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) r = fadd(r, __shfl_xor_sync(0xFFFFFFFFu, r, o));
    }
    return r;   // valid in warp 0
}

// Pairwise tree over leaves j0 .. j0+B (B a power of two), leaves at or past
// cnt are +0, computed left to right with a stack of completed subtrees.
// HALVES: leaf j is part[2j] + part[2j+1]; otherwise part[j].
template <bool HALVES>
__device__ float seq_tree(const float* part, int64_t j0, int64_t B, int64_t cnt)
{
    float stk[40];
    int lvl[40];
    int sp = 0;
    for (int64_t j = j0; j < j0 + B; ++j) {
        float v = 0.0f;
        if (j < cnt) v = HALVES ? fadd(part[2 * j], part[2 * j + 1]) : part[j];
        int lv = 0;
        while (sp > 0 && lvl[sp - 1] == lv) { v = fadd(stk[sp - 1], v); ++lv; --sp; }
        stk[sp] = v; lvl[sp] = lv; ++sp;
    }
    return stk[0];
}

// One CTA per level-1 block (tensor l, block b): the subtree over granule
// sums b*kLevel1Block .. (b+1)*kLevel1Block of the tensor.
__global__ void __launch_bounds__(kNT) k_layer_blocks(const Problem P, const Dev D)
{
    __shared__ float sh[kNT / 32];
    constexpr int64_t kPer = kLevel1Block / kNT;      // leaves per thread
    const int64_t blk = blockIdx.x;
    int lo = 0, hi = P.L - 1;                          // the tensor holding this block
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (D.bbase[mid] <= blk) lo = mid; else hi = mid - 1;
    }
    const int l = lo;
    const int64_t hb = D.hbase[l];
    const int64_t cnt = (D.hbase[l + 1] - hb) / 2;
    const int64_t j0 = (blk - D.bbase[l]) * kLevel1Block + (int64_t)threadIdx.x * kPer;
    const float vx = seq_tree<true>(D.part_x + hb, j0, kPer, cnt);
    const float vu = seq_tree<true>(D.part_u + hb, j0, kPer, cnt);
    const float bx = block_tree256(vx, sh);
    const float bu = block_tree256(vu, sh);
    if (threadIdx.x == 0) {
        D.blk_x[blk] = bx;
        D.blk_u[blk] = bu;
    }
}

__global__ void __launch_bounds__(kNT) k_layer_finish(const Problem P, const Dev D, int first_warmup)
{
    __shared__ float sh[kNT / 32];
    const int l = blockIdx.x;
    const int64_t b0 = D.bbase[l];
    const int64_t nb = D.bbase[l + 1] - b0;
    int64_t p2 = 1;
    while (p2 < nb) p2 <<= 1;
    const int64_t B = p2 > kNT ? p2 / kNT : 1;
    const int64_t j0 = (int64_t)threadIdx.x * B;
    const float vx = seq_tree<false>(D.blk_x + b0, j0, B, nb);
    const float vu = seq_tree<false>(D.blk_u + b0, j0, B, nb);
    const float Sx = block_tree256(vx, sh);
    const float Su = block_tree256(vu, sh);
    if (threadIdx.x == 0) {
        const float ratio = (Sx == 0.0f || Su == 0.0f) ? 1.0f : fdiv(fsqrt(Sx), fsqrt(Su));
        const float c = clip(ratio, P.cmin, P.cmax);
        D.Sx[l] = Sx;
        D.Su[l] = Su;
        D.c_cur[l] = c;
        D.gc[l] = fmul(P.lr, c);
        D.c_bar[l] = first_warmup ? c : fadd(fmul(P.cema, D.c_bar[l]), fmul(P.one_m_cema, c));
    }
}

cudaError_t launch_warmup(const Problem& P, const Dev& D, const Grads& G, float* x,
                          cudaStream_t st, int first_warmup, const cudaEvent_t* ev)
{
    // Half-granule sums that lie outside their tensor are never written and
    // stay at the +0 the context's initialisation left there.
    cudaError_t e;
    if ((e = trace(ev, 0, st)) != cudaSuccess) return e;
    const unsigned grid = (unsigned)((P.N + kBlock - 1) / kBlock);
    switch (G.kind) {
    case kGradF32:  k_warmup_moments<kGradF32><<<grid, kNT, 0, st>>>(P, D, G, x); break;
    case kGradBF16: k_warmup_moments<kGradBF16><<<grid, kNT, 0, st>>>(P, D, G, x); break;
    default:        k_warmup_moments<kGradPhilox><<<grid, kNT, 0, st>>>(P, D, G, x); break;
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = trace(ev, 1, st)) != cudaSuccess) return e;
    if (!P.adam) {   // Adam keeps c = 1 (gc = lr from the initialisation)
        k_layer_blocks<<<(unsigned)P.NB, kNT, 0, st>>>(P, D);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        k_layer_finish<<<(unsigned)P.L, kNT, 0, st>>>(P, D, first_warmup);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if ((e = trace(ev, 2, st)) != cudaSuccess) return e;
    if ((e = launch_update(P, D, x, 0, st)) != cudaSuccess) return e;
    return trace(ev, 3, st);
}

// ---- stage switch and initial layer state ------------------------------------
__global__ void k_layers_reset(const Problem P, const Dev D, int init)
{
    const int l = blockIdx.x * blockDim.x + threadIdx.x;
    if (l >= P.L) return;
    D.r_prev[l] = 1.0f;
    D.Rmax[l] = 0u;
    D.R_last[l] = 0.0f;
    if (init) {
        D.c_bar[l] = 1.0f;
        D.c_cur[l] = 1.0f;
        D.gc[l] = P.lr;
        D.Sx[l] = 0.0f;
        D.Su[l] = 0.0f;
    }
}

cudaError_t launch_freeze(const Problem& P, const Dev& D, cudaStream_t st)
{
    cudaError_t e;
    if ((e = cudaMemcpyAsync(D.v_fresh, D.v, sizeof(float) * P.Np, cudaMemcpyDeviceToDevice, st)))
        return e;
    const size_t fe = P.ebf16 ? 2 : 4;
    if ((e = cudaMemsetAsync(D.e_w, 0, fe * P.Np * P.W, st))) return e;
    if ((e = cudaMemsetAsync(D.e_s, 0, fe * P.Np, st))) return e;
    k_layers_reset<<<(P.L + 255) / 256, 256, 0, st>>>(P, D, 0);
    if ((e = cudaGetLastError())) return e;
    return launch_frozen_denominator(P, D, st);
}

cudaError_t launch_init_layers(const Problem& P, const Dev& D, cudaStream_t st)
{
    k_layers_reset<<<(P.L + 255) / 256, 256, 0, st>>>(P, D, 1);
    return cudaGetLastError();
}

}  // namespace lamb1b
