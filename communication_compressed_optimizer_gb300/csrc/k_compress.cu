// Compression stage of 1-bit LAMB (arXiv 2104.06069): the fused worker +
// server pass and the per-tensor factor.
//
// One CTA owns one chunk of C elements for all W virtual workers, so the
// "communication" of the compressed allreduce (section 5 summary: gather chunk
// k of every worker at server k, average, scatter the average) happens in
// registers: the worker loop accumulates each element's server sum while the
// worker's sign bits are still live, and the packed words and scales are also
// written to the exchange buffers (signs_w, scale_w) as the message.
//
// Thread map (used by every kernel here): thread `tid` of an NT-thread CTA
// holds SLOTS aligned float4 groups, group s at chunk offset s*NT*4 + tid*4.
// Warp w's lanes therefore cover the 128 consecutive elements starting at
// s*NT*4 + w*128, which is one leaf block of the canonical pairwise tree.
#include "lamb1b_internal.cuh"

namespace lamb1b {

// Gradients of elements idx..idx+3 of worker w.  Only the first `nv` of them
// exist (< N); the rest are returned as 0.
template <int GK>
__device__ __forceinline__ void grad4(const Grads& G, int w, int64_t idx, int nv,
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
        if (heavy) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if ((heavy >> c) & 1u)
                    g[c] = fmul(G.heavy_scale, gen::student_t3(G.seed, idx + c, G.t, (uint32_t)w));
        }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c)
        if (c >= nv) g[c] = 0.0f;
}

template <int NT, int SLOTS, int GK>
__global__ void __launch_bounds__(NT) k_compress(const Problem P, const Dev D, const Grads G)
{
    constexpr int NWARP = NT / 32;
    constexpr int C = NT * 4 * SLOTS;
    constexpr int NPART = C / 128;
    __shared__ float red[2][NPART];
    __shared__ uint32_t lmax[kMaxChunkLayers];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t k = blockIdx.x;
    const int64_t base = k * C;
    const int64_t n_k = (base + C <= P.N) ? (int64_t)C : P.N - base;
    const float nkf = (float)n_k;
    const int l0 = D.chunk_l0[k];

    for (int i = tid; i < kMaxChunkLayers; i += NT) lmax[i] = 0u;

    int64_t idx[SLOTS];
    int nv[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        idx[s] = base + s * NT * 4 + tid * 4;
        const int64_t r = P.N - idx[s];
        nv[s] = r >= 4 ? 4 : (r > 0 ? (int)r : 0);
    }

    // Per-element gradient std and Student-t flags (in-kernel gradients only).
    float stdv[SLOTS][4];
    uint32_t heavy[SLOTS];
    if constexpr (GK == kGradPhilox) {
        int l = l0;
        int64_t lend = D.layer_end[l];
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            heavy[s] = 0u;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                stdv[s][c] = 0.0f;
                if (c < nv[s]) {
                    while (idx[s] + c >= lend) { ++l; lend = D.layer_end[l]; }
                    stdv[s][c] = G.layer_std[l];
                    if (G.layer_heavy && G.layer_heavy[l]) heavy[s] |= 1u << c;
                }
            }
        }
    } else {
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            heavy[s] = 0u;
#pragma unroll
            for (int c = 0; c < 4; ++c) stdv[s][c] = 0.0f;
        }
    }

    // beta1 * m_old, kept for the whole chunk (worker momentum and g~).
    float bm[SLOTS][4], acc[SLOTS][4];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        const float4 mo = *reinterpret_cast<const float4*>(D.m + idx[s]);
        bm[s][0] = fmul(P.beta1, mo.x); bm[s][1] = fmul(P.beta1, mo.y);
        bm[s][2] = fmul(P.beta1, mo.z); bm[s][3] = fmul(P.beta1, mo.w);
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[s][c] = 0.0f;
    }

    bool bad = false;
    // ---- phase 1: every worker compresses its chunk k ----------------------
    for (int w = 0; w < P.W; ++w) {
        float z[SLOTS][4];
        float* ew = D.e_w + (int64_t)w * P.Np;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            float g[4];
            grad4<GK>(G, w, idx[s], nv[s], stdv[s], heavy[s], g);
            const float4 e = *reinterpret_cast<const float4*>(ew + idx[s]);
            const float ee[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (P.check_finite && c < nv[s] && !isfinite(g[c])) bad = true;
                const float mw = fadd(bm[s][c], fmul(P.omega1, g[c]));
                z[s][c] = (c < nv[s]) ? fadd(mw, ee[c]) : 0.0f;
            }
            const float t = warp_tree128(fmul(z[s][0], z[s][0]), fmul(z[s][1], z[s][1]),
                                         fmul(z[s][2], z[s][2]), fmul(z[s][3], z[s][3]));
            if (lane == 0) red[w & 1][s * NWARP + warp] = t;
        }
        __syncthreads();
        const float S = tree_over_partials<NPART>(red[w & 1], lane);
        const float sc = fsqrt(fdiv(S, nkf));
        uint32_t* sw = D.signs_w + (int64_t)w * P.words_ld;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            bool pos[4];
            float en[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const bool valid = c < nv[s];
                pos[c] = valid && !(z[s][c] < 0.0f);
                en[c] = valid ? (pos[c] ? fsub(z[s][c], sc) : fadd(z[s][c], sc)) : 0.0f;
                acc[s][c] = fadd(acc[s][c], pos[c] ? sc : -sc);
            }
            const uint32_t word = pack_signs128(pos[0], pos[1], pos[2], pos[3], lane);
            if (lane < 4) sw[(idx[s] - tid * 4 + warp * 128) / 32 + lane] = word;
            *reinterpret_cast<float4*>(ew + idx[s]) = make_float4(en[0], en[1], en[2], en[3]);
        }
        if (tid == 0) D.scale_w[(int64_t)w * P.K + k] = sc;
    }
    if (bad) atomicOr(D.flags, 1u);

    // ---- phases 2 and 3: server average, recompression, scatter -----------
    float y[SLOTS][4];
    const float Wf = (float)P.W;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        const float4 e = *reinterpret_cast<const float4*>(D.e_s + idx[s]);
        const float ee[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
        for (int c = 0; c < 4; ++c)
            y[s][c] = (c < nv[s]) ? fadd(fdiv(acc[s][c], Wf), ee[c]) : 0.0f;
        const float t = warp_tree128(fmul(y[s][0], y[s][0]), fmul(y[s][1], y[s][1]),
                                     fmul(y[s][2], y[s][2]), fmul(y[s][3], y[s][3]));
        if (lane == 0) red[P.W & 1][s * NWARP + warp] = t;
    }
    __syncthreads();
    const float SS = tree_over_partials<NPART>(red[P.W & 1], lane);
    const float ss = fsqrt(fdiv(SS, nkf));

    int l = l0;
    int64_t lend = D.layer_end[l];
    int lcur = -1;
    uint32_t runmax = 0u;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        bool pos[4];
        float es[4], mn[4], vf[4];
        const float4 vfr = *reinterpret_cast<const float4*>(D.v_fresh + idx[s]);
        const float4 vfz = *reinterpret_cast<const float4*>(D.v + idx[s]);
        const float vf_old[4] = {vfr.x, vfr.y, vfr.z, vfr.w};
        const float vz[4] = {vfz.x, vfz.y, vfz.z, vfz.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const bool valid = c < nv[s];
            pos[c] = valid && !(y[s][c] < 0.0f);
            es[c] = valid ? (pos[c] ? fsub(y[s][c], ss) : fadd(y[s][c], ss)) : 0.0f;
            mn[c] = valid ? (pos[c] ? ss : -ss) : 0.0f;
            // reconstructed gradient and fresh second moment
            const float gt = fdiv(fsub(mn[c], bm[s][c]), P.omega1);
            vf[c] = valid ? fadd(fmul(P.beta2, vf_old[c]), fmul(P.omega2, fmul(gt, gt))) : 0.0f;
            if (valid) {
                float rho = fdiv(fadd(fsqrt(vz[c]), P.eps), fadd(fsqrt(vf[c]), P.eps));
                if (rho != rho) rho = __int_as_float(0x7F800000);
                const int64_t i = idx[s] + c;
                while (i >= lend) { ++l; lend = D.layer_end[l]; }
                if (l != lcur) {
                    if (lcur >= 0) {
                        if (lcur - l0 < kMaxChunkLayers) atomicMax(&lmax[lcur - l0], runmax);
                        else atomicMax(&D.Rmax[lcur], runmax);
                    }
                    lcur = l;
                    runmax = 0u;
                }
                runmax = max(runmax, __float_as_uint(rho));
            }
        }
        const uint32_t word = pack_signs128(pos[0], pos[1], pos[2], pos[3], lane);
        if (lane < 4) D.signs_s[(idx[s] - tid * 4 + warp * 128) / 32 + lane] = word;
        *reinterpret_cast<float4*>(D.e_s + idx[s]) = make_float4(es[0], es[1], es[2], es[3]);
        *reinterpret_cast<float4*>(D.m + idx[s]) = make_float4(mn[0], mn[1], mn[2], mn[3]);
        *reinterpret_cast<float4*>(D.v_fresh + idx[s]) = make_float4(vf[0], vf[1], vf[2], vf[3]);
    }
    if (lcur >= 0) {
        if (lcur - l0 < kMaxChunkLayers) atomicMax(&lmax[lcur - l0], runmax);
        else atomicMax(&D.Rmax[lcur], runmax);
    }
    if (tid == 0) D.scale_s[k] = ss;
    __syncthreads();
    const int nl = D.chunk_l1[k] - l0 + 1;
    for (int j = tid; j < nl && j < kMaxChunkLayers; j += NT)
        if (lmax[j]) atomicMax(&D.Rmax[l0 + j], lmax[j]);
}

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

cudaError_t launch_update(const Problem& P, const Dev& D, float* x, cudaStream_t st);

template <int NT, int SLOTS>
static cudaError_t launch_compress_t(const Problem& P, const Dev& D, const Grads& G,
                                     cudaStream_t st)
{
    const dim3 grid((unsigned)P.K);
    switch (G.kind) {
    case kGradF32:   k_compress<NT, SLOTS, kGradF32><<<grid, NT, 0, st>>>(P, D, G); break;
    case kGradBF16:  k_compress<NT, SLOTS, kGradBF16><<<grid, NT, 0, st>>>(P, D, G); break;
    default:         k_compress<NT, SLOTS, kGradPhilox><<<grid, NT, 0, st>>>(P, D, G); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_compress(const Problem& P, const Dev& D, const Grads& G, float* x,
                            cudaStream_t st, const cudaEvent_t* ev)
{
    cudaError_t e;
    if ((e = trace(ev, 0, st)) != cudaSuccess) return e;
    switch (P.C) {
    case 256:  e = launch_compress_t<64, 1>(P, D, G, st); break;
    case 512:  e = launch_compress_t<128, 1>(P, D, G, st); break;
    case 1024: e = launch_compress_t<256, 1>(P, D, G, st); break;
    case 2048: e = launch_compress_t<256, 2>(P, D, G, st); break;
    case 4096: e = launch_compress_t<256, 4>(P, D, G, st); break;
    case 8192: e = launch_compress_t<512, 4>(P, D, G, st); break;
    default:   return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    if ((e = trace(ev, 1, st)) != cudaSuccess) return e;
    k_factor<<<(P.L + 255) / 256, 256, 0, st>>>(P, D);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = trace(ev, 2, st)) != cudaSuccess) return e;
    if ((e = launch_update(P, D, x, st)) != cudaSuccess) return e;
    return trace(ev, 3, st);
}

}  // namespace lamb1b
